"""GB300-native Stable LatentMoE layer forward and Quantile Balancing histogram."""
