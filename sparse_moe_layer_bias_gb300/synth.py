"""Seeded synthetic inputs for the Stable LatentMoE layer and the QB histogram.

This module only draws random numbers and shapes them; it holds none of the
layer's arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle
consume what it produces.  bf16 tensors are produced as torch.bfloat16; use
``bits(t)`` for the uint16 bit patterns the oracle takes.

Recipes (all seeded):
  * activations x ~ N(0, 1), with 1% of the token rows (chosen by the seed)
    scaled by 50 to exercise the SiTU/softcap bounds;
  * every weight ~ N(0, 1/fan_in), drawn in fp64/fp32 and rounded once to bf16;
  * selection bias b_e ~ U(-0.05, 0.05), fp32;
  * K3-shape prefill: router rows scaled by alpha_e so that expert loads follow
    a water-filled Zipf(1.1) law (see ``zipf_router_scales``);
  * K3-shape decode: router weights ~ U(-sqrt(3/latent), sqrt(3/latent));
  * QB sweep: logits ~ N(mu_e, 1) with mu_e ~ N(0, 0.5^2), scores = fp32
    sigmoid of the logits, [T, E] row-major.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import numpy as np
import torch


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    d: int
    latent: int
    n_experts: int
    top_k: int
    inter: int
    n_shared: int
    shared_inter: int
    seed: int
    router: str = "normal"      # "normal" | "zipf" | "uniform"
    beta1: float = 4.0
    beta2: float = 25.0
    rms_eps: float = 1e-6
    norm_after_down: bool = False   # ablation variant: RMSNorm on the latent as well
    expert_fp8: bool = False        # FP8 variant: e4m3 routed experts

    def layer_dict(self) -> dict:
        d = asdict(self)
        for k in ("name", "T", "seed", "router"):
            d.pop(k)
        return d


# The four layer workloads.  K3's widths (7168 -> 3584, 896 experts, 16
# active, 2 shared) are the published model facts; the routed/shared
# intermediate sizes (512 / 1024) and the small shapes are benchmark choices.
TINY = LayerShape("tiny", T=512, d=256, latent=128, n_experts=32, top_k=4, inter=64,
                  n_shared=2, shared_inter=64, seed=1001)
SMALL = LayerShape("small", T=4096, d=1024, latent=512, n_experts=128, top_k=8, inter=128,
                   n_shared=2, shared_inter=256, seed=1002)
K3_PREFILL = LayerShape("k3_prefill", T=8192, d=7168, latent=3584, n_experts=896, top_k=16,
                        inter=512, n_shared=2, shared_inter=1024, seed=1003, router="zipf")
K3_DECODE = LayerShape("k3_decode", T=64, d=7168, latent=3584, n_experts=896, top_k=16,
                       inter=512, n_shared=2, shared_inter=1024, seed=1004, router="uniform")

SHAPES = {s.name: s for s in (TINY, SMALL, K3_PREFILL, K3_DECODE)}

# Quantile Balancing sweep: scores for T tokens x 896 experts, B bins.
QB_SWEEP_T = (65536, 262144, 1048576)
QB_SWEEP_E = 896
QB_SWEEP_B = (1000, 10000)
QB_TOP_K = 16
QB_SEED = 1005


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (as a host numpy array)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """bf16 tensor (host) from uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


def _to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def outlier_rows(T: int, rng: np.random.Generator) -> np.ndarray:
    n = max(1, int(round(0.01 * T))) if T > 0 else 0
    return np.sort(rng.choice(T, size=n, replace=False)) if n else np.zeros(0, np.int64)


def zipf_targets(E: int, k: int, s: float = 1.1, cap: float = 0.5) -> np.ndarray:
    """Per-expert selection probabilities p_e proportional to rank^-s, water-
    filled so that no p_e exceeds ``cap`` and sum(p_e) = k (an expert can be
    chosen at most once per token, so an exact Zipf law is unreachable)."""
    w = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    p = np.zeros(E)
    free = np.ones(E, bool)
    budget = float(k)
    for _ in range(E):
        scale = budget / w[free].sum()
        trial = w * scale
        over = free & (trial > cap)
        if not over.any():
            p[free] = trial[free]
            break
        p[over] = cap
        free &= ~over
        budget = k - p[~free].sum()
    return p


def zipf_router_scales(E: int, k: int, seed: int, n_cal: int = 4096, iters: int = 16) -> np.ndarray:
    """Row scales alpha_e for the router weight so that, with near-isotropic
    unit-variance latents, expert e is among a token's k largest logits with
    about the water-filled Zipf probability.  Calibrated by a multiplicative
    fit on Gaussian surrogate logits alpha_e * g (g ~ N(0,1)); the order of
    alpha_e * g is what decides the top k (the sigmoid is monotone)."""
    target = zipf_targets(E, k)
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((n_cal, E)).astype(np.float32)
    alpha = np.ones(E)
    for _ in range(iters):
        logits = g * alpha.astype(np.float32)
        top = np.argpartition(-logits, k - 1, axis=1)[:, :k]
        load = np.bincount(top.ravel(), minlength=E) / n_cal
        alpha *= np.clip((target + 1e-4) / (load + 1e-4), 0.5, 2.0) ** 0.5
        alpha = np.clip(alpha, 0.05, 12.0)
    perm = rng.permutation(E)      # popular experts at seeded positions, not ids 0..5
    return alpha[perm]


def layer_weights_host(shape: LayerShape) -> dict:
    """All layer inputs generated on the host (numpy, fp64 -> bf16)."""
    rng = np.random.default_rng(shape.seed)
    d, L, E, I = shape.d, shape.latent, shape.n_experts, shape.inter
    S = shape.n_shared * shape.shared_inter

    def normal(shape_, fan_in):
        return _to_bf16(rng.standard_normal(shape_) / math.sqrt(fan_in))

    w = {}
    w["w_down"] = normal((L, d), d)
    wr = rng.standard_normal((E, L)) / math.sqrt(L)
    if shape.router == "zipf":
        wr *= zipf_router_scales(E, shape.top_k, shape.seed)[:, None]
    elif shape.router == "uniform":
        wr = rng.uniform(-math.sqrt(3.0 / L), math.sqrt(3.0 / L), (E, L))
    w["w_router"] = _to_bf16(wr)
    w["w1"] = normal((E, I, L), L)
    w["w2"] = normal((E, I, L), L)
    w["w3"] = normal((E, L, I), I)
    w["ws1"] = normal((S, d), d)
    w["ws2"] = normal((S, d), d)
    w["ws3"] = normal((d, S), shape.shared_inter)
    w["w_up"] = normal((d, L), L)
    return w


def activations_host(shape: LayerShape, T: int | None = None, seed_offset: int = 0):
    """x [T, d] bf16 (1% of rows x50) and bias [E] fp32, on the host."""
    T = shape.T if T is None else T
    rng = np.random.default_rng(shape.seed + 7919 * (1 + seed_offset))
    x = rng.standard_normal((T, shape.d))
    x[outlier_rows(T, rng)] *= 50.0
    bias = rng.uniform(-0.05, 0.05, shape.n_experts).astype(np.float32)
    return _to_bf16(x), torch.from_numpy(bias)


def layer_weights_device(shape: LayerShape, device="cuda") -> dict:
    """Same recipe as ``layer_weights_host`` but drawn on the GPU with torch's
    seeded generator (used for the K3 shapes, ~10 GB of routed weights).
    Values differ from the host recipe; each run's oracle reads back the rows
    it needs from these tensors."""
    gen = torch.Generator(device=device)
    gen.manual_seed(shape.seed)
    d, L, E, I = shape.d, shape.latent, shape.n_experts, shape.inter
    S = shape.n_shared * shape.shared_inter

    def normal(shape_, fan_in):
        out = torch.empty(shape_, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        chunk = 1 << 28
        for i in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - i)
            tmp = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
            flat[i:i + n] = (tmp * (1.0 / math.sqrt(fan_in))).to(torch.bfloat16)
        return out

    w = {}
    w["w_down"] = normal((L, d), d)
    if shape.router == "uniform":
        lim = math.sqrt(3.0 / L)
        u = torch.rand((E, L), generator=gen, device=device, dtype=torch.float32)
        w["w_router"] = ((u * 2.0 - 1.0) * lim).to(torch.bfloat16)
    else:
        wr = torch.randn((E, L), generator=gen, device=device, dtype=torch.float32) / math.sqrt(L)
        if shape.router == "zipf":
            alpha = torch.from_numpy(zipf_router_scales(E, shape.top_k, shape.seed)).to(device)
            wr = wr * alpha.float()[:, None]
        w["w_router"] = wr.to(torch.bfloat16)
    w["w1"] = normal((E, I, L), L)
    w["w2"] = normal((E, I, L), L)
    w["w3"] = normal((E, L, I), I)
    w["ws1"] = normal((S, d), d)
    w["ws2"] = normal((S, d), d)
    w["ws3"] = normal((d, S), shape.shared_inter)
    w["w_up"] = normal((d, L), L)
    return w


def activations_device(shape: LayerShape, T: int | None = None, device="cuda", seed_offset: int = 0):
    T = shape.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(shape.seed + 7919 * (1 + seed_offset))
    x = torch.randn((T, shape.d), generator=gen, device=device, dtype=torch.float32)
    rng = np.random.default_rng(shape.seed + 104729 * (1 + seed_offset))
    rows = torch.from_numpy(outlier_rows(T, rng)).to(device)
    x[rows] *= 50.0
    bias = (torch.rand(shape.n_experts, generator=gen, device=device) * 0.1 - 0.05).float()
    return x.to(torch.bfloat16), bias


def grad_output_host(shape: LayerShape, T: int | None = None, seed_offset: int = 0) -> torch.Tensor:
    """Upstream gradient dy [T, d] bf16, i.i.d. N(0, 1), for the backward pass."""
    T = shape.T if T is None else T
    rng = np.random.default_rng(shape.seed + 15485863 * (1 + seed_offset))
    return _to_bf16(rng.standard_normal((T, shape.d)))


def grad_output_device(shape: LayerShape, T: int | None = None, device="cuda", seed_offset: int = 0):
    """Same distribution as ``grad_output_host``, drawn on the GPU."""
    T = shape.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(shape.seed + 15485863 * (1 + seed_offset))
    return torch.randn((T, shape.d), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def qb_scores(T: int, E: int = QB_SWEEP_E, seed: int = QB_SEED, device="cpu") -> torch.Tensor:
    """fp32 sigmoid scores of logits N(mu_e, 1), mu_e ~ N(0, 0.5^2); [T, E]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    mu = torch.randn(E, generator=gen, device=device, dtype=torch.float32) * 0.5
    out = torch.empty((T, E), dtype=torch.float32, device=device)
    rows = max(1, (1 << 26) // max(E, 1))
    for i in range(0, T, rows):
        n = min(rows, T - i)
        z = torch.randn((n, E), generator=gen, device=device, dtype=torch.float32)
        out[i:i + n] = torch.sigmoid(z + mu)
    return out


def qb_score_stream(T: int, E: int, n_batches: int, seed: int = QB_SEED, device="cpu") -> torch.Tensor:
    """A stationary stream of score batches for closed-loop balancing runs:
    the per-expert logit means mu_e ~ N(0, 0.5^2) are drawn once, every batch
    draws fresh N(0, 1) noise; fp32 sigmoid scores, [n_batches, T, E]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    mu = torch.randn(E, generator=gen, device=device, dtype=torch.float32) * 0.5
    out = torch.empty((n_batches, T, E), dtype=torch.float32, device=device)
    for i in range(n_batches):
        z = torch.randn((T, E), generator=gen, device=device, dtype=torch.float32)
        out[i] = torch.sigmoid(z + mu)
    return out
