"""The benchmark's work model (host logic, no GPU): the per-stage FLOPs add up
to the layer's FLOPs per token, the light/heavy split of the expert W1|W2
stage partitions the experts, and the byte counts follow the stated layout."""
import importlib.util
import os

import numpy as np

from sparse_moe_layer_bias_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def k3_counts(seed=0):
    """Per-expert counts that sum to T*k, Zipf-skewed, a few experts untouched."""
    rng = np.random.default_rng(seed)
    shape = synth.K3_PREFILL
    E, T, k = shape.n_experts, shape.T, shape.top_k
    p = synth.zipf_targets(E, k).astype(np.float64)
    p[:5] = 0.0
    counts = rng.multinomial(T * k, p / p.sum()).astype(np.int64)
    return counts


def test_stage_flops_add_up_to_the_layer():
    bench = load_bench()
    shape = synth.K3_PREFILL
    counts = k3_counts()
    assert counts.sum() == shape.T * shape.top_k
    w = bench.layer_work(shape, shape.T, counts)
    total = sum(v[0] for v in w.values())
    assert abs(total - bench.layer_flops_per_token(shape) * shape.T) <= 1e-9 * total
    # the published-shape figure: 373.42 MFLOP per token
    assert abs(bench.layer_flops_per_token(shape) / 1e6 - 373.42) < 0.01


def test_light_heavy_split_partitions_the_experts():
    bench = load_bench()
    shape = synth.K3_PREFILL
    counts = k3_counts(1)
    L, I = shape.latent, shape.inter
    w = bench.layer_work(shape, shape.T, counts)
    light = (counts > 0) & (counts <= 128)
    heavy = counts > 128
    n_l, n_h = counts[light].sum(), counts[heavy].sum()
    assert w["expert_w12_light"][0] == 4.0 * n_l * L * I
    assert w["expert_w12_heavy"][0] == 4.0 * n_h * L * I
    assert w["expert_w12_light"][1] == light.sum() * 2 * I * L * 2 + shape.T * L * 2 + n_l * I * 2
    assert w["expert_w12_heavy"][1] == heavy.sum() * 2 * I * L * 2 + shape.T * L * 2 + n_h * I * 2
    touched = int((counts > 0).sum())
    n = shape.T * shape.top_k
    assert counts.sum() == n and 0 < light.sum() and 0 < heavy.sum()
    # W3 counts the method's bytes: the touched experts' weights and the
    # activation rows; the o rows this design stores for the combine are not
    # counted (they are an intermediate of the design)
    assert w["expert_w3"][1] == touched * L * I * 2 + n * I * 2
    assert w["combine"][1] == 2.0 * (n * L + shape.T * L)


def test_fp8_bytes_halve_the_weight_streams():
    bench = load_bench()
    shape = synth.K3_PREFILL
    counts = k3_counts(2)
    b16 = bench.layer_work(shape, shape.T, counts)
    b8 = bench.layer_work(shape, shape.T, counts, fp8=True)
    for name in ("expert_w12_light", "expert_w12_heavy", "expert_w3"):
        assert b8[name][0] == b16[name][0]                 # same work
    # the heavy stage is weight-dominated: its bytes come close to halving
    assert b8["expert_w12_heavy"][1] < 0.6 * b16["expert_w12_heavy"][1]
    # W3's activation rows are e4m3 codes too, plus one exponent byte per weight row
    assert b8["expert_w3"][1] < 0.6 * b16["expert_w3"][1]
    for name in ("down", "shared", "router", "up", "combine"):
        assert b8[name] == b16[name]


def test_backward_flops_are_twice_the_forward_plus_recompute():
    """Data plus weight gradients of every GEMM are twice the forward's FLOPs;
    on top, the backward's dense router GEMM runs over E rounded up to 64.
    The SiTU-GLU pre-activations and the router logits come from the training
    forward (no FLOPs counted for them)."""
    bench = load_bench()
    shape = synth.K3_PREFILL
    counts = k3_counts(3)
    T, L, E = shape.T, shape.latent, shape.n_experts
    Ep = -(-E // 64) * 64
    w = bench.backward_work(shape, T, counts)
    executed = sum(v[0] for v in w.values())
    expect = 2 * bench.layer_flops_per_token(shape) * T + 2.0 * T * L * (Ep - E)
    assert abs(executed - expect) <= 1e-9 * expect
    assert all(v[1] > 0 for v in w.values())
