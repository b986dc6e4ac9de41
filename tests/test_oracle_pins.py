"""Pins for the CPU oracle: each test checks it against something other than
itself -- closed forms the pages print, library routines that a special case
reduces to, brute force on tiny inputs, hand-worked fixtures under
tests/golden/, and invariants of the method.  No GPU is needed."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

from sparse_moe_layer_bias_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dec(bits):
    """bf16 bit patterns -> fp64 via torch (independent of the oracle's decode)."""
    return synth.from_bits(np.asarray(bits)).double().numpy()


def bf16_nearest_ok(bits, exact):
    """True where the bf16 value ``bits`` is a nearest bf16 to ``exact``."""
    bits = np.asarray(bits, np.uint16)
    v = dec(bits)
    up = dec((bits.astype(np.int32) + 1).astype(np.uint16))
    dn = dec((bits.astype(np.int32) - 1).astype(np.uint16))
    err = np.abs(v - exact)
    # neighbours on either side (the sign bit makes +-1 move away/toward zero)
    return (err <= np.abs(up - exact) * (1 + 1e-12) + 1e-300) & (err <= np.abs(dn - exact) * (1 + 1e-12) + 1e-300)


def rand_bf16(rng, shape, std=1.0):
    return synth.bits(torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16))


def tiny_cfg(orc, **kw):
    base = dict(d=64, latent=32, n_experts=8, top_k=2, inter=16, n_shared=2, shared_inter=16)
    base.update(kw)
    return orc.LayerConfig(**base)


def tiny_weights(cfg, rng):
    S = cfg.n_shared * cfg.shared_inter
    return {
        "w_down": rand_bf16(rng, (cfg.latent, cfg.d), 1 / math.sqrt(cfg.d)),
        "w_router": rand_bf16(rng, (cfg.n_experts, cfg.latent), 1 / math.sqrt(cfg.latent)),
        "w1": rand_bf16(rng, (cfg.n_experts, cfg.inter, cfg.latent), 1 / math.sqrt(cfg.latent)),
        "w2": rand_bf16(rng, (cfg.n_experts, cfg.inter, cfg.latent), 1 / math.sqrt(cfg.latent)),
        "w3": rand_bf16(rng, (cfg.n_experts, cfg.latent, cfg.inter), 1 / math.sqrt(cfg.inter)),
        "ws1": rand_bf16(rng, (S, cfg.d), 1 / math.sqrt(cfg.d)),
        "ws2": rand_bf16(rng, (S, cfg.d), 1 / math.sqrt(cfg.d)),
        "ws3": rand_bf16(rng, (cfg.d, S), 1 / math.sqrt(cfg.shared_inter)),
        "w_up": rand_bf16(rng, (cfg.d, cfg.latent), 1 / math.sqrt(cfg.latent)),
    }


# --------------------------------------------------------------------- bf16
def test_bf16_rounding_hand_values(orc):
    assert orc.f64_to_bf16(1.0) == 0x3F80
    assert orc.f64_to_bf16(-2.5) == 0xC020
    assert orc.f64_to_bf16(1 + 2 ** -8) == 0x3F80          # tie -> even mantissa 0
    assert orc.f64_to_bf16(1 + 3 * 2 ** -8) == 0x3F82      # tie between 0x3F81 and 0x3F82 -> even
    assert orc.f64_to_bf16(1 + 2 ** -8 + 2 ** -30) == 0x3F81  # just above the tie
    assert orc.f64_to_bf16(3.3895313892515355e38) == 0x7F7F  # largest finite bf16
    assert orc.f64_to_bf16(3.4e38) == 0x7F80                 # rounds past it -> inf
    assert orc.f64_to_bf16(2.0 ** -133) == 0x0001            # smallest subnormal
    assert orc.f64_to_bf16(2.0 ** -134) == 0x0000            # tie with zero -> even
    assert orc.f64_to_bf16(3 * 2.0 ** -134) == 0x0002        # tie -> even
    assert orc.f64_to_bf16(-0.0) == 0x8000
    assert orc.bf16_to_f64(0x3F80) == 1.0
    assert orc.bf16_to_f64(0xC020) == -2.5


def test_bf16_rounding_matches_torch_on_fp32_values(orc):
    # For inputs that are exact fp32 values a single RNE rounding to bf16 is
    # what torch's float32 -> bfloat16 conversion does.
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(1500) * 10.0 ** rng.integers(-30, 30, 1500),
                           rng.standard_normal(500)]).astype(np.float32)
    ref = synth.bits(torch.from_numpy(vals).to(torch.bfloat16))
    got = orc.round_bf16_array(vals.astype(np.float64))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------- scalars
def test_sigmoid_matches_expit_without_overflow(orc):
    for x in [-800.0, -40.0, -3.0, -1e-9, 0.0, 1e-9, 2.0, 35.0, 800.0]:
        assert orc.sigmoid(x) == pytest.approx(float(expit(x)), rel=1e-15, abs=1e-300)


def test_softcap_closed_form_points():
    import oracle as orc
    for beta in (4.0, 25.0):
        assert orc.softcap(0.0, beta) == 0.0
        eps = 1e-6
        deriv = (orc.softcap(eps, beta) - orc.softcap(-eps, beta)) / (2 * eps)
        assert deriv == pytest.approx(1.0, abs=1e-9)
        for x in (0.3, 2.0, 17.0, 300.0):
            assert orc.softcap(-x, beta) == -orc.softcap(x, beta)      # odd
            # bounded in (-beta, beta); fp64 tanh saturates to 1 for large arguments
            assert abs(orc.softcap(x, beta)) < beta if x < 10 else abs(orc.softcap(x, beta)) <= beta
        x = 1e-3                                                       # ~ identity near 0
        assert abs(orc.softcap(x, beta) - x) <= x ** 3 / (3 * beta ** 2) * 1.01
    assert orc.softcap(1e4, 25.0) == pytest.approx(25.0, rel=1e-12)


def test_situ_closed_form_points(orc):
    assert orc.situ(0.0, 4.0) == 0.0
    eps = 1e-6
    assert (orc.situ(eps, 4.0) - orc.situ(-eps, 4.0)) / (2 * eps) == pytest.approx(0.5, abs=1e-9)
    # sigma(x) + sigma(-x) = 1  =>  SiTU(x) - SiTU(-x) = softcap(x)
    for x in (-7.0, -0.4, 0.1, 1.3, 6.0, 40.0):
        assert orc.situ(x, 4.0) - orc.situ(-x, 4.0) == pytest.approx(orc.softcap(x, 4.0), rel=1e-13)
    # beta -> infinity: SiTU -> SiLU(x) = x * sigma(x)   (the SwiGLU gate)
    for x in (-5.0, -1.0, 0.5, 3.0, 9.0):
        assert orc.situ(x, 1e9) == pytest.approx(x * float(expit(x)), rel=1e-12)
    # bounded gate: |SiTU| < beta1; the GLU product below beta1*beta2 = 100
    consts = json.load(open(os.path.join(GOLDEN, "constants.json")))
    b1, b2, bound = consts["beta1"]["value"], consts["beta2"]["value"], consts["product_bound"]["value"]
    xs = np.concatenate([np.linspace(-1e4, 1e4, 2001), np.linspace(-20, 20, 401)])
    worst = max(abs(orc.situ(a, b1) * orc.softcap(b, b2)) for a in xs[::7] for b in xs[::53])
    assert worst <= bound
    assert worst > 0.99 * bound
    assert all(abs(orc.situ(x, b1)) <= b1 for x in xs)
    assert all(abs(orc.situ(x, b1)) < b1 for x in xs if abs(x) < 15)


# --------------------------------------------------------------------- a1, a2
def test_down_proj_is_nearest_bf16_of_the_fp64_matmul(orc):
    rng = np.random.default_rng(1)
    cfg = tiny_cfg(orc)
    x = rand_bf16(rng, (37, cfg.d))
    w = rand_bf16(rng, (cfg.latent, cfg.d), 1 / math.sqrt(cfg.d))
    h = orc.down_proj(cfg, x, w)
    exact = dec(x) @ dec(w).T
    assert h.shape == (37, cfg.latent)
    assert bf16_nearest_ok(h, exact).all()


def test_router_scores(orc):
    rng = np.random.default_rng(2)
    cfg = tiny_cfg(orc, latent=32, n_experts=8)
    h = rand_bf16(rng, (19, cfg.latent))
    # one-hot router rows: logit_e = h_e, so s = sigmoid(h_e) exactly
    eye = np.zeros((cfg.n_experts, cfg.latent), np.float32)
    eye[np.arange(cfg.n_experts), np.arange(cfg.n_experts) * 3] = 1.0
    s = orc.router(cfg, h, synth.bits(torch.from_numpy(eye).to(torch.bfloat16)))
    ref = expit(dec(h)[:, np.arange(cfg.n_experts) * 3]).astype(np.float32)
    assert np.array_equal(s, ref)
    w = rand_bf16(rng, (cfg.n_experts, cfg.latent), 1 / math.sqrt(cfg.latent))
    s = orc.router(cfg, h, w)
    assert np.allclose(s, expit(dec(h) @ dec(w).T), rtol=1e-7, atol=0)


# --------------------------------------------------------------------- a3
def brute_topk(s, b, k):
    T, E = s.shape
    idx = np.zeros((T, k), np.int32)
    for t in range(T):
        u = [(float(np.float32(s[t, e]) + np.float32(b[e])), e) for e in range(E)]
        u.sort(key=lambda p: (-p[0], p[1]))
        idx[t] = [e for _, e in u[:k]]
    return idx


def test_topk_brute_force_and_ties(orc):
    rng = np.random.default_rng(3)
    cfg = tiny_cfg(orc, n_experts=12, top_k=5)
    s = rng.random((40, 12)).astype(np.float32)
    s[::3, 4] = s[::3, 9]                      # planted exact ties (lower id must win)
    s[1, :] = 0.5                              # a row of all-equal scores
    b = (rng.random(12).astype(np.float32) - 0.5) * 0.1
    b[9] = b[4]
    idx, gate, margin = orc.topk(cfg, s, b)
    assert np.array_equal(idx, brute_topk(s, b, 5))
    assert np.array_equal(gate, np.take_along_axis(s, idx.astype(np.int64), 1))   # unbiased gates
    row1 = np.argsort(-(s[1] + b), kind="stable")[:5]
    assert set(idx[1]) == set(row1)
    u = s + b
    srt = -np.sort(-u, axis=1)
    assert np.allclose(margin, srt[:, 4].astype(np.float64) - srt[:, 5].astype(np.float64))


def test_topk_bias_add_is_fp32(orc):
    # s + b done in fp64 would rank expert 1 above expert 0; in fp32 the tiny
    # bias is absorbed (0.5 + 2^-26 == 0.5), the two tie, and the lower id wins.
    cfg = tiny_cfg(orc, n_experts=3, top_k=1)
    s = np.array([[0.5, 0.5, 0.1]], np.float32)
    b = np.array([0.0, 2.0 ** -26, 0.0], np.float32)
    idx, gate, margin = orc.topk(cfg, s, b)
    assert idx[0, 0] == 0 and margin[0] == 0.0
    b2 = np.array([0.0, 2.0 ** -23, 0.0], np.float32)   # representable step: expert 1 wins
    idx, _, _ = orc.topk(cfg, s, b2)
    assert idx[0, 0] == 1


def test_topk_all_experts_margin_inf(orc):
    cfg = tiny_cfg(orc, n_experts=4, top_k=4)
    s = np.random.default_rng(4).random((3, 4)).astype(np.float32)
    idx, gate, margin = orc.topk(cfg, s, np.zeros(4, np.float32))
    assert np.all(np.isinf(margin))
    assert np.array_equal(np.sort(idx, 1), np.tile(np.arange(4), (3, 1)))


# --------------------------------------------------------------------- a4
def test_permute_is_stable_argsort(orc):
    rng = np.random.default_rng(5)
    cfg = tiny_cfg(orc, n_experts=9, top_k=3)
    T = 50
    idx = np.stack([rng.choice(9, 3, replace=False) for _ in range(T)]).astype(np.int32)
    idx[:, :] = np.where(rng.random((T, 3)) < 0.5, idx, idx)   # keep distinct per row
    counts, offsets, perm, inv = orc.permute(cfg, idx)
    flat = idx.ravel()
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(counts, np.bincount(flat, minlength=9))
    assert counts.sum() == T * 3 and offsets[-1] == T * 3
    assert np.array_equal(offsets[1:], np.cumsum(counts))
    assert np.array_equal(inv[perm], np.arange(T * 3))
    assert np.array_equal(perm[inv], np.arange(T * 3))


def test_permute_empty(orc):
    cfg = tiny_cfg(orc, n_experts=5, top_k=2)
    counts, offsets, perm, inv = orc.permute(cfg, np.zeros((0, 2), np.int32))
    assert counts.sum() == 0 and np.all(offsets == 0) and perm.size == 0


# --------------------------------------------------------------------- a5-a7
def numpy_expert_act(h64, w1e, w2e, beta1=None):
    p1 = dec(w1e) @ h64
    p2 = dec(w2e) @ h64
    return p1, p2


def test_routed_reduces_to_swiglu_and_combines(orc):
    rng = np.random.default_rng(6)
    cfg = tiny_cfg(orc, beta1=1e9, beta2=1e9)        # softcaps vanish -> SwiGLU
    w = tiny_weights(cfg, rng)
    T = 11
    h = rand_bf16(rng, (T, cfg.latent))
    idx = np.stack([rng.choice(cfg.n_experts, cfg.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    gate = rng.random((T, cfg.top_k)).astype(np.float32)
    out = orc.routed(cfg, h, idx, gate, w["w1"], w["w2"], w["w3"], want_act=True, want_o=True)
    act, z = out["act"], out["z"]
    H = dec(h)
    zref = np.zeros((T, cfg.latent))
    for t in range(T):
        for j in range(cfg.top_k):
            e = idx[t, j]
            p1, p2 = numpy_expert_act(H[t], w["w1"][e], w["w2"][e])
            swiglu = p1 * expit(p1) * p2
            a = act[t * cfg.top_k + j]
            assert bf16_nearest_ok(a, swiglu).all()
            o = dec(w["w3"][e]) @ dec(a)
            assert np.allclose(out["o"][t * cfg.top_k + j], gate[t, j] * o, rtol=1e-12, atol=1e-14)
            zref[t] += float(gate[t, j]) * o
    assert np.allclose(z, zref, rtol=1e-12, atol=1e-13)


def test_expert_aggregate_from_given_activations(orc):
    """The aggregation step on its own: on the routed experts' own
    activations it gives routed's z bit for bit (same products, same order),
    and on arbitrary activations it equals a numpy sum of gate * W3 act; an
    expert listed twice with opposite gates cancels."""
    rng = np.random.default_rng(61)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    T = 13
    h = rand_bf16(rng, (T, cfg.latent))
    idx = np.stack([rng.choice(cfg.n_experts, cfg.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    gate = rng.random((T, cfg.top_k)).astype(np.float32)
    out = orc.routed(cfg, h, idx, gate, w["w1"], w["w2"], w["w3"], want_act=True)
    z = orc.expert_aggregate(cfg, out["act"], idx, gate, w["w3"])
    assert np.array_equal(z, out["z"])
    act = rand_bf16(rng, (T * cfg.top_k, cfg.inter), 3.0)
    z = orc.expert_aggregate(cfg, act, idx, gate, w["w3"])
    A = dec(act).reshape(T, cfg.top_k, cfg.inter)
    ref = np.zeros((T, cfg.latent))
    for t in range(T):
        for j in range(cfg.top_k):
            ref[t] += float(gate[t, j]) * (dec(w["w3"][idx[t, j]]) @ A[t, j])
    assert np.allclose(z, ref, rtol=1e-12, atol=1e-12)
    # same expert and activation twice, gates g and -g: the token's z is 0
    idx2 = np.tile(np.array([[3, 3]], np.int32), (2, 1))
    g2 = np.array([[0.75, -0.75], [0.5, 0.25]], np.float32)
    act2 = np.repeat(rand_bf16(rng, (2, cfg.inter)), 2, axis=0)
    z2 = orc.expert_aggregate(cfg, act2, idx2, g2, w["w3"])
    assert np.all(z2[0] == 0.0)
    assert np.allclose(z2[1], 0.75 * (dec(w["w3"][3]) @ dec(act2[2])), rtol=1e-12, atol=1e-13)


def test_rmsnorm_unit_rms_and_gate_scale_invariance(orc):
    rng = np.random.default_rng(7)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    T = 9
    h = rand_bf16(rng, (T, cfg.latent))
    idx = np.stack([rng.choice(cfg.n_experts, cfg.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    gate = rng.random((T, cfg.top_k)).astype(np.float32)
    a = orc.routed(cfg, h, idx, gate, w["w1"], w["w2"], w["w3"])
    ms = np.mean(a["z"] ** 2, axis=1)
    assert np.allclose(np.mean(a["r64"] ** 2, axis=1), ms / (ms + cfg.rms_eps), rtol=1e-12)
    assert np.allclose(a["r64"], a["z"] / np.sqrt(ms + cfg.rms_eps)[:, None], rtol=1e-12)
    assert bf16_nearest_ok(a["r"], a["r64"]).all()
    # any positive per-token rescaling of the gates cancels in the norm (up to eps)
    # r(cz)/r(z) = sqrt(ms + eps) / sqrt(ms + eps/c^2), within eps/(2 ms) of 1
    # (c = 4 is a power of two, so the scaled fp32 gates are exact)
    b = orc.routed(cfg, h, idx, (gate * 4.0).astype(np.float32), w["w1"], w["w2"], w["w3"])
    ratio = np.sqrt(ms + cfg.rms_eps) / np.sqrt(ms + cfg.rms_eps / 16.0)
    assert np.allclose(b["r64"], a["r64"] * ratio[:, None], rtol=1e-9, atol=1e-12)
    assert np.all(np.abs(ratio - 1) <= cfg.rms_eps / (2 * ms))
    # z = 0 gives r = 0
    zero = orc.routed(cfg, h, idx, np.zeros_like(gate), w["w1"], w["w2"], w["w3"])
    assert np.all(zero["r64"] == 0.0)


def test_expert_activation_bound_on_outliers(orc):
    rng = np.random.default_rng(8)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    T = 6
    h = rand_bf16(rng, (T, cfg.latent), 200.0)                 # huge latents
    idx = np.tile(np.arange(cfg.top_k, dtype=np.int32), (T, 1))
    gate = np.ones((T, cfg.top_k), np.float32)
    a = orc.routed(cfg, h, idx, gate, w["w1"], w["w2"], w["w3"], want_act=True)
    av = np.abs(dec(a["act"]))
    assert av.max() <= 100.0 and av.max() > 50.0


def test_shared_act_and_up(orc):
    rng = np.random.default_rng(9)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    T = 7
    x = rand_bf16(rng, (T, cfg.d))
    a_s = orc.shared_act(cfg, x, w["ws1"], w["ws2"])
    p1 = dec(x) @ dec(w["ws1"]).T
    p2 = dec(x) @ dec(w["ws2"]).T
    ref = 4.0 * np.tanh(p1 / 4.0) * expit(p1) * 25.0 * np.tanh(p2 / 25.0)
    assert bf16_nearest_ok(a_s, ref).all()
    r = rand_bf16(rng, (T, cfg.latent))
    y = orc.up_shared(cfg, r, a_s, w["w_up"], w["ws3"])
    yref = dec(r) @ dec(w["w_up"]).T + dec(a_s) @ dec(w["ws3"]).T
    assert np.allclose(y, yref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------- whole layer
def numpy_layer_all_experts(cfg, x, w, bias):
    """Independent fp64 numpy layer for top_k == n_experts (every expert is on),
    with the same bf16 rounding points (through torch's rounding)."""
    def rb(a):
        return synth.from_bits(synth.bits(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16))).double().numpy()
    X = dec(x)
    h = rb(X @ dec(w["w_down"]).T)
    s = expit(h @ dec(w["w_router"]).T)
    z = np.zeros((X.shape[0], cfg.latent))
    for e in range(cfg.n_experts):
        p1 = h @ dec(w["w1"][e]).T
        p2 = h @ dec(w["w2"][e]).T
        act = rb(cfg.beta1 * np.tanh(p1 / cfg.beta1) * expit(p1) * cfg.beta2 * np.tanh(p2 / cfg.beta2))
        z += s[:, e:e + 1].astype(np.float32).astype(np.float64) * (act @ dec(w["w3"][e]).T)
    r = rb(z / np.sqrt(np.mean(z ** 2, axis=1, keepdims=True) + cfg.rms_eps))
    q1 = X @ dec(w["ws1"]).T
    q2 = X @ dec(w["ws2"]).T
    a_s = rb(cfg.beta1 * np.tanh(q1 / cfg.beta1) * expit(q1) * cfg.beta2 * np.tanh(q2 / cfg.beta2))
    return r @ dec(w["w_up"]).T + a_s @ dec(w["ws3"]).T


def test_layer_with_all_experts_equals_dense_sum(orc):
    rng = np.random.default_rng(10)
    cfg = tiny_cfg(orc, n_experts=6, top_k=6)
    w = tiny_weights(cfg, rng)
    x = rand_bf16(rng, (13, cfg.d))
    bias = (rng.random(6).astype(np.float32) - 0.5) * 0.1
    out = orc.layer_forward(cfg, x, w, bias)
    ref = numpy_layer_all_experts(cfg, x, w, bias)
    rel = np.linalg.norm(out["y"] - ref) / np.linalg.norm(ref)
    assert rel < 2e-3


def test_layer_zero_up_projection_leaves_shared_only(orc):
    rng = np.random.default_rng(11)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    w["w_up"] = np.zeros_like(w["w_up"])
    x = rand_bf16(rng, (8, cfg.d))
    out = orc.layer_forward(cfg, x, w, np.zeros(cfg.n_experts, np.float32))
    assert np.allclose(out["y"], dec(out["a_s"]) @ dec(w["ws3"]).T, rtol=1e-12, atol=1e-12)


def test_two_shared_experts_equal_one_concatenated(orc):
    rng = np.random.default_rng(12)
    cfg2 = tiny_cfg(orc, n_shared=2, shared_inter=16)
    cfg1 = tiny_cfg(orc, n_shared=1, shared_inter=32)
    w = tiny_weights(cfg2, rng)
    x = rand_bf16(rng, (5, cfg2.d))
    b = np.zeros(cfg2.n_experts, np.float32)
    y2 = orc.layer_forward(cfg2, x, w, b)["y"]
    y1 = orc.layer_forward(cfg1, x, w, b)["y"]
    assert np.array_equal(y1, y2)


def test_layer_is_equivariant_to_expert_relabelling(orc):
    rng = np.random.default_rng(13)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    x = rand_bf16(rng, (10, cfg.d))
    bias = (rng.random(cfg.n_experts).astype(np.float32) - 0.5) * 0.1
    pi = rng.permutation(cfg.n_experts)
    w2 = dict(w)
    for k in ("w_router", "w1", "w2", "w3"):
        w2[k] = np.ascontiguousarray(w[k][pi])
    a = orc.layer_forward(cfg, x, w, bias)
    b = orc.layer_forward(cfg, x, w2, np.ascontiguousarray(bias[pi]))
    assert np.array_equal(pi[b["idx"]], a["idx"])
    assert np.allclose(a["y"], b["y"], rtol=1e-12, atol=1e-12)


def test_layer_is_token_independent(orc):
    rng = np.random.default_rng(14)
    cfg = tiny_cfg(orc)
    w = tiny_weights(cfg, rng)
    x = rand_bf16(rng, (24, cfg.d))
    bias = np.zeros(cfg.n_experts, np.float32)
    full = orc.layer_forward(cfg, x, w, bias)
    sub = [3, 17, 5]
    part = orc.layer_forward(cfg, np.ascontiguousarray(x[sub]), w, bias)
    assert np.array_equal(part["y"], full["y"][sub])
    assert np.array_equal(part["idx"], full["idx"][sub])


# --------------------------------------------------------------------- a9
def test_qb_binning_golden(orc):
    g = json.load(open(os.path.join(GOLDEN, "qb_binning_fp32.json")))
    s = np.array([[c["s"] for c in g["cases"]]], np.float32)
    hist = orc.qb_histogram(s.T.copy(), g["B"], n_cols=1)        # T = cases, one expert
    want = np.zeros(g["B"], np.uint32)
    for c in g["cases"]:
        want[c["bin"]] += 1
    assert np.array_equal(hist[0], want)


def test_qb_histogram_brute_force_and_additivity(orc):
    rng = np.random.default_rng(15)
    T, E, ld, B = 777, 13, 16, 97
    s = rng.random((T, ld)).astype(np.float32)
    s[5, 2] = 1.0
    s[6, 3] = 0.0
    hist = orc.qb_histogram(s, B, n_cols=E)
    ref = np.zeros((E, B), np.uint32)
    bins = np.minimum(B - 1, np.floor(s[:, :E] * np.float32(B)).astype(np.int64))
    for e in range(E):
        np.add.at(ref[e], bins[:, e], 1)
    assert np.array_equal(hist, ref)
    assert hist.sum(dtype=np.uint64) == T * E and np.all(hist.sum(1) == T)
    assert hist[2, B - 1] >= 1 and hist[3, 0] >= 1
    # additivity: hist(A) + hist(B) == hist(A u B)
    h2 = orc.qb_histogram(s[:300], B, n_cols=E)
    orc.qb_histogram(s[300:], B, hist=h2, accumulate=True, n_cols=E)
    assert np.array_equal(h2, hist)


# --------------------------------------------------------------------- a10
def test_qb_quantile_worked_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "qb_worked_example.json")))
    hist = np.array(g["hist"], np.uint32)
    for case in g["cases"]:
        q, b = orc.qb_quantile_bias(hist, case["level"])
        assert np.allclose(q, np.array(case["q"], np.float32), rtol=0, atol=1e-7)
        assert np.allclose(b, -q)


def test_qb_quantile_within_one_bin_of_exact_sort(orc):
    rng = np.random.default_rng(16)
    T, E = 5000, 7
    mu = rng.normal(0, 0.5, E)
    s = expit(rng.standard_normal((T, E)) + mu).astype(np.float32)
    for B in (1000, 10000, 37):
        hist = orc.qb_histogram(s, B)
        for level in (1 - 16 / 896, 0.5, 0.9):
            q, _ = orc.qb_quantile_bias(hist, level)
            r = min(max(math.ceil(level * T), 1), T)
            exact = np.partition(s, r - 1, axis=0)[r - 1]
            assert np.all(np.abs(q.astype(np.float64) - exact) <= 1.0 / B + 1e-6)


def test_qb_bias_sign_flattens_loads(orc):
    """b = -q puts every expert's threshold at its own (1-k/E) quantile, so the
    per-expert loads become nearly equal; the opposite sign makes them worse."""
    rng = np.random.default_rng(17)
    T, E, k = 20000, 64, 4
    s = expit(rng.standard_normal((T, E)) + rng.normal(0, 1.0, E)).astype(np.float32)
    cfg = tiny_cfg(orc, n_experts=E, top_k=k)
    hist = orc.qb_histogram(s, 1000)
    q, b = orc.qb_quantile_bias(hist, 1 - k / E)

    def spread(bias):
        idx, _, _ = orc.topk(cfg, s, bias.astype(np.float32))
        load = np.bincount(idx.ravel(), minlength=E)
        return load.std() / load.mean(), load.max() / load.mean()

    (cv0, mx0), (cv1, mx1), (cv2, mx2) = spread(np.zeros(E)), spread(b), spread(-b)
    assert cv1 < 0.2 * cv0 and mx1 < mx0 / 3          # one QB read flattens the loads
    assert cv2 > cv0 and mx2 > mx0                     # the opposite sign sharpens them


def test_sign_update_closed_forms(orc):
    """The fixed-step rule: under-loaded experts step up, over-loaded ones down,
    experts at the mean stay; mean 2 for loads (3, 1, 2, 2); a non-integer mean
    (1.5) moves both; one fp32 addition per step."""
    b = orc.sign_update(np.array([3, 1, 2, 2], np.int32), 0.5, np.zeros(4, np.float32))
    assert b.tolist() == [-0.5, 0.5, 0.0, 0.0]
    b = orc.sign_update(np.array([1, 2], np.int32), 0.25, np.array([1.0, -1.0], np.float32))
    assert b.tolist() == [1.25, -1.25]
    flat = np.full(7, 9, np.int32)
    b0 = np.linspace(-1, 1, 7).astype(np.float32)
    assert np.array_equal(orc.sign_update(flat, 0.1, b0), b0)
    # fp32 add: 1 + 2^-30 rounds back to 1 in fp32 (it would not in fp64)
    b = orc.sign_update(np.array([0, 5], np.int32), 2.0 ** -30, np.array([1.0, 1.0], np.float32))
    assert b.dtype == np.float32 and b.tolist() == [1.0, 1.0]


def test_closed_loop_qb_settles_in_one_read_sign_steps_slowly(orc):
    """On a stationary stream of skewed score batches, QB sets the biases
    from one batch's quantiles and the next batch is already near balance
    (direct distribution solving); the fixed-step rule needs many steps at a
    small step and moves the loads far less after one."""
    T, E, k = 4000, 64, 4
    cfg = tiny_cfg(orc, n_experts=E, top_k=k)
    batches = synth.qb_score_stream(T, E, 6, seed=5).numpy()

    def max_over_mean(s, bias):
        idx, _, _ = orc.topk(cfg, s, bias)
        load = orc.expert_loads(idx, E)
        return load.max() / load.mean(), load

    m0, _ = max_over_mean(batches[0], np.zeros(E, np.float32))
    _, b_qb = orc.qb_quantile_bias(orc.qb_histogram(batches[0], 1000), 1 - k / E)
    m_qb, _ = max_over_mean(batches[1], b_qb)
    b = np.zeros(E, np.float32)
    m_sign = []
    for i in range(5):
        _, load = max_over_mean(batches[i], b)
        b = orc.sign_update(load, 1e-3, b)
        m_sign.append(max_over_mean(batches[i + 1], b)[0])
    assert m0 > 3.0
    assert m_qb < 1.5
    assert m_sign[0] > 0.8 * m0 and m_sign[-1] < m_sign[0]   # small steps: slow, monotone progress


def test_rms_rows_closed_form(orc):
    """Row RMSNorm on exact bf16 values: (3, 4, 0, 0) has mean square 25/4, so
    it becomes (1.2, 1.6, 0, 0) (rounded once to bf16); a zero row stays zero."""
    cfg = tiny_cfg(orc, rms_eps=0.0)
    h = synth.bits(torch.tensor([[3.0, 4.0, 0.0, 0.0], [0.0, 0.0, 0.0, 0.0]]).to(torch.bfloat16))
    out = dec(orc.rms_rows(cfg, h))
    assert out[1].tolist() == [0.0, 0.0, 0.0, 0.0] and out[0, 2:].tolist() == [0.0, 0.0]
    assert bf16_nearest_ok(orc.rms_rows(cfg, h)[0, :2], np.array([1.2, 1.6])).all()


def test_norm_after_down_makes_routing_scale_free(orc):
    """Ablation variant with the RMSNorm also after the down-projection: the
    latent has unit RMS and routing depends on the token's direction only --
    with eps = 0, x and 4x (exact in bf16) give the same normalised latent,
    scores, chosen experts and aggregate.  Without that norm the same scaling
    changes the routing once a selection bias is present."""
    rng = np.random.default_rng(31)
    cfg = tiny_cfg(orc, n_experts=16, top_k=3, norm_after_down=True, rms_eps=0.0)
    w = tiny_weights(cfg, rng)
    x = rand_bf16(rng, (64, cfg.d))
    x4 = synth.bits(torch.from_numpy(dec(x) * 4.0).to(torch.bfloat16))
    bias = rng.uniform(-0.05, 0.05, cfg.n_experts).astype(np.float32)
    a, b = orc.layer_forward(cfg, x, w, bias), orc.layer_forward(cfg, x4, w, bias)
    for key in ("h", "s", "idx", "r"):
        assert np.array_equal(a[key], b[key]), key
    assert not np.array_equal(a["h_raw"], b["h_raw"])
    hn = dec(a["h"])
    assert np.allclose(np.sqrt(np.mean(hn ** 2, axis=1)), 1.0, atol=2.0 ** -7)
    off = tiny_cfg(orc, n_experts=16, top_k=3, rms_eps=0.0)
    a0, b0 = orc.layer_forward(off, x, w, bias), orc.layer_forward(off, x4, w, bias)
    assert np.array_equal(a0["h"], a0["h_raw"])
    assert not np.array_equal(a0["idx"], b0["idx"])


# --------------------------------------------------------------------- FP8 variant
def test_e4m3_codec_hand_values_and_torch(orc):
    """e4m3 (OCP FP8): 448 is the largest finite value, 2^-6 the smallest
    normal, 2^-9 the subnormal step; ties go to the even code; beyond 448 the
    encoder saturates.  Inside the range it agrees with torch's float8_e4m3fn
    conversion of the same (fp32-exact) values, and decoding agrees too."""
    hand = {448.0: 0x7E, 1.0: 0x38, 2.0 ** -6: 0x08, 2.0 ** -9: 0x01, 1.0625: 0x38, 1.1875: 0x3A,
            -3.0: 0xC4, 0.0: 0x00, 2.0 ** -10: 0x00, 3 * 2.0 ** -11: 0x01, 500.0: 0x7E, -1e9: 0xFE}
    for v, code in hand.items():
        assert int(orc.f64_to_e4m3(v)) == code, v
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(3000) * 10 ** rng.uniform(-3, 2.6, 3000),
                        np.arange(-464.0, 464.0, 0.125)]).astype(np.float32)
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.f64_to_e4m3(x.astype(np.float64)), ref)
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                       # NaN codes
    ref_dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(orc.e4m3_to_f64(codes), ref_dec.astype(np.float64))


def test_fp8_scale_exponent_rule(orc):
    """e is the smallest integer with max|row| <= 448 * 2^e."""
    assert [orc.fp8_exp_for(a) for a in (448.0, 449.0, 224.0, 0.875, 0.8751, 0.0)] == [0, 1, -1, -9, -8, 0]
    rng = np.random.default_rng(9)
    for a in 10 ** rng.uniform(-8, 6, 500):
        e = orc.fp8_exp_for(a)
        assert a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1)


def test_fp8_quantize_rows_matches_torch_and_error_bound(orc):
    rng = np.random.default_rng(10)
    w = rand_bf16(rng, (40, 96), 0.05)
    w[3] = 0                                                     # an all-zero row
    codes, exps = orc.fp8_quantize_rows(w)
    assert exps[3] == 0 and not codes[3].any()
    scaled = dec(w) * np.exp2(-exps.astype(np.float64))[:, None]   # exact power-of-two scaling
    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    back = orc.e4m3_to_f64(codes) * np.exp2(exps.astype(np.float64))[:, None]
    big = np.abs(scaled) >= 2.0 ** -6                            # normal range: half a step, 2^-4 relative
    assert np.all(np.abs(back - dec(w))[big] <= 2.0 ** -4 * np.abs(dec(w))[big])
    assert np.all(np.abs(scaled).max(axis=1)[np.arange(40) != 3] > 224.0)   # the scale uses the top octave


def test_routed_fp8_exact_on_power_of_two_data(orc):
    """With every latent and weight value in {0, +-1/4, +-1/2, +-1, +-2}, every
    quantisation is exact, so the FP8 path equals an independent numpy/torch
    computation: exact products, the SiTU-GLU in fp64, act8 = e4m3(4 act)
    (torch's conversion), o = act8 / 4 . W3, z, and the RMSNorm."""
    rng = np.random.default_rng(11)
    cfg = tiny_cfg(orc, n_experts=6, top_k=2, latent=32, inter=16)
    vals = np.array([0.0, 0.25, -0.25, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0])

    def pick(shape):
        return synth.bits(torch.from_numpy(rng.choice(vals, shape).astype(np.float32)).to(torch.bfloat16))

    T, E, L, I = 10, cfg.n_experts, cfg.latent, cfg.inter
    h = pick((T, L))
    w1, w2, w3 = pick((E, I, L)), pick((E, I, L)), pick((E, L, I))
    idx = np.stack([rng.choice(E, 2, replace=False) for _ in range(T)]).astype(np.int32)
    gate = rng.uniform(0.1, 1.0, (T, 2)).astype(np.float32)
    out = orc.routed_fp8(cfg, h, idx, gate, w1, w2, w3, want_act=True, want_o=True)
    H, W1, W2, W3 = dec(h), dec(w1), dec(w2), dec(w3)
    for t in range(T):
        z = np.zeros(L)
        for j in range(2):
            e, a = idx[t, j], t * 2 + j
            p1, p2 = W1[e] @ H[t], W2[e] @ H[t]
            act = 4.0 * np.tanh(p1 / 4.0) * expit(p1) * 25.0 * np.tanh(p2 / 25.0)
            code = torch.from_numpy((4.0 * act).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(out["act"][a], code)
            o = gate[t, j] * (W3[e] @ (orc.e4m3_to_f64(code) / 4.0))
            assert np.allclose(out["o"][a], o, rtol=1e-12, atol=1e-12)
            z += o
        assert np.allclose(out["z"][t], z, rtol=1e-12, atol=1e-12)
        assert np.allclose(out["r64"][t], z / np.sqrt(np.mean(z ** 2) + cfg.rms_eps), rtol=1e-12)


def test_layer_fp8_keeps_routing_and_stays_near_bf16(orc):
    """The FP8 variant changes only the routed experts: same h, scores and
    choices as the bf16 layer; the output moves by the e4m3 quantisation
    noise (a few percent), not by factors of two."""
    rng = np.random.default_rng(12)
    cfg = tiny_cfg(orc, n_experts=8, top_k=2)
    cfg8 = tiny_cfg(orc, n_experts=8, top_k=2, expert_fp8=True)
    w = tiny_weights(cfg, rng)
    x = rand_bf16(rng, (48, cfg.d))
    bias = np.zeros(8, np.float32)
    a, b = orc.layer_forward(cfg, x, w, bias), orc.layer_forward(cfg8, x, w, bias)
    assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["s"], b["s"])
    rel = np.linalg.norm(b["z"] - a["z"]) / np.linalg.norm(a["z"])
    assert 1e-3 < rel < 0.1


def test_synth_k3_shape_matches_published_constants():
    consts = json.load(open(os.path.join(GOLDEN, "constants.json")))
    k3 = synth.K3_PREFILL
    assert k3.d == consts["hidden"]["value"] and k3.latent == consts["latent"]["value"]
    assert k3.n_experts == consts["routed_experts"]["value"]
    assert k3.top_k == consts["active_experts"]["value"]
    assert k3.n_shared == consts["shared_experts"]["value"]
    assert (k3.beta1, k3.beta2) == (consts["beta1"]["value"], consts["beta2"]["value"])
    p = synth.zipf_targets(896, 16)
    assert abs(p.sum() - 16) < 1e-9 and p.max() <= 0.5 + 1e-12
