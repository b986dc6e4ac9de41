"""Pins for the oracle's backward pass (no GPU).

The oracle's gradient of the unrounded layer (round_mode 0) is checked against
central finite differences of an independent fp64 forward written here with
numpy (its own tanh / exp, a dense loop over tokens and chosen experts), one
random direction per weight and one for x, so a dropped term, a wrong sign or
a transposed operand in any gradient fails.  The rounded mode (the gradient
at the forward's bf16 intermediates) must stay within bf16 rounding of it."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_bias_gb300 import synth

NAMES = oracle.BACKWARD_GRADS


def rand_bf16(rng, shape, std=1.0):
    return synth.bits(torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16))


def dec(bits):
    return synth.from_bits(np.asarray(bits)).double().numpy()


def make_case(seed, **kw):
    """Tiny layer with pre-activations of order one (the SiTU and softcap
    curvature matters), distinct experts per token."""
    shape = dict(d=24, latent=12, n_experts=6, top_k=2, inter=8, n_shared=2, shared_inter=4)
    shape.update(kw)
    extra = {k: shape.pop(k) for k in ("beta1", "beta2", "norm_after_down") if k in shape}
    cfg = oracle.LayerConfig(**shape, **extra)
    rng = np.random.default_rng(seed)
    d, L, E, I, k = cfg.d, cfg.latent, cfg.n_experts, cfg.inter, cfg.top_k
    S = cfg.n_shared * cfg.shared_inter
    T = 5
    w = {"w_down": rand_bf16(rng, (L, d), 2.0 / np.sqrt(d)),
         "w_router": rand_bf16(rng, (E, L), 1.0 / np.sqrt(L)),
         "w1": rand_bf16(rng, (E, I, L), 2.0 / np.sqrt(L)),
         "w2": rand_bf16(rng, (E, I, L), 2.0 / np.sqrt(L)),
         "w3": rand_bf16(rng, (E, L, I), 1.0 / np.sqrt(I)),
         "ws1": rand_bf16(rng, (S, d), 2.0 / np.sqrt(d)),
         "ws2": rand_bf16(rng, (S, d), 2.0 / np.sqrt(d)),
         "ws3": rand_bf16(rng, (d, S), 1.0 / np.sqrt(S)),
         "w_up": rand_bf16(rng, (d, L), 1.0 / np.sqrt(L))}
    x = rand_bf16(rng, (T, d))
    dy = rand_bf16(rng, (T, d))
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    return cfg, w, x, dy, idx


def smooth_loss(cfg, xf, wf, idx, dyf):
    """sum(dy * y) for the unrounded layer, written independently of the
    oracle (numpy fp64)."""
    b1, b2 = cfg.beta1, cfg.beta2
    sig = lambda v: 1.0 / (1.0 + np.exp(-v))
    situ = lambda v: b1 * np.tanh(v / b1) * sig(v)
    cap = lambda v: b2 * np.tanh(v / b2)
    h = xf @ wf["w_down"].T
    if cfg.norm_after_down:   # the ablation variant's RMSNorm after the down-projection
        h = h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + cfg.rms_eps)
    s = sig(h @ wf["w_router"].T)
    z = np.zeros_like(h)
    for t in range(xf.shape[0]):
        for e in idx[t]:
            act = situ(wf["w1"][e] @ h[t]) * cap(wf["w2"][e] @ h[t])
            z[t] += s[t, e] * (wf["w3"][e] @ act)
    r = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True) + cfg.rms_eps)
    a_s = situ(xf @ wf["ws1"].T) * cap(xf @ wf["ws2"].T)
    y = r @ wf["w_up"].T + a_s @ wf["ws3"].T
    return float(np.sum(dyf * y))


@pytest.mark.parametrize("seed,kw", [(1, {}), (2, {"beta1": 1.5, "beta2": 2.0}),
                                     (3, {"top_k": 6}), (8, {"norm_after_down": True}),
                                     (9, {"norm_after_down": True, "beta1": 1.5, "beta2": 2.0})])
def test_backward_matches_finite_differences(seed, kw):
    cfg, w, x, dy, idx = make_case(seed, **kw)
    g = oracle.layer_backward(cfg, x, w, idx, dy, round_mode=0)
    xf, dyf = dec(x), dec(dy)
    wf = {k: dec(v) for k, v in w.items()}
    rng = np.random.default_rng(100 + seed)
    eps = 1e-5
    for name in ("x",) + NAMES:
        base = xf if name == "x" else wf[name]
        v = rng.standard_normal(base.shape) * (np.std(base) + 1e-3)
        def loss_at(sign):
            if name == "x":
                return smooth_loss(cfg, xf + sign * eps * v, wf, idx, dyf)
            w2 = dict(wf)
            w2[name] = wf[name] + sign * eps * v
            return smooth_loss(cfg, xf, w2, idx, dyf)
        fd = (loss_at(1) - loss_at(-1)) / (2 * eps)
        an = float(np.sum(g[name] * v))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_rounded_mode_is_within_bf16_rounding():
    cfg, w, x, dy, idx = make_case(4)
    g0 = oracle.layer_backward(cfg, x, w, idx, dy, round_mode=0)
    g1 = oracle.layer_backward(cfg, x, w, idx, dy, round_mode=1)
    for name in ("x",) + NAMES:
        a, b = g1[name], g0[name]
        rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
        assert rel < 2e-2, (name, rel)
    # the rounding does change the values the gradient is taken at
    assert any(not np.array_equal(g0[n], g1[n]) for n in NAMES)


def test_unchosen_experts_get_no_gradient():
    cfg, w, x, dy, idx = make_case(5, n_experts=8)
    g = oracle.layer_backward(cfg, x, w, idx, dy)
    unused = sorted(set(range(cfg.n_experts)) - set(idx.reshape(-1).tolist()))
    assert unused
    for e in unused:
        for name in ("w1", "w2", "w3", "w_router"):
            assert not np.any(g[name][e]), (name, e)


def test_expert_gradients_from_its_own_tokens_with_compact_experts():
    """One expert's routed gradients (dW1[e], dW2[e], dW3[e], row e of dW_r)
    from the tokens routed to it alone, the other experts those tokens chose
    numbered compactly, equal the full batch's bit for bit: with the routing
    held fixed each assignment's terms depend on its own token only.  The
    sampled check of these gradients at the K3 width rests on it."""
    cfg, w, x, dy, idx = make_case(10, n_experts=8, top_k=3)
    full = oracle.layer_backward(cfg, x, w, idx, dy)
    for e in np.unique(idx):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        used = np.unique(idx[toks])
        compact = {int(u): j for j, u in enumerate(used)}
        cidx = np.vectorize(compact.get, otypes=[np.int32])(idx[toks])
        cw = dict(w, w_router=w["w_router"][used], w1=w["w1"][used], w2=w["w2"][used], w3=w["w3"][used])
        sub = oracle.layer_backward(dataclasses.replace(cfg, n_experts=len(used)), x[toks], cw, cidx, dy[toks])
        j = compact[int(e)]
        for name in ("w1", "w2", "w3", "w_router"):
            np.testing.assert_array_equal(sub[name][j], full[name][e])


def test_up_projection_gradient_is_outer_product_with_normalised_latent():
    """The gradient of the projection after the norm is sum_t dy_t r_t^T with r
    the normalised latent (the oracle's forward r, rounded mode)."""
    cfg, w, x, dy, idx = make_case(6)
    g = oracle.layer_backward(cfg, x, w, idx, dy, round_mode=1)
    h = oracle.down_proj(cfg, x, w["w_down"])
    s = oracle.router(cfg, h, w["w_router"])
    gate = np.take_along_axis(s, idx, axis=1)
    r = oracle.routed(cfg, h, idx, gate, w["w1"], w["w2"], w["w3"])["r"]
    ref = dec(dy).T @ dec(r)
    np.testing.assert_allclose(g["w_up"], ref, rtol=1e-12, atol=1e-12)


def test_token_independence_of_dx():
    """dx of a token depends on that token's x and dy alone."""
    cfg, w, x, dy, idx = make_case(7)
    full = oracle.layer_backward(cfg, x, w, idx, dy, weight_grads=False)["x"]
    for t in (0, 3):
        one = oracle.layer_backward(cfg, x[t:t + 1], w, idx[t:t + 1], dy[t:t + 1], weight_grads=False)["x"]
        np.testing.assert_array_equal(one[0], full[t])


def test_scalar_derivatives():
    """SiTU'(0) = 1/2 and softcap'(0) = 1; both match central differences."""
    assert oracle.situ_grad(0.0, 4.0) == pytest.approx(0.5, abs=1e-15)
    assert oracle.softcap_grad(0.0, 25.0) == 1.0
    for b in (4.0, 25.0, 1.5):
        for x0 in (-30.0, -3.0, -0.4, 0.7, 2.5, 40.0):
            e = 1e-6
            fd = (oracle.situ(x0 + e, b) - oracle.situ(x0 - e, b)) / (2 * e)
            assert oracle.situ_grad(x0, b) == pytest.approx(fd, rel=1e-7, abs=1e-9)
            fd = (oracle.softcap(x0 + e, b) - oracle.softcap(x0 - e, b)) / (2 * e)
            assert oracle.softcap_grad(x0, b) == pytest.approx(fd, rel=1e-7, abs=1e-9)
