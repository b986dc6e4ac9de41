"""Backward pass through the C ABI against the oracle's fp64 gradient.

The oracle takes the GPU forward's routing (top-k is a discrete choice the
gradient does not pass through) and recomputes everything else in fp64 from
the same bf16 inputs; it is itself pinned by finite differences
(test_oracle_backward.py).  Every gradient (dx and the nine weights) must lie
within BWD_REL_FRO in relative Frobenius norm: the GPU path rounds seven
intermediates to bf16 (the SiTU-GLU pre-activations the training forward
keeps, dr, dz, u, dp, the experts' share of dh, dh), each a relative
perturbation of at most 2^-9 (RMS about 2^-9/sqrt(3) = 1.1e-3 per element),
so the expected error is about sqrt(7) * 1.1e-3 = 2.9e-3; the bar leaves a
factor of about 3.  The largest element error must stay within
BWD_MAX_REL of the gradient's largest element.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_bias_gb300 import synth

from layer_check import ACC_REL, S_EVAL, dec, host_bits, oracle_cfg, rel_fro, ws_view

pytestmark = pytest.mark.gpu

BWD_REL_FRO = 1e-2
BWD_MAX_REL = 2e-2


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_moe_layer_bias_gb300 as m
    m.load_library()
    return m


def run_backward(lm, shape, T=None, seed_offset=0):
    w_host = synth.layer_weights_host(shape)
    x_host, b_host = synth.activations_host(shape, T=T, seed_offset=seed_offset)
    T = x_host.shape[0]
    dy_host = synth.grad_output_host(shape, T=T, seed_offset=seed_offset)
    w = {k: v.cuda() for k, v in w_host.items()}
    x, bias, dy = x_host.cuda(), b_host.cuda(), dy_host.cuda()
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    dx, grads = lm.lmoe_backward(h, x, dy, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    lay = lm.lmoe_workspace_layout(h, T)
    idx = ws_view(ws, lay, "topk_idx", torch.int32, (T, shape.top_k)).cpu().numpy()
    return dict(h=h, ws=ws, x_host=x_host, dy_host=dy_host, w_host=w_host, idx=idx, dx=dx, grads=grads)


def compare(name, gpu, ref):
    assert np.all(np.isfinite(gpu)), name
    rf = rel_fro(gpu, ref)
    mx = float(np.max(np.abs(gpu - ref)) / max(np.max(np.abs(ref)), 1e-300))
    assert rf <= BWD_REL_FRO and mx <= BWD_MAX_REL, (name, rf, mx)
    return rf


def check_backward(shape, run):
    cfg = oracle_cfg(shape)
    wb = {k: synth.bits(v) for k, v in run["w_host"].items()}
    ref = oracle.layer_backward(cfg, synth.bits(run["x_host"]), wb, run["idx"], synth.bits(run["dy_host"]))
    errs = {"x": compare("x", dec(host_bits(run["dx"])), ref["x"])}
    for name in oracle.BACKWARD_GRADS:
        errs[name] = compare(name, run["grads"][name].cpu().double().numpy(), ref[name])
    return errs


def test_backward_tiny(lm):
    shape = synth.TINY
    check_backward(shape, run_backward(lm, shape))


@pytest.mark.parametrize("T", [1, 37, 129])
def test_backward_tiny_ragged(lm, T):
    shape = synth.TINY
    check_backward(shape, run_backward(lm, shape, T=T, seed_offset=T))


def test_backward_small(lm):
    # several tiles of every GEMM and a ragged token count
    shape = synth.SMALL
    check_backward(shape, run_backward(lm, shape, T=1000))


@pytest.mark.parametrize("T", [None, 129])
def test_backward_norm_after_down_variant_tiny(lm, T):
    """The ablation variant (RMSNorm after the down-projection as well): its
    gradient also goes through that norm's backward."""
    shape = dataclasses.replace(synth.TINY, norm_after_down=True)
    check_backward(shape, run_backward(lm, shape, T=T, seed_offset=21))


def test_backward_norm_after_down_variant_small(lm):
    shape = dataclasses.replace(synth.SMALL, norm_after_down=True)
    check_backward(shape, run_backward(lm, shape, T=1000, seed_offset=22))


def test_backward_odd_shape(lm):
    """Widths off the usual tiles (see test_gpu_layer.ODD): ragged N tiles,
    E = 10 (the router's transposes take their element-wise tail), k = 3,
    intermediate 192 (dW1 | dW2 rows split inside a 128-row tile)."""
    from test_gpu_layer import ODD
    check_backward(ODD, run_backward(lm, ODD))


def test_backward_odd_split(lm):
    """The training forward and backward with every dense GEMM of the forward
    split over K on the single-CTA variants (see test_gpu_layer.ODD_SPLIT)."""
    from test_gpu_layer import ODD_SPLIT
    check_backward(ODD_SPLIT, run_backward(lm, ODD_SPLIT))


def test_backward_all_experts(lm):
    """k = E: every expert holds all T rows (several 128-row tiles and K
    segments per expert)."""
    from test_gpu_layer import ALL_EXPERTS
    check_backward(ALL_EXPERTS, run_backward(lm, ALL_EXPERTS))


def test_backward_max_routing(lm):
    """E = 1024 (one thread per expert in the segment scan), top-32."""
    from test_gpu_layer import MAX_ROUTING
    check_backward(MAX_ROUTING, run_backward(lm, MAX_ROUTING))


def test_backward_single_expert(lm):
    """E = k = 1: every token's only expert.  Here the norm cancels the gate:
    z = g o, so r = z / sqrt(mean(z^2) + eps) depends on g only through eps,
    and the gate's (hence the router's) true gradient is o . dz with dz =
    dr inv - z (dr . z) inv / (L (ms + eps)), two terms that cancel to a
    relative eps / (ms + eps).  The GPU stores dz in bf16, so its router
    gradient is that cancellation's rounding: each token's dlogit may be off
    by 2^-8 |sigma'(x)| |o| |dz| <= 2^-8 |sigma'(x)| |o| 2 |dr| inv.  Every
    other gradient is compared as in the other layers; the router's against
    that bound (element by element, summed over the tokens)."""
    from test_gpu_layer import SINGLE_EXPERT as shape
    run = run_backward(lm, shape)
    cfg = oracle_cfg(shape)
    wb = {k: synth.bits(v) for k, v in run["w_host"].items()}
    ref = oracle.layer_backward(cfg, synth.bits(run["x_host"]), wb, run["idx"], synth.bits(run["dy_host"]))
    compare("x", dec(host_bits(run["dx"])), ref["x"])
    for name in oracle.BACKWARD_GRADS:
        if name != "w_router":
            compare(name, run["grads"][name].cpu().double().numpy(), ref[name])
    T, L = run["x_host"].shape[0], shape.latent
    lay = lm.lmoe_workspace_layout(run["h"], T)
    h = dec(host_bits(ws_view(run["ws"], lay, "h", torch.bfloat16, (T, L))))
    o = dec(host_bits(ws_view(run["ws"], lay, "o", torch.bfloat16, (T, L))))        # k = 1: one row per token
    logit = h @ dec(wb["w_router"]).T                                                   # [T, 1]
    dsig = 1.0 / (1.0 + np.exp(-logit)) / (1.0 + np.exp(logit))
    dr = dec(synth.bits(run["dy_host"])) @ dec(wb["w_up"])                             # W_up^T dy per token
    z = o                                                                              # z = the one gated row
    inv = 1.0 / np.sqrt(np.mean(z ** 2, axis=1, keepdims=True) + shape.rms_eps)
    per_tok = 2.0 ** -8 * np.abs(dsig) * np.linalg.norm(o, axis=1, keepdims=True) * 2.0 * \
        np.linalg.norm(dr, axis=1, keepdims=True) * inv
    bound = (per_tok * np.abs(h)).sum(axis=0, keepdims=True) + 1e-30
    gw = run["grads"]["w_router"].cpu().double().numpy()
    assert np.all(np.isfinite(gw))
    assert np.all(np.abs(gw - ref["w_router"]) <= bound), np.max(np.abs(gw - ref["w_router"]) / bound)


def test_backward_is_deterministic(lm):
    shape = synth.TINY
    run = run_backward(lm, shape)
    x, dy = run["x_host"].cuda(), run["dy_host"].cuda()
    dx2, g2 = lm.lmoe_backward(run["h"], x, dy, run["ws"])
    torch.cuda.synchronize()
    assert torch.equal(run["dx"], dx2)
    for n, t in run["grads"].items():
        assert torch.equal(t, g2[n]), n


@pytest.mark.parametrize("shape_name", ["tiny", "small"])
def test_backward_gradients_in_16_byte_aligned_buffers(lm, shape_name):
    """The interface promises 16-byte alignment only: gradient buffers 16
    bytes past a 32-byte boundary (TMA store maps and 16-byte stores on them)
    get the same bits as aligned ones."""
    shape = {"tiny": synth.TINY, "small": synth.SMALL}[shape_name]
    run = run_backward(lm, shape, T=300)
    x, dy = run["x_host"].cuda(), run["dy_host"].cuda()
    off = {}
    for n, s in lm.grad_shapes(run["h"]).items():
        numel = int(np.prod(s))
        flat = torch.empty(numel + 8, dtype=torch.float32, device="cuda")
        assert flat.data_ptr() % 32 == 0
        off[n] = flat[4:4 + numel].view(s)
        assert off[n].data_ptr() % 32 == 16
    dx2, _ = lm.lmoe_backward(run["h"], x, dy, run["ws"], grads=off)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(run["h"]) == 0
    assert torch.equal(run["dx"], dx2)
    for n, t in run["grads"].items():
        assert torch.equal(t, off[n]), n


def test_backward_unused_experts_get_zero(lm):
    # few tokens: most of the 32 experts are chosen by none
    shape = synth.TINY
    run = run_backward(lm, shape, T=3, seed_offset=5)
    used = set(run["idx"].reshape(-1).tolist())
    unused = [e for e in range(shape.n_experts) if e not in used]
    assert unused
    for n in ("w1", "w2", "w3", "w_router"):
        g = run["grads"][n].cpu()
        for e in unused:
            assert not torch.any(g[e] != 0), (n, e)


@pytest.mark.parametrize("shape_name", ["tiny", "small"])
def test_training_forward_output_is_the_inference_forward(lm, shape_name):
    """A with_backward handle's forward (whose SiTU-GLU GEMMs also keep their
    pre-activations) gives the inference forward's y and routing bit for bit."""
    shape = synth.SHAPES[shape_name]
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=777))
    T = x.shape[0]
    out = []
    for wb in (False, True):
        h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=wb), w, max_tokens=T)
        ws = lm.alloc_workspace(h, T)
        y = lm.lmoe_forward(h, x, bias, workspace=ws)
        torch.cuda.synchronize()
        assert lm.lmoe_device_status(h) == 0
        lay = lm.lmoe_workspace_layout(h, T)
        assert (lay["pre_act"] >= 0) == wb and (lay["shared_pre_act"] >= 0) == wb
        out.append((y.clone(), ws_view(ws, lay, "topk_idx", torch.int32, (T, shape.top_k)).clone()))
        lm.lmoe_destroy(h)
    assert torch.equal(out[0][0], out[1][0])
    assert torch.equal(out[0][1], out[1][1])


@pytest.mark.parametrize("shape_name,T", [("tiny", 300), ("small", 1000)])
def test_kept_pre_activations_match_their_definition(lm, shape_name, T):
    """pre_act row p (permuted order) holds W1[e] h_t | W2[e] h_t for the
    assignment perm[p] = t * top_k + j, e = idx[t][j], and shared_pre_act row t
    holds Ws1 x_t | Ws2 x_t, each the bf16 rounding of the fp32-accumulated
    product: within 2^-8 relative of the fp64 product of the same bf16
    operands (plus fp32 accumulation error).  logits holds W_router h_t in
    fp32 (within the accumulation error), and the scores are its sigmoid."""
    shape = synth.SHAPES[shape_name]
    w_host = synth.layer_weights_host(shape)
    w = {k: v.cuda() for k, v in w_host.items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=T, seed_offset=3))
    L, I, K = shape.latent, shape.inter, shape.top_k
    S = shape.n_shared * shape.shared_inter
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    torch.cuda.synchronize()
    lay = lm.lmoe_workspace_layout(h, T)
    hl = dec(host_bits(ws_view(ws, lay, "h", torch.bfloat16, (T, L))))
    idx = ws_view(ws, lay, "topk_idx", torch.int32, (T, K)).cpu().numpy()
    perm = ws_view(ws, lay, "perm", torch.int32, (T * K,)).cpu().numpy()
    pre = dec(host_bits(ws_view(ws, lay, "pre_act", torch.bfloat16, (T * K, 2 * I))))
    spre = dec(host_bits(ws_view(ws, lay, "shared_pre_act", torch.bfloat16, (T, 2 * S))))
    tok = perm // K
    ex = idx.reshape(-1)[perm]
    w12 = np.concatenate([dec(synth.bits(w_host["w1"])), dec(synth.bits(w_host["w2"]))], axis=1)   # [E][2I][L]
    ref, absum = np.zeros_like(pre), np.zeros_like(pre)
    for e in np.unique(ex):
        rows = np.nonzero(ex == e)[0]
        ref[rows] = hl[tok[rows]] @ w12[e].T
        absum[rows] = np.abs(hl[tok[rows]]) @ np.abs(w12[e]).T
    assert np.all(np.abs(pre - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * absum)
    xs = dec(synth.bits(x.cpu()))
    ws12 = np.concatenate([dec(synth.bits(w_host["ws1"])), dec(synth.bits(w_host["ws2"]))], axis=0)   # [2S][d]
    sref = xs @ ws12.T
    sabs = np.abs(xs) @ np.abs(ws12).T
    assert np.all(np.abs(spre - sref) <= 2.0 ** -8 * np.abs(sref) + 1e-5 * sabs)
    E = shape.n_experts
    logits = ws_view(ws, lay, "logits", torch.float32, (T, E)).cpu().double().numpy()
    wr = dec(synth.bits(w_host["w_router"]))
    assert np.all(np.abs(logits - hl @ wr.T) <= ACC_REL * (np.abs(hl) @ np.abs(wr).T) + 1e-30)
    scores = ws_view(ws, lay, "scores", torch.float32, (T, E)).cpu().double().numpy()
    assert np.all(np.abs(scores - 1.0 / (1.0 + np.exp(-np.clip(logits, -700.0, 700.0)))) <= S_EVAL)
    lm.lmoe_destroy(h)


def test_backward_needs_a_backward_handle(lm):
    shape = synth.TINY
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=8))
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=8)
    ws = lm.alloc_workspace(h, 8)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_backward(h, x, torch.zeros_like(x), ws, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 1
    torch.cuda.synchronize()


def test_backward_k3_prefill_sampled(lm):
    """K3 prefill (T = 8192) in the configuration the benchmark times: dx on
    sampled tokens (outlier tokens included) against the oracle, which is
    exact per token because dx_t depends on x_t and dy_t alone; dW_up and
    dWs3 on sampled columns against their definition sum_t dy_t r_t^T and
    sum_t dy_t as_t^T on the forward's own r and shared activations; the
    routed weight gradients of sampled experts against the oracle (below);
    every gradient finite."""
    shape = synth.K3_PREFILL
    T, K, L = shape.T, shape.top_k, shape.latent
    S = shape.n_shared * shape.shared_inter
    torch.manual_seed(0)
    w = synth.layer_weights_device(shape)
    x, bias = synth.activations_device(shape)
    dy = synth.grad_output_device(shape)
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    dx, grads = lm.lmoe_backward(h, x, dy, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    lay = lm.lmoe_workspace_layout(h, T)
    idx = ws_view(ws, lay, "topk_idx", torch.int32, (T, K)).cpu().numpy()
    for n, g in grads.items():
        assert bool(torch.isfinite(g).all()), n
    assert bool(torch.isfinite(dx.float()).all())

    rng = np.random.default_rng(3)
    big = torch.nonzero(x.float().abs().amax(dim=1) > 20).flatten().cpu().numpy()   # outlier tokens
    sample = np.unique(np.concatenate([rng.choice(T, 5, replace=False), big[:1]]))
    cfg = oracle_cfg(shape)
    dense = {n: synth.bits(w[n]) for n in ("w_down", "w_router", "ws1", "ws2", "ws3", "w_up")}
    used = np.unique(idx[sample])
    wb = dict(dense)
    for n in ("w1", "w2", "w3"):
        wb[n] = {int(e): synth.bits(w[n][int(e)]) for e in used}
    sm = torch.from_numpy(sample).cuda()
    ref = oracle.layer_backward(cfg, host_bits(x[sm]), wb, idx[sample], host_bits(dy[sm]), weight_grads=False)
    compare("x (sampled tokens)", dec(host_bits(dx[sm])), ref["x"])

    # dW_up and dWs3 on sampled columns, in fp64 on the host from the
    # forward's own bf16 r and shared activations
    dyd = dec(host_bits(dy))
    cols = np.sort(rng.choice(L, 24, replace=False))
    r = dec(host_bits(ws_view(ws, lay, "r", torch.bfloat16, (T, L))))[:, cols]
    compare("w_up (sampled columns)", grads["w_up"].cpu().double().numpy()[:, cols], dyd.T @ r)
    scols = np.sort(rng.choice(S, 24, replace=False))
    a_s = dec(host_bits(ws_view(ws, lay, "shared_act", torch.bfloat16, (T, S))))[:, scols]
    compare("ws3 (sampled columns)", grads["ws3"].cpu().double().numpy()[:, scols], dyd.T @ a_s)

    # dW1[e], dW2[e], dW3[e] and row e of dW_r sum over the assignments to
    # expert e alone, and with the routing held fixed each assignment's terms
    # depend only on its own token: the oracle's backward over exactly the
    # tokens routed to e gives them.  The other experts those tokens chose are
    # numbered compactly (each keeps its own weights and router row, so every
    # token's gates and aggregate are unchanged).  Three of the experts with the
    # fewest tokens keep the oracle's fp64 gradient arrays small.
    E = shape.n_experts
    counts = np.bincount(idx.ravel(), minlength=E)
    touched = np.nonzero(counts)[0]
    picks = touched[np.argsort(counts[touched], kind="stable")[:3]]
    g_all = ws_view(ws, lay, "gates", torch.float32, (T, K)).cpu().numpy()
    expert_grads_match(shape, w, dense, (ws, lay, idx, g_all), x, dy, grads, picks)


def router_row_bound(shape, w, ws, lay, x, dy, idx, gates, e, toks):
    """Element-wise bound on the error of row e of dW_r = sum over the
    assignments a of expert e of dlogit_a * hl_t (hl: the routed latent).
    dlogit_a = sigma'(logit_a) * dg_a with dg_a = o'_a . dz_t (o' = W3[e] act_a,
    the un-gated expert output; dz_t the gradient at the aggregate z_t).  The
    norm's backward makes sum_j g_j dg_j vanish, so a dg_j cancels whenever
    expert j carries much of z_t, and its relative error is not small.  The
    GPU computes it as act . u with u = W3^T dz in bf16, from dz in bf16, from
    dr = W_up^T dy in bf16, with act in bf16: each rounding contributes at
    most 2^-9 of its own magnitude,
        |d dg| <= 2^-9 (3 |u| |act| + |o'| |dz| + 2 |o'| |dr| inv),
    times |sigma'|; the latent itself may take the other bf16 rounding on one
    side (2^-8 |dlogit| |hl|).  Everything is computed in fp64 from the
    forward's own workspace rows."""
    T, K, L, I = shape.T, shape.top_k, shape.latent, shape.inter
    key = "h_norm" if shape.norm_after_down else "h"
    tk = torch.from_numpy(np.asarray(toks)).cuda()
    hl = dec(host_bits(ws_view(ws, lay, key, torch.bfloat16, (T, L))[tk]))
    rows = (np.asarray(toks)[:, None] * K + np.arange(K)[None, :]).reshape(-1)
    o = dec(host_bits(ws_view(ws, lay, "o", torch.bfloat16, (T * K, L))[torch.from_numpy(rows).cuda()]))
    o = o.reshape(len(toks), K, L)
    inv_map = ws_view(ws, lay, "inv", torch.int32, (T * K,)).cpu().numpy()
    wr = dec(synth.bits(w["w_router"][e]))
    w3 = dec(synth.bits(w["w3"][e]))                                    # [L, I]
    wup = dec(synth.bits(w["w_up"]))                                    # [d, L]
    dyd = dec(host_bits(dy[tk]))
    bound = np.zeros(L)
    for i, t in enumerate(toks):
        z = o[i].sum(axis=0)
        inv = 1.0 / np.sqrt(np.mean(z * z) + shape.rms_eps)
        dr = wup.T @ dyd[i]
        dz = inv * dr - z * (dr @ z) * inv ** 3 / L
        for j in np.nonzero(idx[t] == e)[0]:
            a = int(t) * K + int(j)
            act = dec(host_bits(ws_view(ws, lay, "act", torch.bfloat16, (T * K, I))[int(inv_map[a])]))
            op = w3 @ act
            u = w3.T @ dz
            sg = 1.0 / (1.0 + np.exp(-(wr @ hl[i])))
            dsig = sg * (1.0 - sg)
            ddl = dsig * 2.0 ** -9 * (3 * np.linalg.norm(u) * np.linalg.norm(act) +
                                      np.linalg.norm(op) * np.linalg.norm(dz) +
                                      2 * np.linalg.norm(op) * np.linalg.norm(dr) * inv)
            dl = abs(dsig * (op @ dz))
            bound += (ddl + 2.0 ** -8 * dl) * np.abs(hl[i])
    return bound + 1e-30


def expert_grads_match(shape, w, dense, fwd, x, dy, grads, picks):
    """dW1[e], dW2[e], dW3[e] for the experts in `picks` against the oracle's
    backward over exactly the tokens routed to each (the other experts those
    tokens chose numbered compactly; relative tolerance), and row e of dW_r
    against the oracle within router_row_bound.  `fwd`: the forward's
    workspace and layout and its idx, gates."""
    cfg = oracle_cfg(shape)
    ws, lay, idx, gates = fwd
    for e in picks:
        toks = np.nonzero((idx == e).any(axis=1))[0]
        used = np.unique(idx[toks])
        compact = {int(u): j for j, u in enumerate(used)}
        cidx = np.vectorize(compact.get, otypes=[np.int32])(idx[toks])
        cw = dict(dense)
        cw["w_router"] = synth.bits(w["w_router"][torch.from_numpy(used).cuda()])
        for n in ("w1", "w2", "w3"):
            cw[n] = {compact[int(u)]: synth.bits(w[n][int(u)]) for u in used}
        tk = torch.from_numpy(toks).cuda()
        ref = oracle.layer_backward(dataclasses.replace(cfg, n_experts=len(used)), host_bits(x[tk]), cw, cidx,
                                    host_bits(dy[tk]))
        j = compact[int(e)]
        for n in ("w1", "w2", "w3"):
            compare(f"{n}[{e}] ({len(toks)} tokens)", grads[n][int(e)].cpu().double().numpy(), ref[n][j])
        gw = grads["w_router"][int(e)].cpu().double().numpy()
        assert np.all(np.isfinite(gw))
        bound = router_row_bound(shape, w, ws, lay, x, dy, idx, gates, int(e), toks)
        err = np.abs(gw - ref["w_router"][j])
        assert np.all(err <= bound), (e, len(toks), float(np.max(err / bound)))


@pytest.mark.parametrize("norm_after_down", [False, True])
def test_backward_k3_decode(lm, norm_after_down):
    """K3 widths at decode size (T = 64; the training forward splits its dense
    GEMMs over K): dx of every token against the oracle (exact per token), and
    the routed weight gradients of three experts; both layer variants."""
    shape = dataclasses.replace(synth.K3_DECODE, norm_after_down=norm_after_down)
    T, K = shape.T, shape.top_k
    torch.manual_seed(0)
    w = synth.layer_weights_device(shape)
    x, bias = synth.activations_device(shape)
    dy = synth.grad_output_device(shape)
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    dx, grads = lm.lmoe_backward(h, x, dy, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    lay = lm.lmoe_workspace_layout(h, T)
    idx = ws_view(ws, lay, "topk_idx", torch.int32, (T, K)).cpu().numpy()
    for n, g in grads.items():
        assert bool(torch.isfinite(g).all()), n
    cfg = oracle_cfg(shape)
    dense = {n: synth.bits(w[n]) for n in ("w_down", "w_router", "ws1", "ws2", "ws3", "w_up")}
    used = np.unique(idx)
    wb = dict(dense)
    for n in ("w1", "w2", "w3"):
        wb[n] = {int(e): synth.bits(w[n][int(e)]) for e in used}
    ref = oracle.layer_backward(cfg, host_bits(x), wb, idx, host_bits(dy), weight_grads=False)
    compare("x (every token)", dec(host_bits(dx)), ref["x"])
    counts = np.bincount(idx.ravel(), minlength=shape.n_experts)
    touched = np.nonzero(counts)[0]
    picks = touched[np.argsort(-counts[touched], kind="stable")[:1]].tolist()      # the busiest expert
    picks += touched[np.argsort(counts[touched], kind="stable")[:2]].tolist()      # and two with one token
    g_all = ws_view(ws, lay, "gates", torch.float32, (T, K)).cpu().numpy()
    expert_grads_match(shape, w, dense, (ws, lay, idx, g_all), x, dy, grads, picks)


def test_backward_with_forward_outputs_in_caller_buffers(lm):
    """A forward that wrote its routing outputs to caller buffers leaves those
    workspace slots untouched (here: filled with 0xff bytes); the backward
    takes topk_idx and gates from the caller and derives the per-expert counts
    from the workspace's offsets.  It gives the same bits as the default path
    on a copy of that workspace whose routing slots hold the same values."""
    shape = synth.TINY
    T = 64
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=T, seed_offset=9))
    dy = synth.grad_output_host(shape, T=T, seed_offset=9).cuda()
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws2 = lm.alloc_workspace(h, T)
    ws2.fill_(255)
    E, K = shape.n_experts, shape.top_k
    scores = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    lm.lmoe_forward(h, x, bias, workspace=ws2, scores_out=scores, topk_idx_out=idx, gates_out=gates,
                    expert_counts_out=counts)
    torch.cuda.synchronize()
    lay = lm.lmoe_workspace_layout(h, T)
    for key in ("topk_idx", "gates"):      # the slots the forward left alone
        assert torch.all(ws_view(ws2, lay, key, torch.int32, (T, K)) == -1)
    ws = ws2.clone()
    ws_view(ws, lay, "topk_idx", torch.int32, (T, K)).copy_(idx)
    ws_view(ws, lay, "gates", torch.float32, (T, K)).copy_(gates)
    dx_b, g_b = lm.lmoe_backward(h, x, dy, ws2, topk_idx=idx, gates=gates)
    dx_a, g_a = lm.lmoe_backward(h, x, dy, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    assert torch.equal(dx_a, dx_b)
    for n in g_a:
        assert torch.equal(g_a[n], g_b[n]), n


def test_backward_host_errors_enqueue_nothing(lm):
    shape = synth.TINY
    T = 16
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=T))
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    dy = torch.zeros_like(x)
    need = lm.lmoe_backward_workspace_size(h, T)
    with pytest.raises(lm.LmoeError) as e:        # workspace too small
        lm.lmoe_backward(h, x, dy, ws, workspace=torch.empty(need - 256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4
    with pytest.raises(lm.LmoeError) as e:        # forward workspace too small
        lm.lmoe_backward(h, x, dy, ws[:1024])
    assert e.value.status == 4
    with pytest.raises(lm.LmoeError) as e:        # more tokens than the handle was made for
        lm.lmoe_backward_workspace_size(h, T + 1)
    assert e.value.status == 2
    # T = 0 enqueues nothing and succeeds
    dx0, _ = lm.lmoe_backward(h, x[:0], dy[:0], ws, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert dx0.shape[0] == 0
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0


def test_backward_accumulates_into_gradients(lm):
    """accumulate = 1 adds the pass's weight gradients to the buffers: one fp32
    addition per element, so the result equals init + (the overwriting
    pass's gradients) bit for bit, unchosen experts included."""
    shape = synth.TINY
    T = 200
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=T, seed_offset=13))
    dy = synth.grad_output_host(shape, T=T, seed_offset=13).cuda()
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    dx1, g1 = lm.lmoe_backward(h, x, dy, ws)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(17)
    init = {n: torch.randn(t.shape, generator=gen, device="cuda") for n, t in g1.items()}
    acc = {n: t.clone() for n, t in init.items()}
    dx2, _ = lm.lmoe_backward(h, x, dy, ws, grads=acc, accumulate=True)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    assert torch.equal(dx1, dx2)
    for n in g1:
        assert torch.equal(acc[n], init[n] + g1[n]), n


def test_backward_stage_hook_gives_the_same_bits(lm):
    """With the timing hook the backward runs every stage in stream order (no
    side stream); the gradients are the same bits as the overlapped default."""
    shape = synth.TINY
    run = run_backward(lm, shape, T=300, seed_offset=31)
    x, dy = run["x_host"].cuda(), run["dy_host"].cuda()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(lm.BWD_STAGES) + 1)]
    lm.lmoe_set_backward_events(run["h"], evs)
    dx2, g2 = lm.lmoe_backward(run["h"], x, dy, run["ws"])
    torch.cuda.synchronize()
    lm.lmoe_set_backward_events(run["h"], None)
    assert all(evs[j].elapsed_time(evs[j + 1]) >= 0 for j in range(len(evs) - 1))
    assert torch.equal(run["dx"], dx2)
    for n, t in run["grads"].items():
        assert torch.equal(t, g2[n]), n
