"""GPU parity of the Stable LatentMoE forward (through the C ABI) against the
CPU oracle.  Each stage is checked on the GPU's own input to that stage (so a
discontinuous step -- the top-k -- is compared bit for bit), and the layer
output is checked end to end against the oracle's full forward."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_moe_layer_bias_gb300 import synth

from layer_check import (ACC_REL, check_layer_output, check_o, check_r_from_o, check_y_stage, fp8_codes_robust, latent_ambiguity, routing_robust_norm_after_down, score_tol, dec,
                         e4m3_table, host_bits, oracle_cfg, rel_fro, to_e4m3, ulp_bf16, ws_view)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_moe_layer_bias_gb300 as m
    m.load_library()
    return m


def run_host_shape(lm, shape, T=None, seed_offset=0):
    w_host = synth.layer_weights_host(shape)
    x_host, b_host = synth.activations_host(shape, T=T, seed_offset=seed_offset)
    w = {k: v.cuda() for k, v in w_host.items()}
    x, bias = x_host.cuda(), b_host.cuda()
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=x.shape[0])
    ws = lm.alloc_workspace(h, x.shape[0])
    y = lm.lmoe_forward(h, x, bias, workspace=ws)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    layout = lm.lmoe_workspace_layout(h, x.shape[0])
    return dict(h=h, ws=ws, layout=layout, y=y, x_host=x_host, b_host=b_host, w_host=w_host)


def staged_checks(shape, run):
    """Compare every stage with the oracle fed the GPU's own stage inputs."""
    cfg = oracle_cfg(shape)
    T = run["x_host"].shape[0]
    E, K, L, I = shape.n_experts, shape.top_k, shape.latent, shape.inter
    S = shape.n_shared * shape.shared_inter
    ws, lay = run["ws"], run["layout"]
    wb = {k: synth.bits(v) for k, v in run["w_host"].items()}
    xb = synth.bits(run["x_host"])
    bias = run["b_host"].numpy()

    # a1: h within one bf16 ulp of the exact fp64 product
    h_gpu = host_bits(ws_view(ws, lay, "h", torch.bfloat16, (T, L)))
    X, Wd = dec(xb), dec(wb["w_down"])
    exact_h = X @ Wd.T
    absum_h = np.abs(X) @ np.abs(Wd).T
    assert np.all(np.abs(dec(h_gpu) - exact_h) <= ulp_bf16(exact_h) + ACC_REL * absum_h)

    # norm-after-down variant: the routed latent is RMSNorm(h); both sides
    # round the fp64 quotient once to bf16, so it equals the oracle's norm of
    # the GPU's own h bit for bit
    h_lat = h_gpu
    if shape.norm_after_down:
        assert lay["h_norm"] >= 0
        h_lat = host_bits(ws_view(ws, lay, "h_norm", torch.bfloat16, (T, L)))
        assert np.array_equal(h_lat, oracle.rms_rows(cfg, h_gpu))
        assert np.allclose(np.sqrt(np.mean(dec(h_lat) ** 2, axis=1)), 1.0, atol=2.0 ** -7)
    else:
        assert lay["h_norm"] == -1

    # a2: scores on the GPU's routed latent
    s_gpu = ws_view(ws, lay, "scores", torch.float32, (T, E)).cpu().numpy()
    s_ref = oracle.router(cfg, h_lat, wb["w_router"])
    absum_s = np.abs(dec(h_lat)) @ np.abs(dec(wb["w_router"])).T
    assert np.all(np.abs(s_gpu - s_ref) <= score_tol(s_ref, absum_s))

    # a3: top-k on the GPU's scores -- bit-exact
    idx_gpu = ws_view(ws, lay, "topk_idx", torch.int32, (T, K)).cpu().numpy()
    g_gpu = ws_view(ws, lay, "gates", torch.float32, (T, K)).cpu().numpy()
    idx_ref, g_ref, _ = oracle.topk(cfg, s_gpu, bias)
    assert np.array_equal(idx_gpu, idx_ref)
    assert np.array_equal(g_gpu, g_ref)

    # a4: permutation maps on the GPU's idx -- bit-exact
    counts, offsets, perm, inv = oracle.permute(cfg, idx_gpu)
    assert np.array_equal(ws_view(ws, lay, "counts", torch.int32, (E,)).cpu().numpy(), counts)
    assert np.array_equal(ws_view(ws, lay, "offsets", torch.int32, (E + 1,)).cpu().numpy(), offsets)
    assert np.array_equal(ws_view(ws, lay, "perm", torch.int32, (T * K,)).cpu().numpy(), perm)
    assert np.array_equal(ws_view(ws, lay, "inv", torch.int32, (T * K,)).cpu().numpy(), inv)

    # a5/a6: expert activations and gate-weighted outputs on the GPU's h and routing
    if shape.expert_fp8:
        fp8_expert_checks(shape, cfg, run, h_lat, idx_gpu, g_gpu, perm, inv, wb)
    else:
        rt = oracle.routed(cfg, h_lat, idx_gpu, g_gpu, wb["w1"], wb["w2"], wb["w3"], want_act=True, want_o=True)
        act_gpu = dec(host_bits(ws_view(ws, lay, "act", torch.bfloat16, (T * K, I))))
        act_ref = dec(rt["act"])[perm]                       # oracle rows are in assignment order
        # |d act/d p1| <= 1.1 * beta2 and |d act/d p2| <= beta1: the accumulation
        # error of p1, p2 carries over with those factors
        Hd = np.abs(dec(h_lat))
        tok = perm // K
        ex = idx_gpu.reshape(-1)[perm]
        acc_tol = np.zeros_like(act_ref)
        for e in np.unique(ex):
            rows = np.nonzero(ex == e)[0]
            a1 = Hd[tok[rows]] @ np.abs(dec(wb["w1"][e])).T
            a2 = Hd[tok[rows]] @ np.abs(dec(wb["w2"][e])).T
            acc_tol[rows] = ACC_REL * (1.1 * shape.beta2 * a1 + shape.beta1 * a2)
        assert np.all(np.abs(act_gpu - act_ref) <= 2 * ulp_bf16(act_ref) + acc_tol)

        # a6: the gate-weighted expert rows on the GPU's own activations,
        # element by element, and close to the oracle's from its own ones
        act_bits = host_bits(ws_view(ws, lay, "act", torch.bfloat16, (T * K, I)))[inv]   # assignment order
        o_bits = host_bits(ws_view(ws, lay, "o", torch.bfloat16, (T * K, L)))
        check_o(cfg, o_bits, act_bits, idx_gpu, g_gpu, wb["w3"])
        assert rel_fro(dec(o_bits), rt["o"]) <= 5e-3

        # a7: aggregate and RMSNorm on the GPU's own rows o, element by element
        r_bits = host_bits(ws_view(ws, lay, "r", torch.bfloat16, (T, L)))
        z_gpu = check_r_from_o(r_bits, o_bits, K, shape.rms_eps)
        r_gpu = dec(r_bits)
        assert rel_fro(r_gpu, rt["r64"]) <= 5e-3
        # mean(r^2) = ms / (ms + eps): unit RMS unless the aggregate is tiny
        # (a single expert with a gate near 0)
        ms = np.mean(z_gpu ** 2, axis=1)
        assert np.allclose(np.mean(r_gpu ** 2, axis=1), ms / (ms + shape.rms_eps), atol=2e-2)

    # a8': shared-expert activations on x
    sact_gpu = host_bits(ws_view(ws, lay, "shared_act", torch.bfloat16, (T, S)))
    sact_ref = oracle.shared_act(cfg, xb, wb["ws1"], wb["ws2"])
    ds = dec(sact_ref)
    Xa = np.abs(X)
    stol = ACC_REL * (1.1 * shape.beta2 * (Xa @ np.abs(dec(wb["ws1"])).T) +
                      shape.beta1 * (Xa @ np.abs(dec(wb["ws2"])).T))
    assert np.all(np.abs(dec(sact_gpu) - ds) <= 2 * ulp_bf16(ds) + stol)

    # a8: up-projection + shared add on the GPU's r and shared activations,
    # element by element
    y_gpu = run["y"].float().cpu().numpy().astype(np.float64)
    y_stage = check_y_stage(cfg, y_gpu, host_bits(ws_view(ws, lay, "r", torch.bfloat16, (T, L))), sact_gpu,
                            wb["w_up"], wb["ws3"])
    assert rel_fro(y_gpu, y_stage) <= 5e-3


def fp8_expert_checks(shape, cfg, run, h_lat, idx_gpu, g_gpu, perm, inv, wb):
    """FP8 variant, stages a5-a7 on the GPU's own inputs:
    - the e4m3 latent codes and their exponents equal the oracle's quantisation
      of the GPU's latent bit for bit;
    - each activation code is the e4m3 rounding of a value within 2^-9
      (relative, plus 1e-6) of the exact 4*act computed in fp64 from the
      quantised operands (the GPU evaluates the SiTU-GLU in fp32 with
      tanh.approx, ~2^-11 relative, so a value next to a rounding midpoint may
      round to the neighbouring code), and at least 97% of them equal the
      rounding of the exact value;
    - o = gate * act8/4 . W3 (e4m3) on the GPU's codes, element by element,
      and r = RMSNorm(sum of the token's rows o) on the GPU's own rows."""
    ws, lay = run["ws"], run["layout"]
    T = run["x_host"].shape[0]
    L, I, K = shape.latent, shape.inter, shape.top_k
    assert lay["h_fp8"] >= 0 and lay["h_fp8_exp"] >= 0
    h8 = ws[lay["h_fp8"]:lay["h_fp8"] + T * L].view(T, L).cpu().numpy()
    he = ws[lay["h_fp8_exp"]:lay["h_fp8_exp"] + T].cpu().numpy().view(np.int8)
    ref_codes, ref_exps = oracle.fp8_quantize_rows(h_lat)
    assert np.array_equal(h8, ref_codes) and np.array_equal(he, ref_exps)
    tab = e4m3_table()
    Hq = tab[h8] * np.exp2(he.astype(np.float64))[:, None]
    act8 = ws[lay["act"]:lay["act"] + T * K * I].view(T * K, I).cpu().numpy()
    tok, ex = perm // K, idx_gpu.reshape(-1)[perm]
    x_exact = np.zeros((T * K, I))
    o_ref = np.zeros((T * K, L))
    o_abs = np.zeros((T * K, L))
    gates = g_gpu.reshape(-1).astype(np.float64)
    for e in np.unique(ex):
        rows = np.nonzero(ex == e)[0]
        q1, e1 = oracle.fp8_quantize_rows(wb["w1"][e])
        q2, e2 = oracle.fp8_quantize_rows(wb["w2"][e])
        q3, e3 = oracle.fp8_quantize_rows(wb["w3"][e])
        W1 = tab[q1] * np.exp2(e1.astype(np.float64))[:, None]
        W2 = tab[q2] * np.exp2(e2.astype(np.float64))[:, None]
        W3 = tab[q3] * np.exp2(e3.astype(np.float64))[:, None]
        p1, p2 = Hq[tok[rows]] @ W1.T, Hq[tok[rows]] @ W2.T
        situ = shape.beta1 * np.tanh(p1 / shape.beta1) / (1.0 + np.exp(-p1))
        x_exact[rows] = 4.0 * situ * shape.beta2 * np.tanh(p2 / shape.beta2)
        o_ref[perm[rows]] = gates[perm[rows], None] * ((tab[act8[rows]] / 4.0) @ W3.T)
        o_abs[perm[rows]] = gates[perm[rows], None] * (np.abs(tab[act8[rows]] / 4.0) @ np.abs(W3).T)
    tol = 2.0 ** -9 * np.abs(x_exact) + 1e-6
    lo, mid, hi = to_e4m3(x_exact - tol), to_e4m3(x_exact), to_e4m3(x_exact + tol)
    assert np.all((act8 == lo) | (act8 == mid) | (act8 == hi))
    assert np.mean(act8 == mid) >= 0.97
    # o per element: one bf16 rounding plus the e4m3 MMA's accumulation,
    # allowed 2^-9 of gate * |W3| |act| (its internal accumulator width is not
    # documented; the bf16 MMA gets 2^-20)
    o_bits = host_bits(ws_view(ws, lay, "o", torch.bfloat16, (T * K, L)))
    o_tol = ulp_bf16(np.abs(o_ref) + 2.0 ** -9 * o_abs) + 2.0 ** -9 * o_abs
    assert np.all(np.abs(dec(o_bits) - o_ref) <= o_tol), "o"
    assert rel_fro(dec(o_bits), o_ref) <= 5e-3
    check_r_from_o(host_bits(ws_view(ws, lay, "r", torch.bfloat16, (T, L))), o_bits, K, shape.rms_eps)


def end_to_end(shape, run, allow_empty=False):
    """The layer output against the oracle's whole forward from x, over the
    tokens the acceptance bar keeps (routing margin > 1e-4), further
    filtered, in the two variants whose inputs pass a rounding that a correct
    GPU result may take the other way, by the oracle alone: the tokens whose
    oracle routing (norm-after-down) or e4m3 latent codes (FP8) do not change
    when the ambiguous elements of the oracle's own h round the other way."""
    cfg = oracle_cfg(shape)
    wb = {k: synth.bits(v) for k, v in run["w_host"].items()}
    bias = run["b_host"].numpy()
    xb = synth.bits(run["x_host"])
    ref = oracle.layer_forward(cfg, xb, wb, bias)
    also = None
    if shape.norm_after_down or shape.expert_fp8:
        amb, alt = latent_ambiguity(cfg, xb, wb["w_down"], ref["h_raw"])
        also = np.ones(xb.shape[0], bool)
        if shape.norm_after_down:
            also &= routing_robust_norm_after_down(cfg, ref["h_raw"], amb, alt, wb["w_router"], bias, ref["idx"])
        if shape.expert_fp8:
            also &= fp8_codes_robust(ref["h_raw"], amb, alt)
    rf, mx, kept = check_layer_output(run["y"], ref["y"], ref["margin"], also_keep=also, allow_empty=allow_empty)
    return rf, mx, kept, ref


def fp8_from_gpu_latent(shape, run):
    """FP8 variant, every stage after a1 at once: the oracle's FP8 layer run
    from the GPU's own latent h (quantisation, experts, aggregation, norm, up
    and shared experts) against the GPU's y, over every token with routing
    margin > 1e-4 -- including those whose e4m3 codes the end-to-end check
    has to leave out."""
    cfg = oracle_cfg(shape)
    wb = {k: synth.bits(v) for k, v in run["w_host"].items()}
    bias = run["b_host"].numpy()
    T, L = run["x_host"].shape[0], shape.latent
    ws, lay = run["ws"], run["layout"]
    h_gpu = host_bits(ws_view(ws, lay, "h", torch.bfloat16, (T, L)))
    idx_gpu = ws_view(ws, lay, "topk_idx", torch.int32, (T, shape.top_k)).cpu().numpy()
    g_gpu = ws_view(ws, lay, "gates", torch.float32, (T, shape.top_k)).cpu().numpy()
    s_gpu = ws_view(ws, lay, "scores", torch.float32, (T, shape.n_experts)).cpu().numpy()
    rt = oracle.routed_fp8(cfg, h_gpu, idx_gpu, g_gpu, wb["w1"], wb["w2"], wb["w3"])
    a_s = oracle.shared_act(cfg, synth.bits(run["x_host"]), wb["ws1"], wb["ws2"])
    y_ref = oracle.up_shared(cfg, rt["r"], a_s, wb["w_up"], wb["ws3"])
    _, _, margin = oracle.topk(cfg, s_gpu, bias)
    return check_layer_output(run["y"], y_ref, margin)


def test_tiny_layer_stages(lm):
    run = run_host_shape(lm, synth.TINY)
    staged_checks(synth.TINY, run)


def test_tiny_layer_end_to_end(lm):
    run = run_host_shape(lm, synth.TINY)
    rf, mx, kept, ref = end_to_end(synth.TINY, run)
    assert kept >= 0.8 * synth.TINY.T


def test_small_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, synth.SMALL)
    staged_checks(synth.SMALL, run)
    rf, mx, kept, _ = end_to_end(synth.SMALL, run)
    assert kept >= 0.8 * synth.SMALL.T


@pytest.mark.parametrize("T", [1, 3, 33, 127, 129, 200])
def test_tiny_layer_ragged_token_counts(lm, T):
    run = run_host_shape(lm, synth.TINY, T=T, seed_offset=T)
    staged_checks(synth.TINY, run)
    end_to_end(synth.TINY, run)


# The small widths run the down- and the up-projection on CTA pairs (latent
# 512, d = 1024: 256-wide tiles, 256 rows per pair).  Ragged batches: T = 1
# and 129 leave the second CTA of the only pair without rows (129: the first
# CTA full but one row), T = 1000 ends on a pair whose second CTA holds 104.
@pytest.mark.parametrize("T", [1, 129, 1000])
def test_small_layer_ragged_token_counts(lm, T):
    run = run_host_shape(lm, synth.SMALL, T=T, seed_offset=T)
    staged_checks(synth.SMALL, run)
    end_to_end(synth.SMALL, run, allow_empty=T == 1)   # one token may sit within the routing margin


# Widths off the usual tiles: d and the shared width not multiples of 128 (ragged
# N tiles), E = 10 (router tile mostly empty, E not a multiple of 8), k = 3,
# routed intermediate 192 (three 64-feature SiTU-GLU tiles), one shared expert,
# T = 97.
ODD = synth.LayerShape("odd", T=97, d=192, latent=128, n_experts=10, top_k=3, inter=192, n_shared=1,
                       shared_inter=192, seed=1009)


# Every expert chosen by every token (k = E): no routing margin at all, each
# expert holds all T rows.
ALL_EXPERTS = synth.LayerShape("all_experts", T=200, d=256, latent=128, n_experts=8, top_k=8, inter=64,
                               n_shared=2, shared_inter=64, seed=1010)


# The largest routing the library takes: E = 1024 experts, top-32.
MAX_ROUTING = synth.LayerShape("max_routing", T=150, d=256, latent=128, n_experts=1024, top_k=32, inter=64,
                               n_shared=2, shared_inter=64, seed=1011)


# A router as wide as K3's (E = 896 = 4 x 224) at a large batch whose last
# tile is ragged (T = 8200: 65 row tiles of 128, the last one with 8 rows; the
# up-projection's 256-row CTA-pair tiles: 33, the last with 8 rows in its
# first CTA and none in its second), on small widths.
WIDE_ROUTER = synth.LayerShape("wide_router", T=8200, d=256, latent=128, n_experts=896, top_k=16, inter=64,
                               n_shared=2, shared_inter=64, seed=1012)


def test_wide_router_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, WIDE_ROUTER)
    staged_checks(WIDE_ROUTER, run)
    rf, mx, kept, _ = end_to_end(WIDE_ROUTER, run)
    assert kept >= 0.5 * WIDE_ROUTER.T


# Split-K on the single-CTA GEMM variants (the small widths split the 256-wide
# down- and up-projection on CTA pairs): at T = 50 every dense GEMM has a few
# output tiles and at least 8 K blocks, so each splits in two.  The
# up-projection runs 128-wide tiles (d = 576: a ragged last N tile) and its
# second K range straddles the switch from r to the shared activations; the
# shared experts run 64 features per tile (S = 192); the router's 30 columns
# are stored element by element (30 is not a multiple of 4).
ODD_SPLIT = synth.LayerShape("odd_split", T=50, d=576, latent=512, n_experts=30, top_k=5, inter=128,
                             n_shared=1, shared_inter=192, seed=1014)


def test_odd_split_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, ODD_SPLIT)
    staged_checks(ODD_SPLIT, run)
    end_to_end(ODD_SPLIT, run)


# A latent of 8192 (the interface's largest) with k = 16: a token's 16 rows of
# o (256 KB) exceed a CTA's shared memory, so the combine takes its register
# path instead of the bulk copies the other shapes use.
WIDE_LATENT = synth.LayerShape("wide_latent", T=96, d=512, latent=8192, n_experts=24, top_k=16, inter=64,
                               n_shared=1, shared_inter=64, seed=1015)


def test_wide_latent_layer_stages_and_end_to_end(lm):
    assert WIDE_LATENT.top_k * WIDE_LATENT.latent * 2 > 227 * 1024
    run = run_host_shape(lm, WIDE_LATENT)
    staged_checks(WIDE_LATENT, run)
    end_to_end(WIDE_LATENT, run)


# The degenerate routing: one routed expert, chosen by every token (E = k = 1;
# 300 tokens: one pair tile of 256 rows and one of 44 in the W1|W2 GEMM).
SINGLE_EXPERT = synth.LayerShape("single_expert", T=300, d=256, latent=128, n_experts=1, top_k=1, inter=64,
                                 n_shared=2, shared_inter=64, seed=1013)


def test_single_expert_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, SINGLE_EXPERT)
    staged_checks(SINGLE_EXPERT, run)
    rf, mx, kept, _ = end_to_end(SINGLE_EXPERT, run)
    assert kept == SINGLE_EXPERT.T                    # no routing decision to leave out


def test_max_routing_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, MAX_ROUTING)
    staged_checks(MAX_ROUTING, run)
    end_to_end(MAX_ROUTING, run)


def test_all_experts_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, ALL_EXPERTS)
    staged_checks(ALL_EXPERTS, run)
    end_to_end(ALL_EXPERTS, run)


def test_odd_shape_layer_stages_and_end_to_end(lm):
    run = run_host_shape(lm, ODD)
    staged_checks(ODD, run)
    end_to_end(ODD, run)


def test_workspace_for_max_tokens_serves_every_smaller_batch(lm):
    """A workspace sized for max_tokens is large enough for every smaller
    batch, although a smaller batch may split its dense GEMMs over K more
    ways (fewer tiles) and need more partial sums: at the K3 router width
    (E = 896, latent 3584) the router splits 14 ways at 256 tokens and 12 at
    257.  The forward in such a workspace gives the same bits as in one sized
    for its own T."""
    shape = synth.LayerShape("k3_router_width", T=600, d=256, latent=3584, n_experts=896, top_k=16, inter=64,
                             n_shared=1, shared_inter=64, seed=1015)
    w = synth.layer_weights_device(shape)
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=shape.T)
    big = lm.lmoe_workspace_size(h, shape.T)
    sizes = [lm.lmoe_workspace_size(h, t) for t in range(0, shape.T + 1)]
    assert max(sizes) == big and all(a <= b for a, b in zip(sizes, sizes[1:]))
    ws_big = lm.alloc_workspace(h, shape.T)
    x, b = synth.activations_device(shape)
    for t in (64, 255, 256, 257, 384, 512, 513):
        y_big = lm.lmoe_forward(h, x[:t], b, workspace=ws_big)
        y_own = lm.lmoe_forward(h, x[:t], b, workspace=lm.alloc_workspace(h, t))
        torch.cuda.synchronize()
        assert torch.equal(y_big.view(torch.int16), y_own.view(torch.int16)), t
    assert lm.lmoe_device_status(h) == 0


@pytest.mark.parametrize("T", [300, 4096])
def test_caller_output_buffers_get_the_workspace_bits(lm, T):
    """Scores, top-k ids, gates and expert counts written to caller buffers
    equal what a forward without them leaves in its workspace, bit for bit,
    and y is unchanged; at T = 300 the router splits over K, so its scores
    come from the split's finalize."""
    shape = synth.SMALL
    E, K = shape.n_experts, shape.top_k
    w = synth.layer_weights_device(shape)
    x, b = synth.activations_device(shape, T=T, seed_offset=5)
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    y0 = lm.lmoe_forward(h, x, b, workspace=ws)
    torch.cuda.synchronize()
    lay = lm.lmoe_workspace_layout(h, T)
    ref = {"scores": ws_view(ws, lay, "scores", torch.float32, (T, E)).clone(),
           "topk_idx": ws_view(ws, lay, "topk_idx", torch.int32, (T, K)).clone(),
           "gates": ws_view(ws, lay, "gates", torch.float32, (T, K)).clone(),
           "counts": ws_view(ws, lay, "counts", torch.int32, (E,)).clone()}
    s_out = torch.full((T, E), float("nan"), device="cuda")
    i_out = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    g_out = torch.full((T, K), float("nan"), device="cuda")
    c_out = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    ws2 = lm.alloc_workspace(h, T)
    y1 = lm.lmoe_forward(h, x, b, workspace=ws2, scores_out=s_out, topk_idx_out=i_out, gates_out=g_out,
                         expert_counts_out=c_out)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    for got, key in ((s_out, "scores"), (i_out, "topk_idx"), (g_out, "gates"), (c_out, "counts")):
        assert torch.equal(got.view(torch.int32), ref[key].view(torch.int32)), key


def test_forward_is_deterministic(lm):
    """Two forwards of the same batch into two workspaces give the same bits:
    y and every intermediate (no sum depends on thread timing)."""
    shape = synth.SMALL
    T, L, K, I = shape.T, shape.latent, shape.top_k, shape.inter
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, b = (t.cuda() for t in synth.activations_host(shape))
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=T)
    lay = lm.lmoe_workspace_layout(h, T)
    runs = []
    for _ in range(2):
        ws = lm.alloc_workspace(h, T)
        y = lm.lmoe_forward(h, x, b, workspace=ws)
        runs.append((y, ws))
    torch.cuda.synchronize()
    (y1, ws1), (y2, ws2) = runs
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    for key, dt, shp in (("scores", torch.int32, (T, shape.n_experts)), ("topk_idx", torch.int32, (T, K)),
                         ("perm", torch.int32, (T * K,)), ("h", torch.int16, (T, L)),
                         ("act", torch.int16, (T * K, I)), ("o", torch.int16, (T * K, L)), ("r", torch.int16, (T, L))):
        assert torch.equal(ws_view(ws1, lay, key, dt, shp), ws_view(ws2, lay, key, dt, shp)), key


def test_host_errors_enqueue_nothing(lm):
    shape = synth.TINY
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=64)
    x = torch.zeros((65, shape.d), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(shape.n_experts, dtype=torch.float32, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward(h, x, b, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 2                       # T > max_tokens
    x = x[:64]
    small_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward(h, x, b, workspace=small_ws)
    assert e.value.status == 4                       # workspace too small
    bad = dict(shape.layer_dict())
    bad["latent"] = 100
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_create(bad, w, max_tokens=8)
    assert e.value.status == 2
    y = lm.lmoe_forward(h, x[:0], b)                 # T = 0: nothing to do
    assert y.shape[0] == 0


@pytest.mark.parametrize("name,T0", [("tiny", 512), ("small", 300)])
def test_host_io_pipeline_matches_device_forward(lm, name, T0):
    """lmoe_forward_host over several queued batches (ragged T, distinct
    inputs, both staging slots reused) gives the device forward's bits.  At
    the small widths and these batch sizes every dense GEMM splits over K, so
    the queued forwards also share the workspace's partial-sum slot."""
    shape = synth.SHAPES[name]
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=T0)
    ws = lm.alloc_workspace(h, T0)
    io = lm.alloc_host_io(h)
    xs, bs, ys = [], [], []
    for i in range(5):
        x, b = synth.activations_host(shape, T=T0, seed_offset=100 + i)
        T = T0 - 37 * i
        xs.append(x[:T].contiguous().pin_memory())
        bs.append(b.pin_memory())
        ys.append(torch.empty_like(xs[-1]).pin_memory())
    for i in range(5):
        lm.lmoe_forward_host(h, xs[i], bs[i], ys[i], io, ws)
    lm.lmoe_host_wait(h)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    for i in range(5):
        ref = lm.lmoe_forward(h, xs[i].cuda(), bs[i].cuda(), workspace=ws)
        assert torch.equal(ys[i].view(torch.int16), ref.cpu().view(torch.int16)), i
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward_host(h, xs[0], bs[0], ys[0], io[:1024], ws)
    assert e.value.status == 4                       # staging buffer too small


TINY_NORM = dataclasses.replace(synth.TINY, name="tiny_norm_after_down", norm_after_down=True)
SMALL_NORM = dataclasses.replace(synth.SMALL, name="small_norm_after_down", norm_after_down=True)


@pytest.mark.parametrize("T", [None, 1, 129])
def test_norm_after_down_variant_tiny(lm, T):
    """Ablation variant (RMSNorm after the down-projection as well): every
    stage on the GPU's own inputs, and the output end to end."""
    run = run_host_shape(lm, TINY_NORM, T=T, seed_offset=0 if T is None else T)
    staged_checks(TINY_NORM, run)
    end_to_end(TINY_NORM, run, allow_empty=T is not None)


def test_norm_after_down_variant_small(lm):
    run = run_host_shape(lm, SMALL_NORM)
    staged_checks(SMALL_NORM, run)
    rf, mx, kept, _ = end_to_end(SMALL_NORM, run)
    assert kept >= 0.8 * SMALL_NORM.T


def test_norm_after_down_routing_ignores_token_scale(lm):
    """With the variant on and eps = 0, scaling every token by 4 (exact in
    bf16) leaves the routing unchanged on the GPU as well."""
    shape = dataclasses.replace(TINY_NORM, rms_eps=0.0)
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, b = (t.cuda() for t in synth.activations_host(shape))
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=x.shape[0])
    idx1 = torch.empty((x.shape[0], shape.top_k), dtype=torch.int32, device="cuda")
    idx4 = torch.empty_like(idx1)
    lm.lmoe_forward(h, x, b, topk_idx_out=idx1)
    lm.lmoe_forward(h, (x.float() * 4).to(torch.bfloat16), b, topk_idx_out=idx4)
    torch.cuda.synchronize()
    assert torch.equal(idx1, idx4)


def test_bounded_wait_timeout_is_reported_and_context_survives(lm):
    """The failure path without a fault: a bounded mbarrier wait that nothing
    satisfies gives up after its limit and sets the handle's status; the
    status reads LMOE_ERR_TIMEOUT once, clears, and the next forward gives the
    same bits as before."""
    shape = synth.TINY
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, b = (t.cuda() for t in synth.activations_host(shape))
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=x.shape[0])
    y0 = lm.lmoe_forward(h, x, b).clone()
    assert lm.lmoe_device_status(h) == 0
    lm.lmoe_selftest_timeout(h, 2_000_000)
    assert lm.lmoe_device_status(h, clear=True) == 6     # LMOE_ERR_TIMEOUT
    assert lm.lmoe_device_status(h) == 0
    y1 = lm.lmoe_forward(h, x, b)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    with pytest.raises(lm.LmoeError):
        lm.lmoe_selftest_timeout(h, 10)                   # limit below 1 us: rejected on the host


TINY_FP8 = dataclasses.replace(synth.TINY, name="tiny_fp8", inter=128, expert_fp8=True)
SMALL_FP8 = dataclasses.replace(synth.SMALL, name="small_fp8", expert_fp8=True)


@pytest.mark.parametrize("T", [None, 1, 129])
def test_fp8_experts_variant_tiny(lm, T):
    """FP8 variant (e4m3 routed experts): every stage on the GPU's own inputs
    (quantised latent bit-exact, activation codes valid roundings, o, r, y),
    and the output end to end against the oracle's FP8 layer."""
    run = run_host_shape(lm, TINY_FP8, T=T, seed_offset=0 if T is None else T)
    staged_checks(TINY_FP8, run)
    fp8_from_gpu_latent(TINY_FP8, run)
    # with a handful of tokens the oracle-only filter may leave none
    rf, mx, kept, _ = end_to_end(TINY_FP8, run, allow_empty=T is not None)
    if T is None:
        assert kept >= 0.5 * TINY_FP8.T


def test_fp8_experts_variant_small(lm):
    run = run_host_shape(lm, SMALL_FP8)
    staged_checks(SMALL_FP8, run)
    fp8_from_gpu_latent(SMALL_FP8, run)
    rf, mx, kept, _ = end_to_end(SMALL_FP8, run)
    assert kept >= 0.5 * SMALL_FP8.T


def test_fp8_experts_rejects_unaligned_inter(lm):
    shape = dataclasses.replace(synth.TINY, expert_fp8=True)            # inter = 64
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_create(shape.layer_dict(), w, max_tokens=8)
    assert e.value.status == 2
