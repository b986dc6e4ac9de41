"""Shared helpers for the GPU-vs-oracle parity tests (test infrastructure)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from sparse_moe_layer_bias_gb300 import synth

# Tolerances (floating point).  The layer output bar is the one the method
# targets: rel. Frobenius <= 1e-2 and max-abs <= 5e-2 * RMS over tokens whose
# k-th/(k+1)-th biased-score margin exceeds 1e-4.
Y_REL_FRO = 1e-2
Y_MAX_ABS_RMS = 5e-2
MARGIN = 1e-4
# fp32 accumulation: a bf16 result of a K-long dot product may differ from the
# nearest bf16 of the exact value by one ulp plus the accumulation error, which
# under cancellation is bounded by a small multiple of 2^-24 * sum|x_i w_i|.
ACC_REL = 2.0 ** -20
# Router scores from the same bf16 latent: the logit carries the accumulation
# error ACC_REL * sum|h_l w_l|, scaled by the sigmoid's slope s(1-s), plus a
# few fp32 ulps from evaluating the sigmoid itself.
S_EVAL = 1e-6


def score_tol(s, absum):
    s = s.astype(np.float64)
    return s * (1.0 - s) * ACC_REL * absum + S_EVAL


def dec(bits):
    return synth.from_bits(np.asarray(bits)).double().numpy()


def ulp_bf16(v):
    """Spacing of bf16 numbers at |v| (normal range)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def ws_view(ws: torch.Tensor, layout: dict, key: str, dtype, shape):
    off = layout[key]
    assert off >= 0
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    return ws[off:off + n].view(dtype).view(*shape)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return synth.bits(t.cpu())


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_layer_output(y_gpu_bf16: torch.Tensor, y_ref: np.ndarray, margin: np.ndarray, also_keep=None,
                       allow_empty=False):
    """The acceptance test on the layer output; returns (rel_fro, max_abs/rms, kept).

    The layer's output is bf16, so rounding it costs up to half a bf16 ulp of
    |y| by itself; on the x50 outlier tokens |y| reaches ~40x RMS(out), where
    that alone is ~10% of RMS.  The max-abs bar is therefore applied to the
    error beyond the output's own rounding: max(0, |dy| - ulp(y_ref)/2)."""
    yg = y_gpu_bf16.float().cpu().numpy().astype(np.float64)
    keep = margin > MARGIN
    if also_keep is not None:
        keep &= also_keep
    if allow_empty and keep.sum() == 0:
        return float("nan"), float("nan"), 0
    assert keep.sum() > 0, "no token kept" 
    d = np.abs(yg - y_ref)[keep]
    ref = y_ref[keep]
    rf = rel_fro(yg[keep], ref)
    rms = math.sqrt(float(np.mean(ref ** 2)))
    beyond = np.maximum(0.0, d - 0.5 * ulp_bf16(ref))
    mx = float(np.max(beyond)) / rms
    assert rf <= Y_REL_FRO, f"rel Frobenius {rf:.3e}"
    assert mx <= Y_MAX_ABS_RMS, f"max abs / RMS {mx:.3e}"
    return rf, mx, int(keep.sum())


def absum_experts(cfg, act_abs, idx, gate, w_abs):
    """sum_j gate[t, j] * (|W3[e_j]| @ |act_j|) per token and latent channel:
    the scale of the aggregate's accumulation error.  act_abs [T*k, inter]
    (assignment order), w_abs(e) -> |W3[e]| [latent, inter]."""
    T, K = idx.shape
    out = np.zeros((T, cfg.latent))
    flat = idx.reshape(-1)
    g = np.abs(gate.reshape(-1).astype(np.float64))
    for e in np.unique(flat):
        rows = np.nonzero(flat == e)[0]
        contrib = (act_abs[rows] @ w_abs(int(e)).T) * g[rows, None]
        np.add.at(out, rows // K, contrib)
    return out


def check_o(cfg, o_bits, act_bits, idx, gate, w3):
    """a6 on the GPU's own activations, element by element: each gate-weighted
    expert row o (bf16, assignment order) against the oracle's fp64
    gate * W3[e] act on the same bf16 activations.  Bound: one bf16 rounding
    plus the fp32 accumulation of the K = inter dot product (2^-20 of
    gate * |W3| |act|).  Returns the oracle's rows."""
    import dataclasses
    n = idx.size
    one = dataclasses.replace(cfg, top_k=1)          # every assignment on its own
    o_ref = oracle.expert_aggregate(one, act_bits, idx.reshape(n, 1), gate.reshape(n, 1), w3)
    acc = ACC_REL * absum_experts(one, np.abs(dec(act_bits)), idx.reshape(n, 1), gate.reshape(n, 1),
                                  lambda e: np.abs(dec(w3[e])))
    tol = ulp_bf16(np.abs(o_ref) + acc) + acc
    err = np.abs(dec(o_bits) - o_ref)
    assert np.all(err <= tol), f"o: worst error / bound {np.max(err / tol):.3g}"
    return o_ref


def check_r_from_o(r_bits, o_bits, k, eps):
    """a7 on the GPU's own rows o (assignment order): z = the sum of the
    token's k rows, r within one bf16 ulp of the exact z / sqrt(mean(z^2) +
    eps), plus the fp32 summation error of z (k * 2^-24 of sum |o_j|)
    carried through the norm."""
    O = dec(o_bits)
    T = O.shape[0] // k
    O = O.reshape(T, k, -1)
    z = O.sum(axis=1)
    inv = 1.0 / np.sqrt(np.mean(z ** 2, axis=1, keepdims=True) + eps)
    r_exact = z * inv
    tol = ulp_bf16(r_exact) + 2.0 * k * 2.0 ** -24 * np.abs(O).sum(axis=1) * inv + 2.0 ** -20 * np.abs(r_exact)
    err = np.abs(dec(r_bits) - r_exact)
    assert np.all(err <= tol), f"r: worst error / bound {np.max(err / tol):.3g}"
    return z


def check_y_stage(cfg, y_gpu, r_bits, sact_bits, w_up, ws3):
    """a8 on the GPU's own r and shared activations, element by element: y
    within one bf16 ulp plus the fp32 accumulation bound of the exact
    W_up r + Ws3 act_s."""
    y_ref = oracle.up_shared(cfg, r_bits, sact_bits, w_up, ws3)
    acc = ACC_REL * (np.abs(dec(r_bits)) @ np.abs(dec(w_up)).T + np.abs(dec(sact_bits)) @ np.abs(dec(ws3)).T)
    tol = ulp_bf16(np.abs(y_ref) + acc) + acc
    yg = y_gpu.float().cpu().numpy().astype(np.float64) if isinstance(y_gpu, torch.Tensor) else y_gpu
    err = np.abs(yg - y_ref)
    assert np.all(err <= tol), f"y: worst error / bound {np.max(err / tol):.3g}"
    return y_ref


# Oracle-only filters for end-to-end checks whose inputs pass a rounding that
# another correct computation may take the other way.  A bf16 result of a
# K-long dot product accumulated in fp32 (in any order) lies, with
# overwhelming probability, within ROUND_SIGMAS standard deviations of a
# random-walk rounding model of the exact value: sigma ~ 2^-24 * sqrt(K) *
# sqrt(sum_i (x_i w_i)^2).  Elements of the oracle's own bf16 result whose
# exact value lies that close to a rounding midpoint are "ambiguous": a
# correct GPU result may hold the other neighbour there.
ROUND_SIGMAS = 4.0


def bf16_ambiguity(bits, exact, sq_sum, K):
    """(mask, alt): the elements of the oracle's bf16 result ``bits`` (the
    nearest bf16 of ``exact``) that lie within ROUND_SIGMAS * 2^-24 * sqrt(K)
    * sqrt(sq_sum) of a rounding midpoint, and the other neighbour's bits."""
    bits = np.asarray(bits, np.uint16)
    v = dec(bits)
    up = np.where(v >= 0, bits.astype(np.int32) + 1, bits.astype(np.int32) - 1)
    dn = np.where(v > 0, bits.astype(np.int32) - 1, bits.astype(np.int32) + 1)
    alt = np.where(exact > v, up, dn).astype(np.uint16)
    tau = ROUND_SIGMAS * 2.0 ** -24 * math.sqrt(K) * np.sqrt(sq_sum)
    mid = 0.5 * (v + dec(alt))
    mask = (exact != v) & (v != 0) & (np.abs(exact - mid) <= tau)
    return mask, alt


def latent_ambiguity(cfg, x_bits, w_down_bits, h_bits):
    """bf16_ambiguity of the oracle's down-projection h = W_down x."""
    X, Wd = dec(x_bits), dec(w_down_bits)
    return bf16_ambiguity(h_bits, X @ Wd.T, (X ** 2) @ (Wd ** 2).T, cfg.d)


def routing_robust_norm_after_down(cfg, h_bits, amb, alt, w_router, bias, idx, seed=0):
    """Norm-after-down variant: tokens whose oracle routing stays the same
    when the ambiguous elements of the oracle's own h take their other
    rounding -- all of them at once, and two random halves of them.  The
    routed latent RMSNorm(h) depends on the whole row of h, so a last-bit
    change anywhere can move every score; this decides on the oracle's data
    alone which tokens such changes cannot re-route."""
    rng = np.random.default_rng(seed)
    ok = np.ones(h_bits.shape[0], bool)
    ref = np.sort(idx, axis=1)
    for trial in range(3):
        flip = amb if trial == 0 else (amb & (rng.random(amb.shape) < 0.5))
        hp = np.where(flip, alt, h_bits).astype(np.uint16)
        s = oracle.router(cfg, oracle.rms_rows(cfg, hp), w_router)
        ip, _, _ = oracle.topk(cfg, s, bias)
        ok &= np.all(np.sort(ip, axis=1) == ref, axis=1)
    return ok


def fp8_codes_robust(h_bits, amb, alt):
    """FP8 variant: tokens whose e4m3 latent codes (and power-of-two row
    scale) are the same whichever rounding each ambiguous element of the
    oracle's own h takes.  For these the GPU's codes must equal the oracle's;
    the other tokens may differ by a whole e4m3 step in some element."""
    v, a = np.abs(dec(h_bits)), np.abs(dec(alt))
    hi = np.where(amb, np.maximum(v, a), v).max(axis=1)
    lo = np.where(amb, np.minimum(v, a), v).max(axis=1)
    e_hi = np.array([oracle.fp8_exp_for(float(m)) for m in hi])
    e_lo = np.array([oracle.fp8_exp_for(float(m)) for m in lo])
    scale = np.exp2(-e_hi.astype(np.float64))[:, None]
    same = to_e4m3(dec(h_bits) * scale) == to_e4m3(dec(alt) * scale)
    return (e_hi == e_lo) & np.all(same | ~amb, axis=1)


def oracle_cfg(shape: synth.LayerShape) -> oracle.LayerConfig:
    return oracle.LayerConfig(**shape.layer_dict())


_E4M3_VALUES = None


def e4m3_table():
    """fp64 value of each of the 256 e4m3 codes (the oracle's decoder)."""
    global _E4M3_VALUES
    if _E4M3_VALUES is None:
        _E4M3_VALUES = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    return _E4M3_VALUES


def to_e4m3(x):
    """Vectorised e4m3 rounding (torch's float8_e4m3fn conversion; equal to
    the oracle's encoder inside +-448, which is pinned on the CPU)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
