"""CPU oracle for the Stable LatentMoE layer forward and Quantile Balancing.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``sparse_moe_layer_bias_gb300``) never imports it and shares no
code with it.

The arithmetic lives in ``lmoe_oracle.c`` (plain fp64 C, OpenMP over tokens);
this module only compiles it with gcc and marshals numpy arrays through ctypes.
bf16 tensors are passed as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lmoe_oracle.c")
_LIB = os.path.join(_HERE, "liblmoe_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liblmoe_oracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class OrcConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("latent", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("rms_eps", ctypes.c_double)]


@dataclass
class LayerConfig:
    """Shape and constants of one Stable LatentMoE layer."""
    d: int
    latent: int
    n_experts: int
    top_k: int
    inter: int
    n_shared: int
    shared_inter: int
    beta1: float = 4.0
    beta2: float = 25.0
    rms_eps: float = 1e-6
    norm_after_down: bool = False   # ablation variant: RMSNorm on h as well
    expert_fp8: bool = False        # FP8 variant: e4m3 routed experts

    def c(self) -> OrcConfig:
        return OrcConfig(self.d, self.latent, self.n_experts, self.top_k, self.inter,
                         self.n_shared, self.shared_inter, self.beta1, self.beta2, self.rms_eps)


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        cfg = ctypes.POINTER(OrcConfig)
        sig = {
            "orc_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_sigmoid": (ctypes.c_double, [ctypes.c_double]),
            "orc_softcap": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
            "orc_situ": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
            "orc_down_proj": (None, [cfg, _I64, _P, _P, _P]),
            "orc_rms_rows": (None, [_I64, _I64, ctypes.c_double, _P, _P]),
            "orc_router": (None, [cfg, _I64, _P, _P, _P]),
            "orc_topk": (None, [cfg, _I64, _P, _P, _P, _P, _P]),
            "orc_permute": (None, [cfg, _I64, _P, _P, _P, _P, _P]),
            "orc_routed": (None, [cfg, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
            "orc_expert_aggregate": (None, [cfg, _I64, _P, _P, _P, _P, _P]),
            "orc_shared_act": (None, [cfg, _I64, _P, _P, _P, _P]),
            "orc_up_shared": (None, [cfg, _I64, _P, _P, _P, _P, _P]),
            "orc_qb_histogram": (None, [_P, _I64, _I32, _I64, _I32, _P, ctypes.c_int]),
            "orc_qb_quantile_bias": (None, [_P, _I32, _I32, ctypes.c_double, _P, _P]),
            "orc_sign_update": (None, [_P, _I32, ctypes.c_float, _P]),
            "orc_e4m3_to_f64": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_f64_to_e4m3": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_fp8_exp_for": (_I32, [ctypes.c_double]),
            "orc_fp8_quantize_rows": (None, [_P, _I64, _I64, _P, _P]),
            "orc_routed_fp8": (None, [cfg, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
            "orc_softcap_grad": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
            "orc_situ_grad": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
            "orc_backward": (None, [cfg, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int,
                                    ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
            "orc_num_threads": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _need(a, dtype, shape=None):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if shape is not None and tuple(a.shape) != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {tuple(a.shape)}")
    return a


# ---------------------------------------------------------------- scalars
def bf16_to_f64(b: int) -> float:
    return _load().orc_bf16_to_f64(int(b))


def f64_to_bf16(x: float) -> int:
    return _load().orc_f64_to_bf16(float(x))


def round_bf16_array(x: np.ndarray) -> np.ndarray:
    """Element-wise fp64 -> bf16 bit patterns through the oracle's rounding."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).ravel()
    out = np.fromiter((lib.orc_f64_to_bf16(float(v)) for v in flat), dtype=np.uint16,
                      count=flat.size)
    return out.reshape(np.shape(x))


def sigmoid(x: float) -> float:
    return _load().orc_sigmoid(float(x))


def softcap(x: float, beta: float) -> float:
    return _load().orc_softcap(float(x), float(beta))


def situ(x: float, beta: float) -> float:
    return _load().orc_situ(float(x), float(beta))


def softcap_grad(x: float, beta: float) -> float:
    return _load().orc_softcap_grad(float(x), float(beta))


def situ_grad(x: float, beta: float) -> float:
    return _load().orc_situ_grad(float(x), float(beta))


def num_threads() -> int:
    return _load().orc_num_threads()


# ---------------------------------------------------------------- layer steps
def down_proj(cfg: LayerConfig, x, w_down):
    T = x.shape[0]
    x = _need(x, np.uint16, (T, cfg.d))
    w_down = _need(w_down, np.uint16, (cfg.latent, cfg.d))
    h = np.empty((T, cfg.latent), np.uint16)
    c = cfg.c()
    _load().orc_down_proj(ctypes.byref(c), T, _ptr(x), _ptr(w_down), _ptr(h))
    return h


def rms_rows(cfg: LayerConfig, h):
    """Un-weighted RMSNorm of each bf16 row of h (the ablation variant's norm
    after the down-projection); returns bf16 bits."""
    h = _need(h, np.uint16)
    T, L = h.shape
    out = np.empty_like(h)
    _load().orc_rms_rows(T, L, float(cfg.rms_eps), _ptr(h), _ptr(out))
    return out


def router(cfg: LayerConfig, h, w_router):
    T = h.shape[0]
    h = _need(h, np.uint16, (T, cfg.latent))
    w_router = _need(w_router, np.uint16, (cfg.n_experts, cfg.latent))
    s = np.empty((T, cfg.n_experts), np.float32)
    c = cfg.c()
    _load().orc_router(ctypes.byref(c), T, _ptr(h), _ptr(w_router), _ptr(s))
    return s


def topk(cfg: LayerConfig, s, bias):
    T = s.shape[0]
    s = _need(s, np.float32, (T, cfg.n_experts))
    bias = _need(bias, np.float32, (cfg.n_experts,))
    idx = np.empty((T, cfg.top_k), np.int32)
    gate = np.empty((T, cfg.top_k), np.float32)
    margin = np.empty((T,), np.float64)
    c = cfg.c()
    _load().orc_topk(ctypes.byref(c), T, _ptr(s), _ptr(bias), _ptr(idx), _ptr(gate), _ptr(margin))
    return idx, gate, margin


def permute(cfg: LayerConfig, idx):
    T = idx.shape[0]
    idx = _need(idx, np.int32, (T, cfg.top_k))
    n = T * cfg.top_k
    counts = np.empty(cfg.n_experts, np.int32)
    offsets = np.empty(cfg.n_experts + 1, np.int32)
    perm = np.empty(n, np.int32)
    inv = np.empty(n, np.int32)
    c = cfg.c()
    _load().orc_permute(ctypes.byref(c), T, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(perm),
                        _ptr(inv))
    return counts, offsets, perm, inv


def _expert_ptrs(mats, n_experts, shape):
    """Array of per-expert pointers; ``mats`` is an [E, ...] array or a dict
    {expert id: array} holding only the experts that will be used."""
    arr = (_P * n_experts)()
    keep = []
    if isinstance(mats, dict):
        for e, m in mats.items():
            m = _need(m, np.uint16, shape)
            keep.append(m)
            arr[int(e)] = m.ctypes.data
    else:
        mats = _need(mats, np.uint16, (n_experts,) + tuple(shape))
        keep.append(mats)
        step = int(np.prod(shape)) * 2
        for e in range(n_experts):
            arr[e] = mats.ctypes.data + e * step
    return arr, keep


def routed(cfg: LayerConfig, h, idx, gate, w1, w2, w3, want_act=False, want_o=False):
    """Experts + gate-weighted combine + RMSNorm.  Returns a dict with z, r (bf16),
    r64 and optionally act ([T*k, inter] bf16) and o ([T*k, latent] fp64)."""
    T = h.shape[0]
    h = _need(h, np.uint16, (T, cfg.latent))
    idx = _need(idx, np.int32, (T, cfg.top_k))
    gate = _need(gate, np.float32, (T, cfg.top_k))
    if T > 0 and (idx.min() < 0 or idx.max() >= cfg.n_experts):
        raise ValueError("expert index out of range")
    p1, k1 = _expert_ptrs(w1, cfg.n_experts, (cfg.inter, cfg.latent))
    p2, k2 = _expert_ptrs(w2, cfg.n_experts, (cfg.inter, cfg.latent))
    p3, k3 = _expert_ptrs(w3, cfg.n_experts, (cfg.latent, cfg.inter))
    for e in np.unique(idx):
        if not (p1[e] and p2[e] and p3[e]):
            raise ValueError(f"weights of expert {e} were not supplied")
    z = np.empty((T, cfg.latent), np.float64)
    r = np.empty((T, cfg.latent), np.uint16)
    r64 = np.empty((T, cfg.latent), np.float64)
    act = np.empty((T * cfg.top_k, cfg.inter), np.uint16) if want_act else None
    o = np.empty((T * cfg.top_k, cfg.latent), np.float64) if want_o else None
    c = cfg.c()
    _load().orc_routed(ctypes.byref(c), T, _ptr(h), _ptr(idx), _ptr(gate), p1, p2, p3, _ptr(act),
                       _ptr(o), _ptr(z), _ptr(r), _ptr(r64))
    del k1, k2, k3
    out = {"z": z, "r": r, "r64": r64}
    if want_act:
        out["act"] = act
    if want_o:
        out["o"] = o
    return out


def expert_aggregate(cfg: LayerConfig, act, idx, gate, w3):
    """z [T, latent] fp64 = sum_j gate[t, j] * W3[idx[t, j]] act[t*k + j] from
    given bf16 activations ([T*k, inter], assignment order); ``w3`` as in
    ``routed``.  The aggregation step of ``routed`` on its own."""
    T = idx.shape[0]
    idx = _need(idx, np.int32, (T, cfg.top_k))
    gate = _need(gate, np.float32, (T, cfg.top_k))
    act = _need(act, np.uint16, (T * cfg.top_k, cfg.inter))
    if T > 0 and (idx.min() < 0 or idx.max() >= cfg.n_experts):
        raise ValueError("expert index out of range")
    p3, k3 = _expert_ptrs(w3, cfg.n_experts, (cfg.latent, cfg.inter))
    for e in np.unique(idx):
        if not p3[e]:
            raise ValueError(f"weights of expert {e} were not supplied")
    z = np.empty((T, cfg.latent), np.float64)
    c = cfg.c()
    _load().orc_expert_aggregate(ctypes.byref(c), T, _ptr(act), _ptr(idx), _ptr(gate), p3, _ptr(z))
    del k3
    return z


# ---------------------------------------------------------------- FP8 variant
def e4m3_to_f64(codes):
    codes = np.asarray(codes, np.uint8)
    lib = _load()
    return np.array([lib.orc_e4m3_to_f64(int(c)) for c in codes.reshape(-1)]).reshape(codes.shape)


def f64_to_e4m3(x):
    x = np.asarray(x, np.float64)
    lib = _load()
    return np.array([lib.orc_f64_to_e4m3(float(v)) for v in x.reshape(-1)], np.uint8).reshape(x.shape)


def fp8_exp_for(amax: float) -> int:
    return int(_load().orc_fp8_exp_for(float(amax)))


def fp8_quantize_rows(src):
    """bf16 bits [..., R, K] -> (e4m3 codes uint8 [..., R, K], exponents int8 [..., R])."""
    src = np.ascontiguousarray(src, np.uint16)
    K = src.shape[-1]
    R = src.size // K
    codes = np.empty(src.shape, np.uint8)
    exps = np.empty(src.shape[:-1], np.int8)
    _load().orc_fp8_quantize_rows(_ptr(src), R, K, _ptr(codes), _ptr(exps))
    return codes, exps


def _fp8_ptrs(mats, n_experts, shape):
    """Per-expert code and exponent pointers from an [E, R, K] bf16 array or a
    dict {expert: [R, K]} (quantised here, row by row)."""
    codes_arr, exps_arr = (_P * n_experts)(), (_P * n_experts)()
    keep = []
    items = mats.items() if isinstance(mats, dict) else enumerate(_need(mats, np.uint16, (n_experts,) + shape))
    for e, m in items:
        q, x = fp8_quantize_rows(_need(m, np.uint16, shape))
        keep += [q, x]
        codes_arr[int(e)] = q.ctypes.data
        exps_arr[int(e)] = x.ctypes.data
    return codes_arr, exps_arr, keep


def routed_fp8(cfg: LayerConfig, h, idx, gate, w1, w2, w3, want_act=False, want_o=False):
    """FP8 variant of ``routed``: the experts' weights (given as bf16, quantised
    here per row) and operands in e4m3.  ``act`` is the e4m3 code array."""
    T = h.shape[0]
    h = _need(h, np.uint16, (T, cfg.latent))
    idx = _need(idx, np.int32, (T, cfg.top_k))
    gate = _need(gate, np.float32, (T, cfg.top_k))
    q1, e1, k1 = _fp8_ptrs(w1, cfg.n_experts, (cfg.inter, cfg.latent))
    q2, e2, k2 = _fp8_ptrs(w2, cfg.n_experts, (cfg.inter, cfg.latent))
    q3, e3, k3 = _fp8_ptrs(w3, cfg.n_experts, (cfg.latent, cfg.inter))
    for e in np.unique(idx):
        if not (q1[e] and q2[e] and q3[e]):
            raise ValueError(f"weights of expert {e} were not supplied")
    z = np.empty((T, cfg.latent), np.float64)
    r = np.empty((T, cfg.latent), np.uint16)
    r64 = np.empty((T, cfg.latent), np.float64)
    act = np.empty((T * cfg.top_k, cfg.inter), np.uint8) if want_act else None
    o = np.empty((T * cfg.top_k, cfg.latent), np.float64) if want_o else None
    c = cfg.c()
    _load().orc_routed_fp8(ctypes.byref(c), T, _ptr(h), _ptr(idx), _ptr(gate), q1, e1, q2, e2, q3, e3,
                           _ptr(act), _ptr(o), _ptr(z), _ptr(r), _ptr(r64))
    del k1, k2, k3
    out = {"z": z, "r": r, "r64": r64}
    if want_act:
        out["act"] = act
    if want_o:
        out["o"] = o
    return out


def shared_act(cfg: LayerConfig, x, ws1, ws2):
    T = x.shape[0]
    S = cfg.n_shared * cfg.shared_inter
    x = _need(x, np.uint16, (T, cfg.d))
    ws1 = _need(ws1, np.uint16, (S, cfg.d))
    ws2 = _need(ws2, np.uint16, (S, cfg.d))
    a = np.empty((T, S), np.uint16)
    c = cfg.c()
    _load().orc_shared_act(ctypes.byref(c), T, _ptr(x), _ptr(ws1), _ptr(ws2), _ptr(a))
    return a


def up_shared(cfg: LayerConfig, r, a_s, w_up, ws3):
    T = r.shape[0]
    S = cfg.n_shared * cfg.shared_inter
    r = _need(r, np.uint16, (T, cfg.latent))
    a_s = _need(a_s, np.uint16, (T, S))
    w_up = _need(w_up, np.uint16, (cfg.d, cfg.latent))
    ws3 = _need(ws3, np.uint16, (cfg.d, S))
    y = np.empty((T, cfg.d), np.float64)
    c = cfg.c()
    _load().orc_up_shared(ctypes.byref(c), T, _ptr(r), _ptr(a_s), _ptr(w_up), _ptr(ws3), _ptr(y))
    return y


def layer_forward(cfg: LayerConfig, x, w, bias):
    """The whole layer, step by step.  ``w`` maps names to bf16 bit arrays:
    w_down [L,d], w_router [E,L], w1/w2 [E,I,L] (or dicts of used experts),
    w3 [E,L,I], ws1/ws2 [nS*Is,d], ws3 [d,nS*Is], w_up [d,L]."""
    h_raw = down_proj(cfg, x, w["w_down"])
    h = rms_rows(cfg, h_raw) if cfg.norm_after_down else h_raw
    s = router(cfg, h, w["w_router"])
    idx, gate, margin = topk(cfg, s, bias)
    counts, offsets, perm, inv = permute(cfg, idx)
    experts = routed_fp8 if cfg.expert_fp8 else routed
    rt = experts(cfg, h, idx, gate, w["w1"], w["w2"], w["w3"])
    a_s = shared_act(cfg, x, w["ws1"], w["ws2"])
    y = up_shared(cfg, rt["r"], a_s, w["w_up"], w["ws3"])
    return {"h_raw": h_raw, "h": h, "s": s, "idx": idx, "gate": gate, "margin": margin, "counts": counts,
            "offsets": offsets, "perm": perm, "inv": inv, "z": rt["z"], "r": rt["r"],
            "r64": rt["r64"], "a_s": a_s, "y": y}


# ---------------------------------------------------------------- backward
BACKWARD_GRADS = ("w_down", "w_router", "w1", "w2", "w3", "ws1", "ws2", "ws3", "w_up")


def layer_backward(cfg: LayerConfig, x, w, idx, dy, round_mode: int = 1, weight_grads: bool = True):
    """Gradient of the layer for the upstream gradient ``dy`` (bf16 bits
    [T, d]) with the routing ``idx`` ([T, k] int32, from the forward) held
    fixed.  ``round_mode`` 1 takes the gradient at the forward's bf16 / fp32
    roundings (each passing the gradient through); 0 is the smooth, unrounded
    function.  Returns fp64 arrays: "x" [T, d] and, with ``weight_grads``, one
    per weight name in ``BACKWARD_GRADS`` shaped like that weight (w1/w2/w3
    must then be full [E, ...] arrays)."""
    if cfg.expert_fp8:
        raise ValueError("the backward covers the bf16 layer (with or without the norm after the down-projection)")
    T = x.shape[0]
    E, L, I, d = cfg.n_experts, cfg.latent, cfg.inter, cfg.d
    S = cfg.n_shared * cfg.shared_inter
    x = _need(x, np.uint16, (T, d))
    dy = _need(dy, np.uint16, (T, d))
    idx = _need(idx, np.int32, (T, cfg.top_k))
    if T > 0 and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    dense = {k: _need(w[k], np.uint16) for k in ("w_down", "w_router", "ws1", "ws2", "ws3", "w_up")}
    p1, k1 = _expert_ptrs(w["w1"], E, (I, L))
    p2, k2 = _expert_ptrs(w["w2"], E, (I, L))
    p3, k3 = _expert_ptrs(w["w3"], E, (L, I))
    for e in np.unique(idx):
        if not (p1[e] and p2[e] and p3[e]):
            raise ValueError(f"weights of expert {e} were not supplied")
    shapes = {"w_down": (L, d), "w_router": (E, L), "w1": (E, I, L), "w2": (E, I, L),
              "w3": (E, L, I), "ws1": (S, d), "ws2": (S, d), "ws3": (d, S), "w_up": (d, L)}
    out = {"x": np.empty((T, d), np.float64)}
    if weight_grads:
        for k in BACKWARD_GRADS:
            out[k] = np.empty(shapes[k], np.float64)
    g = [_ptr(out.get(k)) for k in BACKWARD_GRADS]
    c = cfg.c()
    _load().orc_backward(ctypes.byref(c), T, _ptr(x), _ptr(idx), _ptr(dy), _ptr(dense["w_down"]),
                         _ptr(dense["w_router"]), p1, p2, p3, _ptr(dense["ws1"]), _ptr(dense["ws2"]),
                         _ptr(dense["ws3"]), _ptr(dense["w_up"]), int(round_mode), int(bool(cfg.norm_after_down)),
                         _ptr(out["x"]), *g)
    del k1, k2, k3
    return out


# ---------------------------------------------------------------- QB
def qb_histogram(scores, B: int, hist=None, accumulate: bool = False, n_cols: int | None = None):
    """Per-expert B-bin histogram of ``scores`` ([T, ld] fp32; the first n_cols
    columns are the experts).  Returns uint32 [E, B]."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    if s.ndim != 2:
        raise ValueError("scores must be 2-D")
    T, ld = s.shape
    E = ld if n_cols is None else int(n_cols)
    if hist is None:
        hist = np.zeros((E, B), np.uint32)
    elif hist.dtype != np.uint32 or hist.shape != (E, B) or not hist.flags.c_contiguous:
        raise ValueError("hist must be a contiguous uint32 [E, B] array")
    _load().orc_qb_histogram(_ptr(s), T, E, ld, B, _ptr(hist), 1 if accumulate else 0)
    return hist


def qb_quantile_bias(hist, level: float):
    hist = _need(hist, np.uint32)
    E, B = hist.shape
    q = np.empty(E, np.float32)
    b = np.empty(E, np.float32)
    _load().orc_qb_quantile_bias(_ptr(hist), E, B, float(level), _ptr(q), _ptr(b))
    return q, b


def sign_update(counts, gamma: float, bias):
    """The fixed-step (SignSGD-like) bias update QB replaces; returns the new
    fp32 bias (the input is not modified)."""
    counts = _need(counts, np.int32)
    out = np.array(bias, dtype=np.float32, copy=True)
    _load().orc_sign_update(_ptr(counts), counts.shape[0], float(np.float32(gamma)), _ptr(out))
    return out


def expert_loads(idx, n_experts: int):
    """Assignments per expert of a top-k index array [T][k] (int32)."""
    return np.bincount(np.asarray(idx).reshape(-1), minlength=n_experts).astype(np.int32)
