"""ctypes binding of liblmoe.so (include/lmoe.h), same names as the C ABI.

Argument marshalling only: every step of the layer and of Quantile Balancing
runs in the library's CUDA kernels.  torch supplies device memory and the
current stream.  If the library is missing, every call raises -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

# LMOE_LIBRARY=debug selects the build with index checks (build.build(debug=True))
_LIB_NAME = "liblmoe_debug.so" if os.environ.get("LMOE_LIBRARY") == "debug" else "liblmoe.so"
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), _LIB_NAME)
_lib = None

STATUS = {0: "LMOE_OK", 1: "LMOE_ERR_INVALID_ARG", 2: "LMOE_ERR_UNSUPPORTED_SHAPE",
          3: "LMOE_ERR_ALIGNMENT", 4: "LMOE_ERR_WORKSPACE", 5: "LMOE_ERR_CUDA",
          6: "LMOE_ERR_TIMEOUT", 7: "LMOE_ERR_NO_DEVICE", 8: "LMOE_ERR_INDEX"}

EXPORTED = ("lmoe_status_string", "lmoe_create", "lmoe_destroy", "lmoe_workspace_size",
            "lmoe_workspace_layout", "lmoe_forward", "lmoe_host_io_size", "lmoe_forward_host",
            "lmoe_host_wait", "lmoe_device_status", "lmoe_set_stage_events", "lmoe_set_backward_events",
            "lmoe_route_static", "lmoe_debug_checks", "lmoe_selftest_index",
            "lmoe_selftest_timeout", "lmoe_backward_workspace_size", "lmoe_backward", "qb_histogram",
            "qb_quantile_bias", "qb_sign_update")

STAGES = ("down", "shared", "router", "topk", "scan", "offsets", "scatter", "expert_w12_light",
          "expert_w12_heavy", "expert_w3", "combine", "up")

BWD_STAGES = ("dr", "shared", "rmsnorm", "expert_u", "expert_glu", "router", "dh_experts", "dh_router", "dh_sum",
              "dx", "transpose", "wgrad_dense", "segments", "wgrad_w3", "wgrad_w12")


class LmoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


class LmoeConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("latent", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("max_tokens", ctypes.c_int64), ("norm_after_down", ctypes.c_int32),
                ("expert_fp8", ctypes.c_int32), ("with_backward", ctypes.c_int32)]


WEIGHT_NAMES = ("w_down", "w_router", "w1", "w2", "w3", "ws1", "ws2", "ws3", "w_up")


class LmoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_NAMES]


class LmoeGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_NAMES] + [("accumulate", ctypes.c_int32)]


class LmoeWsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("h", "scores", "topk_idx", "gates", "counts", "offsets",
                                              "perm", "inv", "act", "o", "r", "shared_act", "h_norm",
                                              "h_fp8", "h_fp8_exp", "pre_act", "shared_pre_act",
                                              "logits")]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load liblmoe.so (built in-tree by build.build()), or with LMOE_LIBRARY=debug
    liblmoe_debug.so (build.build(debug=True)); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "sparse_moe_layer_bias_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.lmoe_status_string.restype = ctypes.c_char_p
    lib.lmoe_status_string.argtypes = [ctypes.c_int]
    lib.lmoe_create.restype = ctypes.c_int
    lib.lmoe_create.argtypes = [ctypes.POINTER(LmoeConfig), ctypes.POINTER(LmoeWeights),
                                ctypes.POINTER(P)]
    lib.lmoe_destroy.restype = ctypes.c_int
    lib.lmoe_destroy.argtypes = [P]
    lib.lmoe_workspace_size.restype = ctypes.c_int
    lib.lmoe_workspace_size.argtypes = [P, I64, ctypes.POINTER(ctypes.c_size_t)]
    lib.lmoe_workspace_layout.restype = ctypes.c_int
    lib.lmoe_workspace_layout.argtypes = [P, I64, ctypes.POINTER(LmoeWsLayout)]
    lib.lmoe_forward.restype = ctypes.c_int
    lib.lmoe_forward.argtypes = [P, P, I64, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.lmoe_backward_workspace_size.restype = ctypes.c_int
    lib.lmoe_backward_workspace_size.argtypes = [P, I64, ctypes.POINTER(ctypes.c_size_t)]
    lib.lmoe_backward.restype = ctypes.c_int
    lib.lmoe_backward.argtypes = [P, P, I64, P, P, P, P, ctypes.c_size_t, P, ctypes.POINTER(LmoeGrads), P,
                                  ctypes.c_size_t, P]
    lib.lmoe_host_io_size.restype = ctypes.c_int
    lib.lmoe_host_io_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
    lib.lmoe_forward_host.restype = ctypes.c_int
    lib.lmoe_forward_host.argtypes = [P, P, I64, P, P, P, P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t, P]
    lib.lmoe_host_wait.restype = ctypes.c_int
    lib.lmoe_host_wait.argtypes = [P, P]
    lib.lmoe_selftest_timeout.restype = ctypes.c_int
    lib.lmoe_selftest_timeout.argtypes = [P, ctypes.c_uint64, P]
    lib.lmoe_device_status.restype = ctypes.c_int
    lib.lmoe_device_status.argtypes = [P, P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.lmoe_set_stage_events.restype = ctypes.c_int
    lib.lmoe_set_stage_events.argtypes = [P, P, ctypes.c_int]
    lib.lmoe_set_backward_events.restype = ctypes.c_int
    lib.lmoe_set_backward_events.argtypes = [P, P, ctypes.c_int]
    lib.lmoe_route_static.restype = ctypes.c_int
    lib.lmoe_route_static.argtypes = [P, I64, I32, I32, P, P, P, P, P, P, P, P]
    lib.lmoe_debug_checks.restype = ctypes.c_int
    lib.lmoe_debug_checks.argtypes = []
    lib.lmoe_selftest_index.restype = ctypes.c_int
    lib.lmoe_selftest_index.argtypes = [P]
    lib.qb_histogram.restype = ctypes.c_int
    lib.qb_histogram.argtypes = [P, I64, I32, I64, I32, P, ctypes.c_int, P]
    lib.qb_sign_update.restype = ctypes.c_int
    lib.qb_sign_update.argtypes = [P, I32, ctypes.c_float, P, P]
    lib.qb_quantile_bias.restype = ctypes.c_int
    lib.qb_quantile_bias.argtypes = [P, I32, I32, ctypes.c_double, P, P, P]
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise LmoeError(fn, status)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, dtype, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def lmoe_status_string(status: int) -> str:
    return load_library().lmoe_status_string(int(status)).decode()


class Handle:
    """Owns an lmoe_handle*; keeps the weight tensors alive (the library keeps
    their pointers)."""

    def __init__(self, ptr, cfg: LmoeConfig, weights: dict):
        self.ptr = ptr
        self.cfg = cfg
        self.weights = weights

    def __del__(self):
        if getattr(self, "ptr", None):
            try:
                lmoe_destroy(self)
            except Exception:
                pass


def lmoe_create(cfg: dict, weights: dict, max_tokens: int) -> Handle:
    """cfg: d, latent, n_experts, top_k, inter, n_shared, shared_inter and
    optional beta1, beta2, rms_eps, norm_after_down, expert_fp8, with_backward.  weights: bf16 CUDA
    tensors named as in lmoe_weights."""
    lib = load_library()
    c = LmoeConfig(int(cfg["d"]), int(cfg["latent"]), int(cfg["n_experts"]), int(cfg["top_k"]),
                   int(cfg["inter"]), int(cfg["n_shared"]), int(cfg["shared_inter"]),
                   float(cfg.get("beta1", 4.0)), float(cfg.get("beta2", 25.0)),
                   float(cfg.get("rms_eps", 1e-6)), int(max_tokens), int(bool(cfg.get("norm_after_down", False))),
                   int(bool(cfg.get("expert_fp8", False))), int(bool(cfg.get("with_backward", False))))
    held = {}
    w = LmoeWeights()
    for n in WEIGHT_NAMES:
        t = _dev(weights[n], torch.bfloat16, n)
        held[n] = t
        setattr(w, n, t.data_ptr())
    out = ctypes.c_void_p()
    _check("lmoe_create", lib.lmoe_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(out)))
    return Handle(out, c, held)


def lmoe_destroy(handle: Handle):
    if handle.ptr:
        lib = load_library()
        st = lib.lmoe_destroy(handle.ptr)
        handle.ptr = None
        _check("lmoe_destroy", st)


def lmoe_workspace_size(handle: Handle, T: int) -> int:
    n = ctypes.c_size_t()
    _check("lmoe_workspace_size", load_library().lmoe_workspace_size(handle.ptr, int(T), ctypes.byref(n)))
    return n.value


def lmoe_workspace_layout(handle: Handle, T: int) -> dict:
    lay = LmoeWsLayout()
    _check("lmoe_workspace_layout", load_library().lmoe_workspace_layout(handle.ptr, int(T), ctypes.byref(lay)))
    return {n: getattr(lay, n) for n, _ in LmoeWsLayout._fields_}


def alloc_workspace(handle: Handle, T: int, device=None) -> torch.Tensor:
    n = lmoe_workspace_size(handle, T)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def lmoe_forward(handle: Handle, x: torch.Tensor, bias: torch.Tensor, y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, scores_out=None, topk_idx_out=None,
                 gates_out=None, expert_counts_out=None, stream=None) -> torch.Tensor:
    lib = load_library()
    x = _dev(x, torch.bfloat16, "x")
    bias = _dev(bias, torch.float32, "bias")
    T = x.shape[0]
    if y is None:
        y = torch.empty_like(x)
    y = _dev(y, torch.bfloat16, "y")
    if workspace is None:
        workspace = alloc_workspace(handle, T, x.device)
    workspace = _dev(workspace, torch.uint8, "workspace")
    st = lib.lmoe_forward(handle.ptr, _ptr(x), T, _ptr(bias), _ptr(y),
                          _ptr(_dev(scores_out, torch.float32, "scores_out")),
                          _ptr(_dev(topk_idx_out, torch.int32, "topk_idx_out")),
                          _ptr(_dev(gates_out, torch.float32, "gates_out")),
                          _ptr(_dev(expert_counts_out, torch.int32, "expert_counts_out")),
                          _ptr(workspace), workspace.numel(), _stream(stream))
    _check("lmoe_forward", st)
    return y


def lmoe_backward_workspace_size(handle: Handle, T: int) -> int:
    n = ctypes.c_size_t()
    _check("lmoe_backward_workspace_size",
           load_library().lmoe_backward_workspace_size(handle.ptr, int(T), ctypes.byref(n)))
    return n.value


def grad_shapes(handle: Handle) -> dict:
    """Shapes of the weight gradients (as the weights)."""
    c = handle.cfg
    S = c.n_shared * c.shared_inter
    return {"w_down": (c.latent, c.d), "w_router": (c.n_experts, c.latent),
            "w1": (c.n_experts, c.inter, c.latent), "w2": (c.n_experts, c.inter, c.latent),
            "w3": (c.n_experts, c.latent, c.inter), "ws1": (S, c.d), "ws2": (S, c.d), "ws3": (c.d, S),
            "w_up": (c.d, c.latent)}


def lmoe_backward(handle: Handle, x: torch.Tensor, dy: torch.Tensor, fwd_workspace: torch.Tensor,
                  dx: torch.Tensor | None = None, grads: dict | None = None, workspace: torch.Tensor | None = None,
                  topk_idx=None, gates=None, accumulate: bool = False, stream=None):
    """Backward of the forward that ran on ``x`` with ``fwd_workspace``.  Pass
    ``topk_idx`` / ``gates`` when that forward wrote them to caller buffers.
    With ``accumulate`` the weight gradients are added to ``grads``' contents.
    Returns (dx bf16 [T, d], dict of fp32 weight gradients)."""
    lib = load_library()
    x = _dev(x, torch.bfloat16, "x")
    dy = _dev(dy, torch.bfloat16, "dy")
    fwd_workspace = _dev(fwd_workspace, torch.uint8, "fwd_workspace")
    T = x.shape[0]
    if dx is None:
        dx = torch.empty_like(x)
    dx = _dev(dx, torch.bfloat16, "dx")
    if grads is None:
        alloc = torch.zeros if accumulate else torch.empty
        grads = {n: alloc(s, dtype=torch.float32, device=x.device) for n, s in grad_shapes(handle).items()}
    g = LmoeGrads()
    for n in WEIGHT_NAMES:
        setattr(g, n, _dev(grads[n], torch.float32, "grad " + n).data_ptr())
    g.accumulate = 1 if accumulate else 0
    if workspace is None:
        workspace = torch.empty(max(lmoe_backward_workspace_size(handle, T), 256), dtype=torch.uint8,
                                device=x.device)
    workspace = _dev(workspace, torch.uint8, "workspace")
    st = lib.lmoe_backward(handle.ptr, _ptr(x), T, _ptr(dy), _ptr(_dev(topk_idx, torch.int32, "topk_idx")),
                           _ptr(_dev(gates, torch.float32, "gates")), _ptr(fwd_workspace),
                           fwd_workspace.numel(), _ptr(dx), ctypes.byref(g), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check("lmoe_backward", st)
    return dx, grads


def _host(t, dtype, name):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def lmoe_host_io_size(handle: Handle) -> int:
    n = ctypes.c_size_t()
    _check("lmoe_host_io_size", load_library().lmoe_host_io_size(handle.ptr, ctypes.byref(n)))
    return n.value


def alloc_host_io(handle: Handle, device=None) -> torch.Tensor:
    return torch.empty(lmoe_host_io_size(handle), dtype=torch.uint8, device=device or "cuda")


def lmoe_forward_host(handle: Handle, x_host: torch.Tensor, bias_host: torch.Tensor, y_host: torch.Tensor,
                      io: torch.Tensor, workspace: torch.Tensor, scores_out=None, topk_idx_out=None,
                      gates_out=None, expert_counts_out=None, stream=None) -> torch.Tensor:
    """Pipelined forward from host tensors (pin them for asynchronous copies).
    Returns y_host, which is complete once `stream` has passed a later
    lmoe_host_wait."""
    lib = load_library()
    x_host = _host(x_host, torch.bfloat16, "x_host")
    bias_host = _host(bias_host, torch.float32, "bias_host")
    y_host = _host(y_host, torch.bfloat16, "y_host")
    if y_host.shape != x_host.shape:
        raise ValueError("y_host must have x_host's shape")
    io = _dev(io, torch.uint8, "io")
    workspace = _dev(workspace, torch.uint8, "workspace")
    st = lib.lmoe_forward_host(handle.ptr, _ptr(x_host), x_host.shape[0], _ptr(bias_host), _ptr(y_host),
                               _ptr(_dev(scores_out, torch.float32, "scores_out")),
                               _ptr(_dev(topk_idx_out, torch.int32, "topk_idx_out")),
                               _ptr(_dev(gates_out, torch.float32, "gates_out")),
                               _ptr(_dev(expert_counts_out, torch.int32, "expert_counts_out")),
                               _ptr(io), io.numel(), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("lmoe_forward_host", st)
    return y_host


def lmoe_host_wait(handle: Handle, stream=None):
    _check("lmoe_host_wait", load_library().lmoe_host_wait(handle.ptr, _stream(stream)))


def lmoe_set_stage_events(handle: Handle, events):
    """events: a list of len(STAGES) + 1 torch.cuda.Event (created with
    enable_timing=True) or None to turn the timing hook off."""
    lib = load_library()
    if events is None:
        handle._event_array = None
        _check("lmoe_set_stage_events", lib.lmoe_set_stage_events(handle.ptr, None, 0))
        return
    for e in events:
        if not e.cuda_event:  # torch creates the cudaEvent_t on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    handle._event_array = arr  # the library keeps the pointer
    handle._events = list(events)
    _check("lmoe_set_stage_events", lib.lmoe_set_stage_events(handle.ptr, arr, len(events)))


def lmoe_set_backward_events(handle: Handle, events):
    """As lmoe_set_stage_events, for the backward's len(BWD_STAGES) + 1 events."""
    lib = load_library()
    if events is None:
        handle._bwd_event_array = None
        _check("lmoe_set_backward_events", lib.lmoe_set_backward_events(handle.ptr, None, 0))
        return
    for e in events:
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    handle._bwd_event_array = arr  # the library keeps the pointer
    handle._bwd_events = list(events)
    _check("lmoe_set_backward_events", lib.lmoe_set_backward_events(handle.ptr, arr, len(events)))


def lmoe_device_status(handle: Handle, clear: bool = True, stream=None) -> int:
    v = ctypes.c_int()
    _check("lmoe_device_status",
           load_library().lmoe_device_status(handle.ptr, _stream(stream), 1 if clear else 0, ctypes.byref(v)))
    return v.value


def lmoe_debug_checks() -> bool:
    return bool(load_library().lmoe_debug_checks())


def lmoe_selftest_index(stream=None):
    _check("lmoe_selftest_index", load_library().lmoe_selftest_index(_stream(stream)))


def lmoe_route_static(scores: torch.Tensor, bias: torch.Tensor, top_k: int, stream=None) -> dict:
    """Top-k + permutation with the library's fixed scratch array (no
    allocation inside the library; the outputs are allocated here by torch)."""
    scores = _dev(scores, torch.float32, "scores")
    bias = _dev(bias, torch.float32, "bias")
    T, E = scores.shape
    dev = scores.device
    out = {"topk_idx": torch.empty((T, top_k), dtype=torch.int32, device=dev),
           "gates": torch.empty((T, top_k), dtype=torch.float32, device=dev),
           "counts": torch.empty(E, dtype=torch.int32, device=dev),
           "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
           "perm": torch.empty(T * top_k, dtype=torch.int32, device=dev),
           "inv": torch.empty(T * top_k, dtype=torch.int32, device=dev)}
    _check("lmoe_route_static", load_library().lmoe_route_static(
        _ptr(scores), T, E, int(top_k), _ptr(bias), _ptr(out["topk_idx"]), _ptr(out["gates"]),
        _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv"]), _stream(stream)))
    return out


def qb_histogram(scores: torch.Tensor, B: int, hist: torch.Tensor | None = None, accumulate: bool = False,
                 n_cols: int | None = None, stream=None) -> torch.Tensor:
    """Per-expert B-bin histogram of a [T, ld] fp32 score tensor (first n_cols
    columns; all by default).  Returns (or accumulates into) uint32 [E, B],
    held in an int32 tensor of the same bits."""
    scores = _dev(scores, torch.float32, "scores")
    T, ld = scores.shape
    E = ld if n_cols is None else int(n_cols)
    if hist is None:
        hist = torch.empty((E, B), dtype=torch.int32, device=scores.device)
    hist = _dev(hist, torch.int32, "hist")
    _check("qb_histogram", load_library().qb_histogram(_ptr(scores), T, E, ld, int(B), _ptr(hist),
                                                       1 if accumulate else 0, _stream(stream)))
    return hist


def qb_quantile_bias(hist: torch.Tensor, level: float, quantile_out=None, bias_out=None, stream=None):
    hist = _dev(hist, torch.int32, "hist")
    E, B = hist.shape
    if bias_out is None:
        bias_out = torch.empty(E, dtype=torch.float32, device=hist.device)
    if quantile_out is None:
        quantile_out = torch.empty(E, dtype=torch.float32, device=hist.device)
    _check("qb_quantile_bias", load_library().qb_quantile_bias(
        _ptr(hist), E, B, float(level), _ptr(_dev(quantile_out, torch.float32, "quantile_out")),
        _ptr(_dev(bias_out, torch.float32, "bias_out")), _stream(stream)))
    return quantile_out, bias_out


def qb_sign_update(counts: torch.Tensor, gamma: float, bias: torch.Tensor, stream=None) -> torch.Tensor:
    """bias[e] += gamma * sign(mean(counts) - counts[e]) in place (the
    fixed-step rule QB replaces); returns bias."""
    counts = _dev(counts, torch.int32, "counts")
    bias = _dev(bias, torch.float32, "bias")
    if counts.numel() != bias.numel():
        raise ValueError("counts and bias must have one entry per expert")
    _check("qb_sign_update", load_library().qb_sign_update(_ptr(counts), counts.numel(), float(gamma),
                                                           _ptr(bias), _stream(stream)))
    return bias


def lmoe_selftest_timeout(handle: Handle, limit_ns: int = 1_000_000, stream=None):
    """Enqueue the bounded-wait self-test (see include/lmoe.h)."""
    _check("lmoe_selftest_timeout", load_library().lmoe_selftest_timeout(handle.ptr, int(limit_ns),
                                                                         _stream(stream)))
