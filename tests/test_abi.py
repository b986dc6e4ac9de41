"""The C-ABI library loads and exports every entry point include/lmoe.h
declares (no compute: this runs without a GPU)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:lmoe|qb)_\w+)\s*\(", text, flags=re.M))
    return names


def test_library_exports_every_declared_symbol():
    from sparse_moe_layer_bias_gb300 import build, binding
    lib_path = build.build()
    lib = ctypes.CDLL(lib_path)
    names = declared_functions()
    assert {"lmoe_create", "lmoe_forward", "lmoe_destroy", "qb_histogram", "qb_quantile_bias"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.EXPORTED) == names


def test_status_strings_without_gpu():
    import sparse_moe_layer_bias_gb300 as lm
    from sparse_moe_layer_bias_gb300 import build
    build.build()
    assert lm.lmoe_status_string(0) == "LMOE_OK"
    assert lm.lmoe_status_string(4) == "LMOE_ERR_WORKSPACE"
    assert lm.lmoe_status_string(99) == "LMOE_ERR_UNKNOWN"


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_layer_bias_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "lmoe_oracle" not in text, f


def test_host_entry_points_reject_bad_arguments_without_gpu():
    """Argument errors return before any CUDA call, so they run here."""
    from sparse_moe_layer_bias_gb300 import build
    lib = ctypes.CDLL(build.build())
    P = ctypes.c_void_p
    lib.lmoe_host_io_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
    lib.lmoe_host_wait.argtypes = [P, P]
    lib.lmoe_forward_host.argtypes = [P, P, ctypes.c_int64, P, P, P, P, P, P, P, ctypes.c_size_t, P,
                                      ctypes.c_size_t, P]
    lib.lmoe_selftest_timeout.argtypes = [P, ctypes.c_uint64, P]
    assert lib.lmoe_selftest_timeout(None, 1000000, None) == 1
    n = ctypes.c_size_t()
    assert lib.lmoe_host_io_size(None, ctypes.byref(n)) == 1
    assert lib.lmoe_host_wait(None, None) == 1
    assert lib.lmoe_forward_host(None, None, 8, None, None, None, None, None, None, None, 0, None, 0,
                                 None) == 1
    lib.lmoe_backward_workspace_size.argtypes = [P, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]
    lib.lmoe_backward.argtypes = [P, P, ctypes.c_int64, P, P, P, P, ctypes.c_size_t, P, P, P,
                                  ctypes.c_size_t, P]
    assert lib.lmoe_backward_workspace_size(None, 8, ctypes.byref(n)) == 1
    assert lib.lmoe_backward(None, None, 8, None, None, None, None, 0, None, None, None, 0, None) == 1


def test_backward_handle_rejects_variants_without_gpu():
    """with_backward covers the bf16 layer (with or without the norm after the
    down-projection): a config that also sets expert_fp8 is rejected while
    validating the config (before any CUDA call)."""
    from sparse_moe_layer_bias_gb300 import build, binding
    lib = ctypes.CDLL(build.build())
    P = ctypes.c_void_p
    lib.lmoe_create.argtypes = [ctypes.POINTER(binding.LmoeConfig), ctypes.POINTER(binding.LmoeWeights),
                                ctypes.POINTER(P)]
    w = binding.LmoeWeights()
    out = P()
    for norm, fp8, expect in ((1, 0, 1), (0, 1, 2), (0, 0, 1)):
        cfg = binding.LmoeConfig(256, 128, 32, 4, 128, 2, 64, 4.0, 25.0, 1e-6, 64, norm, fp8, 1)
        # valid configs: the null weights are what gets rejected
        assert lib.lmoe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(out)) == expect
    cfg = binding.LmoeConfig(256, 128, 32, 4, 128, 2, 64, 4.0, 25.0, 1e-6, 64, 0, 0, 2)
    assert lib.lmoe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(out)) == 1


def test_debug_and_release_builds_without_gpu():
    """The release library compiles the index checks away; the debug build
    (-DLMOE_DEBUG) exports the same entry points and reports its checks.  The
    index self-test returns LMOE_ERR_INVALID_ARG in a release build before any
    CUDA call."""
    from sparse_moe_layer_bias_gb300 import build
    rel = ctypes.CDLL(build.build())
    dbg = ctypes.CDLL(build.build(debug=True))
    for lib, flag in ((rel, 0), (dbg, 1)):
        lib.lmoe_debug_checks.restype = ctypes.c_int
        assert lib.lmoe_debug_checks() == flag
        for n in declared_functions():
            assert hasattr(lib, n), n
    rel.lmoe_selftest_index.argtypes = [ctypes.c_void_p]
    assert rel.lmoe_selftest_index(None) == 1
