"""GB300-native Stable LatentMoE layer (forward and backward) and Quantile Balancing histogram.

The compute lives in liblmoe.so (hand-written CUDA for sm_103a, C ABI in
include/lmoe.h); this package is its ctypes binding plus the seeded input
generators (``synth``).  Importing it does not load the library; the first
call does, and raises if the library has not been built.
"""
from .binding import (  # noqa: F401
    EXPORTED,
    Handle,
    LmoeError,
    alloc_host_io,
    alloc_workspace,
    grad_shapes,
    library_path,
    lmoe_backward,
    lmoe_backward_workspace_size,
    lmoe_create,
    lmoe_debug_checks,
    lmoe_destroy,
    lmoe_device_status,
    lmoe_forward,
    lmoe_forward_host,
    lmoe_host_io_size,
    lmoe_host_wait,
    lmoe_route_static,
    lmoe_selftest_index,
    lmoe_selftest_timeout,
    lmoe_set_stage_events,
    STAGES,
    BWD_STAGES,
    lmoe_set_backward_events,
    lmoe_status_string,
    lmoe_workspace_layout,
    lmoe_workspace_size,
    load_library,
    qb_histogram,
    qb_quantile_bias,
    qb_sign_update,
)
