"""The debug build of the library (-DLMOE_DEBUG: every index a kernel reads
from a device list is checked before use -- the rows the expert GEMMs gather
and scatter, the permutation maps, the tile lists, the backward's column
maps).  It runs in a child process (LMOE_LIBRARY=debug loads
liblmoe_debug.so) over the tiny, small, odd-shape and every-expert (k = E)
layers, forward and backward, the norm-after-down and FP8 forwards and
lmoe_route_static, and no check may fail.  Then the reporting path:
lmoe_selftest_index fails one check on purpose (without touching memory) and
lmoe_device_status must report LMOE_ERR_INDEX once."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import dataclasses, sys
    import torch
    sys.path.insert(0, {root!r})
    import sparse_moe_layer_bias_gb300 as lm
    from sparse_moe_layer_bias_gb300 import synth
    assert lm.lmoe_debug_checks(), "the debug library was not loaded"
    odd = synth.LayerShape("odd", T=97, d=192, latent=128, n_experts=10, top_k=3, inter=192, n_shared=1,
                           shared_inter=192, seed=1009)
    every = synth.LayerShape("all_experts", T=200, d=256, latent=128, n_experts=8, top_k=8, inter=64,
                             n_shared=2, shared_inter=64, seed=1010)
    norm = dataclasses.replace(synth.TINY, name="tiny_norm", norm_after_down=True)
    fp8 = dataclasses.replace(synth.TINY, name="tiny_fp8", inter=128, expert_fp8=True)
    h = None
    for shape, train in ((synth.TINY, True), (synth.SMALL, True), (odd, True), (every, True), (norm, True),
                         (fp8, False)):
        w = {{k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}}
        x, b = (t.cuda() for t in synth.activations_host(shape))
        T = x.shape[0]
        h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=train), w, max_tokens=T)
        ws = lm.alloc_workspace(h, T)
        y = lm.lmoe_forward(h, x, b, workspace=ws)
        if train:
            dy = synth.grad_output_host(shape, T=T).cuda()
            dx, g = lm.lmoe_backward(h, x, dy, ws)
            assert bool(torch.isfinite(dx.float()).all()), shape.name
        torch.cuda.synchronize()
        assert bool(torch.isfinite(y.float()).all()), shape.name
        st = lm.lmoe_device_status(h, clear=False)
        assert st == 0, (shape.name, st)
        print("ok", shape.name, flush=True)
    s = torch.rand((4096, 128), device="cuda")
    lm.lmoe_route_static(s, torch.zeros(128, device="cuda"), 8)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    lm.lmoe_selftest_index()
    assert lm.lmoe_device_status(h, clear=True) == 8      # LMOE_ERR_INDEX
    assert lm.lmoe_device_status(h) == 0
    print("debug checks ok", flush=True)
""")


def test_debug_build_runs_clean_and_reports_a_failed_check():
    from sparse_moe_layer_bias_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, LMOE_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug checks ok" in r.stdout
