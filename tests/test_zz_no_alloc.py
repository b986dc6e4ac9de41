"""lmoe_route_static: the routing step for callers that cannot allocate device
memory (for instance an inference-engine plugin that is given no allocator,
or a serving loop that forbids allocation after start-up).  Its scratch sits
in a fixed array inside the library.  Checked through the C ABI against the
routing that lmoe_forward leaves in its workspace, on two calls in a row (the
second must not see the first call's scratch).  This file is collected last
so that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_bias_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_moe_layer_bias_gb300 as m
    m.load_library()
    return m


def forward_routing(lm, shape, T, seed_offset):
    w = {k: v.cuda() for k, v in synth.layer_weights_host(shape).items()}
    x, bias = (t.cuda() for t in synth.activations_host(shape, T=T, seed_offset=seed_offset))
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=T)
    ws = lm.alloc_workspace(h, T)
    lm.lmoe_forward(h, x, bias, workspace=ws)
    torch.cuda.synchronize()
    lay = lm.lmoe_workspace_layout(h, T)
    E, K = shape.n_experts, shape.top_k

    def view(key, dtype, n):
        return ws[lay[key]:lay[key] + n * 4].view(dtype).clone()

    ref = {"scores": view("scores", torch.float32, T * E).view(T, E),
           "topk_idx": view("topk_idx", torch.int32, T * K).view(T, K),
           "gates": view("gates", torch.float32, T * K).view(T, K),
           "counts": view("counts", torch.int32, E),
           "offsets": view("offsets", torch.int32, E + 1),
           "perm": view("perm", torch.int32, T * K),
           "inv": view("inv", torch.int32, T * K)}
    return ref, bias


def test_route_static_matches_forward_routing_twice(lm):
    # two calls in a row with different problems: the second call's bitmap must
    # start from zero although the array keeps the first call's contents
    for shape, T, off in ((synth.SMALL, 4096, 0), (synth.TINY, 300, 1)):
        ref, bias = forward_routing(lm, shape, T, off)
        got = lm.lmoe_route_static(ref["scores"], bias, shape.top_k)
        torch.cuda.synchronize()
        for key in ("topk_idx", "gates", "counts", "offsets", "perm", "inv"):
            assert torch.equal(got[key], ref[key]), key


def test_route_static_rejects_oversized_problems(lm):
    T, E = 1 << 17, 1024            # bitmaps and prefixes alone: 8 * E * T / 32 bytes = 32 MiB > 8 MiB
    scores = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_route_static(scores, bias, 16)
    assert e.value.status == 2
