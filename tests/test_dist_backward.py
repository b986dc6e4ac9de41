"""Data-parallel backward on two gloo ranks (CPU): each rank takes the
gradient over its own tokens, the weight gradients are summed with the
package's all-reduce helper, and every rank ends with the gradient of the
whole batch -- the single-process gradient over all tokens, up to the fp64
rounding of the sum's order; dx stays per token.  The gradients are the
oracle's (the GPU backward is checked against it elsewhere); this covers the
exchange step."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from sparse_moe_layer_bias_gb300.dist import allreduce_weight_grads

from test_oracle_backward import make_case


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, w, x, dy, idx = make_case(11)
        T = x.shape[0]
        lo, hi = rank * T // world, (rank + 1) * T // world
        g = oracle.layer_backward(cfg, x[lo:hi], w, idx[lo:hi], dy[lo:hi])
        grads = {n: torch.from_numpy(g[n]) for n in oracle.BACKWARD_GRADS}
        allreduce_weight_grads(grads)
        for n, t in grads.items():
            np.save(os.path.join(out_dir, f"{n}_{rank}.npy"), t.numpy())
        np.save(os.path.join(out_dir, f"x_{rank}.npy"), g["x"])
    finally:
        dist.destroy_process_group()


def test_two_rank_weight_gradient_allreduce_gives_the_batch_gradient(tmp_path):
    world = 2
    mp.start_processes(worker, args=(world, free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    cfg, w, x, dy, idx = make_case(11)
    ref = oracle.layer_backward(cfg, x, w, idx, dy)
    T = x.shape[0]
    for r in range(world):
        for n in oracle.BACKWARD_GRADS:
            got = np.load(tmp_path / f"{n}_{r}.npy")
            np.testing.assert_allclose(got, ref[n], rtol=1e-12, atol=1e-12 * np.abs(ref[n]).max())
        lo, hi = r * T // world, (r + 1) * T // world
        np.testing.assert_array_equal(np.load(tmp_path / f"x_{r}.npy"), ref["x"][lo:hi])


def test_grad_allreduce_helper_is_identity_without_process_group():
    g = {"a": torch.ones(3), "b": torch.arange(4.0)}
    out = allreduce_weight_grads({k: v.clone() for k, v in g.items()})
    for k in g:
        assert torch.equal(out[k], g[k])
