"""Data-parallel Quantile Balancing on two gloo ranks (CPU): each rank bins its
own tokens, the histograms are summed with the package's all-reduce helper,
and every rank reads the same biases -- equal to the single-process result
over all tokens.  The binning and the quantile read are the oracle's (the GPU
kernels are checked against it elsewhere); this covers the exchange step."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from sparse_moe_layer_bias_gb300 import synth
from sparse_moe_layer_bias_gb300.dist import qb_allreduce_histogram

T, E, B, K = 6000, 64, 1000, 4


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s = synth.qb_scores(T, E, seed=21).numpy()
        lo, hi = rank * T // world, (rank + 1) * T // world
        local = oracle.qb_histogram(s[lo:hi], B)
        hist = torch.from_numpy(local.astype(np.int32))
        qb_allreduce_histogram(hist)
        _, bias = oracle.qb_quantile_bias(hist.numpy().astype(np.uint32), 1.0 - K / E)
        np.save(os.path.join(out_dir, f"hist{rank}.npy"), hist.numpy())
        np.save(os.path.join(out_dir, f"bias{rank}.npy"), bias)
    finally:
        dist.destroy_process_group()


def test_two_rank_histogram_allreduce_gives_global_biases(tmp_path):
    world = 2
    mp.start_processes(worker, args=(world, free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    s = synth.qb_scores(T, E, seed=21).numpy()
    ref_hist = oracle.qb_histogram(s, B)
    _, ref_bias = oracle.qb_quantile_bias(ref_hist, 1.0 - K / E)
    for r in range(world):
        assert np.array_equal(np.load(tmp_path / f"hist{r}.npy").astype(np.uint32), ref_hist)
        assert np.array_equal(np.load(tmp_path / f"bias{r}.npy"), ref_bias)


def test_allreduce_helper_is_identity_without_process_group():
    h = torch.arange(12, dtype=torch.int32).view(3, 4)
    assert torch.equal(qb_allreduce_histogram(h.clone()), h)
