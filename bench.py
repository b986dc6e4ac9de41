"""Benchmark: the Stable LatentMoE layer forward at K3 prefill shape plus its
Quantile Balancing histogram and bias read, on GB300, through the C ABI.

One step = lmoe_forward over T=8192 tokens (d=7168 -> 3584 latent, 896 routed
experts, top-16, 2 shared experts of 1024, routed intermediate 512) + the
QB histogram (B=1000) of that batch's router scores + the quantile/bias read.
Inputs are seeded synthetic data of that shape (see sparse_moe_layer_bias_gb300
/synth.py); weights (10.3 GB) and activations are resident in HBM.

Also measured in the same run (reported inside the one JSON line):
  * e2e: the same step through the host-memory entry point (lmoe_forward_host):
    x/bias copied in from pinned host memory and y/bias copied back every
    step, inside the timed region, pipelined across steps;
  * the K3 decode layer (T=64) and the QB histogram at T=2^20 x 896;
  * per-stage kernel times from CUDA events on the launching stream, and the
    roofline of the dominant kernel against MEASURED_PEAKS.json;
  * cpu_baseline: the CPU oracle on a bounded sample of the same workload.

`--impl reference` times the CPU oracle (the reference arm) instead.
Multi-GPU (torchrun): every rank runs its own batch ("scaling": "weak"); the
layer needs no exchange, and QB's one exchange step -- the sum of the ranks'
histograms before the quantile read -- is an NCCL all-reduce of [E][B] int32.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_moe_layer_bias_gb300 import synth  # noqa: E402

METRIC = "LatentMoE layer tokens/s & %bf16 TC peak (K3 shape); QB histogram HBM GB/s"
QB_B = 1000
# DRAM read+write / algorithmic bytes, measured with ncu on `--profile-case`
# for the kernels that can be the step's dominant one; a kernel changed since
# its counters were taken has no entry (its traffic is reported as null)
TRAFFIC_RATIO = {"expert_w3": 1.228, "expert_w12_light": 1.021, "expert_w12_heavy": 1.061}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def layer_work(shape, T, counts, fp8=False):
    """Algorithmic FLOPs and bytes per stage for T tokens with per-expert
    assignment counts `counts` (bf16 = 2 bytes; with fp8, the routed experts'
    weights, latent codes and activation codes are 1 byte, plus one exponent
    byte per weight row and token).  The expert W1|W2 GEMM runs as two
    launches: experts with at most 128 rows ("light") and the others."""
    d, L, E, k, I = shape.d, shape.latent, shape.n_experts, shape.top_k, shape.inter
    S = shape.n_shared * shape.shared_inter
    counts = np.asarray(counts)
    n = T * k
    touched = int((counts > 0).sum())
    light = (counts > 0) & (counts <= 128)
    heavy = counts > 128
    w = {}
    w["down"] = (2.0 * T * d * L, 2.0 * (T * d + L * d + T * L))
    w["shared"] = (4.0 * T * d * S, 2.0 * (T * d + 2 * S * d + T * S))
    w["router"] = (2.0 * T * L * E, 2.0 * (T * L + E * L) + 4.0 * T * E)
    w["topk"] = (0.0, 4.0 * T * E + 4.0 * E + 8.0 * n)
    w["scan"] = (0.0, 8.0 * E * math.ceil(T / 32))
    w["offsets"] = (0.0, 8.0 * E)
    w["scatter"] = (0.0, 16.0 * n)
    wb = 1.0 if fp8 else 2.0        # bytes per weight / latent / activation element
    for name, sel in (("expert_w12_light", light), ("expert_w12_heavy", heavy)):
        ne, nr = int(sel.sum()), int(counts[sel].sum())
        # weights of the stage's experts, the latent rows once (the gathered
        # re-reads of a token's row for its several experts hit L2), act out
        byts = ne * 2 * I * (L * wb + (1 if fp8 else 0)) + T * L * wb + nr * I * wb
        w[name] = (4.0 * nr * L * I, byts)
    if fp8:   # the latent's quantisation runs at the start of the light stage
        w["expert_w12_light"] = (w["expert_w12_light"][0], w["expert_w12_light"][1] + 2.0 * T * L + T * (L + 1))
    # W3: the method's bytes, i.e. the touched experts' weights and the
    # activation rows in.  The gate-weighted rows o that this design stores
    # for the combine (2 n L bytes) are an intermediate of the design, not of
    # the method: they show in the launch's measured "traffic", not here.
    w["expert_w3"] = (2.0 * n * I * L, touched * L * (I * wb + (1 if fp8 else 0)) + n * I * wb)
    w["combine"] = (0.0, 2.0 * (n * L + T * L))           # o rows in, r out
    w["up"] = (2.0 * T * (L + S) * d, 2.0 * (T * (L + S) + d * (L + S) + T * d))
    return w


# DRAM read+write over algorithmic bytes of the backward's per-expert weight-
# gradient GEMMs, from ncu on --profile-case --backward
BWD_TRAFFIC_RATIO = {"wgrad_w3": 0.901, "wgrad_w12": 0.944}


def backward_work(shape, T, counts):
    """Algorithmic FLOPs and bytes of each backward stage for T tokens with
    per-expert assignment counts `counts` (bf16 2 bytes, fp32 4 bytes; weight
    gradients are written in fp32).  The routed and shared SiTU-GLU stages
    are element-wise: they read the pre-activations p1 | p2 the training
    forward kept (bf16) and the activation gradient, and write dp1 | dp2."""
    d, L, E, k, I = shape.d, shape.latent, shape.n_experts, shape.top_k, shape.inter
    S = shape.n_shared * shape.shared_inter
    counts = np.asarray(counts)
    n = T * k
    Ep = -(-E // 64) * 64
    touched = int((counts > 0).sum())
    cols = int(((counts + 63) // 64 * 64).sum())      # per-expert segments, padded to 64
    dense = d * L + d * S + 2 * S * d + L * d + E * L  # elements of the six dense weight gradients
    w = {}
    w["dr"] = (2.0 * T * d * (L + S), 2.0 * (T * d + (L + S) * d + T * (L + S)))
    w["shared"] = (0.0, 2.0 * (2 * T * S + T * S + 2 * T * S))
    w["rmsnorm"] = (0.0, 2.0 * (n * L + T * L + T * L))
    w["expert_u"] = (2.0 * n * L * I, 2.0 * (touched * I * L + T * L + n * I))
    # p1 | p2 and u in, dp1 | dp2 out; the row's gate (through perm) in, dgate out
    w["expert_glu"] = (0.0, 2.0 * (2 * n * I + n * I + 2 * n * I) + 12.0 * n)
    # dgate, inv, idx and the kept logit per assignment in, the dense dl row out
    w["router"] = (0.0, 2.0 * T * Ep + 16.0 * n)
    w["dh_experts"] = (4.0 * n * I * L, 2.0 * (touched * 2 * I * L + 2 * n * I + n * L))
    w["dh_router"] = (2.0 * T * Ep * L, 2.0 * (T * Ep + L * Ep) + 4.0 * T * L)
    w["dh_sum"] = (0.0, 2.0 * n * L + 4.0 * T * L + 2.0 * T * L)
    w["dx"] = (2.0 * T * (L + 2 * S) * d, 2.0 * (T * (L + 2 * S) + d * (L + 2 * S) + T * d))
    w["transpose"] = (0.0, 4.0 * T * (2 * d + 3 * L + 3 * S + E))
    w["wgrad_dense"] = (2.0 * T * dense, 2.0 * T * (2 * d + 3 * L + 3 * S + E) + 4.0 * dense)
    w["segments"] = (0.0, 2.0 * cols * (2 * L + 3 * I) + 2.0 * n * (2 * L + 3 * I) + 12.0 * (E - touched) * I * L)
    w["wgrad_w3"] = (2.0 * n * L * I, 4.0 * touched * L * I + 2.0 * cols * (L + I))
    w["wgrad_w12"] = (4.0 * n * I * L, 8.0 * touched * I * L + 2.0 * cols * (2 * I + L))
    return w


def layer_flops_per_token(shape):
    d, L, k, I = shape.d, shape.latent, shape.top_k, shape.inter
    S = shape.n_shared * shape.shared_inter
    return 2.0 * d * L + 2.0 * L * shape.n_experts + 6.0 * k * L * I + 2.0 * L * d + 6.0 * d * S


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        # raw samples go to the system temp directory; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"lmoe_clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for n, v in zip(names[1:], flags[1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[0] for r in rows]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle (CPU)
def oracle_tokens_per_s(shape, w_bits, x_bits, bias, n_tokens, scores_for_qb=None):
    """Time the CPU oracle on n_tokens of the layer (+ QB over scores_for_qb);
    returns (tokens/s, seconds, threads)."""
    import oracle
    cfg = oracle.LayerConfig(**shape.layer_dict())
    t0 = time.perf_counter()
    out = oracle.layer_forward(cfg, x_bits[:n_tokens], w_bits, bias)
    t_layer = time.perf_counter() - t0
    t_qb, qb_tokens = 0.0, 0
    if scores_for_qb is not None:
        t1 = time.perf_counter()
        hist = oracle.qb_histogram(scores_for_qb, QB_B)
        oracle.qb_quantile_bias(hist, 1.0 - shape.top_k / shape.n_experts)
        t_qb = time.perf_counter() - t1
        qb_tokens = scores_for_qb.shape[0]
    per_token = t_layer / n_tokens + (t_qb / qb_tokens if qb_tokens else 0.0)
    del out
    return 1.0 / per_token, t_layer + t_qb, oracle.num_threads()


def host_weights_bits(w):
    return {k: synth.bits(v) for k, v in w.items()}


# ----------------------------------------------------------------------------- reference arm
def bench_config(world):
    """The workload both arms report (the reference arm adds its sample size)."""
    return {"workload": "k3_prefill: Stable LatentMoE layer forward T=8192, d=7168, latent=3584, "
                        "E=896, top-16, I=512, 2 shared experts x 1024 + QB histogram B=1000 + "
                        "quantile bias",
            "T": synth.K3_PREFILL.T, "l2": "inputs larger than L2 (10.3 GB of weights streamed per step)",
            "parallelism": f"dp{world} (QB histograms all-reduced)" if world > 1 else "dp1"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    shape = synth.K3_PREFILL
    w = synth.layer_weights_device(shape)
    x, bias = synth.activations_device(shape)
    wb = host_weights_bits(w)
    del w
    torch.cuda.empty_cache()
    xb = synth.bits(x)
    b = bias.cpu().numpy()
    per_step = max(16, oracle.num_threads())   # one token per host core: the oracle parallelises over tokens
    for i in range(args.warmup):
        oracle_tokens_per_s(shape, wb, xb[i * per_step:], b, per_step)
    t0 = time.perf_counter()
    for i in range(args.steps):
        off = ((args.warmup + i) * per_step) % (shape.T - per_step)
        oracle_tokens_per_s(shape, wb, xb[off:], b, per_step)
    dt = time.perf_counter() - t0
    v = per_step * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(bench_config(world), sample_tokens_per_step=per_step),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{per_step} tokens of the K3 prefill batch per step (fp64 C oracle, OpenMP)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- ncu case
def fp8_experts_variant(lm, stream, steps, warmup, shape, w, x, bias, dshape, wd, xd, bd, peaks):
    """The FP8 expert variant (e4m3 routed experts, kind::f8f6f4 MMA) on the
    same K3 prefill batch and decode batch: forward-only step times, the two
    expert stages' times, and the decode layer's HBM rate on its own bytes."""
    out = {}
    for name, shp, ww, xx, bb in (("prefill", shape, w, x, bias), ("decode", dshape, wd, xd, bd)):
        cfg = dict(shp.layer_dict(), expert_fp8=True)
        h8 = lm.lmoe_create(cfg, ww, max_tokens=shp.T)
        ws8 = lm.alloc_workspace(h8, shp.T)
        y8 = torch.empty_like(xx)
        c8 = torch.empty(shp.n_experts, dtype=torch.int32, device="cuda")
        for _ in range(warmup):
            lm.lmoe_forward(h8, xx, bb, y=y8, workspace=ws8, expert_counts_out=c8, stream=stream)
        torch.cuda.synchronize()
        counts8 = c8.cpu().numpy()
        touched = int((counts8 > 0).sum())
        n = max(steps, 20)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(n):
            lm.lmoe_forward(h8, xx, bb, y=y8, workspace=ws8, expert_counts_out=c8, stream=stream)
        t1.record(stream)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / n
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(lm.STAGES) + 1)] for _ in range(n)]
        for e_ in evs:
            for e in e_:
                e.record(stream)
        torch.cuda.synchronize()
        for i in range(n):
            lm.lmoe_set_stage_events(h8, evs[i])
            lm.lmoe_forward(h8, xx, bb, y=y8, workspace=ws8, expert_counts_out=c8, stream=stream)
        torch.cuda.synchronize()
        lm.lmoe_set_stage_events(h8, None)
        assert lm.lmoe_device_status(h8) == 0
        st = {nm: float(np.mean([ev[j].elapsed_time(ev[j + 1]) for ev in evs])) for j, nm in enumerate(lm.STAGES)}
        work = layer_work(shp, shp.T, counts8, fp8=True)
        byts = sum(v[1] for v in work.values())
        r = {"T": shp.T, "ms": round(ms, 4), "tokens_per_s": shp.T / (ms * 1e-3), "touched_experts": touched}
        for nm in ("expert_w12_light", "expert_w12_heavy", "expert_w3"):
            r[nm + "_ms"] = round(st[nm], 4)
            r[nm + "_gbs"] = round(work[nm][1] / max(st[nm] * 1e-3, 1e-12) / 1e9, 1)
        if name == "decode":
            r["bytes"] = byts
            r["gbs"] = round(byts / (ms * 1e-3) / 1e9, 1)
            r["frac_hbm"] = round(r["gbs"] / peaks["hbm_gbs"], 4)
        out[name] = r
        del h8, ws8
        torch.cuda.empty_cache()
    return out


def backward_pass(lm, stream, steps, warmup, shape, w, x, bias, peaks, peak_src, world=1):
    """The layer's backward at the K3 prefill shape: dx and the fp32 weight
    gradients for an upstream gradient dy ~ N(0, 1), after one forward of the
    same batch.  Timed over `steps` backward passes (weights and activations
    exceed L2), then once more per stage with the timing hook."""
    T = shape.T
    hb = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=T)
    ws = lm.alloc_workspace(hb, T)
    bws = torch.empty(lm.lmoe_backward_workspace_size(hb, T), dtype=torch.uint8, device="cuda")
    grads = {n: torch.empty(sz, dtype=torch.float32, device="cuda") for n, sz in lm.grad_shapes(hb).items()}
    dy = synth.grad_output_device(shape)
    dx = torch.empty_like(x)
    counts = torch.empty(shape.n_experts, dtype=torch.int32, device="cuda")

    def fstep():   # the training forward: also keeps the SiTU-GLU pre-activations
        lm.lmoe_forward(hb, x, bias, workspace=ws, expert_counts_out=counts, stream=stream)

    for _ in range(warmup):
        fstep()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(steps):
        fstep()
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = max_over_ranks(world, f0.elapsed_time(f1) / steps)

    def bstep():
        lm.lmoe_backward(hb, x, dy, ws, dx=dx, grads=grads, workspace=bws, stream=stream)

    for _ in range(warmup):
        bstep()
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(hb) == 0
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(steps):
        bstep()
    b1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, b0.elapsed_time(b1) / steps)   # each rank runs its own batch
    nst = len(lm.BWD_STAGES)
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    for evs in ev_sets:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for evs in ev_sets:
        lm.lmoe_set_backward_events(hb, evs)
        bstep()
    torch.cuda.synchronize()
    lm.lmoe_set_backward_events(hb, None)
    assert lm.lmoe_device_status(hb) == 0
    counts_host = counts.cpu().numpy()
    work = backward_work(shape, T, counts_host)
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    stage_ms = {nm: float(np.mean([ev[j].elapsed_time(ev[j + 1]) for ev in ev_sets]))
                for j, nm in enumerate(lm.BWD_STAGES)}
    stages = {}
    for nm in lm.BWD_STAGES:
        fl, by = work[nm]
        t = stage_ms[nm] * 1e-3
        bound = "tensor" if (fl > 0 and fl / by > ridge) else "hbm"
        if bound == "tensor":
            ach, peak, unit = fl / t / 1e12, peaks["bf16_tflops_sustained"], "TFLOP/s"
        else:
            ach, peak, unit = by / t / 1e9, peaks["hbm_gbs"], "GB/s"
        stages[nm] = {"ms": round(stage_ms[nm], 4), "bound": bound, "achieved": round(ach, 2), "peak": peak,
                      "unit": unit, "frac": round(ach / peak, 4), "share": round(stage_ms[nm] / ms, 4)}
    dom = max(lm.BWD_STAGES, key=lambda nm: stage_ms[nm])
    roof = {k: v for k, v in stages[dom].items() if k not in ("ms", "share")}
    # DRAM bytes per launch: ncu measured the segment GEMMs on the reduced
    # backward case (--profile-case --backward); read+write over the launch's
    # algorithmic bytes there gives the ratio, scaled to this launch
    ratio = BWD_TRAFFIC_RATIO.get(dom)
    roof.update(kernel="backward_" + dom, per_launch={"flop": work[dom][0], "bytes": work[dom][1]},
                traffic=round(ratio * work[dom][1]) if ratio else None,
                traffic_source=("ncu dram__bytes_read.sum + dram__bytes_write.sum on --profile-case --backward, "
                                "ratio to algorithmic bytes scaled to this launch") if ratio else None,
                peak_source=peak_src + (" sustained bf16" if roof["bound"] == "tensor" else " hbm copy"))
    model_flop = 2.0 * layer_flops_per_token(shape) * T      # data + weight gradients of every GEMM
    executed = sum(v[0] for v in work.values())
    out = {"T": T, "ms": round(ms, 4), "tokens_per_s": world * T / (ms * 1e-3),
           "training_forward_ms": round(fwd_ms, 4), "training_step_ms": round(fwd_ms + ms, 4),
           "model_tflops": round(model_flop / (ms * 1e-3) / 1e12, 2),
           "frac_bf16_peak": round(model_flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
           "executed_tflop": round(executed / 1e12, 3), "weight_grad_dtype": "f32",
           "roofline": roof, "stages": stages,
           "gpu_launches_per_pass": 33}
    del hb, ws, bws, grads, dy, dx
    torch.cuda.empty_cache()
    return out


def qb_closed_loop(lm, stream, T=8192, E=896, k=16, n=12):
    """The balancing loop on the GPU over a stationary stream of skewed score
    batches (per-expert logit means mu_e ~ N(0, 0.5^2), fresh noise per batch):
    route batch i with the current bias (top-k kernels), then set the bias from
    batch i by QB (B = 1000 or 10000 bins) or move it by the fixed-step rule.
    Reports max/mean expert load per batch for each rule."""
    batches = synth.qb_score_stream(T, E, n, seed=synth.QB_SEED + 1, device="cuda")
    level = 1.0 - k / E
    rules = {"qb_B1000": ("qb", 1000), "qb_B10000": ("qb", 10000),
             "sign_step1e-3": ("sign", 1e-3), "sign_step1e-2": ("sign", 1e-2)}
    out = {"T": T, "E": E, "top_k": k, "batches": n, "metric": "max/mean expert load per batch"}
    for name, (rule, p) in rules.items():
        b = torch.zeros(E, dtype=torch.float32, device="cuda")
        ratios = []
        for i in range(n):
            counts = lm.lmoe_route_static(batches[i], b, k, stream=stream)["counts"]
            ratios.append(counts.max() / counts.float().mean())
            if rule == "qb":
                _, b = lm.qb_quantile_bias(lm.qb_histogram(batches[i], p, stream=stream), level, stream=stream)
            else:
                lm.qb_sign_update(counts, p, b, stream=stream)
        out[name] = [round(float(r), 3) for r in ratios]
    del batches
    torch.cuda.empty_cache()
    return out


def run_profile_case(args):
    """A few forwards of a reduced K3-width layer (E=256, T=2048, Zipf-skewed
    router like the K3 prefill workload: ~3.3 GB on the device) and a QB
    histogram at T=262144, for ncu captures.  Prints one JSON line with its own
    timing; not a benchmark result."""
    import dataclasses
    import __graft_entry__
    __graft_entry__.build()
    import sparse_moe_layer_bias_gb300 as lm
    if args.backward:
        return run_profile_backward(args, lm)
    shape = dataclasses.replace(synth.K3_PREFILL, name="ncu_case", T=args.profile_tokens,
                                n_experts=args.profile_experts, router="zipf", expert_fp8=bool(args.fp8))
    w = synth.layer_weights_device(shape)
    x, bias = synth.activations_device(shape)
    h = lm.lmoe_create(shape.layer_dict(), w, max_tokens=shape.T)
    ws = lm.alloc_workspace(h, shape.T)
    scores = torch.empty((shape.T, shape.n_experts), dtype=torch.float32, device="cuda")
    sq = synth.qb_scores(262144, 896, device="cuda")
    hq = torch.empty((896, QB_B), dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cnt = torch.empty(shape.n_experts, dtype=torch.int32, device="cuda")
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            e0.record()
        y = lm.lmoe_forward(h, x, bias, workspace=ws, scores_out=scores, expert_counts_out=cnt)
        lm.qb_histogram(sq, QB_B, hist=hq)
    e1.record()
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    work = layer_work(shape, shape.T, cnt.cpu().numpy(), fp8=bool(args.fp8))
    print(json.dumps({"case": "ncu_case", "T": shape.T, "n_experts": shape.n_experts, "fp8": bool(args.fp8),
                      "ms_per_iter": e0.elapsed_time(e1) / max(args.steps, 1),
                      "touched_experts": int((cnt > 0).sum().item()),
                      "algorithmic_bytes": {k: v[1] for k, v in work.items()},
                      "y_finite": bool(torch.isfinite(y.float()).all().item())}), flush=True)
    return 0


def run_profile_backward(args, lm):
    """A few backward passes of a reduced K3-width layer (E=64, T=1024, k=16:
    ~256 rows per expert like the K3 prefill batch; ~4.5 GB on the device
    with the fp32 gradients), for ncu captures.  Not a benchmark result."""
    import dataclasses
    shape = dataclasses.replace(synth.K3_PREFILL, name="ncu_case_backward", T=1024, n_experts=64, router="zipf")
    w = synth.layer_weights_device(shape)
    x, bias = synth.activations_device(shape)
    dy = synth.grad_output_device(shape)
    h = lm.lmoe_create(dict(shape.layer_dict(), with_backward=True), w, max_tokens=shape.T)
    ws = lm.alloc_workspace(h, shape.T)
    bws = torch.empty(lm.lmoe_backward_workspace_size(h, shape.T), dtype=torch.uint8, device="cuda")
    grads = {n: torch.empty(sz, dtype=torch.float32, device="cuda") for n, sz in lm.grad_shapes(h).items()}
    cnt = torch.empty(shape.n_experts, dtype=torch.int32, device="cuda")
    lm.lmoe_forward(h, x, bias, workspace=ws, expert_counts_out=cnt)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            e0.record()
        dx, _ = lm.lmoe_backward(h, x, dy, ws, grads=grads, workspace=bws)
    e1.record()
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(h) == 0
    work = backward_work(shape, shape.T, cnt.cpu().numpy())
    print(json.dumps({"case": "ncu_case_backward", "T": shape.T, "n_experts": shape.n_experts,
                      "ms_per_iter": e0.elapsed_time(e1) / max(args.steps, 1),
                      "touched_experts": int((cnt > 0).sum().item()),
                      "algorithmic_bytes": {k: v[1] for k, v in work.items()},
                      "dx_finite": bool(torch.isfinite(dx.float()).all().item())}), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=128)
    ap.add_argument("--profile-case", action="store_true",
                    help="small case for ncu captures: K3 widths, 256 experts, T=2048 (~3.3 GB)")
    ap.add_argument("--profile-tokens", type=int, default=2048,
                    help="with --profile-case: tokens per forward")
    ap.add_argument("--profile-experts", type=int, default=256,
                    help="with --profile-case: routed experts (fewer experts, more rows per expert; "
                         "128 experts at 4096 tokens: ~512 rows each, like K3 prefill's heavy experts)")
    ap.add_argument("--fp8", action="store_true", help="with --profile-case: the FP8 expert variant")
    ap.add_argument("--backward", action="store_true",
                    help="with --profile-case: backward passes of a K3-width layer with 64 experts, T=1024")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.profile_case:
        return run_profile_case(args)

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    import sparse_moe_layer_bias_gb300 as lm
    from sparse_moe_layer_bias_gb300.dist import qb_allreduce_histogram
    lm.load_library()
    peaks, peak_src = load_peaks()

    shape = synth.K3_PREFILL
    T, E, k = shape.T, shape.n_experts, shape.top_k
    level = 1.0 - k / E
    w = synth.layer_weights_device(shape)
    x, bias = synth.activations_device(shape, seed_offset=rank)
    handle = lm.lmoe_create(shape.layer_dict(), w, max_tokens=T)
    ws = lm.alloc_workspace(handle, T)
    y = torch.empty_like(x)
    scores = torch.empty((T, E), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    hist = torch.empty((E, QB_B), dtype=torch.int32, device="cuda")
    q_out = torch.empty(E, dtype=torch.float32, device="cuda")
    b_new = torch.empty(E, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(xin, bin_, yout):
        lm.lmoe_forward(handle, xin, bin_, y=yout, workspace=ws, scores_out=scores,
                        expert_counts_out=counts, stream=stream)
        lm.qb_histogram(scores, QB_B, hist=hist, stream=stream)
        qb_allreduce_histogram(hist)          # data-parallel QB: sum over ranks (no-op at N=1)
        lm.qb_quantile_bias(hist, level, quantile_out=q_out, bias_out=b_new, stream=stream)

    kernels_per_step = len(lm.STAGES) + 2      # 12 forward kernels + QB histogram + quantile

    for _ in range(args.warmup):
        step(x, bias, y)
    torch.cuda.synchronize()
    assert lm.lmoe_device_status(handle) == 0
    counts_host = counts.cpu().numpy()
    touched = int((counts_host > 0).sum())

    # Headline: K steps with nothing between the kernels but the kernels (the
    # library launches them as programmatic dependent launches, so a kernel's
    # prologue overlaps its predecessor's tail).
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            step(x, bias, y)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(world, ms)
    assert lm.lmoe_device_status(handle) == 0

    # Breakdown: K more steps with a CUDA event before every stage (the events
    # serialise the kernels, so these per-stage times add up to a little more
    # than the headline step)
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(len(lm.STAGES) + 1)]
               for _ in range(args.steps)]
    for evs in ev_sets:       # create the cudaEvent_t handles before use
        for e in evs:
            e.record(stream)
    qb_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        lm.lmoe_set_stage_events(handle, ev_sets[i])
        lm.lmoe_forward(handle, x, bias, y=y, workspace=ws, scores_out=scores,
                        expert_counts_out=counts, stream=stream)
        qb_ev[i][0].record(stream)
        lm.qb_histogram(scores, QB_B, hist=hist, stream=stream)
        qb_allreduce_histogram(hist)
        lm.qb_quantile_bias(hist, level, quantile_out=q_out, bias_out=b_new, stream=stream)
        qb_ev[i][1].record(stream)
    torch.cuda.synchronize()
    lm.lmoe_set_stage_events(handle, None)
    assert lm.lmoe_device_status(handle) == 0

    stage_ms = {}
    for j, name in enumerate(lm.STAGES):
        stage_ms[name] = float(np.mean([ev[j].elapsed_time(ev[j + 1]) for ev in ev_sets]))
    stage_ms["qb"] = float(np.mean([a.elapsed_time(b) for a, b in qb_ev]))
    work = layer_work(shape, T, counts_host)
    stages = {}
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    for name in lm.STAGES:
        fl, by = work[name]
        t = stage_ms[name] * 1e-3
        bound = "tensor" if (fl > 0 and fl / by > ridge) else "hbm"
        if bound == "tensor":
            ach, peak, unit = fl / t / 1e12, peaks["bf16_tflops_sustained"], "TFLOP/s"
        else:
            ach, peak, unit = by / t / 1e9, peaks["hbm_gbs"], "GB/s"
        stages[name] = {"ms": round(stage_ms[name], 4), "bound": bound, "achieved": round(ach, 2),
                        "peak": peak, "unit": unit, "frac": round(ach / peak, 4),
                        "share": round(stage_ms[name] / ms, 4)}
    dom = max(lm.STAGES, key=lambda n: stage_ms[n])
    dfl, dby = work[dom]
    roof = dict(stages[dom])
    roof.pop("ms")
    roof.pop("share")
    roof["kernel"] = dom
    roof["per_launch"] = {"flop": dfl, "bytes": dby}
    # DRAM bytes per launch: the K3 launches are too large for an ncu capture,
    # so ncu measured the same kernels on the reduced K3-width case
    # (--profile-case); DRAM read+write over the launch's algorithmic bytes
    # there (same work model, that run's expert counts) gives the ratio below,
    # and the traffic grows with the touched experts' weights like the bytes.
    roof["traffic"] = round(TRAFFIC_RATIO[dom] * dby) if dom in TRAFFIC_RATIO else None
    roof["traffic_source"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum on --profile-case, "
                              "ratio to algorithmic bytes scaled to this launch") if dom in TRAFFIC_RATIO else None
    roof["peak_source"] = peak_src + (" sustained bf16" if roof["bound"] == "tensor" else " hbm copy")

    total_flop = layer_flops_per_token(shape) * T
    tps = world * T / (ms * 1e-3)
    layer_ms = sum(stage_ms[n] for n in lm.STAGES)
    tflops = total_flop / (layer_ms * 1e-3) / 1e12

    # --------------------------------------------------------------- e2e (host buffers)
    # The library's host-memory entry point, pipelined across steps: every step
    # copies its x and bias in from pinned host memory (input copy stream),
    # runs the forward + QB, and copies y and the new bias back out; a step's
    # input copy overlaps the forward before it, its output copy the one after.
    x_host = x.cpu().pin_memory()
    b_host = bias.cpu().pin_memory()
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    io = lm.alloc_host_io(handle)
    # the new QB bias also goes back to the host each step; its small copy runs
    # on a stream of its own (two slots) so that it never waits, on the compute
    # stream, behind the large output copy on the same copy engine
    bn_dev = [torch.empty(E, dtype=torch.float32, device="cuda") for _ in range(2)]
    bn_host = [torch.empty(E, dtype=torch.float32).pin_memory() for _ in range(2)]
    bn_copied = [torch.cuda.Event(), torch.cuda.Event()]
    bn_stream = torch.cuda.Stream()
    n_e2e = [0]

    def e2e_step():
        j = n_e2e[0] & 1
        n_e2e[0] += 1
        lm.lmoe_forward_host(handle, x_host, b_host, y_host, io, ws, scores_out=scores,
                             expert_counts_out=counts, stream=stream)
        lm.qb_histogram(scores, QB_B, hist=hist, stream=stream)
        qb_allreduce_histogram(hist)          # data-parallel QB: sum over ranks (no-op at N=1)
        stream.wait_event(bn_copied[j])       # the copy that last read bn_dev[j] is done
        lm.qb_quantile_bias(hist, level, quantile_out=q_out, bias_out=bn_dev[j], stream=stream)
        bn_stream.wait_stream(stream)
        with torch.cuda.stream(bn_stream):
            bn_host[j].copy_(bn_dev[j], non_blocking=True)
            bn_copied[j].record(bn_stream)

    for _ in range(args.warmup):
        e2e_step()
    lm.lmoe_host_wait(handle, stream)
    stream.wait_stream(bn_stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    lm.lmoe_host_wait(handle, stream)      # the last step's y has reached host memory
    stream.wait_stream(bn_stream)          # and its bias
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1) / args.steps)
    assert torch.equal(y_host.view(torch.int16), y.cpu().view(torch.int16))
    assert torch.equal(bn_host[(n_e2e[0] - 1) & 1], b_new.cpu())
    h2d = x.numel() * 2 + bias.numel() * 4
    d2h = y.numel() * 2 + E * 4

    # --------------------------------------------------------------- QB histogram sweep
    # T in {65536, 262144, 2^20} x 896 experts, B in {1000, 10000}; every
    # score tensor is larger than L2, so back-to-back launches stream it from HBM
    sweep = []
    for Tq in synth.QB_SWEEP_T:
        sq = synth.qb_scores(Tq, E, device="cuda")
        for Bq in synth.QB_SWEEP_B:
            hq = torch.empty((E, Bq), dtype=torch.int32, device="cuda")
            for _ in range(3):
                lm.qb_histogram(sq, Bq, hist=hq, stream=stream)
            torch.cuda.synchronize()
            q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            nq = max(10, args.steps)
            q0.record(stream)
            for _ in range(nq):
                lm.qb_histogram(sq, Bq, hist=hq, stream=stream)
            q1.record(stream)
            torch.cuda.synchronize()
            ms_q = q0.elapsed_time(q1) / nq
            gbs_q = (4.0 * Tq * E + 4.0 * E * Bq) / (ms_q * 1e-3) / 1e9
            sweep.append({"T": Tq, "E": E, "B": Bq, "ms": round(ms_q, 4), "gbs": round(gbs_q, 1),
                          "frac_hbm": round(gbs_q / peaks["hbm_gbs"], 4)})
            del hq
        del sq
        torch.cuda.empty_cache()
    head = next(p for p in sweep if p["T"] == (1 << 20) and p["B"] == QB_B)
    Tq, qb_ms, qb_gbs = head["T"], head["ms"], head["gbs"]
    qb_loop = qb_closed_loop(lm, stream)

    # --------------------------------------------------------------- decode layer T = 64
    dshape = synth.K3_DECODE
    wd = dict(w)
    lim = math.sqrt(3.0 / dshape.latent)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(dshape.seed)
    wd["w_router"] = ((torch.rand((E, dshape.latent), generator=gen, device="cuda") * 2 - 1) * lim).to(torch.bfloat16)
    hd = lm.lmoe_create(dshape.layer_dict(), wd, max_tokens=dshape.T)
    wsd = lm.alloc_workspace(hd, dshape.T)
    xd, bd = synth.activations_device(dshape)
    yd = torch.empty_like(xd)
    cd = torch.empty(E, dtype=torch.int32, device="cuda")
    for _ in range(args.warmup):
        lm.lmoe_forward(hd, xd, bd, y=yd, workspace=wsd, expert_counts_out=cd, stream=stream)
    torch.cuda.synchronize()
    counts_d = cd.cpu().numpy()
    touched_d = int((counts_d > 0).sum())
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nd = max(20, args.steps)
    d0.record(stream)
    for _ in range(nd):
        lm.lmoe_forward(hd, xd, bd, y=yd, workspace=wsd, expert_counts_out=cd, stream=stream)
    d1.record(stream)
    torch.cuda.synchronize()
    dec_ms = d0.elapsed_time(d1) / nd
    wdec = layer_work(dshape, dshape.T, counts_d)
    dec_bytes = sum(v[1] for v in wdec.values())
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    assert lm.lmoe_device_status(hd) == 0
    # decode breakdown: the same forward with an event before every stage
    # (stream order; the stages' bytes over their times)
    dev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(len(lm.STAGES) + 1)] for _ in range(nd)]
    for evs in dev_sets:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for evs in dev_sets:
        lm.lmoe_set_stage_events(hd, evs)
        lm.lmoe_forward(hd, xd, bd, y=yd, workspace=wsd, expert_counts_out=cd, stream=stream)
    torch.cuda.synchronize()
    lm.lmoe_set_stage_events(hd, None)
    assert lm.lmoe_device_status(hd) == 0
    dec_stages = {}
    for j, name in enumerate(lm.STAGES):
        sm_ = float(np.mean([ev[j].elapsed_time(ev[j + 1]) for ev in dev_sets]))
        dec_stages[name] = {"ms": round(sm_, 4), "gbs": round(wdec[name][1] / (sm_ * 1e-3) / 1e9, 1)}

    # --------------------------------------------------------------- FP8 expert variant
    fp8 = fp8_experts_variant(lm, stream, args.steps, args.warmup, shape, w, x, bias, dshape, wd, xd, bd, peaks)

    # --------------------------------------------------------------- backward pass
    bwd = backward_pass(lm, stream, args.steps, args.warmup, shape, w, x, bias, peaks, peak_src, world)

    # --------------------------------------------------------------- CPU oracle baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        wb = host_weights_bits(w)
        xb = synth.bits(x)
        v, secs, cores = oracle_tokens_per_s(shape, wb, xb, bias.cpu().numpy(), args.cpu_tokens,
                                             scores_for_qb=scores.cpu().numpy())
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "seconds": round(secs, 2),
               "sample": f"{args.cpu_tokens} tokens of the K3 prefill batch through the fp64 C oracle "
                         f"(OpenMP) + the QB histogram/quantile of all {T}x{E} scores"}

    line = {
        "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world),
        "layer_tflops": round(tflops, 2),
        "frac_bf16_peak": round(tflops / peaks["bf16_tflops"], 4),
        "roofline": roof,
        "stages": stages,
        "qb_ms_in_step": round(stage_ms["qb"], 4),
        "qb_hist_sweep": {"T": Tq, "E": E, "B": QB_B, "ms": round(qb_ms, 4), "gbs": round(qb_gbs, 1),
                          "frac_hbm": round(qb_gbs / peaks["hbm_gbs"], 4)},
        "qb_hist_sweep_all": sweep,
        "qb_closed_loop": qb_loop,
        "fp8_experts": fp8,
        "backward": bwd,
        "decode": {"T": dshape.T, "ms": round(dec_ms, 4), "tokens_per_s": dshape.T / (dec_ms * 1e-3),
                   "stages": dec_stages,
                   "touched_experts": touched_d, "bytes": dec_bytes, "gbs": round(dec_gbs, 1),
                   "frac_hbm": round(dec_gbs / peaks["hbm_gbs"], 4)},
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clocks.summary(),
        "peaks": dict(peaks, source=peak_src),
        "cpu_baseline": cpu,
        "touched_experts": touched,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
