"""Benchmark of the low-bit routed-expert FFN layer on GB300.

One step = one pass of the whole layer (route -> permute -> FC1+SwiGLU -> FC2
-> combine) over one batch of synthetic tokens, through libmoe's C ABI.

Default workload: decode — 384 experts, hidden 4096, expert intermediate
2048, top-8 softmax routing, 8 tokens, every expert in the 2-bit codebook
format.  Inputs are larger than L2: step i runs on layer (i mod 4) of four
distinct weight sets (4 x 3.02 GB) with its own token batch, so no step finds
the previous step's weights in the 129 MB L2.

The same run also times the other workloads of the metric, each on its own
layer of weights, as sub-records of the line (``workloads``): prefill_bf16
(8192 tokens, 2-bit experts on the tensor cores), prefill_fp8 (16384 tokens,
MXFP4 experts through the FP8 workspace), prefill_fp8_direct (the same
workload with the MXFP4 experts multiplied as stored, no workspace),
decode_fused (the headline decode as four calls: route, permute, FC1 + FC2
in one launch, combine; the headline runs the whole step as one launch),
decode_unfused (the same with FC1 and FC2 as two calls), decode_mxfp4 (the
decode shapes with MXFP4 experts on the block-scaled FP8 tensor core, MXFP8
tokens), mixed_decode (64 tokens, 2-bit experts plus 64 MXFP4 delta-cache
entries, all in the bf16 profile), mixed_decode_fp8cache (the same with the
cache experts on the block-scaled FP8 tensor core, MXFP8 tokens: their rows
in the fp8 profile) and decode_host (the decode workload with every expert in pinned
host memory and half of them resident on the device: the routed others are
copied over the CPU-GPU link each step).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead: whole layer steps of the same workload, its tokens split over one
process per host core.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; decode weight-stream GB/s and prefill TFLOP/s vs GB300 peak"


def _peaks():
    """Roofline denominators: the measured HBM copy rate and cuBLAS bf16 rates
    of this GPU model (burst: a kernel timed alone or in a short region;
    sustained: seconds-long loops), else the fallback figures.  FP8 has no
    measured figure: 2x the bf16 burst rate (the nominal dense FP8 / BF16
    ratio of the part)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        pk = {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
              "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    else:
        pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}
    pk["fp8_tflops"] = 2.0 * pk["bf16_tflops"]
    return pk


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- workloads
# DRAM bytes per expert-matmul call (dram__bytes_read.sum +
# dram__bytes_write.sum of the kernels one timed call launches, averaged over
# the step's calls, as `achieved` is), from the one-pass ncu captures of the
# full-size workloads summarised under profiles/; reported only while the
# kernels' sources are the ones captured (sha256 over the files named).
_TRAFFIC = {
    "decode": {"bytes": 501.91e6, "src": ['gemv_lut.cu', 'route_common.cuh', 'layer_args.cuh', 'common.cuh', 'internal.cuh'],
              "src_sha256": "49ac8c011b1ca780366e5fd42193ab9bac96178e259908da6cc198d2c684c246"},
    "decode_unfused": {"bytes": 256.4e6, "src": ['gemv_lut.cu', 'common.cuh', 'internal.cuh'],
                      "src_sha256": "199099f071d7a3ab38caf8a3549320951d23e47266d961c1f7c87ae38c50f77f"},
    "decode_mxfp4": {"bytes": 401.82e6, "src": ['gemm_mx.cu', 'tc_common.cuh', 'common.cuh', 'internal.cuh'],
                    "src_sha256": "1a9c10657aee666beceae0f930ecc4cd471d2af6ee8fecee9b83a0d9316c0f85"},
    "mixed_decode": {"bytes": 630.07e6, "src": ['gemv_lut.cu', 'gemm_tmem.cu', 'tc_common.cuh', 'common.cuh', 'internal.cuh'],
                    "src_sha256": "55c25615fb427c34d1a994d6a0c35be2ebd4252e67554f371abad0a6cd464efd"},
    "prefill_bf16": {"bytes": 2301.51e6, "src": ['gemm_tmem.cu', 'tc_common.cuh', 'common.cuh', 'internal.cuh'],
                    "src_sha256": "06ffb5709f2843c3905f50859122a3abba95f5bc1a61cc2fd71750663f4e3906"},
    "prefill_fp8_direct": {"bytes": 4672.7e6, "src": ['gemm_mx.cu', 'tc_common.cuh', 'common.cuh', 'internal.cuh'],
                          "src_sha256": "1a9c10657aee666beceae0f930ecc4cd471d2af6ee8fecee9b83a0d9316c0f85"},
    "prefill_fp8": {"bytes": 1820.26e6, "src": ['gemm_mx.cu', 'tc_common.cuh', 'common.cuh', 'internal.cuh'],
                   "src_sha256": "1a9c10657aee666beceae0f930ecc4cd471d2af6ee8fecee9b83a0d9316c0f85"},
    "decode_host": {"bytes": 246.25e6, "src": ['gemv_lut.cu', 'common.cuh', 'internal.cuh'],
                   "src_sha256": "199099f071d7a3ab38caf8a3549320951d23e47266d961c1f7c87ae38c50f77f"},
    "decode_fused": {"bytes": 502.08e6, "src": ['gemv_lut.cu', 'common.cuh', 'internal.cuh'],
                    "src_sha256": "199099f071d7a3ab38caf8a3549320951d23e47266d961c1f7c87ae38c50f77f"},
    "mixed_decode_fp8cache": {"bytes": 628.21e6, "src": ['gemv_lut.cu', 'gemm_mx.cu', 'tc_common.cuh', 'common.cuh', 'internal.cuh'],
                             "src_sha256": "8d108c4ae4753f82d88326020f24f50382513c22a3697d619de4017e1820ef55"},
}


def _traffic(name):
    import hashlib
    ent = _TRAFFIC.get(name)
    if not ent or ent["bytes"] is None:
        return None
    h = hashlib.sha256()
    for f in ent["src"]:
        try:
            h.update(open(os.path.join(ROOT, "bit_moe_expert_top_gb300", "csrc", f), "rb").read())
        except OSError:
            return None
    return ent["bytes"] if h.hexdigest() == ent["src_sha256"] else None


def flops_per_assignment(w):
    return 6 * w.H * w.I


def build_workload(name, layers, batches, device, tokens=None, experts=None):
    """Device weights (MoELayer per distinct layer) and token batches
    (tokens / experts: a smaller case for profiling captures)."""
    import torch

    from bit_moe_expert_top_gb300 import _lib as L
    from bit_moe_expert_top_gb300 import synth
    from bit_moe_expert_top_gb300.layer import MoELayer

    direct = name.endswith("_direct")  # MXFP4 experts multiplied as stored, no FP8 workspace
    hosted = name.endswith("_host")    # 2-bit experts in host memory, half of them resident on the device
    unfused = name.endswith("_unfused")  # the 2-bit decode's FC1 and FC2 as two calls (not one launch)
    as_mx4 = name.endswith("_mxfp4")     # the workload with MXFP4 experts on the block-scaled tensor core
    four = name.endswith("_fused")       # the 2-bit decode step as four calls (FC1 + FC2 in one launch)
    fp8cache = name.endswith("_fp8cache")  # mixed: the cache experts on the block-scaled FP8 tensor core
    base = name
    for suf in ("_direct", "_host", "_unfused", "_mxfp4", "_fused", "_fp8cache"):
        if name.endswith(suf):
            base = name[:-len(suf)]
    w = synth.get_workload(base)
    if tokens:
        w = w.replace(T=tokens)
    if experts:
        w = w.replace(E=experts, n_hot=min(w.n_hot, experts))
    mls = []
    for l in range(layers):
        if direct or as_mx4:
            ml = MoELayer("mxfp4", w.E, w.H, w.I, w.k, device, mx=synth.make_mxfp4_layer(w, seed=0, layer=l),
                          out_fmt=L.FMT_BF16)
        elif hosted:
            ml = MoELayer("w2host", w.E, w.H, w.I, w.k, device, w2=synth.make_w2_layer(w, 0, l), out_fmt=L.FMT_BF16,
                          resident=range(0, w.E, 2), stage_slots=w.T * w.k)
        elif w.weights == "w2":
            ml = MoELayer("w2", w.E, w.H, w.I, w.k, device, w2=synth.make_w2_layer(w, 0, l), out_fmt=L.FMT_BF16,
                          fused=not unfused, single_launch=not (four or unfused))
        elif w.weights == "mixed":
            ml = MoELayer("mixed", w.E, w.H, w.I, w.k, device, w2=synth.make_w2_layer(w, 0, l),
                          mx=synth.make_mxfp4_layer(w, n=w.n_hot, seed=0, layer=l),
                          expert_slot=synth.hot_experts(w, 0), out_fmt=L.FMT_BF16, cache_fp8=fp8cache)
        else:
            ml = MoELayer("fp8", w.E, w.H, w.I, w.k, device, mx=synth.make_mxfp4_layer(w, seed=0, layer=l),
                          out_fmt=L.FMT_BF16)
        mls.append(ml)
    xs, lgs = [], []
    for bi in range(batches):
        x = synth.make_x(w, 0, tid_offset=bi)
        lg = synth.make_logits(w, 0, x_bits=x, tid_offset=bi)
        xs.append(x)
        lgs.append(lg)
    return w, mls, xs, lgs


# --------------------------------------------------------------------------- ranks
def max_over_ranks(x, device):
    """The largest x over the ranks of the default process group (x itself
    with one rank): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(steps, tokens_per_step, world, seconds):
    """Whole-job throughput: every rank runs `steps` steps of
    `tokens_per_step` tokens (replicas, weak scaling) in `seconds` (the
    slowest rank's time)."""
    return steps * tokens_per_step * world / seconds


# --------------------------------------------------------------------------- GPU arm
def _decode_like(w):
    return w.T * w.k < 4096


def measure(name, args, device, world, layers, *, clocks=None, tokens=None, experts=None):
    """Time `steps` layer steps of workload `name` from a CUDA graph.

    Returns the record of the workload (tokens/s, ms per step, the roofline
    of the expert matmuls from per-launch CUDA-event durations, e2e through
    the API) and the objects the caller may reuse."""
    import torch
    import torch.distributed as dist

    from bit_moe_expert_top_gb300 import _lib as L

    batches = max(layers, 4)
    w, mls, xs_h, lgs_h = build_workload(name, layers, batches, device, tokens, experts)
    xs = [torch.from_numpy(x.view(np.int16)).to(device) for x in xs_h]
    lgs = [torch.from_numpy(lg).to(device) for lg in lgs_h]
    bufs = [ml.buffers(w.T) for ml in mls]

    def step(i, ev=None):
        li = i % layers
        return mls[li].step(xs[i % batches], lgs[i % batches], bufs[li], ev)

    # algorithmic work of every (layer, batch) pairing used by the timed steps
    work_bytes, staged = {}, {}
    for i in range(batches):
        li = i % layers
        step(i)
        torch.cuda.synchronize()
        off = bufs[li].offsets.cpu().numpy()
        work_bytes[i] = mls[li].touched_weight_bytes(off)
        if i == 0:
            group_rows = np.diff(off)
        staged[i] = mls[li].staged_bytes(off) if mls[li].fmt == "w2host" else 0
        if L.moe_get_error(bufs[li].dev_err) != 0:
            raise RuntimeError(f"{name}: device error flags set during warm-up")

    # The timed steps run from a CUDA graph: S consecutive steps (layer i mod
    # L, batch i mod B) captured once, replayed K/S times.  A second graph of
    # the same steps carries an event pair around every expert matmul (the
    # roofline's per-kernel durations); it is replayed after the timed
    # region, because event nodes between kernels would serialise the
    # programmatic launches of the timed graph.
    steps = args.steps
    S = max(d for d in range(1, min(steps, 64) + 1) if steps % d == 0)
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(S):
            step(i)
    graph_ev = []
    g_ev = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g_ev):
        for i in range(S):
            step(i, graph_ev)
    torch.cuda.synchronize()
    for _ in range(max(1, args.warmup // S + 1)):
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()

    # Clock samples: nvidia-smi cannot sample a region of a few ms, so the
    # sampler runs over a window of ~1 s of the same replays that contains
    # the timed region (replays before and after it keep the GPU under load).
    if clocks is not None:
        clocks.start()
        _spin(g, 0.5)
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps // S):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    clk = None
    if clocks is not None:
        _spin(g, 0.5)
        clk = clocks.stop()
        clk["window"] = "~1 s of the same graph replays around the timed region"
    if world > 1:
        dist.barrier()
    for _ in range(2):  # the event graph: the last replay's durations are read below
        g_ev.replay()
    torch.cuda.synchronize()

    mm_ms = sum(a.elapsed_time(b) for _, a, b in graph_ev)
    n_mm = len(graph_ev)
    per_label = {}
    for label, a, b in graph_ev:
        per_label.setdefault(label, []).append(a.elapsed_time(b) * 1e3)
    kernels_us = {k: round(sum(v) / len(v), 2) for k, v in per_label.items()}
    graph_bytes = sum(work_bytes[i % batches] for i in range(S))
    tot_bytes = sum(work_bytes[i % batches] for i in range(steps))
    A = w.A
    tot_flops = steps * A * flops_per_assignment(w)
    t_max = max_over_ranks(ms, device)
    value = job_tokens_per_s(steps, w.T, world, t_max / 1e3)

    peaks = _peaks()
    decode = _decode_like(w)
    traffic = _traffic(name) if tokens is None and experts is None else None
    if decode:
        achieved = graph_bytes / (mm_ms / 1e3) / 1e9
        single = any(lbl == "w2_layer_single_launch" for lbl, _, _ in graph_ev)
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": ("the single-launch layer kernel (routing, grouping, FC1+FC2, combine)" if single else
                           "expert matmuls (FC1+FC2 launches of the step)"),
                "peak_src": f"{peaks['src']} HBM copy rate",
                "bytes_per_launch": round(graph_bytes / n_mm), "launch_us": round(mm_ms / n_mm * 1e3, 2)}
    else:
        fp8 = w.weights == "mxfp4"
        peak = peaks["fp8_tflops"] if fp8 else peaks["bf16_tflops"]
        achieved = S * A * flops_per_assignment(w) / (mm_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": "expert matmuls (FC1+FC2 launches of the step)",
                "peak_src": (f"2 x {peaks['src']} bf16 burst rate (nominal FP8/BF16 ratio)" if fp8 else
                             f"{peaks['src']} bf16 burst rate (the timed region is well under a second)"),
                "flops_per_step": A * flops_per_assignment(w), "launch_us": round(mm_ms / n_mm * 1e3, 2),
                "step_frac": round(tot_flops / (t_max / 1e3) / 1e12 / peak, 4)}
    rec = {"value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(t_max / steps, 5),
           "config": {"workload": name, "weight_path": mls[0].fmt, "E": w.E, "H": w.H, "I": w.I, "k": w.k, "T": w.T, "weights": w.weights,
                      "l2": (f"inputs larger than L2: {layers} distinct layers of weights rotated per step"
                             if layers > 1 else "inputs larger than L2: one layer of weights "
                             f"({_layer_gb(mls[0]):.1f} GB) and 4 token batches rotated per step"),
                      "launch": f"CUDA graph of {S} steps replayed {steps // S} times"},
           "weight_stream_gbs": round(tot_bytes / (t_max / 1e3) / 1e9 / world, 1) if decode else None,
           "tflops": round(tot_flops / (t_max / 1e3) / 1e12, 2),
           "roofline": roof, "kernels_us": kernels_us,
           "gpu_launches": steps * launches_per_step(mls[0], w.T)}
    # the expert group sizes of the first token batch (rows per expert)
    edges = [0, 1, 16, 64, 256, 1024, 4096, 1 << 30]
    rec["groups"] = {"min": int(group_rows.min()), "max": int(group_rows.max()),
                     "empty": int((group_rows == 0).sum()), "touched": int((group_rows > 0).sum()),
                     "hist_edges": edges[:-1], "hist": np.histogram(group_rows, bins=edges)[0].tolist()}
    if mls[0].fmt == "w2host":
        sb = sum(staged[i % batches] for i in range(steps))
        rec["host_resident"] = {"resident_experts": mls[0].R, "staging_slots": mls[0].S,
                                "staged_bytes_per_step": round(sb / steps),
                                "link_gbs": round(sb / (t_max / 1e3) / 1e9, 1),
                                "note": "weights of the routed experts without a device slot, copied from pinned "
                                        "host memory each step"}
    if clk is not None:
        rec["clocks"] = clk
    if not args.no_e2e:
        rec["e2e"] = run_e2e(args, w, mls, bufs, xs_h, lgs_h, device, world)
    del g, g_ev, graph_ev
    return rec, (w, mls, bufs)


def _spin(g, seconds):
    import torch
    t = time.perf_counter()
    while time.perf_counter() - t < seconds:
        g.replay()
        torch.cuda.synchronize()


def _layer_gb(ml):
    n = 0
    for a in ("c1k", "s1k", "c2k", "s2k", "q1", "e1", "q2", "e2"):
        t = getattr(ml, a, None)
        if t is not None:
            n += t.numel() * t.element_size()
    return n / 1e9


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from bit_moe_expert_top_gb300 import _lib as L

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    L.lib()

    head, _ = measure(args.workload, args, device, world, args.layers, clocks=ClockSampler(local),
                      tokens=args.tokens, experts=args.experts)
    subs = {}
    if args.sub and args.tokens is None and args.experts is None:
        for name in args.sub.split(","):
            if name and name != args.workload:
                torch.cuda.empty_cache()
                rec, objs = measure(name, args, device, world, 1)
                del objs
                subs[name] = rec
                torch.cuda.empty_cache()
    cfg = dict(head["config"], parallelism=f"replicas{world}")
    res = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "weight_stream_gbs": head["weight_stream_gbs"], "tflops": head["tflops"],
        "roofline": head["roofline"], "kernels_us": head["kernels_us"], "e2e": head.get("e2e"),
        "gpu_launches": head["gpu_launches"] + sum(r["gpu_launches"] for r in subs.values()),
        "clocks": head.get("clocks"),
    }
    res["groups"] = head["groups"]
    if "host_resident" in head:
        res["host_resident"] = head["host_resident"]
    if subs:
        res["workloads"] = subs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.workload, steps=1)
        # the oracle beside two more configurations, on 16-token samples, in
        # the sub-records of those names (the FP8 profile's oracle takes about
        # a minute of one core per token: left out of the default run)
        for name in ("mixed_decode", "prefill_bf16"):
            if name in subs:
                subs[name]["cpu_baseline"] = cpu_baseline(name, steps=1, max_tokens=16)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()


def launches_per_step(ml, T):
    """Kernel launches of one layer step on the path the layer takes:
    route + permute (+ the row gather) + combine, and per expert matmul the
    table GEMV with its summing kernel (2-bit decode) or one tensor-core
    kernel, plus two workspace conversions per expert batch on the FP8 path."""
    tc = ml.use_gemm(T)
    if ml.fmt == "w2" and ml.single_launch and not tc and T * ml.k <= 256 and ml.k <= 16 and ml.E <= 1024:
        return 1  # the whole step in one launch
    if ml.fmt == "w2" and ml.fused and not tc:  # route, permute, fused FC1+FC2, combine
        return 4
    if ml.fmt == "w2":
        return 6 if tc else 7
    if ml.fmt == "mixed":  # route, permute (+ gather), 2 x (table GEMV + sums), 2 x cache-expert matmul, combine
        gather = ml.mx_tensor_path() or ml.cache_fp8
        return 3 + (1 if gather else 0) + 2 * 2 + 2 * 1
    if ml.fmt == "mxfp4":
        return 6
    if ml.fmt == "w2host":  # route, permute, stage select, fill, combine + 3 (4 with side SMs) x (table GEMV + sums)
        return 5 + 2 * (4 if ml.side_sms > 0 else 3)
    nb = (ml.E + ml.batch - 1) // ml.batch
    return 4 + 4 * nb


def run_e2e(args, w, mls, bufs, xs_h, lgs_h, device, world):
    """The same steps end to end through the library's API, each inside the
    timed region: the token batch and the router logits copied in from pinned
    host memory, the layer step as its chain of C-ABI calls (``MoELayer.step``),
    and the layer output read back to pinned host memory.  The copies run on
    two copy streams (in, out) ordered by events, so that step i+1's inputs
    and step i's output move while the GPU computes (each of the L layers has
    its own device input and output buffers; step i uses layer i mod L).
    `graph` repeats the measurement with each step replayed from a captured
    one-step graph instead of the calls."""
    import torch
    steps = max(1, min(args.steps, args.e2e_steps))
    layers = len(mls)
    batches = len(xs_h)
    hx = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_h]
    hl = [torch.from_numpy(l).pin_memory() for l in lgs_h]
    dx = [torch.empty_like(hx[0], device=device) for _ in range(layers)]
    dl = [torch.empty_like(hl[0], device=device) for _ in range(layers)]
    out_h = [torch.empty(bufs[0].out.shape, dtype=bufs[0].out.dtype).pin_memory() for _ in range(layers)]
    main = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(layers)]
    in_free = [torch.cuda.Event() for _ in range(layers)]
    out_ready = [torch.cuda.Event() for _ in range(layers)]
    out_free = [torch.cuda.Event() for _ in range(layers)]

    def piped(i, run):
        li = i % layers
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[li])  # the last step on this layer has read its inputs
            dx[li].copy_(hx[i % batches], non_blocking=True)
            dl[li].copy_(hl[i % batches], non_blocking=True)
            in_ready[li].record(s_in)
        main.wait_event(in_ready[li])
        main.wait_event(out_free[li])  # the last step's output on this layer has been read back
        out = run(li)
        in_free[li].record(main)
        out_ready[li].record(main)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[li])
            out_h[li].copy_(out, non_blocking=True)
            out_free[li].record(s_out)

    def eager(li):
        return mls[li].step(dx[li], dl[li], bufs[li])

    for li in range(layers):  # events start recorded: nothing to wait for
        for ev in (in_free[li], out_free[li]):
            ev.record(main)
    for i in range(min(steps, 3)):  # warm: host-side caches of the calls
        piped(i, eager)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        piped(i, eager)
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, device)

    graphs = []
    for li in range(layers):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            out = mls[li].step(dx[li], dl[li], bufs[li])
        graphs.append((g, out))
    torch.cuda.synchronize()

    def replay(li):
        g, out = graphs[li]
        g.replay()
        return out

    t0 = time.perf_counter()
    for i in range(steps):
        piped(i, replay)
    torch.cuda.synchronize()
    dtg = max_over_ranks(time.perf_counter() - t0, device)
    return {"value": round(job_tokens_per_s(steps, w.T, world, dt), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(hx[0].numel() * 2 + hl[0].numel() * 4),
            "d2h_bytes_per_step": int(out_h[0].numel() * out_h[0].element_size()), "steps": steps,
            "path": ("pinned host -> device copies on a copy stream, the layer's C-ABI calls, device -> pinned "
                     "host on a second copy stream, every step; copies overlap the neighbouring steps' kernels"),
            "graph": {"value": round(job_tokens_per_s(steps, w.T, world, dtg), 1), "unit": "tokens/s",
                      "path": "as above with the step replayed from a captured one-step CUDA graph"}}


# --------------------------------------------------------------------------- CPU oracle
# The oracle (numpy, float64) timed on the host cores: a layer step's tokens
# are split over one process per core (at most one per token); each process
# prepares its experts' stored weights untimed, then every step starts on a
# barrier and the step's time is the slowest process's.

def _oracle_prepare(workload, tokens):
    from bit_moe_expert_top_gb300 import synth
    from oracle import codecs as C
    from oracle import moe as M
    w = synth.get_workload(workload)
    x = synth.make_x(w, 0)
    logits = synth.make_logits(w, 0, x_bits=x)
    ids = M.route(logits, w.k)[0][tokens]
    raw = {}
    if w.weights == "w2":
        for e in np.unique(ids):
            raw[int(e)] = synth.make_w2_expert(w, int(e), 0, 0)

        def acc(e):
            c1, s1, c2, s2 = raw[e]
            return C.decode_w2(c1, s1), C.decode_w2(c2, s2)
        prof = "bf16"
    elif w.weights == "mixed":
        slot = synth.hot_experts(w, 0)
        for e in np.unique(ids):
            raw[int(e)] = (synth.make_mxfp4_expert(w, int(slot[e]), 0, 0) if slot[e] >= 0 else
                           synth.make_w2_expert(w, int(e), 0, 0))

        def acc(e):
            a, b, c, d = raw[e]
            if slot[e] >= 0:
                return C.decode_mxfp4(a, b), C.decode_mxfp4(c, d)
            return C.decode_w2(a, b), C.decode_w2(c, d)
        prof = "bf16"
    else:
        for e in np.unique(ids):
            raw[int(e)] = synth.make_mxfp4_expert(w, int(e), 0, 0)

        def acc(e):
            q1, s1, q2, s2 = raw[e]
            return C.e4m3_value(C.mxfp4_to_e4m3(q1, s1)), C.e4m3_value(C.mxfp4_to_e4m3(q2, s2))
        prof = "fp8"
    return w, x, logits, acc, prof


def _oracle_proc(workload, tokens, steps, barrier, conn):
    from oracle import moe as M
    w, x, logits, acc, prof = _oracle_prepare(workload, tokens)
    for _ in range(steps):
        barrier.wait()
        t0 = time.perf_counter()
        M.layer(x, logits, w.k, acc, profile=prof, tokens=tokens)
        conn.send(time.perf_counter() - t0)
    conn.close()


def oracle_steps(workload, steps, max_tokens=None):
    """Run `steps` oracle steps of `workload` (all its tokens, or the first
    `max_tokens`) on the host cores; returns (per-step seconds, processes,
    host cores, tokens per step)."""
    import multiprocessing as mp
    from bit_moe_expert_top_gb300 import synth
    w = synth.get_workload(workload)
    ntok = w.T if max_tokens is None else min(w.T, max_tokens)
    cores = len(os.sched_getaffinity(0))
    procs = max(1, min(cores, ntok))
    chunks = [c.tolist() for c in np.array_split(np.arange(ntok), procs)]
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        barrier = ctx.Barrier(procs)
        pipes, ps = [], []
        for c in chunks:
            rd, wr = ctx.Pipe(duplex=False)
            p = ctx.Process(target=_oracle_proc, args=(workload, c, steps, barrier, wr), daemon=True)
            p.start()
            wr.close()
            pipes.append(rd)
            ps.append(p)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    times = []
    for _ in range(steps):
        times.append(max(rd.recv() for rd in pipes))
    for p in ps:
        p.join(timeout=60)
    return times, procs, cores, ntok


def cpu_baseline(workload, steps=1, max_tokens=None):
    """The oracle on the host cores, whole layer steps of `workload` (or a
    bounded sample of `max_tokens` of its tokens)."""
    from bit_moe_expert_top_gb300 import synth
    w = synth.get_workload(workload)
    max_tok = w.T if _decode_like(w) else 16   # prefill steps: a bounded token sample
    if max_tokens is not None:
        max_tok = min(max_tok, max_tokens)
    try:
        times, procs, cores, ntok = oracle_steps(workload, steps, max_tok)
    except Exception as e:  # reported, not fatal to the GPU line
        return {"value": None, "unit": "tokens/s", "cores": 0, "kind": "oracle", "sample": f"failed: {e}"}
    t = statistics.median(times)
    return {"value": round(ntok / t, 4), "unit": "tokens/s", "cores": procs, "host_cores": cores, "kind": "oracle",
            "sample": (f"{'all ' if ntok == w.T else ''}{ntok} of {w.T} tokens of one {workload} layer per step, "
                       f"split over {procs} processes (numpy fp64, 1 BLAS thread each), median of {steps} "
                       f"step(s), {t:.2f} s per step")}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from bit_moe_expert_top_gb300 import synth
    w = synth.get_workload(args.workload)
    max_tok = w.T if _decode_like(w) else 16
    times, procs, cores, ntok = oracle_steps(args.workload, args.warmup + args.steps, max_tok)
    timed = times[args.warmup:]
    t = statistics.median(timed)
    value = ntok / t
    sample = (f"{'all ' if ntok == w.T else ''}{ntok} of {w.T} tokens of one {args.workload} layer per step, "
              f"split over {procs} processes (numpy fp64, 1 BLAS thread each)")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "E": w.E, "H": w.H, "I": w.I, "k": w.k, "T": w.T,
                      "weights": w.weights, "tokens_per_step": ntok},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": procs, "host_cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=["tiny", "decode", "mixed_decode", "prefill_bf16", "prefill_fp8", "prefill_fp8_direct",
                             "decode_host", "decode_unfused", "decode_mxfp4", "decode_fused",
                             "mixed_decode_fp8cache"])
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--sub", default="decode_fused,decode_unfused,decode_mxfp4,prefill_bf16,prefill_fp8,prefill_fp8_direct,"
                                     "mixed_decode,mixed_decode_fp8cache,decode_host",
                    help="other workloads timed in the same run as sub-records ('' for none)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (small cases for profiler captures)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the workload's expert count (small cases for profiler captures)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
