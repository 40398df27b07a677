"""Benchmark of the low-bit routed-expert FFN layer on GB300.

One step = one pass of the whole layer (route -> permute -> FC1+SwiGLU -> FC2
-> combine) over one batch of synthetic tokens, through libmoe's C ABI.

Default workload: decode — 384 experts, hidden 4096, expert intermediate
2048, top-8 softmax routing, 8 tokens, every expert in the 2-bit codebook
format.  Inputs are larger than L2: step i runs on layer (i mod 4) of four
distinct weight sets (4 x 3.02 GB) with its own token batch, so no step finds
the previous step's weights in the 129 MB L2.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead (a bounded sample of the same workload on the host cores).
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
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


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
                                          "--format=csv,noheader,nounits", "-lms", "100"],
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
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, mean of
# the FC1 and FC2 launches) of the dominant kernel, from the ncu captures
# summarised under profiles/; reported only while the kernel source is the
# one that was captured (sha256 of the file named).
_TRAFFIC = {
    "decode": {"bytes": 250.31e6, "src": "gemv_lut.cu",
               "src_sha256": "8415d1fcfcc286234ba3f206d24193dda346e22e404a9c5f80995019f668640f"},
    "prefill_bf16": {"bytes": 2312.48e6, "src": "gemm_tmem.cu",
                     "src_sha256": "c76ee4c57ee6b3e3352415b0bf3e9cc8766c3baf143397685942f1bdf29fe09e"},
}


def _traffic(w):
    import hashlib
    ent = _TRAFFIC.get(w.name)
    if not ent or ent["bytes"] is None:
        return None
    src = os.path.join(ROOT, "bit_moe_expert_top_gb300", "csrc", ent["src"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return ent["bytes"] if digest == ent["src_sha256"] else None


def flops_per_assignment(w):
    return 6 * w.H * w.I


def build_workload(name, layers, batches, device, tokens=None):
    """Device weights (MoELayer per distinct layer) and token batches
    (tokens: a smaller token count for profiling captures)."""
    import torch

    from bit_moe_expert_top_gb300 import _lib as L
    from bit_moe_expert_top_gb300 import synth
    from bit_moe_expert_top_gb300.layer import MoELayer

    w = synth.get_workload(name)
    if tokens:
        w = w.replace(T=tokens)
    mls = []
    for l in range(layers):
        if w.weights == "w2":
            ml = MoELayer("w2", w.E, w.H, w.I, w.k, device, w2=synth.make_w2_layer(w, 0, l), out_fmt=L.FMT_BF16)
        elif w.weights == "mixed":
            ml = MoELayer("mixed", w.E, w.H, w.I, w.k, device, w2=synth.make_w2_layer(w, 0, l),
                          mx=synth.make_mxfp4_layer(w, n=w.n_hot, seed=0, layer=l),
                          expert_slot=synth.hot_experts(w, 0), out_fmt=L.FMT_BF16)
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

    layers = args.layers
    batches = max(layers, 4)
    w, mls, xs_h, lgs_h = build_workload(args.workload, layers, batches, device, args.tokens)
    xs = [torch.from_numpy(x.view(np.int16)).to(device) for x in xs_h]
    lgs = [torch.from_numpy(lg).to(device) for lg in lgs_h]
    bufs = [ml.buffers(w.T) for ml in mls]

    def step(i, ev=None):
        li = i % layers
        return mls[li].step(xs[i % batches], lgs[i % batches], bufs[li], ev)

    # algorithmic work of every (layer, batch) pairing used by the timed steps
    work_bytes = {}
    for i in range(batches):
        li = i % layers
        step(i)
        torch.cuda.synchronize()
        off = bufs[li].offsets.cpu().numpy()
        work_bytes[i] = mls[li].touched_weight_bytes(off)
        if L.moe_get_error(bufs[li].dev_err) != 0:
            raise RuntimeError("device error flags set during warm-up")

    # ---- the timed steps run from a CUDA graph: S consecutive steps (layer
    # i mod L, batch i mod B) captured once; the timed region replays it K/S
    # times.  A second graph of the same steps carries an event pair around
    # every expert matmul (the roofline's per-kernel durations); it is
    # replayed after the timed region, because event nodes between kernels
    # would serialise the programmatic launches of the timed graph.
    S = max(d for d in range(1, min(args.steps, 64) + 1) if args.steps % d == 0)
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

    clocks = ClockSampler(local)
    clocks.start()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps // S):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    for _ in range(2):  # the event graph: the last replay's durations are read below
        g_ev.replay()
    torch.cuda.synchronize()

    # per-launch durations of the expert matmul kernels (the dominant ones),
    # from the event pairs of the event graph's last replay
    mm_ms = sum(a.elapsed_time(b) for _, a, b in graph_ev)
    n_mm = len(graph_ev)
    per_label = {}
    for label, a, b in graph_ev:
        per_label.setdefault(label, []).append(a.elapsed_time(b) * 1e3)
    kernels_us = {k: round(sum(v) / len(v), 2) for k, v in per_label.items()}
    graph_bytes = sum(work_bytes[i % batches] for i in range(S))
    tot_bytes = sum(work_bytes[i % batches] for i in range(args.steps))
    A = w.A
    tot_flops = args.steps * A * flops_per_assignment(w)

    t_max = max_over_ranks(ms, device)
    value = job_tokens_per_s(args.steps, w.T, world, t_max / 1e3)

    peaks = _peaks()
    decode = w.T * w.k < 4096
    traffic = _traffic(w) if args.tokens is None else None
    if decode:
        achieved = graph_bytes / (mm_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": "expert matmuls (moe_w2_mm FC1+FC2)", "peak_src": peaks["src"],
                "bytes_per_launch": round(graph_bytes / n_mm), "launch_us": round(mm_ms / n_mm * 1e3, 2)}
    else:
        achieved = S * A * flops_per_assignment(w) / (mm_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops_sustained"], 4), "traffic": traffic,
                "kernel": "expert matmuls", "peak_src": peaks["src"], "launch_us": round(mm_ms / n_mm * 1e3, 2)}

    # ---------------- end to end: host buffers through the public API
    e2e = run_e2e(args, w, mls, bufs, xs_h, lgs_h, device, world)

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "E": w.E, "H": w.H, "I": w.I, "k": w.k, "T": w.T,
                   "weights": w.weights, "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2: {layers} distinct layers of weights rotated per step",
                   "launch": f"CUDA graph of {S} steps replayed {args.steps // S} times"},
        "weight_stream_gbs": round(tot_bytes / (t_max / 1e3) / 1e9 / world, 1) if decode else None,
        "tflops": round(tot_flops / (t_max / 1e3) / 1e12, 2),
        "roofline": roof,
        "kernels_us": kernels_us,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step(mls[0], w.T),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_sample)
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
    if ml.fmt == "w2":
        return 6 if tc else 7
    if ml.fmt == "mixed":
        mx_tc = ml.mx_tensor_path()
        return 3 + (1 if mx_tc else 0) + 2 * 2 + 2 * 1
    nb = (ml.E + ml.batch - 1) // ml.batch
    return 4 + 4 * nb


def run_e2e(args, w, mls, bufs, xs_h, lgs_h, device, world):
    """The same steps through the public API with the token batch copied in
    from pinned host memory and the layer output read back, every step inside
    the timed region (the step itself replays a captured one-step graph)."""
    import torch
    steps = max(1, min(args.steps, args.e2e_steps))
    layers = len(mls)
    batches = len(xs_h)
    hx = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_h]
    hl = [torch.from_numpy(l).pin_memory() for l in lgs_h]
    dx = [torch.empty_like(hx[0], device=device) for _ in range(layers)]
    dl = [torch.empty_like(hl[0], device=device) for _ in range(layers)]
    out_h = torch.empty(bufs[0].out.shape, dtype=bufs[0].out.dtype).pin_memory()
    graphs = []
    torch.cuda.synchronize()
    for li in range(layers):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            out = mls[li].step(dx[li], dl[li], bufs[li])
        graphs.append((g, out))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        li = i % layers
        dx[li].copy_(hx[i % batches], non_blocking=True)
        dl[li].copy_(hl[i % batches], non_blocking=True)
        g, out = graphs[li]
        g.replay()
        out_h.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, device)
    return {"value": round(job_tokens_per_s(steps, w.T, world, dt), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(hx[0].numel() * 2 + hl[0].numel() * 4),
            "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()), "steps": steps}


# --------------------------------------------------------------------------- CPU oracle
def cpu_baseline(workload, sample_tokens):
    """Time the oracle on a bounded sample in a fresh single-threaded process."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", workload, "--cpu-sample", str(sample_tokens)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"failed: {r.stderr.strip()[-200:]}"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_sample(workload, ntok):
    from bit_moe_expert_top_gb300 import synth
    from oracle import moe as M
    w = synth.get_workload(workload)
    x = synth.make_x(w, 0)
    logits = synth.make_logits(w, 0, x_bits=x)
    tokens = list(range(min(ntok, w.T)))
    if w.weights == "w2":
        ids = M.route(logits, w.k)[0][tokens]
        raw = {}
        for e in np.unique(ids):
            raw[int(e)] = synth.make_w2_expert(w, int(e), 0, 0)

        def acc(e):
            c1, s1, c2, s2 = raw[e]
            from oracle import codecs as C
            return C.decode_w2(c1, s1), C.decode_w2(c2, s2)
        prof = "bf16"
    elif w.weights == "mixed":
        slot = synth.hot_experts(w, 0)
        from oracle import codecs as C

        def acc(e):
            if slot[e] >= 0:
                q1, s1, q2, s2 = synth.make_mxfp4_expert(w, int(slot[e]), 0, 0)
                return C.decode_mxfp4(q1, s1), C.decode_mxfp4(q2, s2)
            c1, s1, c2, s2 = synth.make_w2_expert(w, e, 0, 0)
            return C.decode_w2(c1, s1), C.decode_w2(c2, s2)
        prof = "bf16"
    else:
        from oracle import codecs as C

        def acc(e):
            q1, s1, q2, s2 = synth.make_mxfp4_expert(w, e, 0, 0)
            return C.e4m3_value(C.mxfp4_to_e4m3(q1, s1)), C.e4m3_value(C.mxfp4_to_e4m3(q2, s2))
        prof = "fp8"
    t0 = time.perf_counter()
    M.layer(x, logits, w.k, acc, profile=prof, tokens=tokens)
    dt = time.perf_counter() - t0
    return {"value": round(len(tokens) / dt, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(tokens)} of {w.T} tokens of one {workload} layer (routing over all tokens), "
                      f"{dt:.1f} s, numpy fp64, 1 thread"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from bit_moe_expert_top_gb300 import synth
    w = synth.get_workload(args.workload)
    vals = []
    for _ in range(args.warmup + args.steps):
        vals.append(cpu_baseline(args.workload, args.cpu_sample))
    timed = [v for v in vals[args.warmup:] if v.get("value")]
    value = statistics.median([v["value"] for v in timed]) if timed else None
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * w.T / value, 3) if value else None, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "E": w.E, "H": w.H, "I": w.I, "k": w.k, "T": w.T,
                      "weights": w.weights},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                            "sample": timed[0]["sample"] if timed else "failed"},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=["tiny", "decode", "mixed_decode", "prefill_bf16", "prefill_fp8"])
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (small cases for profiler captures)")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-sample", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        print(json.dumps(oracle_sample(args.oracle_sample, args.cpu_sample)))
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
