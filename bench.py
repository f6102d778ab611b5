"""Throughput of the MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one whole layer forward (router GEMM + softmax/top-k + stats,
scan, permute, expert FFN GEMM1 + GELU, GEMM2, combine) over one batch of
the workload, inputs resident in HBM. Every rank runs an independent
replica on its own GPU (the layer needs no exchange for its output), the
timed region is bracketed by a barrier and a device synchronisation, and
rank 0 prints one JSON line with the max-over-ranks time.

`--impl reference` times the CPU oracle as it stands on this host's cores
on a bounded token sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "MoE layer fwd tokens/s; grouped-GEMM TFLOP/s & permute GB/s vs GB300 peaks"
DEFAULT_WORKLOAD = "large_expert"
L2_BYTES = 129 * 2 ** 20
# DRAM bytes (read + write) per grouped-GEMM launch, averaged over GEMM1 and
# GEMM2, from the ncu capture summarised in profiles/ (null until captured
# for the current kernel).
TRAFFIC = {"large_expert": 17.7e9}
TRAFFIC_FP8 = {"large_expert": 4.85e9}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------ accounting ----

def algorithmic_work(w: W.Workload, n_kept: int, n_tokens_any: int, fp8: bool = False) -> dict:
    """What each stage must move or compute (not what it happens to move):
    router reads x and the gate and writes indices/weights; permute reads
    each token row that has a kept slot once and writes each kept row once
    (dispatch bytes of the comm bottleneck page, section 2.1, with drops
    removed); GEMM1/GEMM2 are 2*N*H*h FLOP each (4*H*h per token-expert,
    section 2.2); combine reads each kept row and writes each token row.
    With FP8 the permute writes e4m3 rows (1 byte per value) and a 4-byte
    scale per kept row, and the combine reads e4m3 rows with a 4-byte scale
    per 128-column block."""
    T, H, E, k, h = w.T, w.H, w.E, w.k, w.h
    permute = 2 * H * n_tokens_any + ((H + 4) * n_kept if fp8 else 2 * H * n_kept)
    combine_in = (H + 4 * -(-H // 128)) * n_kept if fp8 else 2 * H * n_kept
    return {
        "route_bytes": 2 * T * H + 2 * H * E + 8 * T * k,
        "route_flop": 2 * T * H * E,
        "permute_bytes": permute,
        "gemm1_flop": 2 * n_kept * H * h,
        "gemm2_flop": 2 * n_kept * h * H,
        "combine_bytes": combine_in + 2 * H * T,
    }


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- our arm ----

def run_ours(args, rank, world, local_rank):
    import top_routing_expert_gb300 as moe

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.build()
    moe.load_library()
    w = W.get(args.workload)
    inp = W.make_inputs(w, seed=rank)
    s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s, device=dev, fp8=args.fp8)
    d = {kk: (v.to(dev) if v is not None else None) for kk, v in inp.items()}
    T, E, k = w.T, w.E, w.k
    y = torch.empty((T, w.H), dtype=torch.bfloat16, device=dev)
    aux = torch.zeros(1, dtype=torch.float32, device=dev)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    dest = torch.zeros((T, k), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    q = None
    if args.fp8:
        # weights are parameters: quantised once, before the timed region
        q = moe.Fp8Weights(d["W1"], d["W2"])
        torch.cuda.synchronize(dev)

        def step(events=None, strm=None):
            moe.moe_layer_fwd_fp8(s, d["x"], d["gate"], d["bias"], q, y, aux=aux,
                                  offsets=offsets, dest_row=dest, dev_status=status, ws=ws,
                                  stream=strm or stream, events=events)
    elif args.gumbel is None:
        def step(events=None, strm=None):
            moe.moe_layer_fwd(s, d["x"], d["gate"], d["bias"], d["W1"], d["W2"], y, aux=aux,
                              offsets=offsets, dest_row=dest, dev_status=status, ws=ws,
                              stream=strm or stream, events=events)
    else:
        # the training router: uniforms drawn once, outside the timed region
        gen = torch.Generator(device=dev).manual_seed(rank + 1)
        noise = torch.rand((T, E), generator=gen, device=dev, dtype=torch.float32)

        def step(events=None, strm=None):
            moe.moe_layer_fwd_gumbel(s, d["x"], d["gate"], d["bias"], noise, args.gumbel,
                                     d["W1"], d["W2"], y, aux=aux, offsets=offsets,
                                     dest_row=dest, dev_status=status, ws=ws,
                                     stream=strm or stream, events=events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # per-stage events, recorded once so that their handles exist
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.LAYER_NUM_EVENTS)]
          for _ in range(args.steps)]
    for row in ev:
        for e in row:
            e.record(stream)
    # inputs re-read every step; below 2x L2 they could stay cached, so then
    # L2 is flushed between steps and each step is timed by its own events
    in_bytes = sum(v.numel() * v.element_size() for v in d.values() if v is not None)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) \
        if in_bytes < 2 * L2_BYTES else None
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(float(i))
        step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if flush is None:
        ms = t0.elapsed_time(t1) / args.steps
    else:
        ms = sum(ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps)) / args.steps
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    stage_ms = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)) / args.steps
                for j in range(moe.LAYER_NUM_EVENTS - 1)]
    st = int(status.item())
    n_kept = int(offsets[E].item())
    any_kept = int((dest >= 0).any(dim=1).sum().item())

    # the end-to-end leg times the inference layer; skipped for the training router
    e2e = None if (args.no_e2e or args.gumbel is not None) else \
        run_e2e(args, moe, s, inp, d, y, aux, ws, stream, dev, world, q)
    dense = None if (args.fp8 or args.gumbel is not None) else \
        run_dense_ffn(args, moe, w, d, stream, dev, flush is not None)
    graph = run_graph(args, step, stream, dev, flush) if args.graph else None
    if rank != 0:
        return None
    l2 = (f"L2 flushed between steps ({2 * L2_BYTES >> 20} MB write); steps timed by their own events"
          if flush is not None else
          f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB re-read per step); no flush")
    line = report(args, w, world, ms, stage_ms, clk, st, n_kept, any_kept, e2e, inp, l2, dense)
    if graph is not None:
        line["graph_replay"] = {"ms_per_step": round(graph, 4),
                                "value": round(w.T * world / (graph / 1e3), 1), "unit": "tokens/s",
                                "what": "the same step captured once in a CUDA graph and replayed"}
    return line


def run_graph(args, step, stream, dev, flush):
    """The same layer step captured once in a CUDA graph and replayed: the
    host's launch work leaves the loop (it matters for the small,
    launch-bound layers). Timed like the main loop, without per-stage
    events."""
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step(strm=side)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(strm=torch.cuda.current_stream(dev))
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    cur = torch.cuda.current_stream(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(cur)
        g.replay()
        ev[i][1].record(cur)
    t1.record(cur)
    torch.cuda.synchronize(dev)
    if flush is None:
        return t0.elapsed_time(t1) / args.steps
    return sum(a.elapsed_time(b) for a, b in ev) / args.steps


def run_dense_ffn(args, moe, w, d, stream, dev, flush_l2):
    """The secondary metric of the module notes' benchmark protocol (section
    5.3): the MoE layer's time over that of one dense FFN of width h on the
    same T tokens, run by the same grouped-GEMM kernels with E = 1 (expert 0's
    weights, every token kept)."""
    T, H, h = w.T, w.H, w.h
    s1 = moe.MoeShape.make(T, H, 1, 1, h, 1.0)
    ws1 = moe.Workspace(s1, device=dev)
    off = torch.tensor([0, T], dtype=torch.int32, device=dev)
    W1 = d["W1"][:1].contiguous()
    W2 = d["W2"][:1].contiguous()
    act = torch.empty((T, h), dtype=torch.bfloat16, device=dev)
    yd = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush_l2 else None
    n = max(3, min(args.steps, 30))
    for _ in range(3):
        moe.moe_expert_ffn(s1, d["x"], off, W1, W2, act, yd, ws=ws1, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    torch.cuda.synchronize(dev)
    for i in range(n):
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(stream)
        moe.moe_expert_ffn(s1, d["x"], off, W1, W2, act, yd, ws=ws1, stream=stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / n


def run_e2e(args, moe, s, inp, d, y, aux, ws, stream, dev, world, q=None):
    """End to end through the public API with host buffers: every step is one
    micro-batch of moe_layer_fwd_host - its tokens copied in from pinned host
    memory, the layer, its output and aux copied back to the host - with the
    copies of neighbouring micro-batches overlapping the layer on three
    streams. Timed from before the first copy-in to after the last copy-out."""
    T, H = inp["x"].shape
    pipe = moe.HostPipeline(s, device=dev, fp8=q is not None)
    x_host = inp["x"].pin_memory()
    y_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    aux_host = torch.empty(max(args.steps, args.warmup), dtype=torch.float32).pin_memory()

    def run(n):
        if q is not None:
            return pipe.run([x_host] * n, [y_host] * n, d["gate"], d["bias"], q, None, aux_host)
        return pipe.run([x_host] * n, [y_host] * n, d["gate"], d["bias"], d["W1"], d["W2"],
                        aux_host)

    run(args.warmup).synchronize()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0.record(pipe.streams[1])
    out = run(args.steps)
    e1.record(out)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    return {"ms": e2e_ms, "h2d": T * H * 2, "d2h": T * H * 2 + 4}


def report(args, w, world, ms, stage_ms, clk, st, n_kept, any_kept, e2e, inp, l2, dense=None):
    T, k = w.T, w.k
    pk = peaks()
    work = algorithmic_work(w, n_kept, any_kept, fp8=args.fp8)
    names = ["route", "scan", "permute", "gemm1", "gemm2", "combine"]
    stage = dict(zip(names, stage_ms))
    kern = {}
    for nm, key, unit in [("route", "route_bytes", "GB/s"), ("permute", "permute_bytes", "GB/s"),
                          ("combine", "combine_bytes", "GB/s"), ("gemm1", "gemm1_flop", "TFLOP/s"),
                          ("gemm2", "gemm2_flop", "TFLOP/s")]:
        sec = stage[nm] / 1e3
        if unit == "GB/s":
            a = work[key] / sec / 1e9
            kern[nm] = {"ms": round(stage[nm], 4), "achieved": round(a, 1), "unit": unit,
                        "frac_of_measured_hbm": round(a / pk["hbm_gbs"], 3)}
        else:
            a = work[key] / sec / 1e12
            kern[nm] = {"ms": round(stage[nm], 4), "achieved": round(a, 1), "unit": unit,
                        "frac_of_measured_bf16": round(a / pk["bf16_tflops"], 3)}
    kern["scan"] = {"ms": round(stage["scan"], 4)}
    gemm_ms = stage["gemm1"] + stage["gemm2"]
    gemm_tf = (work["gemm1_flop"] + work["gemm2_flop"]) / (gemm_ms / 1e3) / 1e12
    # the GEMM runs inside a ~1 s loop of back-to-back layer steps under the
    # power cap: the sustained bf16 figure is its roofline (burst also given)
    peak = pk["bf16_tflops_sustained"] or pk["bf16_tflops"]
    burst = pk["bf16_tflops"]
    kind = f"{pk['source']} bf16 sustained"
    if args.fp8:
        # e4m3 runs at twice the bf16 tensor rate (nominal 4.5 vs 2.25 PFLOP/s dense)
        peak, burst = 2 * peak, 2 * burst
        kind = f"{pk['source']} bf16 sustained x 2 (nominal e4m3/bf16 ratio)"
        for nm in ("gemm1", "gemm2"):
            kern[nm]["frac_of_measured_fp8"] = round(kern[nm]["frac_of_measured_bf16"] / 2, 3)
        kern["gemm1"]["includes"] = "GEMM1 + act row quantisation"
    roofline = {"kernel": "grouped GEMM (expert FFN GEMM1+GELU and GEMM2 launches)",
                "bound": "tensor", "achieved": round(gemm_tf, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(gemm_tf / peak, 4),
                "peak_kind": kind,
                "frac_of_burst": round(gemm_tf / burst, 4),
                "traffic": (TRAFFIC_FP8 if args.fp8 else TRAFFIC).get(w.name)}
    tokens = T * world
    line = {
        "metric": METRIC, "value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {**w.describe(), "parallelism": f"replicas x{world} (no exchange)",
                   "router": "inference (top-k of logits)" if args.gumbel is None
                   else f"training (Gumbel noise, temperature {args.gumbel})",
                   "expert_ffn": "FP8 e4m3 dispatch + FFN + combine, per-row/per-column/"
                                 "128-column-block fp32 scales"
                   if args.fp8 else "bf16",
                   "l2": l2},
        "clocks": clk,
        "e2e": None if e2e is None else {
            "value": round(tokens / (e2e["ms"] / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(e2e["ms"], 4), "h2d_bytes_per_step": e2e["h2d"],
            "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": (8 if args.fp8 else 7) * args.steps,
        "roofline": roofline,
        "kernels": kern,
        "routing": {"kept_rows": n_kept, "assignments": T * k, "dropped": T * k - n_kept,
                    "dev_status": st},
    }
    if dense is not None:
        line["moe_vs_dense_ffn"] = {
            "dense_ffn_ms": round(dense, 4), "ratio": round(ms / dense, 3),
            "what": "layer time / one dense FFN (h) over the same T tokens, same kernels, E=1",
            "ideal_from_flops": round(n_kept / T, 3)}
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(OracleInputs(w, inp, fp8=args.fp8), args.cpu_tokens)
    return line


# ------------------------------------------------------------ CPU oracle ----

class OracleInputs:
    """Float64 copies of a workload's inputs for the oracle, made once
    (outside any timed region): the oracle works on float64 arrays."""

    def __init__(self, w: W.Workload, inp: dict, fp8: bool = False):
        import numpy as np
        from oracle import moe_oracle as O
        f64 = lambda t: t.float().numpy().astype(np.float64)
        self.w = w
        self.x = inp["x"]
        self.gate = f64(inp["gate"])
        self.bias = None if inp["bias"] is None else inp["bias"].numpy()
        self.fp8 = fp8
        if fp8:
            # weights quantised once, as the GPU arm does before timing
            self.Q1 = [O.quantize_weights_fp8(f64(inp["W1"][e])) for e in range(w.E)]
            self.Q2 = [O.quantize_weights_fp8(f64(inp["W2"][e])) for e in range(w.E)]
        else:
            self.W1 = [f64(inp["W1"][e]) for e in range(w.E)]
            self.W2 = [f64(inp["W2"][e]) for e in range(w.E)]
        self._f64 = f64


def cpu_baseline(oi: OracleInputs, n_tokens: int) -> dict:
    """The oracle as it stands, one layer forward of a bounded token sample of
    the workload (its own capacity on the sample), timed on this host."""
    from oracle import moe_oracle as O

    w = oi.w
    n = min(n_tokens, w.T)
    x = oi._f64(oi.x[:n])
    t0 = time.perf_counter()
    if oi.fp8:
        r = O.route_from_logits(O.router_logits(x, oi.gate, oi.bias), w.k)
        d = O.dispatch_plan(r.idx, w.E, O.capacity(n, w.E, w.k, w.cf))
        O.token_outputs_fp8(x, r.idx, r.w, d.dest_row >= 0, oi.Q1, oi.Q2)
    else:
        O.layer_forward(x, oi.gate, oi.bias, oi.W1, oi.W2, w.k, w.cf)
    dt = time.perf_counter() - t0
    # numpy's BLAS runs the matmuls on the process's cores; the other steps
    # are single-threaded numpy
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(n / dt, 2), "unit": "tokens/s", "cores": cores,
            "threads": "BLAS matmuls on all listed cores, other oracle steps on one",
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"one oracle layer forward{' (FP8 path)' if oi.fp8 else ''} of the "
                      f"first {n} of {w.T} tokens "
                      f"(float64 numpy, capacity from the sample's own T)"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = W.get(args.workload)
    # every step is one bounded oracle sample; keep the whole run short
    n = max(16, args.cpu_tokens // max(1, args.steps + args.warmup))
    oi = OracleInputs(w, W.make_inputs(w, seed=0))
    for _ in range(args.warmup):
        cpu_baseline(oi, n)
    vals = [cpu_baseline(oi, n) for _ in range(args.steps)]
    secs = sum(v["seconds"] for v in vals)
    value = n * args.steps / secs
    cb = dict(vals[-1])
    cb["value"] = round(value, 2)
    cb["sample"] = f"{args.steps} oracle layer forwards of the first {n} of {w.T} tokens each " \
                   f"(float64 numpy, capacity from the sample's own T)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "parallelism": "host cores"},
        "cpu_baseline": cb,
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=W.WORKLOAD_ORDER + list(W.PROFILE_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=6144)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph and replayed")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 (e4m3) dispatch and expert FFN (weights quantised before timing)")
    ap.add_argument("--gumbel", type=float, default=None, metavar="TAU",
                    help="time the layer with the Gumbel training router at temperature TAU")
    args = ap.parse_args()
    if args.fp8 and args.gumbel is not None:
        ap.error("--fp8 and --gumbel are separate benchmark lines")
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
