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
import datetime
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
TRAFFIC = {"large_expert": 7.92e9}
TRAFFIC_FP8 = {"large_expert": 4.43e9}


def launches_per_step(w: W.Workload, fp8: bool) -> int:
    """Kernels one layer step launches: router, scan, gather, GEMM1, GEMM2,
    combine, plus a gate transpose unless E >= 64 is a multiple of 8 (the
    router then reads the gate as given) and the act row quantisation with
    FP8."""
    return 6 + (not (w.E >= 64 and w.E % 8 == 0)) + (1 if fp8 else 0)


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
    """nvidia-smi sampling of SM clocks, power and throttle reasons every
    50 ms for the whole run; `window(t0, t1)` summarises the samples taken
    between two host times (the timed regions start and end with a device
    synchronisation, so host time brackets them)."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.rows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # the first sample must exist before any timed region starts
        t_end = time.time() + 5.0
        while time.time() < t_end and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def settle(self):
        """Lets a sample land after a timed region ends."""
        if self.proc is not None:
            time.sleep(2.5 * self.PERIOD_MS / 1e3)

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                self.rows.append([ts] + parts[1:])
        os.unlink(self.path)
        self.proc = None

    def window(self, t0: float, t1: float):
        if not self.rows:
            return None
        rows = [r for r in self.rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        num = lambda v: v.replace(".", "", 1).isdigit()
        sm = [float(r[2]) for r in rows if num(r[2])]
        mx = [float(r[3]) for r in self.rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "period_ms": self.PERIOD_MS}


# ------------------------------------------------------------- our arm ----

class Layer:
    """One layer configuration ready to run: shape, workspace, outputs and a
    `step(events, strm)` that enqueues one whole layer forward."""

    def __init__(self, moe, w: W.Workload, d: dict, dev, fp8=False, gumbel=None, seed=1):
        self.w, self.d, self.fp8, self.gumbel = w, d, fp8, gumbel
        T, E, k = w.T, w.E, w.k
        self.s = s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
        self.ws = ws = moe.Workspace(s, device=dev, fp8=fp8)
        self.y = y = torch.empty((T, w.H), dtype=torch.bfloat16, device=dev)
        self.aux = aux = torch.zeros(1, dtype=torch.float32, device=dev)
        self.offsets = offsets = torch.zeros(E + 1, dtype=torch.int32, device=dev)
        self.dest = dest = torch.zeros((T, k), dtype=torch.int32, device=dev)
        self.status = status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.q = None
        if fp8:
            # weights are parameters: quantised once, before any timed region
            self.q = q = moe.Fp8Weights(d["W1"], d["W2"])
            torch.cuda.synchronize(dev)

            def step(events=None, strm=None):
                moe.moe_layer_fwd_fp8(s, d["x"], d["gate"], d["bias"], q, y, aux=aux,
                                      offsets=offsets, dest_row=dest, dev_status=status, ws=ws,
                                      stream=strm, events=events)
        elif gumbel is None:
            def step(events=None, strm=None):
                moe.moe_layer_fwd(s, d["x"], d["gate"], d["bias"], d["W1"], d["W2"], y,
                                  aux=aux, offsets=offsets, dest_row=dest, dev_status=status,
                                  ws=ws, stream=strm, events=events)
        else:
            # the training router: uniforms drawn once, outside the timed region
            gen = torch.Generator(device=dev).manual_seed(seed)
            noise = torch.rand((T, E), generator=gen, device=dev, dtype=torch.float32)

            def step(events=None, strm=None):
                moe.moe_layer_fwd_gumbel(s, d["x"], d["gate"], d["bias"], noise, gumbel,
                                         d["W1"], d["W2"], y, aux=aux, offsets=offsets,
                                         dest_row=dest, dev_status=status, ws=ws,
                                         stream=strm, events=events)
        self.step = step

    def input_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.d.values() if v is not None)


def time_layer(moe, L: Layer, stream, dev, steps, warmup, world, clocks=None) -> dict:
    """W untimed steps, then exactly K timed steps bracketed by a barrier and
    a device synchronisation on both sides; per-stage CUDA events on the
    launching stream. Inputs re-read every step: below 2x L2 they could stay
    cached, so then L2 is flushed between steps and each step is timed by its
    own events."""
    strm = stream
    for _ in range(warmup):
        L.step(strm=strm)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.LAYER_NUM_EVENTS)]
          for _ in range(steps)]
    for row in ev:
        for e in row:
            e.record(strm)
    in_bytes = L.input_bytes()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) \
        if in_bytes < 2 * L2_BYTES else None
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    L.status.zero_()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    h0 = time.time()
    t0.record(strm)
    for i in range(steps):
        if flush is not None:
            flush.fill_(float(i))
        L.step(ev[i], strm)
    t1.record(strm)
    torch.cuda.synchronize(dev)
    h1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    if flush is None:
        ms = t0.elapsed_time(t1) / steps
    else:
        ms = sum(ev[i][0].elapsed_time(ev[i][-1]) for i in range(steps)) / steps
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    stage_ms = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps
                for j in range(moe.LAYER_NUM_EVENTS - 1)]
    if clocks is not None:
        clocks.settle()
    l2 = (f"L2 flushed between steps ({2 * L2_BYTES >> 20} MB write); steps timed by their own "
          f"events" if flush is not None else
          f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB re-read per step); no flush")
    return {"ms": ms, "stage_ms": stage_ms, "status": int(L.status.item()),
            "n_kept": int(L.offsets[L.w.E].item()),
            "any_kept": int((L.dest >= 0).any(dim=1).sum().item()),
            "host_window": (h0, h1), "l2": l2, "steps": steps}


def run_ours(args, rank, world, local_rank):
    import top_routing_expert_gb300 as moe

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.build()
    moe.load_library()
    w = W.get(args.workload)
    inp = W.make_inputs(w, seed=rank)
    d = {kk: (v.to(dev) if v is not None else None) for kk, v in inp.items()}
    stream = torch.cuda.current_stream(dev)
    L = Layer(moe, w, d, dev, fp8=args.fp8, gumbel=args.gumbel, seed=rank + 1)
    clocks = ClockSampler(local_rank)
    clocks.start()
    m = time_layer(moe, L, stream, dev, args.steps, args.warmup, world, clocks)

    # the end-to-end leg times the inference layer; skipped for the training router
    e2e = None if (args.no_e2e or args.gumbel is not None) else \
        run_e2e(args, moe, L.s, inp, d, stream, dev, world, L.q)
    dense = None if (args.fp8 or args.gumbel is not None) else \
        run_dense_ffn(args, moe, w, d, stream, dev, m["l2"].startswith("L2 flushed"))
    graph = None
    if args.graph:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) \
            if m["l2"].startswith("L2 flushed") else None
        graph = run_graph(args, L.step, stream, dev, flush)
    extra = pipelined = None
    if world == 1 and not args.no_extra and args.workload == DEFAULT_WORKLOAD and \
            not args.fp8 and args.gumbel is None:
        extra = run_extra(args, moe, L, stream, dev, clocks)
        pipelined = run_pipelined(args, moe, L, stream, dev)
    clocks.stop()
    if rank != 0:
        return None
    line = report(args, w, world, m, clocks.window(*m["host_window"]), e2e, inp, dense)
    if graph is not None:
        line["graph_replay"] = {"ms_per_step": round(graph, 4),
                                "value": round(w.T * world / (graph / 1e3), 1), "unit": "tokens/s",
                                "what": "the same step captured once in a CUDA graph and replayed"}
    if pipelined is not None:
        line["device_pipeline"] = pipelined
    if extra is not None:
        line["per_workload"] = [
            {**kernel_report(x["w"], x["m"], x["fp8"]), "clocks": clocks.window(*x["m"]["host_window"])}
            for x in extra]
    return line


EXTRA_WORKLOADS = [("imbalanced", False), ("fine_grained", False), ("many_expert", False),
                   ("large_expert", True)]
# micro-batches of the on-device two-stream pipeline (each of the workload's T)
PIPELINED = [("fine_grained", 4), ("large_expert", 2)]


def run_extra(args, moe, headline: Layer, stream, dev, clocks):
    """The other layer configurations, timed like the headline after it (a
    few steps each): the skewed, the fine-grained and the many-expert layer
    in bf16 (inputs drawn on the device with the same distributions), and
    the headline layer again with the FP8 dispatch, FFN and combine."""
    out = []
    steps = max(3, min(args.steps, 20))
    for name, fp8 in EXTRA_WORKLOADS:
        w = W.get(name)
        if name == headline.w.name:
            d = headline.d
        else:
            d = W.make_inputs_on_device(w, dev, seed=11)
        L = Layer(moe, w, d, dev, fp8=fp8)
        m = time_layer(moe, L, stream, dev, steps, args.warmup, 1, clocks)
        out.append({"w": w, "m": m, "fp8": fp8})
        del L, d
        torch.cuda.empty_cache()
    return out


def run_pipelined(args, moe, headline: Layer, stream, dev):
    """The dual-stream micro-batch pipeline on the device (the comm
    bottleneck page's section 5.2 overlap, with the on-device dispatch and
    combine in the role of the all-to-alls): n micro-batches of the
    workload's T tokens through moe_layer_fwd_pipelined, against the same n
    micro-batches as back-to-back moe_layer_fwd calls. Each is timed from
    before the first kernel to after the last, a few repetitions."""
    out = []
    reps = max(2, min(args.steps, 5))
    for name, n in PIPELINED:
        w = W.get(name)
        d = headline.d if name == headline.w.name else W.make_inputs_on_device(w, dev, seed=11)
        s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
        x_all = d["x"].repeat(n, 1).contiguous()
        y_all = torch.empty_like(x_all)
        pipe = moe.DevicePipeline(s, device=dev)
        L = Layer(moe, w, d, dev)

        def pipelined():
            pipe.run(n, x_all, d["gate"], d["bias"], d["W1"], d["W2"], y_all)
            stream.wait_stream(pipe.streams[0])

        def sequential():
            for i in range(n):
                moe.moe_layer_fwd(s, x_all[i * w.T:(i + 1) * w.T], d["gate"], d["bias"], d["W1"],
                                  d["W2"], y_all[i * w.T:(i + 1) * w.T], ws=L.ws, stream=stream)

        res = {}
        for key, fn in (("sequential", sequential), ("pipelined", pipelined)):
            for _ in range(2):
                fn()
            torch.cuda.synchronize(dev)
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(reps):
                fn()
            t1.record(stream)
            torch.cuda.synchronize(dev)
            res[key] = t0.elapsed_time(t1) / (reps * n)
        out.append({"workload": name, "n_micro": n, "tokens_per_micro_batch": w.T,
                    "ms_per_micro_batch": round(res["pipelined"], 4),
                    "sequential_ms_per_micro_batch": round(res["sequential"], 4),
                    "speedup": round(res["sequential"] / res["pipelined"], 4),
                    "value": round(w.T / (res["pipelined"] / 1e3), 1), "unit": "tokens/s"})
        del pipe, L, x_all, y_all, d
        torch.cuda.empty_cache()
    return out


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


def run_e2e(args, moe, s, inp, d, stream, dev, world, q=None):
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


def kernel_report(w: W.Workload, m: dict, fp8: bool) -> dict:
    """Per-kernel times (from the layer's stage events) against their
    rooflines, and the grouped GEMM (GEMM1 + GEMM2) against the measured
    dense bf16 peak: the burst figure, since every timed region here is
    well under a second of back-to-back steps (the sustained figure, for
    seconds-long runs at the power cap, is given beside it)."""
    pk = peaks()
    work = algorithmic_work(w, m["n_kept"], m["any_kept"], fp8=fp8)
    names = ["route", "scan", "permute", "gemm1", "gemm2", "combine"]
    stage = dict(zip(names, m["stage_ms"]))
    kern = {}
    for nm, key, unit in [("route", "route_bytes", "GB/s"), ("permute", "permute_bytes", "GB/s"),
                          ("combine", "combine_bytes", "GB/s"), ("gemm1", "gemm1_flop", "TFLOP/s"),
                          ("gemm2", "gemm2_flop", "TFLOP/s")]:
        sec = max(stage[nm], 1e-6) / 1e3
        if unit == "GB/s":
            a = work[key] / sec / 1e9
            kern[nm] = {"ms": round(stage[nm], 4), "achieved": round(a, 1), "unit": unit,
                        "frac_of_measured_hbm": round(a / pk["hbm_gbs"], 3)}
        else:
            a = work[key] / sec / 1e12
            peak = pk["bf16_tflops"] * (2 if fp8 else 1)
            kern[nm] = {"ms": round(stage[nm], 4), "achieved": round(a, 1), "unit": unit,
                        "frac_of_measured_peak": round(a / peak, 3)}
    kern["scan"] = {"ms": round(stage["scan"], 4)}
    if fp8:
        kern["gemm1"]["includes"] = "GEMM1 + act row quantisation"
    gemm_ms = stage["gemm1"] + stage["gemm2"]
    gemm_tf = (work["gemm1_flop"] + work["gemm2_flop"]) / (max(gemm_ms, 1e-6) / 1e3) / 1e12
    burst, sustained = pk["bf16_tflops"], pk["bf16_tflops_sustained"] or pk["bf16_tflops"]
    kind = f"{pk['source']} bf16 burst (cuBLAS, best of 10)"
    if fp8:
        # e4m3 runs at twice the bf16 tensor rate (nominal 4.5 vs 2.25 PFLOP/s dense)
        burst, sustained = 2 * burst, 2 * sustained
        kind = f"{pk['source']} bf16 burst x 2 (nominal e4m3/bf16 ratio)"
    roofline = {"kernel": "grouped GEMM (expert FFN GEMM1+GELU and GEMM2 launches)",
                "bound": "tensor", "achieved": round(gemm_tf, 1), "peak": burst,
                "unit": "TFLOP/s", "frac": round(gemm_tf / burst, 4), "peak_kind": kind,
                "frac_of_sustained": round(gemm_tf / sustained, 4),
                "traffic": (TRAFFIC_FP8 if fp8 else TRAFFIC).get(w.name)}
    return {"workload": w.name, "dtype": "e4m3 (fp32 accumulate)" if fp8 else "bf16",
            "config": w.describe(), "ms_per_step": round(m["ms"], 4), "steps": m["steps"],
            "value": round(w.T / (m["ms"] / 1e3), 1), "unit": "tokens/s",
            "roofline": roofline, "kernels": kern, "l2": m["l2"],
            "routing": {"kept_rows": m["n_kept"], "assignments": w.T * w.k,
                        "dropped": w.T * w.k - m["n_kept"], "dev_status": m["status"]}}


def report(args, w, world, m, clk, e2e, inp, dense=None):
    T = w.T
    kr = kernel_report(w, m, args.fp8)
    ms = m["ms"]
    tokens = T * world
    line = {
        "metric": METRIC, "value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": kr["dtype"], "data": "synthetic",
        "config": {**w.describe(), "parallelism": f"replicas x{world} (no exchange)",
                   "router": "inference (top-k of logits)" if args.gumbel is None
                   else f"training (Gumbel noise, temperature {args.gumbel})",
                   "expert_ffn": "FP8 e4m3 dispatch + FFN + combine, per-row/per-column/"
                                 "128-column-block fp32 scales"
                   if args.fp8 else "bf16",
                   "l2": m["l2"]},
        "clocks": clk,
        "e2e": None if e2e is None else {
            "value": round(tokens / (e2e["ms"] / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(e2e["ms"], 4), "h2d_bytes_per_step": e2e["h2d"],
            "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": launches_per_step(w, args.fp8) * args.steps,
        "roofline": kr["roofline"],
        "kernels": kr["kernels"],
        "routing": kr["routing"],
    }
    if dense is not None:
        line["moe_vs_dense_ffn"] = {
            "dense_ffn_ms": round(dense, 4), "ratio": round(ms / dense, 3),
            "what": "layer time / one dense FFN (h) over the same T tokens, same kernels, E=1",
            "ideal_from_flops": round(m["n_kept"] / T, 3)}
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(OracleInputs(w, inp, fp8=args.fp8), args.cpu_tokens)
        if not args.fp8:
            line["cpu_baseline_one_core"] = cpu_baseline_one_core(w, max(64, args.cpu_tokens // 12))
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


def cpu_baseline_one_core(w: W.Workload, n_tokens: int) -> dict:
    """The oracle on ONE host core: a child process with single-threaded
    BLAS pinned to one core runs one oracle layer forward of n tokens drawn
    with the workload's recipe (its own inputs: n tokens, the full expert
    weights)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-core",
                            w.name, str(n_tokens)], env=env, capture_output=True, text=True,
                           timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.TimeoutExpired, ValueError, IndexError) as e:
        return {"unavailable": f"one-core oracle run failed: {type(e).__name__}"}


def oracle_one_core_child(name: str, n: int):
    from oracle import moe_oracle as O
    import numpy as np
    w = W.get(name)
    ws = W.custom(n, w.H, w.E, w.k, w.h, w.cf, w.bias, name=f"{name}_sample")
    inp = W.make_inputs(ws, seed=0)
    f64 = lambda t: t.float().numpy().astype(np.float64)
    x, gate = f64(inp["x"]), f64(inp["gate"])
    bias = None if inp["bias"] is None else inp["bias"].numpy()
    W1 = [f64(inp["W1"][e]) for e in range(w.E)]
    W2 = [f64(inp["W2"][e]) for e in range(w.E)]
    core = min(os.sched_getaffinity(0))
    os.sched_setaffinity(0, {core})
    t0 = time.perf_counter()
    O.layer_forward(x, gate, bias, W1, W2, w.k, w.cf)
    dt = time.perf_counter() - t0
    print(json.dumps({"value": round(n / dt, 2), "unit": "tokens/s", "cores": 1,
                      "kind": "oracle", "seconds": round(dt, 3),
                      "sample": f"one oracle layer forward of {n} tokens drawn with the {name} "
                                f"recipe (float64 numpy, BLAS single-threaded, pinned to one "
                                f"core, capacity from the sample's own T)"}))


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
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload lines after the headline")
    ap.add_argument("--oracle-one-core", nargs=2, metavar=("WORKLOAD", "TOKENS"),
                    help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_one_core:
        oracle_one_core_child(args.oracle_one_core[0], int(args.oracle_one_core[1]))
        return
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
