"""Benchmark of the decode hot path (dq_gemm + gqa_decode_attn) on GB300.

One step = every call of the workload once. The default workload is the
long-context step of the 70B fixture: paged GQA attention (64 q / 8 KV heads)
over 8 sequences of 131072 tokens (4 GiB of bf16 KV) plus the four 70B
projections (QKV, O, gate+up, down) at M = 8 in FP8-E4M3 and in INT4 g128.
Weights and KV are resident in HBM; every step reads them once. The other
workloads (the tiny case, the 8B layer at batch 1, the 70B layer at batch 32,
speculative verify, and the FP8-cache steps) are measured after it, one at a
time, and reported as sub-records of the same JSON line.

Metric: effective HBM GB/s = algorithmic bytes of the step (weights with their
scales/zeros, activations, outputs, K/V, q, block table) / step time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--no-subrecords]
Under torchrun (N > 1) every rank runs an independent replica of the chosen
workload (the path has no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from memory_bound_decode_dq_gb300 import bounds, configs, synth  # noqa: E402

WTYPE_NAMES = configs.WTYPE_NAMES
DEFAULT_WORKLOAD = "longctx_70b_b8"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=[w.__name__ for w in configs.ALL])
    p.add_argument("--graph-steps", type=int, default=50, help="steps unrolled per CUDA graph")
    p.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps (capped at 2000)")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-call-protocol", action="store_true",
                   help="skip the per-call graph protocol (50 back-to-back calls, L2-cold copies)")
    p.add_argument("--no-subrecords", action="store_true",
                   help="measure the chosen workload only (no sub-records of the other workloads)")
    p.add_argument("--min-load-s", type=float, default=1.5,
                   help="repeat the K-step timed run until about this much load has passed")
    p.add_argument("--sub-min-load-s", type=float, default=0.3, help="the same for each sub-record")
    return p.parse_args()


def workload(name):
    return {w.__name__: w for w in configs.ALL}[name]()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def csrc_hash() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "memory_bound_decode_dq_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms for the
    whole run; window() summarises the samples taken inside a wall-clock
    interval (a timed region, or one call's replays)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None
        self.lock = threading.Lock()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) >= 10:
                with self.lock:
                    self.lines.append((time.time(), parts))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def window(self, t0, t1, brief=False):
        """Median SM clock, the largest maximum clock, the throttle reasons
        seen and the sample count over [t0, t1] (wall clock)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)  # let the reader thread take the samples of the interval's end
        with self.lock:
            use = [p for ts, p in self.lines if t0 - 0.06 <= ts <= t1 + 0.06]
        sm = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for p in use if p[3].replace(".", "").isdigit()]
        reasons = sorted({name for p in use for name, val in zip(self.REASONS, p[6:10])
                          if val.strip().lower() == "active"})
        d = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
             "reasons": reasons, "samples": len(use)}
        if not brief:
            d["samples_in_timed_region"] = len(use)
            d["sm_mhz_min"] = min(sm) if sm else None
        return d

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()


# ------------------------------------------------------- device workload ----

class Call:
    def __init__(self, name, kind, nbytes, flops, fn, launches, clone=None):
        self.name, self.kind, self.nbytes, self.flops, self.fn, self.launches = name, kind, nbytes, flops, fn, launches
        # clone() -> a call of the same shape on fresh copies of the resident
        # operands (weights, KV pools) and the same small inputs and outputs
        self.clone = clone


def build_calls(wl, dev, dqd):
    """Inputs drawn on the device, outputs and workspaces preallocated; returns
    the calls of one step and the host-visible inputs/outputs for e2e."""
    import torch
    calls = []
    io = []  # (name, device input tensors, device output tensors)
    for c in wl.gemms:
        seed = wl.seed
        x = synth.normal_bf16(seed, c.name + ".x", (c.m, c.k), device=dev)
        if c.wtype == configs.W_INT4_G128:
            wq = synth.int4_weight(seed, c.name, c.n, c.k, device=dev)
            weight = dqd.Weight.int4(dqd.pack_int4_g128(wq.codes, wq.scales, wq.zeros))
            del wq
        else:
            if c.outliers:
                w = synth.bf16_weight_outliers_device(seed, c.name, c.n, c.k, 0.02, c.outliers, 20.0, dev)
            else:
                w = synth.normal_bf16(seed, c.name, (c.n, c.k), 0.02, device=dev)
            if c.wtype == configs.W_BF16:
                weight = dqd.Weight.bf16(w)
            else:
                codes, scales = dqd.quant_fp8_rowwise(w)
                weight = dqd.Weight.fp8(codes, scales)
                del w
        y = torch.empty((c.m, c.n), dtype=torch.bfloat16, device=dev)
        need = dqd.dq_gemm_workspace_bytes(weight, c.m)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev) if need else None

        def fn(weight=weight, x=x, y=y, ws=ws):
            dqd.dq_gemm(weight, x, y=y, ws=ws)

        def clone(weight=weight, x=x, y=y, ws=ws):
            wc = dqd.Weight(weight.type, weight.n, weight.k, weight.data.clone(),
                            None if weight.scales is None else weight.scales.clone(),
                            None if weight.zeros is None else weight.zeros.clone())
            return lambda: dqd.dq_gemm(wc, x, y=y, ws=ws)
        calls.append(Call(c.name, "dq_gemm", bounds.dq_gemm_bytes(c.wtype, c.m, c.n, c.k),
                          bounds.dq_gemm_flops(c.m, c.n, c.k), fn, 1, clone))
        io.append((c.name, [x], [y]))
    for a in wl.attns:
        seed = wl.seed
        ctx = list(a.context)
        table, nblk = synth.block_table(seed, a.name + ".table", ctx, a.shuffle)
        shape = (nblk, a.hkv, 16, a.d)
        if a.kv_fp8:
            kp = synth.e4m3_codes(seed, a.name + ".k", shape, device=dev)
            vp = synth.e4m3_codes(seed, a.name + ".v", shape, device=dev)
        else:
            kp = synth.normal_bf16(seed, a.name + ".k", shape, 1.0, device=dev)
            vp = synth.normal_bf16(seed, a.name + ".v", shape, 1.0, device=dev)
        q = synth.normal_bf16(seed, a.name + ".q", (a.batch, a.width, a.hq, a.d), device=dev)
        table_t = torch.from_numpy(table).to(dev)
        ctx_t = torch.tensor(ctx, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        maxc = max(ctx)
        if a.kv_fp8:
            need = dqd.gqa_decode_attn_fp8kv_workspace_bytes(a.batch, a.width, a.hq, a.hkv, a.d, maxc)
        else:
            need = dqd.gqa_decode_attn_workspace_bytes(a.batch, a.width, a.hq, a.hkv, a.d, maxc)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev) if need else None

        def attn_call(kp, vp, q=q, table_t=table_t, ctx_t=ctx_t, out=out, ws=ws, maxc=maxc, a=a):
            if a.kv_fp8:
                return lambda: dqd.gqa_decode_attn_fp8kv(q, kp, vp, table_t, ctx_t, maxc, a.k_scale, a.v_scale,
                                                         out=out, ws=ws)
            return lambda: dqd.gqa_decode_attn(q, kp, vp, table_t, ctx_t, maxc, out=out, ws=ws)

        def clone(kp=kp, vp=vp, attn_call=attn_call):
            return attn_call(kp.clone(), vp.clone())
        calls.append(Call(a.name, "gqa_decode_attn_fp8kv" if a.kv_fp8 else "gqa_decode_attn",
                          bounds.attn_bytes(ctx, a.width, a.hq, a.hkv, a.d,
                                            kv_bytes_per_element=1 if a.kv_fp8 else 2),
                          bounds.attn_flops(ctx, a.width, a.hq, a.d), attn_call(kp, vp), 2 if need else 1, clone))
        io.append((a.name, [q, table_t, ctx_t], [out]))
    for rc in getattr(wl, "ropes", ()):
        ctx = list(rc.context)
        table, nblk = synth.block_table(wl.seed, rc.name + ".table", ctx, True)
        rows = rc.batch * rc.width
        qkv = synth.normal_bf16(wl.seed, rc.name + ".qkv", (rows, (rc.hq + 2 * rc.hkv) * rc.d), device=dev)
        kp = torch.zeros((nblk, rc.hkv, 16, rc.d), dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        table_t = torch.from_numpy(table).to(dev)
        ctx_t = torch.tensor(ctx, dtype=torch.int32, device=dev)
        q_out = torch.empty((rc.batch, rc.width, rc.hq, rc.d), dtype=torch.bfloat16, device=dev)

        def rope_call(x, kp=kp, vp=vp, table_t=table_t, ctx_t=ctx_t, q_out=q_out, rc=rc):
            return lambda: dqd.rope_kv_append(x, rc.batch, rc.width, rc.hq, rc.hkv, kp, vp, table_t, ctx_t,
                                              rope_base=rc.rope_base, q_out=q_out)

        def rclone(x=qkv, rope_call=rope_call):
            return rope_call(x.clone())
        calls.append(Call(rc.name, "rope_kv_append", bounds.rope_append_bytes(rows, rc.hq, rc.hkv, rc.d), 0.0,
                          rope_call(qkv), 1, rclone))
        io.append((rc.name, [qkv, table_t, ctx_t], [q_out]))
    for qc in getattr(wl, "qkv_ropes", ()):
        seed = wl.seed
        ctx = list(qc.context)
        table, nblk = synth.block_table(seed, qc.name + ".table", ctx, True)
        rows, n = qc.batch * qc.width, (qc.hq + 2 * qc.hkv) * qc.d
        x = synth.normal_bf16(seed, qc.name + ".x", (rows, qc.k), device=dev)
        if qc.wtype == configs.W_INT4_G128:
            wq = synth.int4_weight(seed, qc.name, n, qc.k, device=dev)
            weight = dqd.Weight.int4(dqd.pack_int4_g128(wq.codes, wq.scales, wq.zeros))
            del wq
        else:
            weight = dqd.Weight.bf16(synth.normal_bf16(seed, qc.name, (n, qc.k), 0.02, device=dev))
        kp = torch.zeros((nblk, qc.hkv, 16, qc.d), dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        table_t = torch.from_numpy(table).to(dev)
        ctx_t = torch.tensor(ctx, dtype=torch.int32, device=dev)
        q_out = torch.empty((qc.batch, qc.width, qc.hq, qc.d), dtype=torch.bfloat16, device=dev)
        need = dqd.dq_gemm_workspace_bytes(weight, rows)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev) if need else None

        def qkv_call(weight, x=x, kp=kp, vp=vp, table_t=table_t, ctx_t=ctx_t, q_out=q_out, ws=ws, qc=qc):
            return lambda: dqd.dq_gemm_qkv_rope_append(weight, x, qc.batch, qc.width, qc.hq, qc.hkv, kp, vp,
                                                       table_t, ctx_t, rope_base=qc.rope_base, q_out=q_out, ws=ws)

        def qclone(weight=weight, qkv_call=qkv_call):
            return qkv_call(dqd.Weight(weight.type, weight.n, weight.k, weight.data.clone(),
                                       None if weight.scales is None else weight.scales.clone(),
                                       None if weight.zeros is None else weight.zeros.clone()))
        calls.append(Call(qc.name, "dq_gemm_qkv_rope_append",
                          bounds.qkv_rope_append_bytes(qc.wtype, rows, qc.k, qc.hq, qc.hkv, qc.d),
                          bounds.dq_gemm_flops(rows, n, qc.k), qkv_call(weight), 1, qclone))
        io.append((qc.name, [x, table_t, ctx_t], [q_out]))
    for v in getattr(wl, "verifies", ()):
        import numpy as np
        logits = synth.normal_bf16(wl.seed, v.name + ".logits", (v.batch, v.width, v.vocab), device=dev)
        draft = torch.from_numpy(synth.rng(wl.seed, v.name + ".draft").integers(
            0, v.vocab, (v.batch, v.width - 1)).astype(np.int32)).to(dev)
        ctx_v = torch.full((v.batch,), 1 << 30, dtype=torch.int32, device=dev)  # updated in place
        vout = torch.empty((v.batch, v.width), dtype=torch.int32, device=dev)
        vcnt = torch.empty((v.batch,), dtype=torch.int32, device=dev)

        def verify_call(lg, draft=draft, ctx_v=ctx_v, vout=vout, vcnt=vcnt):
            return lambda: dqd.spec_verify_greedy(lg, draft, ctx_v, out=vout, count=vcnt)

        def vclone(lg=logits, verify_call=verify_call):
            return verify_call(lg.clone())
        calls.append(Call(v.name, "spec_verify_greedy", bounds.verify_bytes(v.batch, v.width, v.vocab), 0.0,
                          verify_call(logits), 2, vclone))
        io.append((v.name, [logits, draft], [vout, vcnt]))
    return calls, io


def working_set_bytes(calls):
    return sum(c.nbytes for c in calls)


def _graph(calls, dev, nsteps, with_events=False):
    """A CUDA graph of nsteps steps (every call once per step); with_events
    puts a timing event on either side of every call."""
    import torch
    evs = []
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in calls:
            c.fn()
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        for _ in range(nsteps):
            row = []
            for c in calls:
                if with_events:
                    e0 = torch.cuda.Event(enable_timing=True, external=True)
                    e1 = torch.cuda.Event(enable_timing=True, external=True)
                    e0.record()
                    c.fn()
                    e1.record()
                    row.append((e0, e1))
                else:
                    c.fn()
            evs.append(row)
    return g, evs


def timed_steps(calls, dev, K, graph_steps, world, min_load_s, max_runs=5000):
    """The timed region: exactly K steps, replayed from plain CUDA graphs of
    up to graph_steps unrolled steps (kernels back to back, so a kernel may
    overlap the tail of the one before it, as in a decode loop), bracketed by
    a barrier and a synchronise on both sides and timed with CUDA events on
    the replay stream. The K-step run is repeated until about min_load_s of
    load has passed (at least 5 runs); ms_per_step is the median run."""
    import torch
    import torch.distributed as dist
    G = max(1, min(graph_steps, K))
    full, rem = divmod(K, G)
    graph = _graph(calls, dev, G)[0]
    graph_rem = _graph(calls, dev, rem)[0] if rem else None
    for _ in range(2):
        graph.replay()
        if graph_rem is not None:
            graph_rem.replay()
    torch.cuda.synchronize()

    def one_run():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(full):
            graph.replay()
        if graph_rem is not None:
            graph_rem.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        if world > 1:
            dist.barrier()
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    first = one_run()
    runs = max(5, min(max_runs, math.ceil(min_load_s * 1e3 / max(first, 1e-3))))
    if world > 1:  # every rank runs the same number of timed runs
        t = torch.tensor([runs], dtype=torch.int64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        runs = int(t.item())
    wall0 = time.time()
    ms = [one_run() for _ in range(runs)]
    wall1 = time.time()
    del graph, graph_rem
    qs = sorted(ms)
    return {"K": K, "graph_steps": G, "runs": runs, "run_ms": ms,
            "ms_per_step": statistics.median(ms) / K,
            "min_ms_per_step": qs[0] / K, "max_ms_per_step": qs[-1] / K,
            "p10_ms_per_step": qs[int(0.1 * (len(qs) - 1))] / K, "p90_ms_per_step": qs[int(0.9 * (len(qs) - 1))] / K,
            "wall": (wall0, wall1)}


def evented_pass(calls, dev, K, graph_steps):
    """Per-call device durations inside the step, from a separate pass after
    the timed region: one graph of the step with a timing event on either side
    of every call (the events break the overlap between consecutive kernels,
    so each duration carries its kernel's launch and drain)."""
    import torch
    G = max(1, min(graph_steps, K))
    try:
        g, events = _graph(calls, dev, G, with_events=True)
    except Exception:
        return {}, None
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    per_call = {}
    for i, c in enumerate(calls):
        d = [events[s][i][0].elapsed_time(events[s][i][1]) for s in range(G)]
        per_call[c.name] = sum(d) / len(d)
    return per_call, e0.elapsed_time(e1) / G


def measure_workload(name, args, rank, world, dev, dqd, sampler, min_load_s, e2e=True, protocol=True):
    """Build one workload, warm it up, time it (timed_steps), then the evented
    pass, the end-to-end step through the binding and each call alone."""
    import torch
    wl = workload(name)
    calls, io = build_calls(wl, dev, dqd)
    step_bytes = sum(c.nbytes for c in calls)
    launches_per_step = sum(c.launches for c in calls)
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 3)):  # eager warm-up steps (also sets kernel attributes before capture)
        for c in calls:
            c.fn()
    torch.cuda.synchronize()
    sampler.mark("begin")
    tm = timed_steps(calls, dev, args.steps, args.graph_steps, world, min_load_s)
    sampler.mark("end")
    per_call, evented_ms = evented_pass(calls, dev, args.steps, args.graph_steps)
    res = dict(wl=wl, calls=calls, step_bytes=step_bytes, launches=launches_per_step, timing=tm,
               per_call=per_call, evented_ms=evented_ms, clocks=sampler.window(*tm["wall"]))
    res["e2e"] = run_e2e(args, calls, io, dev, dqd, step_bytes, world) if e2e else None
    res["proto"] = call_protocol(calls, dev, sampler) if protocol else {}
    return res


def call_protocol(calls, dev, sampler=None, n_calls=50, min_reps=7, min_s=0.25):
    """Per-call device time, each call on its own: n_calls back-to-back calls
    captured in a CUDA graph, rotating through copies of the resident operands
    so that the copies span at least 4x the L2 (cold lines every call); the
    graph is replayed at least min_reps times and for at least min_s seconds,
    each replay timed with CUDA events; the clocks sampled over those replays
    go with the record. Also the latency of one call launched alone (events
    around a single eager call)."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20))
    out = {}
    for c in calls:
        copies = max(1, min(64, math.ceil(4 * l2 / max(c.nbytes, 1)), int((8 << 30) // max(c.nbytes, 1))))
        fns = [c.fn] + [c.clone() for _ in range(copies - 1)] if c.clone else [c.fn]
        n = max(n_calls, len(fns))
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for f in fns:
                f()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                fns[i % len(fns)]()
        g.replay()
        torch.cuda.synchronize()
        times = []
        w0 = time.time()
        while len(times) < min_reps or (time.time() - w0 < min_s and len(times) < 10000):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / n)
        w1 = time.time()
        single = []
        for _ in range(10):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            c.fn()
            e1.record()
            torch.cuda.synchronize()
            single.append(e0.elapsed_time(e1) * 1e3)
        out[c.name] = {"median": statistics.median(times), "min": min(times), "copies": len(fns), "calls": n,
                       "replays": len(times), "single": statistics.median(single),
                       "clocks": sampler.window(w0, w1, brief=True) if sampler is not None else None}
        del g, fns
        torch.cuda.empty_cache()
    return out


def run_e2e(args, calls, io, dev, dqd, step_bytes, world):
    """End to end through the public API, every step: copy the step's inputs
    (activations, queries, block table, context lengths) from pinned host
    memory, make every call through the Python binding and the C ABI
    (argument checks, planning and launch on each call), copy every output
    back to pinned host memory and synchronise; timed on the host clock.
    Weights and KV stay resident: they are model and cache state, not per-step
    inputs. The inputs and outputs live in one buffer per dtype, as an
    engine's step buffers would, so each direction is one copy per dtype.

    The same step captured once as a CUDA graph (its copies from and to the
    pinned host buffers are nodes of the graph, so every replay moves that
    step's bytes), replayed and synchronised per step, is reported beside it
    under "graph": the host work of the binding is then paid once, at capture."""
    import torch
    import torch.distributed as dist

    def arenas(tensors):
        """Re-points the given device tensors (their contents kept) into one
        contiguous device buffer per dtype; returns (device buffer, pinned host
        twin holding the same bytes) pairs."""
        by_dtype = {}
        for t in tensors:
            by_dtype.setdefault(t.dtype, []).append(t)
        pairs = []
        for dt, ts in by_dtype.items():
            n = sum(t.numel() for t in ts)
            dbuf = torch.empty(n, dtype=dt, device=dev)
            hbuf = torch.empty(n, dtype=dt, pin_memory=True)
            off = 0
            for t in ts:
                if not t.is_contiguous():
                    raise ValueError("e2e inputs and outputs must be contiguous")
                k = t.numel()
                dbuf[off:off + k].copy_(t.reshape(-1))
                t.set_(dbuf.untyped_storage(), off, t.shape, t.stride())
                off += k
            hbuf.copy_(dbuf)
            pairs.append((dbuf, hbuf))
        torch.cuda.synchronize()
        return pairs

    in_pairs = arenas([t for _, ins, _ in io for t in ins])
    out_pairs = arenas([t for _, _, outs in io for t in outs])
    h2d = sum(d.numel() * d.element_size() for d, _ in in_pairs)
    d2h = sum(d.numel() * d.element_size() for d, _ in out_pairs)
    steps = args.e2e_steps or min(args.steps, 2000)

    def issue():
        for d, h in in_pairs:
            d.copy_(h, non_blocking=True)
        for c in calls:
            c.fn()
        for d, h in out_pairs:
            h.copy_(d, non_blocking=True)

    def one_step_eager():
        issue()
        torch.cuda.current_stream().synchronize()

    graph = None
    try:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            issue()
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            issue()
    except Exception:
        graph = None

    def one_step_graph():
        graph.replay()
        torch.cuda.current_stream().synchronize()

    def timed(step_fn, n):
        for _ in range(3):
            step_fn()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            step_fn()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        t = torch.tensor([dt], dtype=torch.float64, device=dev)
        if world > 1:
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    dt = timed(one_step_eager, steps)
    out = {"value": round(step_bytes * steps * world / dt / 1e9, 3), "unit": "GB/s",
           "ms_per_step": round(1e3 * dt / steps, 4), "steps": steps,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "mode": ("eager: every step copies its inputs from pinned host memory, makes every call through "
                    "the Python binding and the C ABI, copies its outputs back and synchronises")}
    if graph is not None:
        dtg = timed(one_step_graph, steps)
        out["graph"] = {"value": round(step_bytes * steps * world / dtg / 1e9, 3), "unit": "GB/s",
                        "ms_per_step": round(1e3 * dtg / steps, 4), "steps": steps,
                        "mode": "the same step captured once as a CUDA graph (copies included), replayed per step"}
    return out


# ------------------------------------------------------------ CPU oracle ----

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: every call is
    evaluated on a random subset of its output rows (same shapes and
    distributions), the subset sized so that one run costs about budget_s
    seconds. Inputs are drawn once; run() times only the oracle calls."""

    def __init__(self, wl, budget_s, seed=1234):
        import numpy as np

        import oracle
        oracle.build()
        self.oracle = oracle
        rng = np.random.default_rng(seed)
        costs = [c.m * c.n * c.k for c in wl.gemms] + \
                [sum(a.context) * a.width * a.hq * a.d * 2 for a in wl.attns] + \
                [v.batch * v.width * v.vocab for v in getattr(wl, "verifies", ())] + \
                [200 * r.batch * r.width * (r.hq + 2 * r.hkv) * r.d for r in getattr(wl, "ropes", ())] + \
                [r.batch * r.width * (r.hq + 2 * r.hkv) * r.d * r.k for r in getattr(wl, "qkv_ropes", ())]
        rate = 1.5e8 * max(1, oracle.num_threads())  # oracle multiply-adds per second, roughly
        self.frac = frac = min(1.0, budget_s * rate / float(sum(costs)))
        self.jobs, self.covered = [], 0.0
        for c in wl.gemms:
            rows = max(1, int(round(c.n * frac)))
            x = synth.normal_bf16(wl.seed, c.name + ".x", (c.m, c.k))
            if c.wtype == configs.W_INT4_G128:
                args = (rng.integers(0, 16, (rows, c.k), dtype=np.uint8),
                        synth.uniform_bf16(wl.seed, c.name + ".s", (rows, c.k // 128), 0.005, 0.02),
                        rng.integers(0, 16, (rows, c.k // 128), dtype=np.uint8))
            else:
                w = synth.f32_to_bf16_bits(rng.standard_normal((rows, c.k), dtype=np.float32) * 0.02)
                args = (w, None, None) if c.wtype == configs.W_BF16 else oracle.quant_fp8_rowwise(w) + (None,)
            self.jobs.append(lambda c=c, args=args, x=x: oracle.dq_gemm(c.wtype, *args, x))
            self.covered += bounds.dq_gemm_bytes(c.wtype, c.m, c.n, c.k) * rows / c.n
        for a in wl.attns:
            # one (sequence, kv head) group: its heads at every verify position
            G = a.hq // a.hkv
            b = int(rng.integers(0, a.batch))
            ctx = [a.context[b]]
            if a.kv_fp8:
                kv = synth.paged_kv_fp8(seed, a.name + ".cpu", ctx, 1, a.d, shuffle=a.shuffle)
            else:
                kv = synth.paged_kv(seed, a.name + ".cpu", ctx, 1, a.d, shuffle=a.shuffle)
            q = synth.normal_bf16(seed, a.name + ".cpu.q", (1, a.width, G, a.d))
            rows_all = a.batch * a.width * a.hq
            want = max(1, int(round(rows_all * frac)))
            # cost of a row in this group relative to an average row
            rel = a.context[b] / (sum(a.context) / a.batch)
            nrows = max(1, min(a.width * G, int(round(want / max(rel, 1e-9)))))
            pick = np.sort(rng.choice(a.width * G, nrows, replace=False))
            if a.kv_fp8:
                self.jobs.append(lambda kv=kv, q=q, pick=pick, a=a: oracle.gqa_decode_attn_fp8kv(
                    q, kv.k_codes, kv.v_codes, kv.block_table, kv.context_lens, 1, 1 / math.sqrt(a.d),
                    a.k_scale, a.v_scale, rows=pick))
            else:
                self.jobs.append(lambda kv=kv, q=q, pick=pick, d=a.d: oracle.gqa_decode_attn(
                    q, kv.k_pool, kv.v_pool, kv.block_table, kv.context_lens, 1, 1 / math.sqrt(d), rows=pick))
            per_row = bounds.attn_bytes(a.context, a.width, a.hq, a.hkv, a.d,
                                        kv_bytes_per_element=1 if a.kv_fp8 else 2) / rows_all
            self.covered += per_row * rel * nrows
        for rc in getattr(wl, "ropes", ()):
            ntok = max(1, int(round(rc.batch * rc.width * frac)))
            ctx_s = np.asarray(rc.context[:1], np.int32)
            tbl, nb = synth.block_table(seed, rc.name + ".cpu.table", ctx_s)
            qkv = synth.normal_bf16(seed, rc.name + ".cpu", (ntok, (rc.hq + 2 * rc.hkv) * rc.d))
            self.jobs.append(lambda qkv=qkv, ntok=ntok, rc=rc, ctx_s=ctx_s, tbl=tbl, nb=nb: oracle.rope_kv_append(
                qkv, 1, ntok, rc.hq, rc.hkv, rc.rope_base, np.maximum(ctx_s, ntok), tbl, nb))
            self.covered += bounds.rope_append_bytes(ntok, rc.hq, rc.hkv, rc.d)
        for qc in getattr(wl, "qkv_ropes", ()):
            # the projection on a random subset of its output rows, then the
            # rotation of the whole q and k heads those rows fall in
            n = (qc.hq + 2 * qc.hkv) * qc.d
            heads = max(1, int(round((qc.hq + 2 * qc.hkv) * frac)))
            rows = heads * qc.d
            tokens = qc.batch * qc.width
            x = synth.normal_bf16(wl.seed, qc.name + ".x", (tokens, qc.k))
            if qc.wtype == configs.W_INT4_G128:
                args = (rng.integers(0, 16, (rows, qc.k), dtype=np.uint8),
                        synth.uniform_bf16(wl.seed, qc.name + ".s", (rows, qc.k // 128), 0.005, 0.02),
                        rng.integers(0, 16, (rows, qc.k // 128), dtype=np.uint8))
            else:
                args = (synth.f32_to_bf16_bits(rng.standard_normal((rows, qc.k), dtype=np.float32) * 0.02),
                        None, None)
            pos = np.repeat(np.asarray([c - qc.width + i for c in qc.context for i in range(qc.width)],
                                       np.float64), heads)

            def job(qc=qc, args=args, x=x, pos=pos, heads=heads, tokens=tokens):
                y = oracle.dq_gemm(qc.wtype, *args, x)
                oracle.rope(y.reshape(tokens * heads, qc.d), pos, qc.rope_base)
            self.jobs.append(job)
            self.covered += bounds.qkv_rope_append_bytes(qc.wtype, tokens, qc.k, qc.hq, qc.hkv, qc.d) * rows / n
        for v in getattr(wl, "verifies", ()):
            # one request's verify block (its w logit rows), one in ``reqs``
            reqs = max(1, int(round(v.batch * frac)))
            lg = synth.normal_bf16(seed, v.name + ".cpu", (reqs, v.width, v.vocab))
            dr = rng.integers(0, v.vocab, (reqs, v.width - 1)).astype(np.int32)
            self.jobs.append(lambda lg=lg, dr=dr: oracle.spec_verify_greedy(lg, dr))
            self.covered += bounds.verify_bytes(v.batch, v.width, v.vocab) * reqs / v.batch
        self.threads = oracle.num_threads()
        self.desc = (f"oracle on a random {frac:.4g} of every projection's output rows and on "
                     f"sampled query rows of one (sequence, kv head) per attention call; "
                     f"{self.threads} OpenMP threads")

    def run(self) -> float:
        t0 = time.perf_counter()
        for j in self.jobs:
            j()
        return time.perf_counter() - t0


def run_reference(args, rank, world):
    if world > 1:
        # the other ranks do no work, so rank 0's oracle takes the host's cores
        # (torchrun sets OMP_NUM_THREADS=1 for every process)
        import oracle
        oracle.build()
        oracle.set_num_threads(len(os.sched_getaffinity(0)))
    wl = workload(args.workload)
    total_steps = args.steps + args.warmup
    # the whole reference run ends within a few minutes
    per_step_budget = max(0.002, min(2.0, 150.0 / max(1, total_steps)))
    sample = OracleSample(wl, per_step_budget)
    for _ in range(args.warmup):
        sample.run()
    secs = sum(sample.run() for _ in range(args.steps))
    value = sample.covered * args.steps / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": sample.threads, "kind": "oracle",
                         "sample": sample.desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


METRIC = "effective HBM GB/s (% of GB300 peak) and us/call for dq_gemm + gqa_decode_attn"
# Nominal HBM3e bandwidth of the part (the measured copy peak is the roofline's denominator).
HBM_NOMINAL_GBS = 8000.0


def cpu_model() -> str:
    """The host CPU's model string (x86 'model name', Arm implementer/part)."""
    try:
        txt = open("/proc/cpuinfo").read()
    except Exception:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for line in txt.splitlines():
            if line.lower().startswith(key.lower()) and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = [line.split(":", 1)[1].strip() for line in txt.splitlines()
             if line.startswith(("CPU implementer", "CPU part")) and ":" in line][:2]
    return "arm " + " ".join(parts) if parts else "unknown"


def traffic_for(kernel_call_name, workload_name):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    ent = d.get(workload_name, {}).get(kernel_call_name)
    if not ent or ent.get("csrc_hash") != csrc_hash():
        return None
    return ent.get("dram_bytes")


SUB_WORKLOADS = ("tiny", "llama3_8b_b1", "dense70b_b32", "verify_8b", "longctx_70b_b8_fp8kv",
                 "int4_70b_b32_fp8kv")


def call_records(calls, per_call, proto, hbm, tf):
    """Per-call records: the in-step evented duration and, when measured,
    the call alone (back-to-back in a CUDA graph, L2-cold copies)."""
    out = {}
    for c in calls:
        us = per_call.get(c.name, 0.0) * 1e3
        gbs = c.nbytes / (us * 1e-6) / 1e9 if us > 0 else None
        info = {"us": round(us, 3), "GB/s": round(gbs, 1) if gbs else None,
                "frac_hbm": round(gbs / hbm, 4) if gbs else None, "bytes": int(c.nbytes)}
        pr = proto.get(c.name)
        if pr:
            med = pr["median"]
            info["alone"] = {"us_median": round(med, 3), "us_min": round(pr["min"], 3),
                             "GB/s": round(c.nbytes / (med * 1e-6) / 1e9, 1),
                             "frac_hbm": round(c.nbytes / (med * 1e-6) / 1e9 / hbm, 4),
                             "frac_hbm_nominal": round(c.nbytes / (med * 1e-6) / 1e9 / HBM_NOMINAL_GBS, 4),
                             "TFLOP/s": round(c.flops / (med * 1e-6) / 1e12, 2),
                             "frac_tensor_bf16": round(c.flops / (med * 1e-6) / 1e12 / tf, 4),
                             "copies": pr["copies"], "calls": pr["calls"], "replays": pr["replays"],
                             "single_launch_us": round(pr["single"], 3), "clocks": pr["clocks"]}
        out[c.name] = info
    return out


def summary(r, world, hbm, tf):
    """The step-level figures of one measured workload."""
    tm = r["timing"]
    step_s = tm["ms_per_step"] / 1e3
    value = r["step_bytes"] * world / step_s / 1e9
    return {
        "workload": r["wl"].name, "value": round(value, 2), "unit": "GB/s",
        "ms_per_step": round(tm["ms_per_step"], 5), "steps": tm["K"], "timed_runs": tm["runs"],
        "ms_per_step_spread": {"min": round(tm["min_ms_per_step"], 5), "p10": round(tm["p10_ms_per_step"], 5),
                               "p90": round(tm["p90_ms_per_step"], 5), "max": round(tm["max_ms_per_step"], 5)},
        "frac_of_peak": round(value / world / hbm, 4), "frac_of_nominal": round(value / world / HBM_NOMINAL_GBS, 4),
        "step_bytes": int(r["step_bytes"]), "launches_per_step": r["launches"],
        "evented_ms_per_step": round(r["evented_ms"], 5) if r["evented_ms"] else None,
        "clocks": r["clocks"],
        "e2e": r["e2e"],
        "per_call": call_records(r["calls"], r["per_call"], r["proto"], hbm, tf),
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, rank, world)
        return

    import gc

    import torch
    import torch.distributed as dist
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    from memory_bound_decode_dq_gb300 import dqd
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    hbm, tf, tf_sus, peak_src = peaks()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    r = measure_workload(args.workload, args, rank, world, dev, dqd, sampler, args.min_load_s,
                         protocol=not args.no_call_protocol)
    head = summary(r, world, hbm, tf)
    wl, calls = r["wl"], r["calls"]
    per_call = r["per_call"]
    dom = max(calls, key=lambda c: per_call.get(c.name, 0.0)) if per_call else None
    roof = None
    if dom is not None and per_call.get(dom.name, 0) > 0:
        dur = per_call[dom.name] / 1e3
        ach = dom.nbytes / dur / 1e9
        alone = head["per_call"][dom.name].get("alone")
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": traffic_for(dom.name, wl.name),
                "kernel": dom.kind, "call": dom.name, "peak_source": peak_src,
                "algorithmic_bytes": int(dom.nbytes), "us_per_launch": round(per_call[dom.name] * 1e3, 3),
                "duration_from": "CUDA events on the launching stream around every launch of the call "
                                 "in a graph of the step, a pass after the timed region",
                "alone_us_median": alone["us_median"] if alone else None,
                "alone_frac": alone["frac_hbm"] if alone else None}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # about cpu_seconds of oracle work: a sample sized for a third of
        # it, run at least 3 times and until the budget is spent
        sample = OracleSample(wl, args.cpu_seconds / 3)
        secs, runs = 0.0, 0
        while runs < 3 or (secs < args.cpu_seconds and runs < 1000):
            secs += sample.run()
            runs += 1
        cpu = {"value": round(runs * sample.covered / secs / 1e9, 4), "unit": "GB/s", "cores": sample.threads,
               "cpu_model": cpu_model(), "kind": "oracle",
               "sample": sample.desc + f"; {runs} runs, {secs:.1f} s"}
    ws_mb = working_set_bytes(calls) / 1e6
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size / 1e6
    launches = r["launches"]
    G = r["timing"]["graph_steps"]
    del r, calls, per_call, dom
    gc.collect()
    torch.cuda.empty_cache()

    # the other workloads, one at a time, as sub-records (one replica: N = 1)
    subs = {}
    if world == 1 and not args.no_subrecords:
        for name in SUB_WORKLOADS:
            if workload(name).name == wl.name:
                continue
            rs = measure_workload(name, args, rank, world, dev, dqd, sampler, args.sub_min_load_s,
                                  protocol=not args.no_call_protocol)
            subs[name] = summary(rs, world, hbm, tf)
            del rs
            gc.collect()
            torch.cuda.empty_cache()
    if rank == 0:
        sampler.stop()
        line = {
            "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "calls": list(head["per_call"]),
                       "l2": f"inputs larger than L2: every step streams {ws_mb:.0f} MB once ({ws_mb / l2:.1f}x the {l2:.0f} MB L2)",
                       "timing": (f"each timed run is exactly {args.steps} steps replayed from CUDA graphs of {G} "
                                  f"steps (kernels back to back), with a barrier and a synchronise on both sides "
                                  f"and CUDA events on the replay stream; {head['timed_runs']} runs, ms_per_step "
                                  f"is the median run (max over ranks); per-call durations come from a separate "
                                  f"evented pass after the timed runs"),
                       "parallelism": f"replicas x{world}"},
            "frac_of_peak": head["frac_of_peak"],
            "frac_of_nominal": head["frac_of_nominal"],
            "timed_runs": head["timed_runs"],
            "ms_per_step_spread": head["ms_per_step_spread"],
            "per_call": head["per_call"],
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": head["e2e"],
            "gpu_launches": launches * args.steps,
            "gpu_launches_per_step": launches,
            "clocks": head["clocks"],
            "timing_detail": {"evented_ms_per_step": head["evented_ms_per_step"]},
            "workloads": subs,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
