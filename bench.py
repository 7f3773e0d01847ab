#!/usr/bin/env python3
"""KIVI hot-path benchmark on GB300.

One step = one pass of the whole hot path over one batch of the Qwen3-8B-like
single-layer workload (B=1, H_kv=8, 32 query heads, D=128, 2238-token prompt,
4-bit, G=32, residual_length=128):
  1. flush the oldest 2080 tokens of K and V into the packed store (one launch),
  2. append the 158-token fp16 tail to the K and V residual windows (one launch),
  3. dequantize the packed K and V stores back to fp16 (one launch),
  4. fused dequantize-and-attend decode of one query token per head (split over
     the cached tokens; the last CTA of each head merges the splits).
Steps 2 and 4 run on a side stream (4 after the flush), beside step 3.
value = algorithmic HBM bytes of the step / device time per step (GB/s).

Inputs rotate through a pool of independent instances whose total size is
several times the L2 cache, so no step finds its inputs in L2. Steps are
captured in CUDA graphs of 8 consecutive steps on 8 distinct instances; the
timed region replays them (K steps in all) between two CUDA events. Each op's
average launch duration is timed the same way on graphs of 8 launches of that
op alone.

--impl reference times the plain CPU oracle on the same workload and metric.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
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

METRIC = "KIVI flush/dequant/decode-attend HBM GB/s (% of peak); decode tokens/s"
FALLBACK_HBM_GBS = 6800.0


# --profile-case NAME: (op kind, B, S_q, n_res, bits); flush cases use the named workload
# (with the group size a _gNN suffix names)
PROFILE_CASES = {
    "flush_long2bit": ("flush", 0, 0, 0, 2),
    "flush_long2bit_g128": ("flush", 0, 0, 0, 2),
    "decode_b1_16k": ("decode", 1, 16384 - 128, 128, 4),
    "decode_b32_4k": ("decode", 32, 4032, 64, 4),
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", default="qwen8b", choices=["tiny", "qwen8b", "long2bit"])
    p.add_argument("--pool", type=int, default=0, help="instances in the rotating pool (0 = auto)")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--e2e-streams", type=int, default=2,
                   help="streams the end-to-end instances alternate between (copies of one overlap the others)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--hashes", action="store_true", help="print the source hash of each op and exit")
    p.add_argument("--stream", action="store_true",
                   help="instead of the step line: the 36-layer streaming serving simulation (tokens/s)")
    p.add_argument("--stream-steps", type=int, default=3072, help="decode steps of --stream (multiple of 32)")
    p.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                   help="run one op on one case a few times, untimed (a target for ncu captures)")
    p.add_argument("--sweep", nargs="?", const="all", choices=["all", "decode", "flush"],
                   help="instead of the step line: per-op GB/s at larger sizes and a decode S_kv sweep "
                        "('decode': the decode cases only; 'flush': flush, dequant and fake quantization only)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# workload accounting
# ---------------------------------------------------------------------------

def op_bytes(w, n_flush: int, n_res: int, meta_bytes: int = 6) -> dict:
    """Algorithmic HBM bytes per step, per op (each tensor read or written once).
    meta_bytes: scale + zero per group (6 with fp32 scales, 4 with fp16)."""
    el = w.BH * n_flush * w.D                     # flushed elements per tensor
    packed = w.bits / 8 + meta_bytes / w.G        # code bits + scale + zero per group
    flush = 2 * el * (2 + packed)                 # K and V: read fp16, write codes + metadata
    dequant = 2 * el * (packed + 2)               # read codes + metadata, write fp16
    append = 2 * 2 * w.BH * n_res * w.D * 2       # K and V tail rows: read + write
    # decode: per (kv head, store token) K+V codes + key metadata (6 B per channel
    # per 32 tokens) + value metadata (6 B per 32-channel group)
    per_tok = 2 * w.D * w.bits / 8 + w.D * meta_bytes / w.G + (w.D // w.G) * meta_bytes
    decode = (w.BH * n_flush * per_tok + w.BH * n_res * w.D * 2 * 2
              + w.B * w.Hq * w.D * 2 + w.B * w.Hq * w.D * 4)
    return {"flush_kv": flush, "residual_append": append, "dequant_kv": dequant, "decode_attend": decode}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over all ranks (a job takes as long as its slowest rank)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_step: float, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `bytes_per_step`
    within `elapsed_ms` (the max over ranks)."""
    return world * bytes_per_step * steps / (elapsed_ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(files) -> str:
    """First 16 hex digits of the sha256 of the op's CUDA sources."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "kivi_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(files, op: str):
    """DRAM bytes per launch of an op from an ncu capture (profiles/traffic.txt
    lines 'op sha bytes'), or None if the op's sources changed since."""
    try:
        sha = source_hash(files)
        for ln in open(os.path.join(ROOT, "profiles", "traffic.txt")):
            parts = ln.split()
            if len(parts) >= 3 and not ln.startswith("#") and parts[0] == op and parts[1] == sha:
                return float(parts[2])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GB300 arm
# ---------------------------------------------------------------------------

class Instance:
    """Device buffers of one independent copy of the workload."""

    def __init__(self, w, seed, device, kv, synth):
        import torch
        self.kv = kv
        self.w = w
        self.k, self.v, self.q = synth.prefill_inputs_torch(w, seed, device)
        self.n_flush = kv.kivi_flush_count(w.S, w.R, w.G)
        self.n_res = w.S - self.n_flush
        self.res_cap = w.R + w.G
        self.kst = kv.KiviStore(0, w.BH, self.n_flush, w.D, w.G, w.bits, device=device)
        self.vst = kv.KiviStore(1, w.BH, self.n_flush, w.D, w.G, w.bits, device=device)
        self.kres = torch.zeros((w.BH, self.res_cap, w.D), dtype=torch.float16, device=device)
        self.vres = torch.zeros_like(self.kres)
        self.kdq = torch.empty((w.BH, self.n_flush, w.D), dtype=torch.float16, device=device)
        self.vdq = torch.empty_like(self.kdq)
        self.out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=device)
        need = kv.kivi_decode_workspace_size(w.B, w.Hq, w.Hkv, self.n_flush, self.n_res, w.D)
        self.ws = kv.kivi_decode_workspace(need, device)
        self.side = torch.cuda.Stream(device=device)
        self.flushed = torch.cuda.Event()

    def step(self, join=True):
        """One pass of the hot path. The flush and the dequant run on the
        current stream; the residual append and the decode (which needs the
        flushed store) run on a side stream beside the dequant; the side
        stream joins the current one at the end (or, with join=False, when the
        caller joins it, so independent steps may overlap)."""
        import torch
        kv, w = self.kv, self.w
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            kv.kivi_residual_append_kv(self.k[:, self.n_flush:], self.v[:, self.n_flush:], self.kres, self.vres,
                                       0, self.n_res)
        kv.kivi_flush_kv(self.k, self.v, w.R, self.kst, self.vst)
        self.flushed.record(main)
        kv.kivi_dequant_kv(self.kst, self.vst, self.n_flush, kout=self.kdq, vout=self.vdq)
        with torch.cuda.stream(self.side):
            self.side.wait_event(self.flushed)
            kv.kivi_decode_attend(self.q, self.kst, self.vst, self.n_flush, self.kres, self.vres, self.n_res,
                                  w.Hkv, w.sm_scale, out=self.out, workspace=self.ws)
        if join:
            main.wait_stream(self.side)

    def nbytes(self):
        ts = [self.k, self.v, self.q, self.kres, self.vres, self.kdq, self.vdq, self.out, self.ws,
              self.kst.codes, self.kst.scale, self.kst.zero, self.vst.codes, self.vst.scale, self.vst.zero]
        return sum(t.numel() * t.element_size() for t in ts)


OPS = ["flush_kv", "residual_append", "dequant_kv", "decode_attend"]
GRAPH_STEPS = 8
OP_KERNEL_FILES = {"flush_kv": ["flush.cu"], "residual_append": ["residual.cu"], "dequant_kv": ["dequant.cu"],
                   "decode_attend": ["decode_pair.cu", "decode_merge.cuh", "decode_common.cuh"]}
LAUNCHES = {"flush_kv": 1, "residual_append": 1, "dequant_kv": 1, "decode_attend": 1}


def workload_label(w) -> str:
    """The step's workload, named the same way by both arms."""
    return ("%s: single-layer prefill flush + residual append + dequant + decode "
            "(B=%d, H_kv=%d, Hq=%d, D=%d, S=%d, bits=%d, G=%d, residual_length=%d)"
            % (w.name, w.B, w.Hkv, w.Hq, w.D, w.S, w.bits, w.G, w.R))


def run_gb300(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import kivi_kv_cache_gb300 as kv
    from kivi_kv_cache_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)

    probe = Instance(w, 1000 * rank + 0, dev, kv, synth)
    inst_bytes = probe.nbytes()
    # pool: a multiple of GRAPH_STEPS independent instances, >= 4x L2 in total
    pool = args.pool or int(min(64, max(2, math.ceil(4 * l2 / inst_bytes))))
    pool = max(GRAPH_STEPS, (pool + GRAPH_STEPS - 1) // GRAPH_STEPS * GRAPH_STEPS)
    insts = [probe] + [Instance(w, 1000 * rank + i, dev, kv, synth) for i in range(1, pool)]
    launches_per_step = sum(LAUNCHES.values())

    # eager warm-up; then CUDA graphs of GRAPH_STEPS consecutive steps, each on
    # its own instance (a graph launch costs microseconds; steps inside a graph
    # follow each other with programmatic dependent launch), plus one-step
    # graphs for a remainder of K that is not a multiple of GRAPH_STEPS
    for i in range(max(1, args.warmup)):
        insts[i % pool].step()
    torch.cuda.synchronize()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def steps(j):
        group = insts[j * GRAPH_STEPS:(j + 1) * GRAPH_STEPS]
        for inst in group:
            inst.step(join=False)
        for inst in group:
            torch.cuda.current_stream().wait_stream(inst.side)

    multi = [capture(lambda j=j: steps(j)) for j in range(pool // GRAPH_STEPS)]
    single = [capture(lambda I=I: I.step()) for I in insts]
    for i in range(max(1, args.warmup // GRAPH_STEPS)):
        multi[i % len(multi)].replay()
    torch.cuda.synchronize()

    gpu_id = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local_rank)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    n_multi, n_rest = divmod(args.steps, GRAPH_STEPS)
    start.record()
    for i in range(n_multi):
        multi[i % len(multi)].replay()
    for i in range(n_rest):
        single[i % pool].replay()
    end.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clock = clocks.stop()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)

    # per-op average launch duration: CUDA events on the launching stream
    # around replays of a graph of GRAPH_STEPS launches of that op alone, on
    # consecutive instances of the same rotating pool and with the step's
    # launch configuration
    op_fns = {
        "flush_kv": lambda I: kv.kivi_flush_kv(I.k, I.v, w.R, I.kst, I.vst),
        "residual_append": lambda I: kv.kivi_residual_append_kv(I.k[:, I.n_flush:], I.v[:, I.n_flush:], I.kres,
                                                                 I.vres, 0, I.n_res),
        "dequant_kv": lambda I: kv.kivi_dequant_kv(I.kst, I.vst, I.n_flush, kout=I.kdq, vout=I.vdq),
        "decode_attend": lambda I: kv.kivi_decode_attend(I.q, I.kst, I.vst, I.n_flush, I.kres, I.vres, I.n_res,
                                                         w.Hkv, w.sm_scale, out=I.out, workspace=I.ws),
    }
    op_ms = {}
    reps = max(4, min(200, args.steps // GRAPH_STEPS))
    for op, fn in op_fns.items():
        gs = [capture(lambda j=j, fn=fn: [fn(insts[j * GRAPH_STEPS + t]) for t in range(GRAPH_STEPS)])
              for j in range(pool // GRAPH_STEPS)]
        for g in gs:
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            gs[i % len(gs)].replay()
        e1.record()
        torch.cuda.synchronize()
        op_ms[op] = e0.elapsed_time(e1) / (reps * GRAPH_STEPS)
        del gs

    ob = op_bytes(w, probe.n_flush, probe.n_res)
    step_bytes = sum(ob.values())
    ms_per_step = elapsed_ms / args.steps
    value = job_gbs(world, step_bytes, args.steps, elapsed_ms)
    peak, peak_kind = measured_peaks()
    ops = {}
    for op in OPS:
        gbs = ob[op] / (op_ms[op] * 1e-3) / 1e9
        ops[op] = {"us": round(op_ms[op] * 1e3, 3), "bytes": int(ob[op]), "GB/s": round(gbs, 1),
                   "frac_of_peak": round(gbs / peak, 4)}
    dom = max(OPS, key=lambda o: op_ms[o])
    achieved = ob[dom] / (op_ms[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": peak_kind + " hbm_gbs (copy, burst)", "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": read_traffic(OP_KERNEL_FILES[dom], dom)}

    # end to end: host inputs (pinned) -> device, the step, result -> host.
    # Each instance's public-API calls (the copies of its K, V and q from
    # pinned host buffers, the step, the copy of its output back) are
    # captured once as a CUDA graph, as a serving loop would; graphs of
    # independent instances alternate between two streams, so the copies of
    # one step overlap the kernels of the other. Every step moves its inputs
    # and its result through the copy engines inside the timed region.
    e2e = None
    if args.e2e_steps > 0:
        nl = max(1, args.e2e_streams)
        ne = min(pool, max(2 * nl, 4))  # instances: two per stream, at least 4
        hk = [insts[i].k.cpu().pin_memory() for i in range(ne)]
        hv = [insts[i].v.cpu().pin_memory() for i in range(ne)]
        hq = [insts[i].q.cpu().pin_memory() for i in range(ne)]
        hout = [torch.empty((w.B, w.Hq, w.D), dtype=torch.float32).pin_memory() for _ in range(ne)]
        lanes = [torch.cuda.Stream(dev) for _ in range(nl)]

        def e2e_step(i):
            insts[i].k.copy_(hk[i], non_blocking=True)
            insts[i].v.copy_(hv[i], non_blocking=True)
            insts[i].q.copy_(hq[i], non_blocking=True)
            insts[i].step()
            hout[i].copy_(insts[i].out, non_blocking=True)

        e2e_graphs = []
        for i in range(ne):
            lane = lanes[i % nl]
            lane.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(lane):
                e2e_step(i)  # eager once on this stream before the capture
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=lane):
                    e2e_step(i)
            e2e_graphs.append(g)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        main = torch.cuda.current_stream()
        s0.record(main)
        for lane in lanes:
            lane.wait_stream(main)
        for j in range(args.e2e_steps):
            i = j % ne
            with torch.cuda.stream(lanes[i % nl]):
                e2e_graphs[i].replay()
        for lane in lanes:
            main.wait_stream(lane)
        s1.record(main)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s0.elapsed_time(s1), world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (hk[0], hv[0], hq[0]))
        e2e = {"value": round(job_gbs(world, step_bytes, args.e2e_steps, e2e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout[0].numel() * 4),
               "ms_per_step": round(e2e_ms / args.e2e_steps, 5),
               "how": "per-instance CUDA graphs of the public-API calls: pinned H2D copies of K, V, q, the step, "
                      "D2H of the output; %d streams alternate instances so copies overlap kernels" % nl}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle(w, args.cpu_seconds)

    decode_s = op_ms["decode_attend"] * 1e-3
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_label(w),
                   "n_flush": probe.n_flush, "n_res": probe.n_res,
                   "l2": "rotating pool of %d independent instances, %.0f MB total (L2 %d MB)"
                         % (pool, pool * inst_bytes / 2 ** 20, l2 >> 20),
                   "timing": "graphs of %d steps on distinct instances, K steps between CUDA events" % GRAPH_STEPS,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "ops": ops,
        "decode_tokens_per_s": round(w.B / decode_s, 1),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock,
        "peak_hbm_gbs": peak,
        "per_op_timing": "CUDA events around graphs of %d back-to-back launches of the op" % GRAPH_STEPS,
    }
    return line


# ---------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def cpu_oracle_step(w, k, v, q, threads):
    """One step of the workload on the CPU oracle, one KV head per thread."""
    import numpy as np

    import oracle
    n = oracle.flush_count(w.S, w.R, w.G)
    n_res = w.S - n
    gq = w.Hq // w.Hkv

    def head(bh):
        b, hk = divmod(bh, w.Hkv)
        ks = oracle.Store(0, 1, n, w.D, w.G, w.bits)
        vs = oracle.Store(1, 1, n, w.D, w.G, w.bits)
        oracle.flush(0, k[bh:bh + 1], n, ks)
        oracle.flush(1, v[bh:bh + 1], n, vs)
        kres = np.zeros((1, w.R + w.G, w.D), np.float16)
        vres = np.zeros_like(kres)
        oracle.residual_append(kres, 0, np.ascontiguousarray(k[bh:bh + 1, n:]), n_res)
        oracle.residual_append(vres, 0, np.ascontiguousarray(v[bh:bh + 1, n:]), n_res)
        oracle.dequant(ks, n)
        oracle.dequant(vs, n)
        qh = np.ascontiguousarray(q[b:b + 1, hk * gq:(hk + 1) * gq])
        return oracle.decode_attend(qh, ks, vs, n, kres, vres, n_res, 1, w.sm_scale)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(head, range(w.BH)))


def cpu_oracle(w, seconds, steps=None):
    """Time the oracle on host cores: whole steps until `seconds` (or `steps`)."""
    from kivi_kv_cache_gb300 import synth
    import oracle
    oracle.build()
    k, v, q = synth.prefill_inputs(w)
    threads = max(1, min(os.cpu_count() or 1, w.BH))
    cpu_oracle_step(w, k, v, q, threads)  # warm (page in, build)
    n = oracle.flush_count(w.S, w.R, w.G)
    step_bytes = sum(op_bytes(w, n, w.S - n).values())
    done, t0 = 0, time.perf_counter()
    times = []
    while True:
        t = time.perf_counter()
        cpu_oracle_step(w, k, v, q, threads)
        times.append(time.perf_counter() - t)
        done += 1
        if (steps is not None and done >= steps) or (steps is None and time.perf_counter() - t0 >= seconds):
            break
    total = sum(times)
    return {"value": round(step_bytes * done / total / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d whole steps of the %s workload (C oracle, one KV head per thread), %.1f s"
                      % (done, w.name, total),
            "ms_per_step": round(1e3 * total / done, 3)}


def run_reference(args, rank, world):
    from kivi_kv_cache_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    import oracle
    oracle.build()
    k, v, q = synth.prefill_inputs(w)
    threads = max(1, min(os.cpu_count() or 1, w.BH))
    for _ in range(max(0, args.warmup)):
        cpu_oracle_step(w, k, v, q, threads)
    steps = max(1, args.steps)
    # keep the reference arm to a bounded number of whole steps
    t = time.perf_counter()
    cpu_oracle_step(w, k, v, q, threads)
    one = time.perf_counter() - t
    steps = max(1, min(steps, int(120.0 / max(one, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(steps):
        cpu_oracle_step(w, k, v, q, threads)
    el = time.perf_counter() - t0
    n = oracle.flush_count(w.S, w.R, w.G)
    step_bytes = sum(op_bytes(w, n, w.S - n).values())
    value = step_bytes * steps / el / 1e9
    sample = "%d whole steps of the %s workload (C oracle, one KV head per thread)" % (steps, w.name)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * el / steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_label(w), "note": "plain C CPU oracle as the reference arm"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_sweep(args):
    """Per-op throughput at larger sizes (one JSON line per measurement).

    Each measurement: a rotating pool of independent inputs totalling more than
    4x L2, CUDA graphs of 8 launches of the op on distinct pool entries, CUDA
    events around R graph replays; GB/s = algorithmic bytes / mean duration."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import kivi_kv_cache_gb300 as kv
    from kivi_kv_cache_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)
    peak, kind = measured_peaks()

    def timed(fns, nbytes, label, extra):
        gs = []
        for j in range(len(fns) // 8):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for f in fns[8 * j:8 * j + 8]:
                    f()
            gs.append(g)
        for g in gs:
            g.replay()
        torch.cuda.synchronize()
        reps = max(8, 400 // len(gs))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            gs[i % len(gs)].replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * 8)
        gbs = nbytes / (us * 1e-6) / 1e9
        line = {"op": label, "us": round(us, 3), "bytes": int(nbytes), "GB/s": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4), "peak": peak, "peak_kind": kind}
        line.update(extra)
        print(json.dumps(line), flush=True)

    def pool_count(bytes_each):
        return max(8, min(64, int(math.ceil(4 * l2 / max(bytes_each, 1) / 8)) * 8))

    # flush / dequant at the long-context 2-bit and qwen8b sizes; head dims 64
    # and 256 at the long 2-bit size with the same element count (16 or 4 KV heads)
    # (workload, G, D, fp16 scales)
    shapes = (("qwen8b", 32, 128, False), ("long2bit", 32, 128, False), ("long2bit", 64, 128, False),
              ("long2bit", 128, 128, False), ("long2bit", 32, 64, False), ("long2bit", 64, 64, False),
              ("long2bit", 32, 256, False), ("long2bit", 128, 256, False), ("long2bit", 32, 128, True))
    for name, G, D, hs in (shapes if args.sweep in ("all", "flush") else ()):
        w = dataclasses.replace(synth.WORKLOADS[name], G=G, D=D, Hkv=synth.WORKLOADS[name].Hkv * 128 // D,
                                Hq=synth.WORKLOADS[name].Hq * 128 // D)
        n = kv.kivi_flush_count(w.S, w.R, w.G)
        meta = 4 if hs else 6  # bytes of scale + zero per group
        per = w.BH * w.S * w.D * 2 * 2 + 2 * w.BH * n * (w.D * w.bits // 8 + w.D * meta // w.G) + w.BH * n * w.D * 4
        P = pool_count(per)
        ks, vs, kd, vd, xs = [], [], [], [], []
        for i in range(P):
            k, v, _ = synth.prefill_inputs_torch(w, 7000 + i, dev)
            xs.append((k, v))
            ks.append(kv.KiviStore(0, w.BH, n, w.D, w.G, w.bits, device=dev, scale_f16=hs))
            vs.append(kv.KiviStore(1, w.BH, n, w.D, w.G, w.bits, device=dev, scale_f16=hs))
            kd.append(torch.empty((w.BH, n, w.D), dtype=torch.float16, device=dev))
            vd.append(torch.empty_like(kd[-1]))
        ob = op_bytes(w, n, w.S - n, meta_bytes=4 if hs else 6)
        timed([lambda i=i: kv.kivi_flush_kv(xs[i][0], xs[i][1], w.R, ks[i], vs[i]) for i in range(P)],
              ob["flush_kv"], "flush_kv", {"workload": name, "tokens": n, "bits": w.bits, "G": G, "D": D, "scale_f16": hs,
                                                   "pool": P})
        timed([lambda i=i: kv.kivi_dequant_kv(ks[i], vs[i], n, kout=kd[i], vout=vd[i]) for i in range(P)],
              ob["dequant_kv"], "dequant_kv", {"workload": name, "tokens": n, "bits": w.bits, "G": G, "D": D, "scale_f16": hs,
                                                     "pool": P})
        # fake quantization of the same tokens: read 2 B and write 2 B per element of K and V (the kd/vd
        # buffers hold the n flushed tokens, so the S - n fp16 tokens are not part of this launch)
        timed([lambda i=i: kv.kivi_fake_quant_kv(xs[i][0][:, :n], xs[i][1][:, :n], 0, kout=kd[i], vout=vd[i],
                                                 G=G, bits=w.bits, scale_f16=hs) for i in range(P)],
              2 * w.BH * n * w.D * 4, "fake_quant_kv", {"workload": name, "tokens": n, "bits": w.bits, "G": G,
                                                        "D": D, "scale_f16": hs, "pool": P})
        del ks, vs, kd, vd, xs
        torch.cuda.empty_cache()
    if args.sweep == "flush":
        return

    # decode over a packed store + fp16 residual
    # (B, packed tokens, fp16 residual tokens, bits): the qwen8b decode, the long-context and batched
    # decodes, and the streaming workload's S_kv sweep (128 / 512 / 2048 / 8192 / 16384 at B=1 and B=16)
    cases = [(1, 2080, 158, 4), (1, 4096 - 128, 128, 4), (1, 8192 - 128, 128, 4), (1, 16384 - 128, 128, 4),
             (1, 32768 - 128, 128, 2), (32, 4032, 64, 4), (16, 2048 - 128, 128, 4), (16, 16384 - 128, 128, 4),
             (1, 0, 128, 4), (1, 512 - 128, 128, 4), (1, 2048 - 128, 128, 4),
             (16, 0, 128, 4), (16, 512 - 128, 128, 4), (16, 8192 - 128, 128, 4)]
    # 8, 6 and 3 query heads per KV head (sub-groups of up to 4 heads)
    cases += [(1, 16384 - 128, 128, 4, 64), (32, 4032, 64, 4, 64), (1, 4096 - 128, 128, 4, 64),
              (32, 4032, 64, 4, 48), (32, 4032, 64, 4, 24)]
    # stores of group size 64 and 128
    cases += [(1, 2080, 158, 4, 32, 64), (1, 16384 - 128, 128, 4, 32, 64), (1, 16384 - 128, 128, 4, 32, 128),
              (32, 4032, 64, 4, 32, 64), (32, 4032, 64, 4, 32, 128), (1, 32768 - 128, 128, 2, 32, 128)]
    # head dims 64 and 256
    cases += [(1, 16384 - 128, 128, 4, 32, 32, 64), (32, 4032, 64, 4, 32, 32, 64),
              (1, 16384 - 128, 128, 4, 32, 32, 256), (32, 4032, 64, 4, 32, 32, 256)]
    # fp16 scale storage (160 bytes per 4-bit token instead of 176)
    cases += [(1, 2080, 158, 4, 32, 32, 128, True), (1, 16384 - 128, 128, 4, 32, 32, 128, True),
              (32, 4032, 64, 4, 32, 32, 128, True)]
    for case in cases:
        B, S_q, n_res, bits = case[:4]
        Hq = case[4] if len(case) > 4 else 32
        G = case[5] if len(case) > 5 else 32
        D = case[6] if len(case) > 6 else 128
        hs = case[7] if len(case) > 7 else False
        w = synth.Workload("decode", B=B, Hkv=8, Hq=Hq, D=D, S=S_q + n_res, bits=bits, G=G, R=0,
                           n_outlier=4, outlier_scale=8.0, seed=11)
        s_cap = max(1, -(-S_q // G)) * G
        meta = 4 if hs else 6  # bytes of scale + zero per group
        per_tok = 2 * w.D * bits / 8 + w.D * meta / w.G + (w.D // w.G) * meta
        nbytes = w.BH * S_q * per_tok + w.BH * n_res * w.D * 4 + B * w.Hq * w.D * 6
        P = pool_count(nbytes)
        entries = []
        for i in range(P):
            k, v, q = synth.prefill_inputs_torch(w, 9000 + i, dev)
            gk = kv.KiviStore(0, w.BH, s_cap, w.D, w.G, bits, device=dev, scale_f16=hs)
            gv = kv.KiviStore(1, w.BH, s_cap, w.D, w.G, bits, device=dev, scale_f16=hs)
            if S_q > 0:
                kv.kivi_flush_kv(k, v, 0, gk, gv, n_tokens=S_q)
            kr = k[:, S_q:].contiguous()
            vr = v[:, S_q:].contiguous()
            out = torch.empty((B, w.Hq, w.D), dtype=torch.float32, device=dev)
            need = kv.kivi_decode_workspace_size(B, w.Hq, w.Hkv, S_q, n_res, w.D)
            ws = kv.kivi_decode_workspace(need, dev)
            entries.append((q, gk, gv, kr, vr, out, ws))
            del k, v
        torch.cuda.synchronize()
        fns = [lambda e=e: kv.kivi_decode_attend(e[0], e[1], e[2], S_q, e[3], e[4], n_res, w.Hkv, w.sm_scale,
                                                 out=e[5], workspace=e[6]) for e in entries]
        timed(fns, nbytes, "decode_attend", {"B": B, "Hkv": 8, "Hq": Hq, "S_kv": S_q + n_res, "bits": bits,
                                             "G": G, "D": D, "scale_f16": hs, "pool": P, "tokens_per_s": None})
        del entries, fns
        torch.cuda.empty_cache()

    # two-pass "decode-once" against the fused decode (B=1 and B=32, 4032
    # packed + 64 fp16 tokens): the store changes only when a flush folds G
    # tokens in, so a two-pass decoder dequantizes it once per G steps and
    # attends over an all-fp16 cache every step. Reported: the fused decode,
    # the dequant, the fp16 attend (the same decode kernels over S_q = 0 and
    # S_kv fp16 tokens) and the two-pass cost per step, attend + dequant / G.
    for B in (1, 32):
        S_q, n_res = 4032, 64
        S = S_q + n_res
        w = synth.Workload("twopass", B=B, Hkv=8, Hq=32, D=128, S=S, bits=4, G=32, R=0, n_outlier=4,
                           outlier_scale=8.0, seed=12)
        k, v, q = synth.prefill_inputs_torch(w, 41, dev)
        gk = kv.KiviStore(0, w.BH, S_q, w.D, w.G, 4, device=dev)
        gv = kv.KiviStore(1, w.BH, S_q, w.D, w.G, 4, device=dev)
        kv.kivi_flush_kv(k, v, 0, gk, gv, n_tokens=S_q)
        kr, vr = k[:, S_q:].contiguous(), v[:, S_q:].contiguous()
        kd = torch.empty((w.BH, S_q, w.D), dtype=torch.float16, device=dev)
        vd = torch.empty_like(kd)
        kfull = torch.cat([kd, kr], dim=1)  # the fp16 cache the attend reads (contents: any fp16)
        vfull = torch.cat([vd, vr], dim=1)
        del k, v
        out = torch.empty((B, w.Hq, w.D), dtype=torch.float32, device=dev)
        ws = kv.kivi_decode_workspace(max(kv.kivi_decode_workspace_size(B, w.Hq, w.Hkv, S_q, n_res, w.D),
                                          kv.kivi_decode_workspace_size(B, w.Hq, w.Hkv, 0, S, w.D)), dev)
        per_tok = 2 * w.D * 4 / 8 + w.D * 6 / w.G + (w.D // w.G) * 6
        fused_b = w.BH * S_q * per_tok + w.BH * n_res * w.D * 4 + B * w.Hq * w.D * 6
        deq_b = 2 * w.BH * S_q * w.D * (2 + 4 / 8 + 6 / w.G)
        att_b = w.BH * S * w.D * 4 + B * w.Hq * w.D * 6
        res = {}
        for label, fn, nbytes in (
                ("fused", lambda: kv.kivi_decode_attend(q, gk, gv, S_q, kr, vr, n_res, w.Hkv, w.sm_scale, out=out,
                                                        workspace=ws), fused_b),
                ("dequant", lambda: kv.kivi_dequant_kv(gk, gv, S_q, kout=kd, vout=vd), deq_b),
                ("fp16_attend", lambda: kv.kivi_decode_attend(q, gk, gv, 0, kfull, vfull, S, w.Hkv, w.sm_scale,
                                                              out=out, workspace=ws), att_b)):
            g = torch.cuda.CUDAGraph()
            fn()
            torch.cuda.synchronize()
            with torch.cuda.graph(g):
                for _ in range(8):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            reps = 25
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            res[label] = e0.elapsed_time(e1) * 1e3 / (reps * 8)
            res[label + "_GB/s"] = round(nbytes / (res[label] * 1e-6) / 1e9, 1)
        two_pass = res["fp16_attend"] + res["dequant"] / w.G
        print(json.dumps({"op": "decode_two_pass_vs_fused", "B": B, "S_kv": S, "bits": 4,
                          "fused_us": round(res["fused"], 3), "dequant_us": round(res["dequant"], 3),
                          "fp16_attend_us": round(res["fp16_attend"], 3),
                          "two_pass_us_per_step": round(two_pass, 3),
                          "fused_over_two_pass": round(two_pass / res["fused"], 3),
                          "GB/s": {k2: v2 for k2, v2 in res.items() if k2.endswith("GB/s")},
                          "note": "two-pass per step = fp16 attend + dequant / G (one dequant per G steps); "
                                  "L2 not flushed between launches: one instance, 8 launches per graph"}),
              flush=True)
        del gk, gv, kr, vr, kd, vd, kfull, vfull, ws
        torch.cuda.empty_cache()

    # batched decode, 30 consecutive steps: B=32 sequences of 4032 packed + 64
    # fp16 tokens; each step appends one token per sequence to the residual
    # window (n_res 64 -> 93, no flush) and decodes one query token per head
    B, S_q, n0, steps = 32, 4032, 64, 30
    w = synth.Workload("batched", B=B, Hkv=8, Hq=32, D=128, S=S_q + n0 + steps, bits=4, G=32, R=0,
                       n_outlier=4, outlier_scale=8.0, seed=4)
    k, v, _ = synth.prefill_inputs_torch(w, 31, dev)
    gk = kv.KiviStore(0, w.BH, S_q, w.D, w.G, 4, device=dev)
    gv = kv.KiviStore(1, w.BH, S_q, w.D, w.G, 4, device=dev)
    kv.kivi_flush_kv(k, v, 0, gk, gv, n_tokens=S_q)
    res_cap = 128
    kres = torch.zeros((w.BH, res_cap, w.D), dtype=torch.float16, device=dev)
    vres = torch.zeros_like(kres)
    kv.kivi_residual_append_kv(k[:, S_q:S_q + n0], v[:, S_q:S_q + n0], kres, vres, 0)
    new_k = k[:, S_q + n0:].contiguous()
    new_v = v[:, S_q + n0:].contiguous()
    del k, v
    gen = torch.Generator(device=dev)
    gen.manual_seed(32)
    qs = torch.randn((steps, B, w.Hq, w.D), generator=gen, device=dev).to(torch.float16)
    out = torch.empty((B, w.Hq, w.D), dtype=torch.float32, device=dev)
    ws = kv.kivi_decode_workspace(kv.kivi_decode_workspace_size(B, w.Hq, w.Hkv, S_q, n0 + steps, w.D), dev)

    def run_steps():
        for i in range(steps):
            kv.kivi_residual_append_kv(new_k[:, i:i + 1], new_v[:, i:i + 1], kres, vres, n0 + i)
            kv.kivi_decode_attend(qs[i], gk, gv, S_q, kres[:, :n0 + i + 1], vres[:, :n0 + i + 1], n0 + i + 1,
                                  w.Hkv, w.sm_scale, out=out, workspace=ws)

    run_steps()  # eager warm-up (loads the kernels, sets attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_steps()
    g.replay()
    torch.cuda.synchronize()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * steps)
    per_step = sum(B * w.Hkv * S_q * (2 * w.D * 4 / 8 + w.D * 6 / w.G + (w.D // w.G) * 6) +
                   B * w.Hkv * (n0 + i + 1) * w.D * 4 + B * w.Hq * w.D * 6 + B * w.Hkv * w.D * 2 * 2 * 2
                   for i in range(steps)) / steps
    gbs = per_step / (us * 1e-6) / 1e9
    print(json.dumps({"op": "batched_decode_steps", "B": B, "S_kv": S_q + n0, "steps": steps,
                      "us_per_step": round(us, 3), "tokens_per_s": round(B / (us * 1e-6), 1),
                      "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "peak": peak,
                      "peak_kind": kind, "step": "append 1 token (K, V) + decode"}), flush=True)


def run_stream(args):
    """Streaming serving simulation of the KV-cache work: 36 layers, B=16,
    H_kv=8, Hq=32, D=128, 4-bit, G=32, R=128, context growing from 1024 tokens
    by one token per step. Every layer-step appends the new token's K and V to
    the fp16 residual window, flushes G tokens into the packed store and
    compacts the window when it reaches R + G tokens, and decodes one query
    token per head. The launches of each 32-step flush cycle (all layers) are
    captured in a CUDA graph beforehand; the timed region replays them all.
    tokens/s = B * steps / time (KV-cache work only: no projections or MLP)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import kivi_kv_cache_gb300 as kv
    from kivi_kv_cache_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = measured_peaks()
    L, B, Hkv, Hq, D, G, R, bits = 36, 16, 8, 32, 128, 32, 128, 4
    ctx0 = 1024
    steps = (args.stream_steps // G) * G
    BH = B * Hkv
    s_cap = ctx0 + steps
    res_cap = R + G
    w = synth.Workload("stream", B=B, Hkv=Hkv, Hq=Hq, D=D, S=ctx0, bits=bits, G=G, R=R, n_outlier=4,
                       outlier_scale=8.0, seed=5)
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    new_k = torch.randn((BH, G, D), generator=gen, device=dev).to(torch.float16)  # tokens appended, cyclically
    new_v = torch.randn((BH, G, D), generator=gen, device=dev).to(torch.float16)
    qs = torch.randn((G, B, Hq, D), generator=gen, device=dev).to(torch.float16)
    layers = []
    for l in range(L):
        k, v, _ = synth.prefill_inputs_torch(w, 100 + l, dev)
        ks = kv.KiviStore(0, BH, s_cap, D, G, bits, device=dev)
        vs = kv.KiviStore(1, BH, s_cap, D, G, bits, device=dev)
        S_q = kv.kivi_flush_kv(k, v, R, ks, vs)
        kres = torch.zeros((BH, res_cap, D), dtype=torch.float16, device=dev)
        vres = torch.zeros_like(kres)
        n_res = kv.kivi_residual_append_kv(k[:, S_q:], v[:, S_q:], kres, vres, 0)
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
        layers.append({"ks": ks, "vs": vs, "kres": kres, "vres": vres, "S_q": S_q, "n_res": n_res, "out": out})
        del k, v
    need = max(kv.kivi_decode_workspace_size(B, Hq, Hkv, sq, nr, D)  # the largest plan of any step
               for sq in range(ctx0 - R, s_cap + 1, G) for nr in range(R, R + G + 1))
    ws = kv.kivi_decode_workspace(need, dev)

    def layer_step(st, i):
        st["n_res"] = kv.kivi_residual_append_kv(new_k[:, i % G:i % G + 1], new_v[:, i % G:i % G + 1], st["kres"],
                                                 st["vres"], st["n_res"])
        if st["n_res"] >= R + G:
            n = kv.kivi_flush_kv(st["kres"], st["vres"], R, st["ks"], st["vs"], s_off=st["S_q"],
                                 n_tokens=st["n_res"])
            st["S_q"] += n
            st["n_res"] = kv.kivi_residual_compact_kv(st["kres"], st["vres"], st["n_res"], n)
        nr = st["n_res"]
        kv.kivi_decode_attend(qs[i % G], st["ks"], st["vs"], st["S_q"], st["kres"][:, :nr], st["vres"][:, :nr],
                              nr, Hkv, w.sm_scale, out=st["out"], workspace=ws)

    # warm-up on a copy of nothing: one eager cycle would change the state, so
    # run the first cycle eagerly only to load the kernels, then restart it
    snapshot = [(st["S_q"], st["n_res"]) for st in layers]
    for st in layers:
        layer_step(st, 0)
    torch.cuda.synchronize()
    for st, (sq, nr) in zip(layers, snapshot):  # the appended token is overwritten by the replay
        st["S_q"], st["n_res"] = sq, nr
    graphs = []
    for c in range(steps // G):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(G):
                for st in layers:
                    layer_step(st, c * G + j)
        graphs.append(g)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    print(json.dumps({"op": "stream_simulation", "layers": L, "B": B, "Hkv": Hkv, "Hq": Hq, "D": D, "bits": bits,
                      "G": G, "R": R, "context": [ctx0, ctx0 + steps], "steps": steps,
                      "ms": round(ms, 3), "tokens_per_s": round(B * steps / (ms * 1e-3), 1),
                      "us_per_layer_step": round(ms * 1e3 / (steps * L), 3),
                      "flushes_per_layer": steps // G, "peak": peak, "peak_kind": kind,
                      "note": "KV-cache work only (append, flush, compact, decode per layer-step); "
                              "no projections or MLP"}), flush=True)


def run_profile_case(name: str, reps: int = 3):
    """A few untimed launches of one op, for profiler captures of a size the
    step bench does not run."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import kivi_kv_cache_gb300 as kv
    from kivi_kv_cache_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kind, B, S_q, n_res, bits = PROFILE_CASES[name]
    if kind == "flush":
        parts = name.split("_")
        w = synth.WORKLOADS[parts[1]]
        if len(parts) > 2 and parts[2].startswith("g"):
            w = dataclasses.replace(w, G=int(parts[2][1:]))
        n = kv.kivi_flush_count(w.S, w.R, w.G)
        k, v, _ = synth.prefill_inputs_torch(w, 1, dev)
        ks = kv.KiviStore(0, w.BH, n, w.D, w.G, w.bits, device=dev)
        vs = kv.KiviStore(1, w.BH, n, w.D, w.G, w.bits, device=dev)
        for _ in range(reps):
            kv.kivi_flush_kv(k, v, w.R, ks, vs)
    else:
        w = synth.Workload("decode", B=B, Hkv=8, Hq=32, D=128, S=S_q + n_res, bits=bits, G=32, R=0,
                           n_outlier=4, outlier_scale=8.0, seed=4)
        k, v, q = synth.prefill_inputs_torch(w, 2, dev)
        gk = kv.KiviStore(0, w.BH, S_q, w.D, w.G, bits, device=dev)
        gv = kv.KiviStore(1, w.BH, S_q, w.D, w.G, bits, device=dev)
        kv.kivi_flush_kv(k, v, 0, gk, gv, n_tokens=S_q)
        kr = k[:, S_q:].contiguous()
        vr = v[:, S_q:].contiguous()
        del k, v
        ws = kv.kivi_decode_workspace(kv.kivi_decode_workspace_size(B, w.Hq, w.Hkv, S_q, n_res, w.D), dev)
        for _ in range(reps):
            kv.kivi_decode_attend(q, gk, gv, S_q, kr, vr, n_res, w.Hkv, w.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    print("ok", name)


def main():
    args = parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.stream:
        run_stream(args)
        return
    if args.hashes:
        for op, files in OP_KERNEL_FILES.items():
            print(op, source_hash(files))
        return
    if args.sweep:
        run_sweep(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl")
    line = run_gb300(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
