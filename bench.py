#!/usr/bin/env python3
"""KIVI hot-path benchmark on GB300.

One step = one pass of the whole hot path over one batch of the long-context
2-bit workload (B=1, H_kv=8, 32 query heads, D=128, S=32768, 2-bit, G=32,
residual_length=128), the single-sequence point (B=1, H_kv=8, S_kv >= 4096)
that the throughput targets are stated at:
  1. flush the oldest 32640 tokens of K and V into the packed store (one launch),
  2. append the 128-token fp16 tail to the K and V residual windows (one launch),
  3. dequantize the packed K and V stores back to fp16 (one launch),
  4. fused dequantize-and-attend decode of one query token per head (split over
     the cached tokens; the last CTA of each head merges the splits).
Steps 2 and 4 run on a side stream (4 after the flush), beside step 3.
value = algorithmic HBM bytes of the step / device time per step (GB/s).

Inputs rotate through a pool of independent instances whose total size is
several times the L2 cache, so no step finds its inputs in L2. Steps are
captured in CUDA graphs of 8 consecutive steps on 8 distinct instances; the
timed region replays them (K steps in all) between two CUDA events. Each op's
launch duration is timed on graphs of 8 launches of that op alone: the median
of 21 samples per op, taken in turn with the other ops, at least 256 launches
and 50 ms of device time per op in all.

On one GPU the same JSON line also carries, each timed on its own:
  * "qwen8b": the Qwen3-8B-like single-layer step (2238-token prompt, 4-bit);
  * "batched_decode": 32 sequences of 4096 cached tokens, 30 steps that each
    append one token per sequence and decode (tokens/s);
  * "stream": 36 layers, B=16, context 1024 -> 4096, an incremental flush
    whenever a window fills, a decode every layer-step (tokens/s);
  * "decode_b1": single-sequence decodes at 4096, 8192 and 16384 tokens
    (4-bit) and 32768 (2-bit), plain and with KIVI_DECODE_STORE_READY (a
    sequence of decodes: the preceding kernel never writes the store).

--impl reference times the plain CPU oracle on the same workload and metric.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import json
import math
import os
import platform
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
NOMINAL_HBM_GBS = 7900.0  # HBM3e nominal, quoted beside the measured peak
GRAPH_STEPS = 8
GRAPH_BRANCHES = 4  # parallel stream branches per timed graph (two steps each)
MIN_OP_LAUNCHES = 256
MIN_OP_MS = 50.0
OP_ROUNDS = 21  # interleaved timing samples per op of the step (the median is reported)


# --profile-case NAME: (op kind, B, S_q, n_res, bits); flush cases use the named workload
# (with the group size a _gNN suffix names)
PROFILE_CASES = {
    "flush_long2bit": ("flush", 0, 0, 0, 2),
    "flush_long2bit_g64": ("flush", 0, 0, 0, 2),
    "flush_long2bit_g128": ("flush", 0, 0, 0, 2),
    "flush_long2bit_f16s": ("flush", 0, 0, 0, 2),
    "flush_qwen8b": ("flush", 0, 0, 0, 4),
    "decode_b1_4k": ("decode", 1, 4096 - 128, 128, 4),
    "decode_b1_16k": ("decode", 1, 16384 - 128, 128, 4),
    "decode_b1_32k_2bit": ("decode", 1, 32768 - 128, 128, 2),
    "decode_b32_4k": ("decode", 32, 4032, 64, 4),
    "step_long2bit": ("step", 0, 0, 0, 2),
    "step_qwen8b": ("step", 0, 0, 0, 4),
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=16)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", default="long2bit", choices=["tiny", "qwen8b", "long2bit"])
    p.add_argument("--pool", type=int, default=0, help="instances in the rotating pool (0 = auto)")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--e2e-streams", type=int, default=2,
                   help="streams the end-to-end instances alternate between (copies of one overlap the others)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the qwen8b, batched, stream and B=1 decode sub-objects of the line")
    p.add_argument("--hashes", action="store_true", help="print the source hash of each op and exit")
    p.add_argument("--stream", action="store_true",
                   help="instead of the step line: the 36-layer streaming serving simulation (tokens/s)")
    p.add_argument("--stream-steps", type=int, default=3072, help="decode steps of the stream simulation "
                                                                   "(multiple of 32)")
    p.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                   help="run one op on one case a few times, untimed (a target for ncu captures)")
    p.add_argument("--sweep", nargs="?", const="all", choices=["all", "decode", "flush", "twopass"],
                   help="instead of the step line: per-op GB/s at larger sizes and a decode S_kv sweep "
                        "('decode': the decode cases only; 'flush': flush, dequant and fake quantization only; "
                        "'twopass': the fused decode against dequantize-once + fp16 attend over S_kv x B)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# workload accounting
# ---------------------------------------------------------------------------

def decode_bytes(B, Hkv, Hq, D, G, bits, S_q, n_res, meta_bytes=6) -> float:
    """Algorithmic bytes of one decode: per (KV head, store token) the K and V
    codes plus the key metadata (meta_bytes per channel per G tokens) and the
    value metadata (meta_bytes per G-channel group); 4 D bytes per (KV head,
    residual token); q (fp16) and out (fp32) once."""
    per_tok = 2 * D * bits / 8 + D * meta_bytes / G + (D // G) * meta_bytes
    return B * Hkv * S_q * per_tok + B * Hkv * n_res * D * 4 + B * Hq * D * 6


def op_bytes(w, n_flush: int, n_res: int, meta_bytes: int = 6) -> dict:
    """Algorithmic HBM bytes per step, per op (each tensor read or written once).
    meta_bytes: scale + zero per group (6 with fp32 scales, 4 with fp16)."""
    el = w.BH * n_flush * w.D                     # flushed elements per tensor
    packed = w.bits / 8 + meta_bytes / w.G        # code bits + scale + zero per group
    flush = 2 * el * (2 + packed)                 # K and V: read fp16, write codes + metadata
    dequant = 2 * el * (packed + 2)               # read codes + metadata, write fp16
    append = 2 * 2 * w.BH * n_res * w.D * 2       # K and V tail rows: read + write
    decode = decode_bytes(w.B, w.Hkv, w.Hq, w.D, w.G, w.bits, n_flush, n_res, meta_bytes)
    return {"flush_kv": flush, "residual_append": append, "dequant_kv": dequant, "decode_attend": decode}


def op_read_bytes(w, n_flush: int, n_res: int, meta_bytes: int = 6) -> dict:
    """The read share of op_bytes (what a DRAM read counter should see)."""
    el = w.BH * n_flush * w.D
    packed = w.bits / 8 + meta_bytes / w.G
    dec = decode_bytes(w.B, w.Hkv, w.Hq, w.D, w.G, w.bits, n_flush, n_res, meta_bytes) - w.B * w.Hq * w.D * 4
    return {"flush_kv": 2 * el * 2, "residual_append": 2 * w.BH * n_res * w.D * 2, "dequant_kv": 2 * el * packed,
            "decode_attend": dec}


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


def read_traffic(files, op: str, workload: str):
    """DRAM bytes per launch of an op at a workload from an ncu capture
    (profiles/traffic.txt lines 'op workload sha read_bytes write_bytes'), as
    {"read": r, "write": w}, or None if there is no capture of the op's
    current sources at that workload."""
    try:
        sha = source_hash(files)
        for ln in open(os.path.join(ROOT, "profiles", "traffic.txt")):
            parts = ln.split()
            if (len(parts) >= 5 and not ln.startswith("#") and parts[0] == op and parts[1] == workload
                    and parts[2] == sha):
                return {"read": float(parts[3]), "write": float(parts[4])}
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
# device timing helpers
# ---------------------------------------------------------------------------

def capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_graphs(graphs, launches_per_graph: int, min_launches: int = MIN_OP_LAUNCHES, min_ms: float = MIN_OP_MS):
    """Mean device time (ms) per launch over replays of `graphs` in turn (each
    graph holds launches_per_graph launches on distinct pool entries): at
    least min_launches launches and min_ms of device time, CUDA events on the
    current stream around the replays."""
    import torch
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    per_graph = max(e0.elapsed_time(e1) / len(graphs), 1e-4)
    reps = max(len(graphs), math.ceil(min_launches / launches_per_graph), math.ceil(min_ms / per_graph))
    e0.record()
    for i in range(reps):
        graphs[i % len(graphs)].replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * launches_per_graph)


def pool_count(bytes_each: float, l2: int, lo: int = 8, hi: int = 64) -> int:
    """Independent pool entries (a multiple of 8) totalling more than 4x L2."""
    return max(lo, min(hi, int(math.ceil(4 * l2 / max(bytes_each, 1) / 8)) * 8))


def l2_bytes(dev) -> int:
    import torch
    return getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)


# ---------------------------------------------------------------------------
# the single-layer step (flush, append, dequant, decode)
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

    def op(self, name):
        kv, w = self.kv, self.w
        if name == "flush_kv":
            kv.kivi_flush_kv(self.k, self.v, w.R, self.kst, self.vst)
        elif name == "residual_append":
            kv.kivi_residual_append_kv(self.k[:, self.n_flush:], self.v[:, self.n_flush:], self.kres, self.vres, 0,
                                       self.n_res)
        elif name == "dequant_kv":
            kv.kivi_dequant_kv(self.kst, self.vst, self.n_flush, kout=self.kdq, vout=self.vdq)
        else:
            kv.kivi_decode_attend(self.q, self.kst, self.vst, self.n_flush, self.kres, self.vres, self.n_res, w.Hkv,
                                  w.sm_scale, out=self.out, workspace=self.ws)

    def step(self):
        """One pass of the hot path. The flush and the dequant run on the
        current stream; the residual append and the decode (which needs the
        flushed store) run on a side stream beside the dequant; the side
        stream joins the current one at the end."""
        import torch
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            self.op("residual_append")
        self.op("flush_kv")
        self.flushed.record(main)
        self.op("dequant_kv")
        with torch.cuda.stream(self.side):
            self.side.wait_event(self.flushed)
            self.op("decode_attend")
        main.wait_stream(self.side)

    def nbytes(self):
        ts = [self.k, self.v, self.q, self.kres, self.vres, self.kdq, self.vdq, self.out, self.ws,
              self.kst.codes, self.kst.scale, self.kst.zero, self.vst.codes, self.vst.scale, self.vst.zero]
        return sum(t.numel() * t.element_size() for t in ts)


OPS = ["flush_kv", "residual_append", "dequant_kv", "decode_attend"]
OP_KERNEL_FILES = {"flush_kv": ["flush.cu"], "residual_append": ["residual.cu"], "dequant_kv": ["dequant.cu"],
                   "decode_attend": ["decode_pair.cu", "decode_mma.cuh", "decode_merge.cuh", "decode_common.cuh"]}
LAUNCHES = {"flush_kv": 1, "residual_append": 1, "dequant_kv": 1, "decode_attend": 1}


def workload_label(w) -> str:
    """The step's workload, named the same way by both arms."""
    return ("%s: single-layer prefill flush + residual append + dequant + decode "
            "(B=%d, H_kv=%d, Hq=%d, D=%d, S=%d, bits=%d, G=%d, residual_length=%d)"
            % (w.name, w.B, w.Hkv, w.Hq, w.D, w.S, w.bits, w.G, w.R))


class StepBench:
    """A rotating pool of instances of one workload, with CUDA graphs of
    GRAPH_STEPS steps (and of GRAPH_STEPS launches of each op) over distinct
    instances."""

    def __init__(self, kv, synth, w, dev, rank, pool_arg=0):
        self.kv, self.w, self.dev = kv, w, dev
        probe = Instance(w, 1000 * rank + 0, dev, kv, synth)
        self.inst_bytes = probe.nbytes()
        l2 = l2_bytes(dev)
        self.l2 = l2
        pool = pool_arg or int(min(64, max(2, math.ceil(4 * l2 / self.inst_bytes))))
        self.pool = max(GRAPH_STEPS, (pool + GRAPH_STEPS - 1) // GRAPH_STEPS * GRAPH_STEPS)
        self.insts = [probe] + [Instance(w, 1000 * rank + i, dev, kv, synth) for i in range(1, self.pool)]
        self.n_flush, self.n_res = probe.n_flush, probe.n_res

    def warm_and_capture(self, warmup):
        import torch
        for i in range(max(1, warmup)):
            self.insts[i % self.pool].step()
        torch.cuda.synchronize()

        branches = [torch.cuda.Stream(device=self.dev) for _ in range(GRAPH_BRANCHES)]

        def steps(j):
            # the graph's independent steps on GRAPH_BRANCHES parallel stream
            # branches (step t on branch t % GRAPH_BRANCHES; within a step the
            # flush -> dequant chain and, after the flush, the decode), all
            # joined at the end of the graph
            group = self.insts[j * GRAPH_STEPS:(j + 1) * GRAPH_STEPS]
            cur = torch.cuda.current_stream()
            for b in branches:
                b.wait_stream(cur)
            for t, inst in enumerate(group):
                with torch.cuda.stream(branches[t % GRAPH_BRANCHES]):
                    inst.step()
            for b in branches:
                cur.wait_stream(b)

        self.multi = [capture(lambda j=j: steps(j)) for j in range(self.pool // GRAPH_STEPS)]
        self.single = [capture(lambda I=I: I.step()) for I in self.insts]
        for i in range(max(1, warmup // GRAPH_STEPS)):
            self.multi[i % len(self.multi)].replay()
        torch.cuda.synchronize()

    def time_steps(self, steps, before=None):
        """Device ms of exactly `steps` steps between two CUDA events."""
        import torch
        if before:
            before()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        n_multi, n_rest = divmod(steps, GRAPH_STEPS)
        start.record()
        for i in range(n_multi):
            self.multi[i % len(self.multi)].replay()
        for i in range(n_rest):
            self.single[i % self.pool].replay()
        end.record()
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    def op_times(self, rounds=OP_ROUNDS):
        """Device ms per launch of each op: the median of `rounds` samples per
        op, taken in turn (flush, append, dequant, decode, flush, ...). A
        sample is CUDA events around replays of graphs of GRAPH_STEPS
        launches of the op alone on consecutive instances of the pool, with
        the step's launch configuration; each sample takes at least
        1/rounds of MIN_OP_LAUNCHES launches and of MIN_OP_MS."""
        import torch
        graphs, reps = {}, {}
        for op in OPS:
            gs = [capture(lambda j=j, op=op: [self.insts[j * GRAPH_STEPS + t].op(op) for t in range(GRAPH_STEPS)])
                  for j in range(self.pool // GRAPH_STEPS)]
            per_graph = max(time_graphs(gs, GRAPH_STEPS, min_launches=1, min_ms=0.0) * GRAPH_STEPS, 1e-4)
            reps[op] = max(len(gs), math.ceil(MIN_OP_LAUNCHES / (rounds * GRAPH_STEPS)),
                           math.ceil(MIN_OP_MS / (rounds * per_graph)))
            graphs[op] = gs
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        samples = {op: [] for op in OPS}
        for _ in range(rounds):
            for op in OPS:
                gs, n = graphs[op], reps[op]
                e0.record()
                for i in range(n):
                    gs[i % len(gs)].replay()
                e1.record()
                torch.cuda.synchronize()
                samples[op].append(e0.elapsed_time(e1) / (n * GRAPH_STEPS))
        del graphs
        return {op: statistics.median(samples[op]) for op in OPS}

    def summary(self, op_ms, peak, steps=None, elapsed_ms=None, world=1):
        w = self.w
        ob = op_bytes(w, self.n_flush, self.n_res)
        ops = {}
        for op in OPS:
            gbs = ob[op] / (op_ms[op] * 1e-3) / 1e9
            ops[op] = {"us": round(op_ms[op] * 1e3, 3), "bytes": int(ob[op]), "GB/s": round(gbs, 1),
                       "frac_of_peak": round(gbs / peak, 4)}
        d = {"workload": workload_label(w), "n_flush": self.n_flush, "n_res": self.n_res, "ops": ops,
             "step_bytes": int(sum(ob.values())),
             "decode_tokens_per_s": round(w.B / (op_ms["decode_attend"] * 1e-3), 1),
             "pool": "rotating pool of %d independent instances, %.0f MB total (L2 %d MB)"
                     % (self.pool, self.pool * self.inst_bytes / 2 ** 20, self.l2 >> 20)}
        if steps:
            d["steps"] = steps
            d["ms_per_step"] = round(elapsed_ms / steps, 6)
            d["GB/s"] = round(job_gbs(world, sum(ob.values()), steps, elapsed_ms), 2)
        return d


# ---------------------------------------------------------------------------
# decode cases, the batched decode and the streaming simulation
# ---------------------------------------------------------------------------

def time_decode_case(kv, synth, dev, B, S_q, n_res, bits, Hq=32, G=32, D=128, hs=False, Hkv=8, peak=None,
                     store_ready=False):
    """Mean device time of one decode over a rotating pool of independent
    stores (more than 4x L2 in total): graphs of 8 launches on distinct
    entries, at least 256 launches and 50 ms. store_ready: the decodes take
    KIVI_DECODE_STORE_READY (the preceding kernel is another decode, which
    does not write their stores)."""
    import torch
    w = synth.Workload("decode", B=B, Hkv=Hkv, Hq=Hq, D=D, S=S_q + n_res, bits=bits, G=G, R=0,
                       n_outlier=4, outlier_scale=8.0, seed=11)
    s_cap = max(1, -(-S_q // G)) * G
    meta = 4 if hs else 6
    nbytes = decode_bytes(B, Hkv, w.Hq, D, G, bits, S_q, n_res, meta)
    P = pool_count(nbytes, l2_bytes(dev))
    entries = []
    for i in range(P):
        k, v, q = synth.prefill_inputs_torch(w, 9000 + i, dev)
        gk = kv.KiviStore(0, w.BH, s_cap, D, G, bits, device=dev, scale_f16=hs)
        gv = kv.KiviStore(1, w.BH, s_cap, D, G, bits, device=dev, scale_f16=hs)
        if S_q > 0:
            kv.kivi_flush_kv(k, v, 0, gk, gv, n_tokens=S_q)
        kr = k[:, S_q:].contiguous()
        vr = v[:, S_q:].contiguous()
        out = torch.empty((B, w.Hq, D), dtype=torch.float32, device=dev)
        need = kv.kivi_decode_workspace_size(B, w.Hq, w.Hkv, S_q, n_res, D)
        entries.append((q, gk, gv, kr, vr, out, kv.kivi_decode_workspace(need, dev)))
        del k, v
    torch.cuda.synchronize()

    def fn(e):
        kv.kivi_decode_attend(e[0], e[1], e[2], S_q, e[3], e[4], n_res, w.Hkv, w.sm_scale, out=e[5], workspace=e[6],
                              store_ready=store_ready)

    for e in entries:
        fn(e)
    gs = [capture(lambda j=j: [fn(entries[8 * j + t]) for t in range(8)]) for j in range(P // 8)]
    ms = time_graphs(gs, 8)
    us = ms * 1e3
    gbs = nbytes / (ms * 1e-3) / 1e9
    plan = kv.kivi_decode_plan_info(B, w.Hq, w.Hkv, S_q, n_res, D, G, bits, hs)
    d = {"B": B, "Hkv": Hkv, "Hq": w.Hq, "S_kv": S_q + n_res, "S_q": S_q, "n_res": n_res, "bits": bits, "G": G,
         "D": D, "scale_f16": hs, "store_ready": store_ready, "us": round(us, 3), "bytes": int(nbytes),
         "GB/s": round(gbs, 1), "pool": P,
         "tokens_per_s": round(B / (ms * 1e-3), 1), "plan": plan}
    if peak:
        d["frac_of_peak"] = round(gbs / peak, 4)
    del entries, gs
    torch.cuda.empty_cache()
    return d


def run_batched(kv, synth, dev, peak, instances=2):
    """The batched decode workload: B=32 sequences, H_kv=8, 32 query heads,
    4096 cached tokens each (4032 packed + 64 fp16: a layer cache with
    residual_length 64 prefilled with 4096 tokens), then 30 steps that each
    append one token per sequence (kivi_cache_append) and decode one query
    token per head (kivi_cache_decode). Independent caches alternate step by
    step (their stores total more than L2, as the layers of a model would),
    so no step finds its store in L2. tokens/s = sequences * steps / time."""
    import torch
    w = synth.WORKLOADS["batched"]
    R, steps = 64, w.steps
    caches, toks, wss = [], [], []
    gen = torch.Generator(device=dev)
    gen.manual_seed(32)
    for i in range(instances):
        k, v, _ = synth.prefill_inputs_torch(w, 31 + i, dev)
        c = kv.KiviCache(w.BH, w.S_q, w.D, w.G, w.bits, R, device=dev)
        assert c.prefill(k, v) == w.S_q and c.n_res == w.n_res
        del k, v
        nk = torch.randn((steps, w.BH, 1, w.D), generator=gen, device=dev).half()
        nv = torch.randn((steps, w.BH, 1, w.D), generator=gen, device=dev).half()
        qs = torch.randn((steps, w.B, w.Hq, w.D), generator=gen, device=dev).half()
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
        need = kv.kivi_decode_workspace_size(w.B, w.Hq, w.Hkv, w.S_q, w.n_res + steps, w.D)
        caches.append(c)
        toks.append((nk, nv, qs, out))
        wss.append(kv.kivi_decode_workspace(need, dev))
    states = [c.state() for c in caches]

    def run_steps():
        for s in range(steps):
            for c, (nk, nv, qs, out), ws in zip(caches, toks, wss):
                c.append(nk[s], nv[s])
                c.decode(qs[s], w.Hkv, w.sm_scale, out=out, workspace=ws)

    run_steps()  # eager warm-up (loads the kernels, sets attributes)
    torch.cuda.synchronize()
    for c, st in zip(caches, states):
        c.set_state(*st)
    g = capture(run_steps)  # every replay appends the same tokens at the same rows
    for c, st in zip(caches, states):
        c.set_state(*st)
    ms = time_graphs([g], instances * steps, min_launches=1, min_ms=200.0)  # per (cache, step)
    us = ms * 1e3
    per_step = sum(decode_bytes(w.B, w.Hkv, w.Hq, w.D, w.G, w.bits, w.S_q, w.n_res + i + 1)
                   + w.BH * w.D * 2 * 2 * 2 for i in range(steps)) / steps
    gbs = per_step / (ms * 1e-3) / 1e9
    return {"workload": "batched: B=32, H_kv=8, Hq=32, D=128, 4-bit, G=32, 4032 packed + 64 fp16 tokens, "
                        "30 steps of append 1 token + decode",
            "us_per_step": round(us, 3), "tokens_per_s": round(w.B / (ms * 1e-3), 1),
            "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "bytes_per_step": int(per_step),
            "l2": "%d independent caches alternate step by step (%.0f MB of stores)"
                  % (instances, instances * w.BH * w.S_q * 176 / 2 ** 20)}


def run_stream_sim(kv, synth, dev, peak, steps=3072, L=36):
    """The streaming serving simulation of the KV-cache work: L layers, B=16,
    H_kv=8, Hq=32, D=128, 4-bit, G=32, R=128, context growing from 1024
    tokens by one token per step. Each layer-step is kivi_cache_append of the
    new token's K and V (which flushes G tokens into the store whenever the
    window reaches R + G tokens; the window buffer holds R + 4G tokens, so
    the remaining R tokens move back to its row 0 once per 4 flushes) and
    kivi_cache_decode of one query token per head. The launches of each 32-step flush cycle (all
    layers) are captured in a CUDA graph beforehand; the timed region replays
    them all. tokens/s = B * steps / time (KV-cache work only: no projections
    or MLP)."""
    import torch
    B, Hkv, Hq, D, G, R, bits = 16, 8, 32, 128, 32, 128, 4
    ctx0 = 1024
    steps = (steps // G) * G
    BH = B * Hkv
    s_cap = ctx0 + steps
    w = synth.Workload("stream", B=B, Hkv=Hkv, Hq=Hq, D=D, S=ctx0, bits=bits, G=G, R=R, n_outlier=4,
                       outlier_scale=8.0, seed=5)
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    new_k = torch.randn((BH, G, D), generator=gen, device=dev).to(torch.float16)  # tokens appended, cyclically
    new_v = torch.randn((BH, G, D), generator=gen, device=dev).to(torch.float16)
    qs = torch.randn((G, B, Hq, D), generator=gen, device=dev).to(torch.float16)
    caches, outs = [], []
    for layer in range(L):
        k, v, _ = synth.prefill_inputs_torch(w, 100 + layer, dev)
        c = kv.KiviCache(BH, s_cap, D, G, bits, R, res_cap=R + 4 * G, device=dev)
        c.prefill(k, v)
        caches.append(c)
        outs.append(torch.empty((B, Hq, D), dtype=torch.float32, device=dev))
        del k, v
    S_q0, n_res0 = caches[0].state()[:2]
    need = max(kv.kivi_decode_workspace_size(B, Hq, Hkv, sq, nr, D)  # the largest plan of any step
               for sq in range(S_q0, s_cap + 1, G) for nr in range(R, R + G + 1))
    ws = kv.kivi_decode_workspace(need, dev)

    def layer_step(c, out, i):
        c.append(new_k[:, i % G:i % G + 1], new_v[:, i % G:i % G + 1])
        c.decode(qs[i % G], Hkv, w.sm_scale, out=out, workspace=ws)

    # one eager layer-step per layer loads the kernels; the counters are then
    # restored (the graphs rewrite the appended rows)
    snapshot = [c.state() for c in caches]
    for c, out in zip(caches, outs):
        layer_step(c, out, 0)
    torch.cuda.synchronize()
    for c, st in zip(caches, snapshot):
        c.set_state(*st)
    graphs = []
    for cyc in range(steps // G):
        graphs.append(capture(lambda cyc=cyc: [layer_step(c, out, cyc * G + j)
                                               for j in range(G) for c, out in zip(caches, outs)]))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    # algorithmic bytes: the decodes, the appends and the flushes (the window
    # compaction moves are not counted)
    total = 0.0
    S_q, n_res = S_q0, n_res0
    flush_b = 2 * BH * G * D * (2 + bits / 8 + 6 / G)
    for i in range(steps):
        n_res += 1
        total += BH * D * 2 * 2 * 2
        if n_res >= R + G:
            S_q += G
            n_res -= G
            total += flush_b
        total += decode_bytes(B, Hkv, Hq, D, G, bits, S_q, n_res)
    total *= L
    assert (S_q, n_res) == caches[0].state()[:2]
    gbs = total / (ms * 1e-3) / 1e9
    return {"workload": "stream: %d layers, B=16, H_kv=8, Hq=32, D=128, 4-bit, G=32, R=128, context %d -> %d"
                        % (L, ctx0, ctx0 + steps),
            "steps": steps, "ms": round(ms, 3), "tokens_per_s": round(B * steps / (ms * 1e-3), 1),
            "us_per_layer_step": round(ms * 1e3 / (steps * L), 3), "flushes_per_layer": steps // G,
            "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "note": "KV-cache work only (append and decode per layer-step, a flush every 32 steps, the window "
                    "moved back to its row 0 every 128 steps); no projections or MLP; bytes exclude the "
                    "window moves"}


# ---------------------------------------------------------------------------
# the GB300 arm
# ---------------------------------------------------------------------------

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
    peak, peak_kind = measured_peaks()

    sb = StepBench(kv, synth, w, dev, rank, args.pool)
    sb.warm_and_capture(args.warmup)

    gpu_id = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local_rank)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.2)
    barrier = (lambda: torch.distributed.barrier()) if world > 1 else None
    elapsed_ms = sb.time_steps(args.steps, before=barrier)
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    # per-op average launch duration (CUDA events on the launching stream,
    # graphs of GRAPH_STEPS launches of the op alone), in the same clock window
    op_ms = sb.op_times()
    clock = clocks.stop()

    summ = sb.summary(op_ms, peak)
    ob = op_bytes(w, sb.n_flush, sb.n_res)
    step_bytes = sum(ob.values())
    ms_per_step = elapsed_ms / args.steps
    value = job_gbs(world, step_bytes, args.steps, elapsed_ms)
    dom = max(OPS, key=lambda o: op_ms[o])
    achieved = ob[dom] / (op_ms[dom] * 1e-3) / 1e9
    traffic = read_traffic(OP_KERNEL_FILES[dom], dom, w.name)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": peak_kind + " hbm_gbs (copy, burst)", "unit": "GB/s", "nominal_peak": NOMINAL_HBM_GBS,
                "frac": round(achieved / peak, 4),
                "traffic": None if traffic is None else traffic["read"] + traffic["write"],
                "traffic_read": None if traffic is None else traffic["read"],
                "algorithmic_bytes": int(ob[dom]),
                "algorithmic_read_bytes": int(op_read_bytes(w, sb.n_flush, sb.n_res)[dom]),
                "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch at this workload; "
                                "writes a launch leaves in L2 are not counted"}

    # end to end: host inputs (pinned) -> device, the step, result -> host.
    # Each instance's public-API calls (the copies of its K, V and q from
    # pinned host buffers, the step, the copy of its output back) are
    # captured once as a CUDA graph, as a serving loop would; graphs of
    # independent instances alternate between streams, so the copies of
    # one step overlap the kernels of another. Every step moves its inputs
    # and its result through the copy engines inside the timed region.
    e2e = None
    insts = sb.insts
    if args.e2e_steps > 0:
        nl = max(1, args.e2e_streams)
        ne = min(sb.pool, max(2 * nl, 4))  # instances: two per stream, at least 4
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
        del e2e_graphs, hk, hv, hq
    del sb, insts
    torch.cuda.empty_cache()

    # the other workloads (one GPU only; each timed on its own)
    extra = {}
    if world == 1 and not args.no_extra:
        if w.name != "qwen8b":
            sq = StepBench(kv, synth, synth.WORKLOADS["qwen8b"], dev, rank)
            sq.warm_and_capture(16)
            q_steps = 2000
            q_ms = sq.time_steps(q_steps)
            extra["qwen8b"] = sq.summary(sq.op_times(), peak, q_steps, q_ms)
            del sq
            torch.cuda.empty_cache()
        extra["batched_decode"] = run_batched(kv, synth, dev, peak)
        torch.cuda.empty_cache()
        extra["stream"] = run_stream_sim(kv, synth, dev, peak, args.stream_steps)
        torch.cuda.empty_cache()
        extra["decode_b1"] = [time_decode_case(kv, synth, dev, 1, S - 128, 128, bits, peak=peak, store_ready=sr)
                              for S, bits in ((4096, 4), (8192, 4), (16384, 4), (32768, 2)) for sr in (False, True)]
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle(w, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_label(w),
                   "n_flush": summ["n_flush"], "n_res": summ["n_res"],
                   "l2": summ["pool"],
                   "timing": "graphs of %d independent steps on distinct instances over %d stream branches, "
                             "K steps between CUDA events" % (GRAPH_STEPS, GRAPH_BRANCHES),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "ops": summ["ops"],
        "decode_tokens_per_s": summ["decode_tokens_per_s"],
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(LAUNCHES.values()) * args.steps,
        "clocks": clock,
        "peak_hbm_gbs": peak,
        "per_op_timing": "median of %d samples per op taken in turn with the other ops; a sample is CUDA events "
                         "around graphs of %d back-to-back launches of the op on distinct instances; at least %d "
                         "launches and %.0f ms per op" % (OP_ROUNDS, GRAPH_STEPS, MIN_OP_LAUNCHES, MIN_OP_MS),
    }
    line.update(extra)
    return line


# ---------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name from /proc/cpuinfo (implementer and part on
    Arm, whose cpuinfo has no model name)."""
    impl = part = None
    try:
        for ln in open("/proc/cpuinfo"):
            key, _, val = ln.partition(":")
            key, val = key.strip().lower(), val.strip()
            if key == "model name":
                return val
            if key == "cpu implementer" and impl is None:
                impl = val
            if key == "cpu part" and part is None:
                part = val
    except OSError:
        pass
    if impl or part:
        return "%s implementer %s part %s" % (platform.machine(), impl, part)
    return platform.processor() or platform.machine()


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

    if threads == 1:
        for bh in range(w.BH):
            head(bh)
        return
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(head, range(w.BH)))


def _time_oracle(w, k, v, q, threads, seconds, min_steps=1):
    done, times, t0 = 0, [], time.perf_counter()
    while True:
        t = time.perf_counter()
        cpu_oracle_step(w, k, v, q, threads)
        times.append(time.perf_counter() - t)
        done += 1
        if done >= min_steps and time.perf_counter() - t0 >= seconds:
            break
    return done, sum(times)


def cpu_oracle(w, seconds):
    """Time the oracle on the host cores: whole steps for about seconds / 2
    with one KV head per thread on up to BH threads, then whole steps for
    about seconds / 2 on one thread."""
    from kivi_kv_cache_gb300 import synth
    import oracle
    oracle.build()
    k, v, q = synth.prefill_inputs(w)
    threads = max(1, min(os.cpu_count() or 1, w.BH))
    cpu_oracle_step(w, k, v, q, threads)  # warm (page in, build)
    n = oracle.flush_count(w.S, w.R, w.G)
    step_bytes = sum(op_bytes(w, n, w.S - n).values())
    done, total = _time_oracle(w, k, v, q, threads, seconds / 2)
    done1, total1 = _time_oracle(w, k, v, q, 1, seconds / 2)
    return {"value": round(step_bytes * done / total / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d whole steps of the %s workload (C oracle, one KV head per thread), %.1f s"
                      % (done, w.name, total),
            "ms_per_step": round(1e3 * total / done, 3),
            "single_thread": {"value": round(step_bytes * done1 / total1 / 1e9, 4), "unit": "GB/s",
                              "ms_per_step": round(1e3 * total1 / done1, 3),
                              "sample": "%d whole steps on one thread, %.1f s" % (done1, total1)},
            "cpu_model": cpu_model(), "host_cores": os.cpu_count()}


def run_reference(args, rank, world):
    from kivi_kv_cache_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    import oracle
    oracle.build()
    k, v, q = synth.prefill_inputs(w)
    threads = max(1, min(os.cpu_count() or 1, w.BH))
    t = time.perf_counter()
    cpu_oracle_step(w, k, v, q, threads)  # one warm-up step, also the size of a step
    one = time.perf_counter() - t
    for _ in range(max(0, min(args.warmup, 2) - 1)):
        cpu_oracle_step(w, k, v, q, threads)
    # a bounded sample of whole steps (about a minute at most)
    steps = max(1, min(args.steps, int(60.0 / max(one, 1e-3))))
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
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# sweeps
# ---------------------------------------------------------------------------

def run_sweep(args):
    """Per-op throughput at larger sizes (one JSON line per measurement).

    Each measurement: a rotating pool of independent inputs totalling more than
    4x L2, CUDA graphs of 8 launches of the op on distinct pool entries, CUDA
    events around at least 256 launches and 50 ms; GB/s = algorithmic bytes /
    mean duration."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import kivi_kv_cache_gb300 as kv
    from kivi_kv_cache_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = l2_bytes(dev)
    peak, kind = measured_peaks()

    def emit(label, nbytes, ms, extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        line = {"op": label, "us": round(ms * 1e3, 3), "bytes": int(nbytes), "GB/s": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4), "peak": peak, "peak_kind": kind}
        line.update(extra)
        print(json.dumps(line), flush=True)

    def timed(fns, nbytes, label, extra):
        gs = [capture(lambda j=j: [f() for f in fns[8 * j:8 * j + 8]]) for j in range(len(fns) // 8)]
        emit(label, nbytes, time_graphs(gs, 8), extra)
        del gs

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
        P = pool_count(per, l2)
        ks, vs, kd, vd, xs = [], [], [], [], []
        for i in range(P):
            k, v, _ = synth.prefill_inputs_torch(w, 7000 + i, dev)
            xs.append((k, v))
            ks.append(kv.KiviStore(0, w.BH, n, w.D, w.G, w.bits, device=dev, scale_f16=hs))
            vs.append(kv.KiviStore(1, w.BH, n, w.D, w.G, w.bits, device=dev, scale_f16=hs))
            kd.append(torch.empty((w.BH, n, w.D), dtype=torch.float16, device=dev))
            vd.append(torch.empty_like(kd[-1]))
        ob = op_bytes(w, n, w.S - n, meta_bytes=meta)
        ex = {"workload": name, "tokens": n, "bits": w.bits, "G": G, "D": D, "scale_f16": hs, "pool": P}
        timed([lambda i=i: kv.kivi_flush_kv(xs[i][0], xs[i][1], w.R, ks[i], vs[i]) for i in range(P)],
              ob["flush_kv"], "flush_kv", ex)
        timed([lambda i=i: kv.kivi_dequant_kv(ks[i], vs[i], n, kout=kd[i], vout=vd[i]) for i in range(P)],
              ob["dequant_kv"], "dequant_kv", ex)
        # fake quantization of the same tokens: read 2 B and write 2 B per element of K and V (the kd/vd
        # buffers hold the n flushed tokens, so the S - n fp16 tokens are not part of this launch)
        timed([lambda i=i: kv.kivi_fake_quant_kv(xs[i][0][:, :n], xs[i][1][:, :n], 0, kout=kd[i], vout=vd[i],
                                                 G=G, bits=w.bits, scale_f16=hs) for i in range(P)],
              2 * w.BH * n * w.D * 4, "fake_quant_kv", ex)
        del ks, vs, kd, vd, xs
        torch.cuda.empty_cache()

    if args.sweep in ("all", "decode"):
        # decode over a packed store + fp16 residual
        # (B, packed tokens, fp16 residual tokens, bits[, Hq, G, D, fp16 scales]): the qwen8b decode, the
        # long-context and batched decodes, and the streaming workload's S_kv sweep (128 / 512 / 2048 /
        # 8192 / 16384 at B=1 and B=16)
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
            d = time_decode_case(kv, synth, dev, B, S_q, n_res, bits, Hq=case[4] if len(case) > 4 else 32,
                                 G=case[5] if len(case) > 5 else 32, D=case[6] if len(case) > 6 else 128,
                                 hs=case[7] if len(case) > 7 else False, peak=peak)
            d.update({"op": "decode_attend", "peak": peak, "peak_kind": kind})
            print(json.dumps(d), flush=True)
        print(json.dumps(dict(op="batched_decode_steps", **run_batched(kv, synth, dev, peak))), flush=True)

    if args.sweep in ("all", "twopass"):
        run_twopass_sweep(kv, synth, dev, peak, kind)


def run_twopass_sweep(kv, synth, dev, peak, kind):
    """Two-pass "decode-once" against the fused decode over S_kv x B, every
    arm over its own rotating pool of independent inputs (L2-cold). The
    store changes only when a flush folds G tokens in, so a two-pass decoder
    dequantizes it once per G steps and attends over an all-fp16 cache every
    step: its cost per step is attend + dequant / G. The fp16 attend arm runs
    the decode kernels over S_q = 0 and S_kv fp16 tokens. Also reported: the
    two-pass cost at the HBM bound (its bytes at the measured peak), a lower
    bound for any fp16 attend kernel."""
    import torch
    l2 = l2_bytes(dev)
    G, bits, D, Hkv, Hq, n_res = 32, 4, 128, 8, 32, 64
    for B in (1, 16, 32):
        for S in (512, 1024, 2048, 3072, 4096, 8192):
            S_q = S - n_res
            fused = time_decode_case(kv, synth, dev, B, S_q, n_res, bits, peak=peak)
            att = time_decode_case(kv, synth, dev, B, 0, S, bits, peak=peak)
            # dequant of the S_q store tokens, rotating pool
            w = synth.Workload("twopass", B=B, Hkv=Hkv, Hq=Hq, D=D, S=S, bits=bits, G=G, R=0, n_outlier=4,
                               outlier_scale=8.0, seed=12)
            deq_b = 2 * w.BH * S_q * D * (2 + bits / 8 + 6 / G)
            P = pool_count(deq_b, l2)
            ent = []
            for i in range(P):
                k, v, _ = synth.prefill_inputs_torch(w, 500 + i, dev, S=S_q)
                gk = kv.KiviStore(0, w.BH, S_q, D, G, bits, device=dev)
                gv = kv.KiviStore(1, w.BH, S_q, D, G, bits, device=dev)
                kv.kivi_flush_kv(k, v, 0, gk, gv)
                ent.append((gk, gv, k, v))  # the inputs' buffers take the fp16 output
            gs = [capture(lambda j=j: [kv.kivi_dequant_kv(e[0], e[1], S_q, kout=e[2], vout=e[3])
                                       for e in ent[8 * j:8 * j + 8]]) for j in range(P // 8)]
            deq_ms = time_graphs(gs, 8)
            del gs, ent
            torch.cuda.empty_cache()
            two = att["us"] + deq_ms * 1e3 / G
            bound = (att["bytes"] + deq_b / G) / (peak * 1e9) * 1e6
            print(json.dumps({"op": "decode_two_pass_vs_fused", "B": B, "S_kv": S, "S_q": S_q, "n_res": n_res,
                              "bits": bits, "fused_us": fused["us"], "fp16_attend_us": att["us"],
                              "dequant_us": round(deq_ms * 1e3, 3), "two_pass_us_per_step": round(two, 3),
                              "two_pass_at_hbm_bound_us": round(bound, 3),
                              "fused_over_two_pass": round(two / fused["us"], 3),
                              "fused_over_two_pass_bound": round(bound / fused["us"], 3),
                              "fused_GB/s": fused["GB/s"], "fp16_attend_GB/s": att["GB/s"], "peak": peak,
                              "peak_kind": kind, "note": "every arm over a rotating pool (L2-cold)"}), flush=True)


def run_stream(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import kivi_kv_cache_gb300 as kv
    from kivi_kv_cache_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = measured_peaks()
    d = run_stream_sim(kv, synth, dev, peak, args.stream_steps)
    d.update({"op": "stream_simulation", "peak": peak, "peak_kind": kind})
    print(json.dumps(d), flush=True)


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
    if kind == "step":  # one instance of the bench's step, eagerly (flush, append, dequant, decode)
        inst = Instance(synth.WORKLOADS[name.split("_")[1]], 1, dev, kv, synth)
        for _ in range(reps):
            inst.step()
    elif kind == "flush":
        parts = name.split("_")
        w = synth.WORKLOADS[parts[1]]
        if len(parts) > 2 and parts[2].startswith("g"):
            w = dataclasses.replace(w, G=int(parts[2][1:]))
        hs = parts[-1] == "f16s"  # fp16 scale storage
        n = kv.kivi_flush_count(w.S, w.R, w.G)
        k, v, _ = synth.prefill_inputs_torch(w, 1, dev)
        ks = kv.KiviStore(0, w.BH, n, w.D, w.G, w.bits, device=dev, scale_f16=hs)
        vs = kv.KiviStore(1, w.BH, n, w.D, w.G, w.bits, device=dev, scale_f16=hs)
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
