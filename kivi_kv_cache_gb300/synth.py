"""Seeded synthetic inputs for the KIVI workloads.

This module holds no quantization or attention arithmetic: it only draws
random fp16 tensors with the shapes and value distributions of the workloads
the KIVI pages measure, so the same bytes can feed the CUDA path and the CPU
oracle.

Distributions (the pages measure real models; these stand in for them):
  * keys:    N(0, 1) with a fixed set of outlier channels scaled by a factor
             (keys carry a few channels with consistently huge magnitudes --
             VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM
             Exactly 0% Faster", "What we're actually optimizing");
  * values:  N(0, 1);
  * queries: N(0, 1).
All draws come from ``numpy.random.default_rng(seed)`` and are rounded to fp16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hkv: int
    Hq: int
    D: int
    S: int                 # tokens in the prefill call (or cached tokens)
    bits: int
    G: int
    R: int                 # residual_length
    n_outlier: int
    outlier_scale: float
    seed: int
    # batched decode: tokens already flushed / residual tokens / steps
    S_q: int = 0
    n_res: int = 0
    steps: int = 0
    # streaming: layers, context range and decode-sweep lengths
    layers: int = 1
    ctx_end: int = 0
    sweep: tuple = ()

    @property
    def BH(self) -> int:
        return self.B * self.Hkv

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    # Tiny correctness case: 2 heads, 256 tokens, the first 128 flushed.
    "tiny": Workload("tiny", B=1, Hkv=2, Hq=2, D=128, S=256, bits=4, G=32, R=128,
                     n_outlier=4, outlier_scale=10.0, seed=1),
    # Qwen3-8B-like single layer: GQA 32:8, D=128, 2238-token prompt, 4-bit.
    "qwen8b": Workload("qwen8b", B=1, Hkv=8, Hq=32, D=128, S=2238, bits=4, G=32, R=128,
                       n_outlier=4, outlier_scale=8.0, seed=2),
    # Long context, 2-bit.
    "long2bit": Workload("long2bit", B=1, Hkv=8, Hq=32, D=128, S=32768, bits=2, G=32, R=128,
                         n_outlier=4, outlier_scale=8.0, seed=3),
    # Batched decode: 32 sequences of 4096 cached tokens (4032 packed + 64 fp16).
    "batched": Workload("batched", B=32, Hkv=8, Hq=32, D=128, S=4096, bits=4, G=32, R=128,
                        n_outlier=4, outlier_scale=8.0, seed=4, S_q=4032, n_res=64, steps=30),
    # Streaming serving: 36 layers, B=16, context 1024 -> 4096.
    "stream": Workload("stream", B=16, Hkv=8, Hq=32, D=128, S=1024, bits=4, G=32, R=128,
                       n_outlier=4, outlier_scale=8.0, seed=5, layers=36, ctx_end=4096,
                       sweep=(128, 512, 2048, 8192, 16384)),
}


def outlier_channels(w: Workload) -> np.ndarray:
    """The fixed outlier channel indices of a workload (same for every head)."""
    rng = np.random.default_rng(10_000 + w.seed)
    return np.sort(rng.choice(w.D, size=w.n_outlier, replace=False))


def keys(rng: np.random.Generator, shape, D: int, channels: np.ndarray, factor: float) -> np.ndarray:
    x = rng.standard_normal(size=tuple(shape) + (D,), dtype=np.float32)
    x[..., channels] *= np.float32(factor)
    return x.astype(np.float16)


def normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=tuple(shape), dtype=np.float32).astype(np.float16)


def prefill_inputs(w: Workload, S: int | None = None, seed: int | None = None):
    """K, V [B*Hkv, S, D] fp16 and q [B, Hq, D] fp16 for a prefill-then-decode call."""
    S = w.S if S is None else S
    rng = np.random.default_rng(w.seed if seed is None else seed)
    ch = outlier_channels(w)
    k = keys(rng, (w.BH, S), w.D, ch, w.outlier_scale)
    v = normal(rng, (w.BH, S, w.D))
    q = normal(rng, (w.B, w.Hq, w.D))
    return k, v, q


def step_tokens(rng: np.random.Generator, w: Workload, n: int = 1):
    """n new tokens of K, V [B*Hkv, n, D] and one query [B, Hq, D]."""
    ch = outlier_channels(w)
    k = keys(rng, (w.BH, n), w.D, ch, w.outlier_scale)
    v = normal(rng, (w.BH, n, w.D))
    q = normal(rng, (w.B, w.Hq, w.D))
    return k, v, q


def prefill_inputs_torch(w: Workload, seed: int, device, S: int | None = None):
    """Device-side draw with the same distributions as prefill_inputs (for
    large input pools; seeded with torch's generator, so the values differ
    from the numpy draw of the same seed)."""
    import torch
    S = w.S if S is None else S
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    ch = torch.as_tensor(outlier_channels(w), device=device)
    k = torch.randn((w.BH, S, w.D), generator=g, device=device, dtype=torch.float32)
    k[..., ch] *= w.outlier_scale
    v = torch.randn((w.BH, S, w.D), generator=g, device=device, dtype=torch.float32)
    q = torch.randn((w.B, w.Hq, w.D), generator=g, device=device, dtype=torch.float32)
    return k.half(), v.half(), q.half()
