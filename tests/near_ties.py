"""Quantizer groups whose quotients sit on or next to a half-integer.

KIVI's codes are q = rint(RN(RN(x - min) / scale)) with round half to even
(VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly 0%
Faster", "Three ways to be off by one bit", #2: exact .5 quotients are common
in real quantization). A kernel that approximates the quotient must take the
same decision as the IEEE division at and near those half-integers. This
module builds such groups for the tests: for a (min, max) pair it lists every
fp16 value x in [min, max] whose fp32 quotient (x - min) / scale lies within
2^-14 of k + 1/2 (exact ties included), and those just outside that band
(2^-14 to 2^-11 away), using numpy's IEEE fp32 arithmetic only.

Test infrastructure: it shares nothing with the CUDA path or the oracle.
"""
from __future__ import annotations

import numpy as np

BAND = 2.0 ** -14

_ALL_F16 = None


def all_finite_f16() -> np.ndarray:
    """Every finite fp16 value, ascending, as float32."""
    global _ALL_F16
    if _ALL_F16 is None:
        h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
        h = h[np.isfinite(h)].astype(np.float32)
        _ALL_F16 = np.unique(h)  # -0.0 and +0.0 collapse
    return _ALL_F16


def group_scale(lo: np.float32, hi: np.float32, bits: int, scale_f16: bool) -> np.float32:
    """RN32(RN32(hi - lo) / (2^bits - 1)), rounded to fp16 when stored as fp16."""
    s = np.float32(np.float32(hi - lo) / np.float32((1 << bits) - 1))
    return np.float32(np.float16(s)) if scale_f16 else s


def quotient_distance(x: np.ndarray, lo: np.float32, s: np.float32) -> np.ndarray:
    """|frac(RN32(RN32(x - lo) / s)) - 1/2| for each x (float64)."""
    q = (x.astype(np.float32) - lo) / s  # numpy fp32: IEEE subtraction and division
    q = q.astype(np.float64)
    return np.abs(q - np.floor(q) - 0.5)


def candidates(lo: float, hi: float, bits: int, scale_f16: bool):
    """(near, edge, scale): fp16 values of [lo, hi] whose quotient is within
    the band of a half-integer, those just outside it (up to 2^-11), and the
    group's scale."""
    v = all_finite_f16()
    lo32, hi32 = np.float32(np.float16(lo)), np.float32(np.float16(hi))
    s = group_scale(lo32, hi32, bits, scale_f16)
    if not s > 0:
        return v[:0], v[:0], s
    x = v[(v >= lo32) & (v <= hi32)]
    d = quotient_distance(x, lo32, s)
    return x[d < BAND], x[(d >= BAND) & (d < 2.0 ** -11)], s


def tie_configs(rng: np.random.Generator, bits: int, scale_f16: bool, configs: int = 48):
    """(lo, hi, near, edge) for `configs` (min, max) pairs that have near-tie
    candidates: ranges over several decades, some on a coarse grid where
    exact ties abound."""
    out = []
    while len(out) < configs:
        if rng.random() < 0.3:
            lo = float(rng.integers(-8, 8)) * 0.25
            hi = lo + float(rng.integers(1, 40)) * 0.25
        else:
            lo = float(rng.standard_normal() * 10 ** rng.uniform(-2, 1.5))
            hi = lo + float(10 ** rng.uniform(-2.5, 2))
        lo16, hi16 = np.float16(lo), np.float16(hi)
        if not (np.isfinite(lo16) and np.isfinite(hi16)) or hi16 <= lo16:
            continue
        near, edge, _ = candidates(float(lo16), float(hi16), bits, scale_f16)
        if len(near) == 0:
            continue
        out.append((lo16, hi16, near, edge))
    return out


def tie_groups(rng: np.random.Generator, n: int, G: int, bits: int, scale_f16: bool, configs: int = 48):
    """n groups of G fp16 values: each holds its min and max once and G - 2
    values drawn from the near-tie (70 %) and band-edge candidates of one
    (min, max) pair, in random order. Returns (groups [n, G] fp16, number of
    near-tie elements)."""
    cfg = tie_configs(rng, bits, scale_f16, configs)
    which = rng.integers(len(cfg), size=n)
    out = np.empty((n, G), np.float16)
    n_near = 0
    for ci, (lo, hi, near, edge) in enumerate(cfg):
        idx = np.nonzero(which == ci)[0]
        if len(idx) == 0:
            continue
        pick_near = rng.choice(near, size=(len(idx), G - 2))
        if len(edge):
            pick_edge = rng.choice(edge, size=(len(idx), G - 2))
            use_near = rng.random((len(idx), G - 2)) < 0.7
            vals = np.where(use_near, pick_near, pick_edge)
        else:
            use_near = np.ones((len(idx), G - 2), bool)
            vals = pick_near
        n_near += int(use_near.sum())
        rows = np.concatenate([np.full((len(idx), 1), lo, np.float32), np.full((len(idx), 1), hi, np.float32),
                               vals.astype(np.float32)], axis=1)
        perm = np.argsort(rng.random((len(idx), G)), axis=1)
        out[idx] = np.take_along_axis(rows, perm, axis=1).astype(np.float16)
    return out, n_near
