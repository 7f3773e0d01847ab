"""The flush kernel's scale and fast quotient, restated from their derivation
and checked on the CPU.

KIVI's code is q = rint(RN(a / s)) with a = RN(x - min) and s the group's
scale RN((max - min) / (2^bits - 1)), rounded half to even (VeloxQuant-MLX
blog, "A 5.65x Metal Kernel That Made My LLM Exactly 0% Faster", "What we're
actually optimizing"; "Three ways to be off by one bit", #2: exact .5
quotients are common in real quantization).

The scale: the kernel divides by the constant L = 2^bits - 1 with one
multiply by c = RN(1 / L), the fma remainder x - q L and one fma correction.
test_scale_division_every_fp32 checks, with a C program that uses IEEE float
division and fmaf, that this equals RN(x / L) for every non-negative finite
fp32 x, for L = 3 and 15.

The quotient avoids the IEEE division for all but near-ties:
 (1) r = 1 / s to within 1 ulp (rcp.approx.f32): r = (1 / s)(1 + e) with
     |e| <= 2^-23, so the exact product a r differs from a / s by at most
     (a / s) 2^-23;
 (2) RN(a / s) differs from a / s by at most half an ulp;
     with fp32 scales a / s <= 2^bits - 1 < 16, so (1) + (2) gives
     |a r - RN(a / s)| <= 2^-19 + 2^-21 < 2^-18; with fp16 scales a subnormal
     scale lets the quotient reach about 1.5 (2^bits - 1) < 32, and the bound
     is 2^-18 + 2^-20 < 2^-17;
 (3) one fma rounds a r half to even (q = rint(a r)) and a second measures
     f = RN32(a r - q); when |f| <= 1/2 - 2^-14, a r is at least
     2^-14 - 2^-26 from the nearest half-integer, farther than RN(a / s) can
     stray, so rint(RN(a / s)) = q; otherwise the kernel divides.
The tests draw (a, s) as the quantizer forms them, from random fp16 groups
and from near-tie groups (tests/near_ties.py), and check (1)-(3) with exact
float64 arithmetic (a r is exact in float64: 24 x 24 significant bits) for r
= RN(1 / s) and for its neighbours one ulp below and above (the extremes a
1-ulp reciprocal can return)."""
import numpy as np
import pytest

import near_ties


def _check(a: np.ndarray, s: np.ndarray, scale_f16: bool):
    """(1)-(3) for fp32 arrays a >= 0, s > 0, for r = RN(1/s) and its two
    1-ulp neighbours; returns the fast-path mask of r = RN(1/s)."""
    r0 = (np.float32(1.0) / s).astype(np.float32)
    qd = (a / s).astype(np.float32).astype(np.float64)    # RN32(a / s)
    assert np.all(qd < (32.0 if scale_f16 else 16.0))
    bound = 2.0 ** -17 if scale_f16 else 2.0 ** -18
    masks = []
    for r in (r0, np.nextafter(r0, np.float32(0)), np.nextafter(r0, np.float32(np.inf))):
        ar = a.astype(np.float64) * r.astype(np.float64)  # exact
        assert np.all(np.abs(ar - qd) <= bound), float(np.max(np.abs(ar - qd)))
        q = np.rint(ar)                                   # fma RN(a r + 2^23) - 2^23: half to even
        f = (ar - q).astype(np.float32)                   # fma RN(a r - q): exact difference, one rounding
        fast = np.abs(f) <= np.float32(0.5 - 2.0 ** -14)
        assert np.array_equal(q[fast], np.rint(qd)[fast])
        masks.append(fast)
    return masks[0]


def _random_pairs(rng, n, bits, scale_f16):
    """(a, s) of random fp16 groups: min and max over several decades, x in between."""
    lo = (rng.standard_normal(n) * 10 ** rng.uniform(-3, 2, n)).astype(np.float16).astype(np.float32)
    hi = (lo + 10 ** rng.uniform(-3, 2.5, n)).astype(np.float16).astype(np.float32)
    ok = np.isfinite(hi) & (hi > lo)
    lo, hi = lo[ok], hi[ok]
    x = (lo + rng.random(len(lo)).astype(np.float32) * (hi - lo)).astype(np.float16).astype(np.float32)
    x = np.clip(x, lo, hi)
    s = ((hi - lo) / np.float32((1 << bits) - 1)).astype(np.float32)
    if scale_f16:
        s = s.astype(np.float16).astype(np.float32)
    keep = s > 0
    a = (x - lo).astype(np.float32)
    # the group maximum itself: the largest quotient of the group
    a = np.concatenate([a[keep], (hi - lo)[keep]])
    return a, np.concatenate([s[keep], s[keep]])


@pytest.mark.parametrize("bits,scale_f16", [(2, False), (4, False), (2, True), (4, True)])
def test_fast_quotient_on_random_groups(bits, scale_f16):
    rng = np.random.default_rng(100 + bits + 10 * scale_f16)
    a, s = _random_pairs(rng, 2_000_000, bits, scale_f16)
    fast = _check(a, s, scale_f16)
    # divisions: exact and near ties, common where a range spans few fp16 steps
    assert fast.mean() > 0.9


@pytest.mark.parametrize("bits,scale_f16", [(2, False), (4, False), (2, True), (4, True)])
def test_fast_quotient_on_near_ties(bits, scale_f16):
    """Every fp16 value whose quotient lies within 2^-14 of a half-integer
    (exact ties included) takes the division, and those just outside the
    band take the fast path with the right code."""
    rng = np.random.default_rng(200 + bits + 10 * scale_f16)
    n_tie = n_near = n_edge = 0
    for lo, hi, near, edge in near_ties.tie_configs(rng, bits, scale_f16, configs=160):
        s = near_ties.group_scale(np.float32(lo), np.float32(hi), bits, scale_f16)
        for xs, is_near in ((near, True), (edge, False)):
            if len(xs) == 0:
                continue
            a = (xs - np.float32(lo)).astype(np.float32)
            fast = _check(a, np.full(len(a), s, np.float32), scale_f16)
            d = near_ties.quotient_distance(xs, np.float32(lo), s)
            if is_near:
                # within the band: the kernel must not trust the product
                assert not fast.any()
                n_near += len(xs)
                n_tie += int((d == 0).sum())
            else:
                n_edge += len(xs)
    assert n_tie > 50 and n_near > 300 and n_edge > 1000, (n_tie, n_near, n_edge)


def test_scale_division_every_fp32(tmp_path):
    """The kernel's scale RN(x / L) (multiply by RN(1/L), fma remainder, fma
    correction) equals the IEEE quotient for every non-negative finite fp32 x,
    L = 3 and 15 (tests/div_levels_check.c, on all host cores)."""
    import os
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "div_levels_check.c")
    exe = str(tmp_path / "div_levels_check")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-pthread", "-o", exe, src, "-lm"], check=True)
    res = subprocess.run([exe, str(os.cpu_count() or 1)], capture_output=True, text=True, timeout=900)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout
