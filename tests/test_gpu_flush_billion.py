"""The flush against the oracle over more than 10^9 elements, bit-exact.

The flush kernel computes each scale by a multiply and two fmas, each code
from the product a * r (r = 1 / s to within 1 ulp), and falls back to an
IEEE division only for quotients within 2^-14 of a half-integer (the scale
division and the bound are checked in tests/test_guard_band.py). Ties are
common in real data (VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My
LLM Exactly 0% Faster", "Three ways to be off by one bit", #2), so both paths
must agree with the oracle's division everywhere. Eight chunks of 16 heads x
32768 tokens x 128 channels of K and V (1.07 x 10^9 elements) are flushed,
2- and 4-bit, fp32 and fp16 scale storage; in each, one key column group in
16 and one value row group in 16 is replaced by a near-tie group (min, max
and 30 values whose quotients lie within 2^-14 of a half-integer, exact ties
included, or just outside that band). Codes, scales and zeros must equal the
oracle's bit for bit."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import near_ties
import oracle
import kivi_kv_cache_gb300 as kv

pytestmark = pytest.mark.gpu

BH, S, D, G = 16, 32768, 128, 32
CHUNKS = [(4, False), (2, False), (4, True), (2, True), (4, False), (2, False), (4, True), (2, False)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _chunk(rng, bits, hs):
    k = rng.standard_normal((BH, S, D), dtype=np.float32)
    k[..., rng.choice(D, 4, replace=False)] *= 8.0  # outlier channels
    k = k.astype(np.float16)
    v = rng.standard_normal((BH, S, D), dtype=np.float32).astype(np.float16)
    n_cols = BH * (S // G) * D
    pick = rng.choice(n_cols, n_cols // 16, replace=False)
    groups, near_k = near_ties.tie_groups(rng, len(pick), G, bits, hs)
    bh, rest = np.divmod(pick, (S // G) * D)
    gi, ch = np.divmod(rest, D)
    k.reshape(BH, S // G, G, D)[bh, gi, :, ch] = groups
    n_rows = BH * S * (D // G)
    pick = rng.choice(n_rows, n_rows // 16, replace=False)
    groups, near_v = near_ties.tie_groups(rng, len(pick), G, bits, hs)
    bh, rest = np.divmod(pick, S * (D // G))
    t, j = np.divmod(rest, D // G)
    v.reshape(BH, S, D // G, G)[bh, t, j, :] = groups
    return k, v, near_k + near_v


def test_flush_bit_exact_over_a_billion_elements():
    rng = np.random.default_rng(2026)
    dev = torch.device("cuda")
    total = near = 0
    threads = max(1, min(16, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for ci, (bits, hs) in enumerate(CHUNKS):
            k, v, n_near = _chunk(rng, bits, hs)
            ks = kv.KiviStore(0, BH, S, D, G, bits, device=dev, scale_f16=hs)
            vs = kv.KiviStore(1, BH, S, D, G, bits, device=dev, scale_f16=hs)
            assert kv.kivi_flush_kv(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), 0, ks, vs) == S

            def head(args):
                axis, x, bh = args
                st = oracle.Store(axis, 1, S, D, G, bits, scale_f16=hs)
                oracle.flush(axis, x[bh:bh + 1], S, st)
                return axis, bh, st

            refs = list(ex.map(head, [(a, x, bh) for a, x in ((0, k), (1, v)) for bh in range(BH)]))
            got = {0: (ks.codes.cpu().numpy(), ks.scale.cpu().numpy(), ks.zero.cpu().numpy()),
                   1: (vs.codes.cpu().numpy(), vs.scale.cpu().numpy(), vs.zero.cpu().numpy())}
            for axis, bh, st in refs:
                codes, scale, zero = got[axis]
                assert np.array_equal(codes[bh], st.codes[0]), (ci, axis, bh, "codes")
                assert np.array_equal(scale[bh].view(np.uint8), st.scale[0].view(np.uint8)), (ci, axis, bh, "scale")
                assert np.array_equal(zero[bh].view(np.uint16), st.zero[0].view(np.uint16)), (ci, axis, bh, "zero")
            total += 2 * k.size
            near += n_near
            del ks, vs, k, v, refs, got
            torch.cuda.empty_cache()
    assert total >= 10 ** 9 and near > 10 ** 6, (total, near)
