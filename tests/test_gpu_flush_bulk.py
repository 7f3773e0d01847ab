"""Long flushes at group size 32 stage their items with bulk tensor copies
(more items than one wave of the cp.async grid); shorter ones and fake
quantization use cp.async. Parity of the bulk-copy path at every head dim,
both bit widths and both scale storages, on a ragged tail (residual length
0, S not a multiple of 32), adversarial rows, a strided view into a larger
cache and a store offset: codes, scales and zeros bit-exact with the oracle.
Sizes: 16 heads x 4103 tokens gives 4128 to 16464 items, above the 2432 of
one cp.async wave on 152 SMs."""
import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(rng, BH, S_max, D):
    k = synth.keys(rng, (BH, S_max), D, np.array([3, D // 2, D - 1]), 8.0)
    v = synth.normal(rng, (BH, S_max, D))
    # edge rows: a constant channel, an exact grid with half-integer quotients, the fp16 extremes
    k[0, :, 0] = np.float16(3.0)
    k[0, :32, 1] = (np.arange(32) % 16 * 0.5).astype(np.float16)
    k[1, :, 2] = np.float16(65504.0)
    k[1, ::2, 2] = np.float16(-65504.0)
    v[0, 6, :] = (np.arange(D) % 4 * 0.25).astype(np.float16)
    v[1, 9, :] = np.float16(6e-8)
    v[1, 9, ::3] = np.float16(-6e-8)
    # subnormal fp16 scales, whose codes are clipped (4-bit: 20 -> 15, 2-bit: 4 -> 3)
    tiny = 2.0 ** -24
    v[0, 12, :] = (np.arange(D) % 21 * tiny).astype(np.float16)
    v[0, 13, :] = (np.arange(D) % 5 * tiny).astype(np.float16)
    k[0, :, 5] = (np.arange(S_max) % 21 * tiny).astype(np.float16)
    k[0, :, 6] = (np.arange(S_max) % 5 * tiny).astype(np.float16)
    return k, v


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("bits,scale_f16", [(2, False), (4, False), (2, True), (4, True)])
def test_bulk_copy_flush_matches_oracle(D, bits, scale_f16):
    rng = np.random.default_rng(1000 + D + 10 * bits + int(scale_f16))
    BH, S, S_max, s_off = 16, 4103, 4160, 64   # ragged last group of 7 tokens; heads S_max tokens apart
    k, v = _inputs(rng, BH, S_max, D)
    s_cap = s_off + 4128
    ks = kv.KiviStore(0, BH, s_cap, D, 32, bits, device="cuda", scale_f16=scale_f16)
    vs = kv.KiviStore(1, BH, s_cap, D, 32, bits, device="cuda", scale_f16=scale_f16)
    kt = torch.from_numpy(k).cuda()[:, :S]       # a view: head stride S_max tokens
    vt = torch.from_numpy(v).cuda()[:, :S]
    assert kv.kivi_flush_kv(kt, vt, 0, ks, vs, s_off=s_off) == S
    torch.cuda.synchronize()
    for axis, x, gs in ((0, k, ks), (1, v, vs)):
        ref = oracle.flush(axis, np.ascontiguousarray(x[:, :S]), S,
                           oracle.Store(axis, BH, s_cap, D, 32, bits, scale_f16=scale_f16), s_off=s_off)
        assert np.array_equal(gs.codes.cpu().numpy(), ref.codes), "codes differ (axis %d)" % axis
        sc = gs.scale.cpu().numpy()
        assert np.array_equal(sc.view(np.uint16 if scale_f16 else np.uint32),
                              ref.scale.view(np.uint16 if scale_f16 else np.uint32)), "scales differ (axis %d)" % axis
        assert np.array_equal(gs.zero.cpu().numpy().view(np.uint16), ref.zero.view(np.uint16)), \
            "zeros differ (axis %d)" % axis
    assert kv.kivi_wait_timeouts() == 0
