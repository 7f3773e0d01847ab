"""GPU parity of the fp16 scale storage option (KIVI_SCALE_F16): the flush
rounds each scale to fp16 and computes the codes with it; dequant, fake
quantization and the fused decode read the fp16 scales. Codes, packed bytes,
fp16 scales, zeros and fp16 outputs must equal the oracle's bit for bit; the
decode must lie within 2e-3 of the float64 oracle. The adversarial rows include
groups whose fp16 scale underflows to 0 and groups whose subnormal fp16 scale
clips the largest code."""
import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 2e-3
TINY = 2.0 ** -24  # the smallest fp16 subnormal


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint16), np.asarray(b).view(np.uint16))


def assert_store_equal(gpu, ref, what=""):
    assert np.array_equal(host(gpu.codes), ref.codes), "packed codes differ " + what
    assert host(gpu.scale).dtype == np.float16 and ref.scale.dtype == np.float16
    assert same(host(gpu.scale), ref.scale), "fp16 scales differ " + what
    assert same(host(gpu.zero), ref.zero), "zeros differ " + what


def adversarial(rng, BH, S, D):
    x = synth.normal(rng, (BH, S, D))
    x[0, :, 0] = np.float16(3.0)                                   # constant key channel
    x[0, 5, :] = np.float16(-2.0)                                  # constant value row
    x[0, 6, :] = (np.arange(D) % 4 * 0.25).astype(np.float16)
    x[0, 11, :] = (np.arange(D) % 31 * 0.5).astype(np.float16)
    x[1 % BH, :, 2] = np.float16(65504.0)
    x[1 % BH, ::2, 2] = np.float16(-65504.0)                       # full fp16 range
    x[1 % BH, 9, :] = np.float16(6e-8)
    x[1 % BH, 9, ::3] = np.float16(-6e-8)                          # scale underflows to 0
    x[0, 12, :] = (np.arange(D) % 21 * TINY).astype(np.float16)    # 4-bit: subnormal scale clips 20 -> 15
    x[0, 13, :] = (np.arange(D) % 5 * TINY).astype(np.float16)     # 2-bit: clips 4 -> 3
    x[0, :, 5] = (np.arange(S) % 21 * TINY).astype(np.float16)     # the same down a key channel
    x[0, :, 6] = (np.arange(S) % 5 * TINY).astype(np.float16)
    x[0, :, 7] = (np.arange(S) % 2 * 0.5).astype(np.float16)       # 0 / 0.5 grid: scale 1/30 -> fp16
    return x


def flush_both(axis, x, R, G, bits):
    BH, S, D = x.shape
    n = kv.kivi_flush_count(S, R, G)
    s_cap = max(G, -(-n // G) * G)
    gs = kv.KiviStore(axis, BH, s_cap, D, G, bits, device=DEV, scale_f16=True)
    fn = kv.kivi_flush_keys if axis == 0 else kv.kivi_flush_values
    assert fn(dev(x), R, gs) == n
    rs = oracle.Store(axis, BH, s_cap, D, G, bits, scale_f16=True)
    if n:
        oracle.flush(axis, x, n, rs)
    return n, gs, rs


@pytest.mark.parametrize("D,G", [(128, 32), (128, 64), (128, 128), (64, 32), (256, 128)])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_flush_dequant_scale_f16(D, G, bits, axis):
    rng = np.random.default_rng(1100 + D + G + bits + axis)
    for S, R in [(1, 0), (63, 0), (300, 0), (700, 128)]:
        BH = int(rng.integers(1, 4))
        x = synth.keys(rng, (BH, S), D, np.array([3, D - 1]), 10.0) if axis == 0 else synth.normal(rng, (BH, S, D))
        n, gs, rs = flush_both(axis, x, R, G, bits)
        assert_store_equal(gs, rs, "D=%d G=%d S=%d" % (D, G, S))
        if n:
            assert same(host(kv.kivi_dequant(gs, n)), oracle.dequant(rs, n)), (D, G, S)
    x = adversarial(rng, 3, 2 * G + 17, D)
    n, gs, rs = flush_both(axis, x, 0, G, bits)
    assert_store_equal(gs, rs, "adversarial D=%d G=%d" % (D, G))
    assert same(host(kv.kivi_dequant(gs, n)), oracle.dequant(rs, n))


@pytest.mark.parametrize("G", [32, 128])
def test_fused_kv_flush_dequant_and_fake_quant_scale_f16(G):
    w = synth.WORKLOADS["qwen8b"]
    k, v, _ = synth.prefill_inputs(w)
    n = kv.kivi_flush_count(w.S, w.R, G)
    ks = kv.KiviStore(0, w.BH, n, w.D, G, w.bits, device=DEV, scale_f16=True)
    vs = kv.KiviStore(1, w.BH, n, w.D, G, w.bits, device=DEV, scale_f16=True)
    assert kv.kivi_flush_kv(dev(k), dev(v), w.R, ks, vs) == n
    rk = oracle.flush(0, k, n, oracle.Store(0, w.BH, n, w.D, G, w.bits, scale_f16=True))
    rv = oracle.flush(1, v, n, oracle.Store(1, w.BH, n, w.D, G, w.bits, scale_f16=True))
    assert_store_equal(ks, rk, "keys")
    assert_store_equal(vs, rv, "values")
    kd, vd = kv.kivi_dequant_kv(ks, vs, n)
    assert same(host(kd), oracle.dequant(rk, n)) and same(host(vd), oracle.dequant(rv, n))
    # fake quantization with fp16 scales: the flushed tokens become exactly
    # that dequantization, the rest are copied
    kout, vout, nq = kv.kivi_fake_quant_kv(dev(k), dev(v), w.R, G=G, bits=w.bits, scale_f16=True)
    assert nq == n
    kref, vref = k.copy(), v.copy()
    kref[:, :n] = oracle.dequant(rk, n)
    vref[:, :n] = oracle.dequant(rv, n)
    assert same(host(kout), kref) and same(host(vout), vref)


@pytest.mark.parametrize("D,G", [(128, 32), (128, 128), (64, 64), (256, 32)])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("B,hq,hkv,S_q,n_res", [
    (2, 8, 8, 70, 9),        # ragged last key group
    (2, 32, 8, 4096, 37),    # 4 heads per KV head, several splits (the warp-pair plan is not used)
    (1, 24, 8, 1000, 200),   # sub-groups
    (1, 4, 4, 2080, 158),    # the qwen8b decode's shape per KV head
])
def test_decode_scale_f16(D, G, bits, B, hq, hkv, S_q, n_res):
    rng = np.random.default_rng(1200 + D + G + bits + S_q + hq)
    BH = B * hkv
    k = synth.keys(rng, (BH, S_q + n_res), D, np.array([3, D // 2, D - 1]), 8.0)
    v = synth.normal(rng, (BH, S_q + n_res, D))
    if S_q > 40:
        k[0, :32, 5] = (np.arange(32) % 21 * TINY).astype(np.float16)  # a clipped key group
        v[0, 12, :] = (np.arange(D) % 21 * TINY).astype(np.float16)    # clipped value groups
    q = synth.normal(rng, (B, hq, D))
    s_cap = max(G, -(-S_q // G) * G)
    gk = kv.KiviStore(0, BH, s_cap, D, G, bits, device=DEV, scale_f16=True)
    gv = kv.KiviStore(1, BH, s_cap, D, G, bits, device=DEV, scale_f16=True)
    kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=S_q)
    rk = oracle.flush(0, k, S_q, oracle.Store(0, BH, s_cap, D, G, bits, scale_f16=True))
    rv = oracle.flush(1, v, S_q, oracle.Store(1, BH, s_cap, D, G, bits, scale_f16=True))
    assert_store_equal(gk, rk, "keys")
    assert_store_equal(gv, rv, "values")
    kr, vr = np.ascontiguousarray(k[:, S_q:]), np.ascontiguousarray(v[:, S_q:])
    sm = 1.0 / np.sqrt(D)
    out = host(kv.kivi_decode_attend(dev(q), gk, gv, S_q, dev(kr), dev(vr), n_res, hkv, sm)).astype(np.float64)
    ref = oracle.decode_attend(q, rk, rv, S_q, kr, vr, n_res, hkv, sm)
    err = np.max(np.abs(out - ref))
    assert err <= TOL, err
