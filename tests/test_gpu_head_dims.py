"""GPU parity of the flush, dequant, fake quantization, residual window and
fused decode at head dims 64 and 256 (the kernels are templated on D; D = 128
is covered by the other parity files). Codes, packed bytes, scales, zeros and
fp16 outputs must equal the oracle's bit for bit; the decode must lie within
2e-3 of the float64 oracle."""
import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (D, G) pairs the library supports besides D = 128: a value group lies within
# one token row, so G <= D
SHAPES = [(64, 32), (64, 64), (256, 32), (256, 64), (256, 128)]


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
    assert np.array_equal(host(gpu.scale).view(np.uint32), ref.scale.view(np.uint32)), "scales differ " + what
    assert np.array_equal(host(gpu.zero).view(np.uint16), ref.zero.view(np.uint16)), "zeros differ " + what


def outliers(D):
    return np.array([3, D // 2, D // 2 + 1, D - 1])


def adversarial(rng, BH, S, D):
    """Rows and columns that pin the edge cases: constant groups, an exact
    grid with half-integer quotients, -0, the full fp16 range, subnormals."""
    x = synth.normal(rng, (BH, S, D))
    x[0, :, 0] = np.float16(3.0)
    x[0, 5, :] = np.float16(-2.0)
    x[0, :32, 1] = (np.arange(32) % 16 * 0.5).astype(np.float16)
    x[0, 6, :] = (np.arange(D) % 4 * 0.25).astype(np.float16)
    x[0, 7, :32] = np.float16(0.0)
    x[0, 7, 0] = np.float16(-0.0)
    x[1 % BH, :, 2] = np.float16(65504.0)
    x[1 % BH, ::2, 2] = np.float16(-65504.0)
    x[1 % BH, 9, :] = np.float16(6e-8)
    x[1 % BH, 9, ::3] = np.float16(-6e-8)
    x[0, 11, :] = (np.arange(D) % 31 * 0.5).astype(np.float16)
    x[0, :32, 4] = (np.arange(32) % 31 * 0.5).astype(np.float16)
    return x


def flush_both(axis, x, R, G, bits):
    BH, S, D = x.shape
    n = kv.kivi_flush_count(S, R, G)
    s_cap = max(G, -(-n // G) * G)
    gs = kv.KiviStore(axis, BH, s_cap, D, G, bits, device=DEV)
    fn = kv.kivi_flush_keys if axis == 0 else kv.kivi_flush_values
    assert fn(dev(x), R, gs) == n
    rs = oracle.Store(axis, BH, s_cap, D, G, bits)
    if n:
        oracle.flush(axis, x, n, rs)
    return n, gs, rs


@pytest.mark.parametrize("D,G", SHAPES)
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_flush_dequant_head_dims(D, G, bits, axis):
    """Ragged lengths (residual_length 0 flushes every token), residual
    windows and the adversarial rows; store and dequant bit-exact."""
    rng = np.random.default_rng(500 + D + G + bits + axis)
    for S, R in [(1, 0), (31, 0), (64, 0), (129, 0), (300, 0), (700, 128)]:
        BH = int(rng.integers(1, 5))
        x = synth.keys(rng, (BH, S), D, outliers(D), 10.0) if axis == 0 else synth.normal(rng, (BH, S, D))
        n, gs, rs = flush_both(axis, x, R, G, bits)
        assert n == oracle.flush_count(S, R, G)
        assert_store_equal(gs, rs, "D=%d G=%d S=%d" % (D, G, S))
        if n:
            assert same(host(kv.kivi_dequant(gs, n)), oracle.dequant(rs, n)), (D, G, S)
    x = adversarial(rng, 3, 2 * G + 17, D)
    n, gs, rs = flush_both(axis, x, 0, G, bits)
    assert_store_equal(gs, rs, "adversarial D=%d G=%d" % (D, G))
    assert same(host(kv.kivi_dequant(gs, n)), oracle.dequant(rs, n))


@pytest.mark.parametrize("D,G", SHAPES)
def test_fused_kv_flush_and_dequant_head_dims(D, G):
    """One launch for keys and values, into a store offset of a strided view."""
    rng = np.random.default_rng(600 + D + G)
    BH, S, R = 5, 1100, 128
    k = synth.keys(rng, (BH, S + 40), D, outliers(D), 8.0)
    v = synth.normal(rng, (BH, S + 40, D))
    n = kv.kivi_flush_count(S, R, G)
    s_cap = -(-(n + G) // G) * G
    ks = kv.KiviStore(0, BH, s_cap, D, G, 4, device=DEV)
    vs = kv.KiviStore(1, BH, s_cap, D, G, 4, device=DEV)
    gk, gv = dev(k), dev(v)
    # tokens 40 .. 40 + S of each head (head stride S + 40) land at store token G
    assert kv.kivi_flush_kv(gk[:, 40:], gv[:, 40:], R, ks, vs, s_off=G, n_tokens=S) == n
    rk = oracle.Store(0, BH, s_cap, D, G, 4)
    rv = oracle.Store(1, BH, s_cap, D, G, 4)
    oracle.flush(0, k, n, rk, s_off=G, t0=40)
    oracle.flush(1, v, n, rv, s_off=G, t0=40)
    assert_store_equal(ks, rk, "keys")
    assert_store_equal(vs, rv, "values")
    kd, vd = kv.kivi_dequant_kv(ks, vs, G + n)
    assert same(host(kd)[:, G:], oracle.dequant(rk, G + n)[:, G:])
    assert same(host(vd)[:, G:], oracle.dequant(rv, G + n)[:, G:])


@pytest.mark.parametrize("D,G", SHAPES)
@pytest.mark.parametrize("bits", [2, 4])
def test_fake_quant_head_dims(D, G, bits):
    """Quantize-then-dequantize fp16 for the tokens a flush would take, the
    rest copied; keys and values in one launch, and in place."""
    rng = np.random.default_rng(700 + D + G + bits)
    for S, R in [(100, 0), (700, 128)]:
        k = synth.keys(rng, (3, S), D, outliers(D), 10.0)
        v = synth.normal(rng, (3, S, D))
        kout, vout, n = kv.kivi_fake_quant_kv(dev(k), dev(v), R, G=G, bits=bits)
        assert n == oracle.flush_count(S, R, G)
        for axis, x, out in ((0, k, kout), (1, v, vout)):
            ref = x.copy()
            if n:
                rs = oracle.Store(axis, 3, -(-n // G) * G, D, G, bits)
                oracle.flush(axis, x, n, rs)
                ref[:, :n] = oracle.dequant(rs, n)
            assert same(host(out), ref), (D, G, bits, S, axis)
        gv = dev(v)
        out, n2 = kv.kivi_fake_quant_values(gv, R, out=gv, G=G, bits=bits)  # in place
        assert n2 == n and same(host(gv), host(vout))


@pytest.mark.parametrize("D", [64, 256])
def test_residual_head_dims(D):
    rng = np.random.default_rng(800 + D)
    res = synth.normal(rng, (6, 160, D))
    src = synth.normal(rng, (6, 50, D))
    g_res, ref = dev(res), res.copy()
    assert kv.kivi_residual_append(dev(src), g_res, 100, n_new=37) == 137
    oracle.residual_append(ref, 100, src, 37)
    assert same(host(g_res), ref)
    for n_res, n_drop in ((137, 32), (105, 100), (5, 2), (160, 1)):
        g = dev(ref)
        kv.kivi_residual_compact(g, n_res, n_drop)
        r2 = ref.copy()
        oracle.residual_compact(r2, n_res, n_drop)
        assert same(host(g), r2), (n_res, n_drop)
    kres, vres = dev(res), dev(res[::-1].copy())
    rk, rv = res.copy(), res[::-1].copy()
    kv.kivi_residual_append_kv(dev(src), dev(src[:, ::-1].copy()), kres, vres, 90, n_new=50)
    oracle.residual_append(rk, 90, src, 50)
    oracle.residual_append(rv, 90, src[:, ::-1].copy(), 50)
    kv.kivi_residual_compact_kv(kres, vres, 140, 64)
    oracle.residual_compact(rk, 140, 64)
    oracle.residual_compact(rv, 140, 64)
    assert same(host(kres), rk) and same(host(vres), rv)


TOL = 2e-3  # decode max-abs error against the float64 oracle


def decode_both(D, G, bits, B, hq, hkv, S_q, n_res, seed, noalloc=False):
    """Flush K and V of S_q tokens on both sides, then decode one query per
    head over the store plus n_res fp16 tokens; returns (gpu, oracle)."""
    rng = np.random.default_rng(seed)
    BH = B * hkv
    k = synth.keys(rng, (BH, S_q + n_res), D, outliers(D), 8.0)
    v = synth.normal(rng, (BH, S_q + n_res, D))
    q = synth.normal(rng, (B, hq, D))
    sm_scale = 1.0 / np.sqrt(D)
    s_cap = max(G, -(-S_q // G) * G)
    gk = kv.KiviStore(0, BH, s_cap, D, G, bits, device=DEV)
    gv = kv.KiviStore(1, BH, s_cap, D, G, bits, device=DEV)
    rk = oracle.Store(0, BH, s_cap, D, G, bits)
    rv = oracle.Store(1, BH, s_cap, D, G, bits)
    if S_q:
        kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=S_q)
        oracle.flush(0, k, S_q, rk)
        oracle.flush(1, v, S_q, rv)
    kr = np.ascontiguousarray(k[:, S_q:])
    vr = np.ascontiguousarray(v[:, S_q:])
    fn = kv.kivi_decode_attend_noalloc if noalloc else kv.kivi_decode_attend
    out = fn(dev(q), gk, gv, S_q, dev(kr), dev(vr), n_res, hkv, sm_scale)
    ref = oracle.decode_attend(q, rk, rv, S_q, kr, vr, n_res, hkv, sm_scale)
    return host(out).astype(np.float64), ref


DECODE_SHAPES = [
    (2, 8, 8, 70, 9),        # ragged last key group; a tile of 6 valid tokens
    (2, 32, 8, 4096, 37),    # 4 heads per KV head, several splits per head
    (1, 24, 8, 1000, 200),   # 3 heads per KV head (sub-groups), ragged store
    (1, 16, 2, 16384, 100),  # sub-groups of a long cache: more splits than a cluster holds
    (3, 4, 4, 64, 0),        # store only
    (1, 8, 8, 0, 37),        # fp16 residual only
]


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("big_g", [False, True])
@pytest.mark.parametrize("B,hq,hkv,S_q,n_res", DECODE_SHAPES)
def test_decode_head_dims(D, bits, big_g, B, hq, hkv, S_q, n_res):
    """The fused decode at head dims 64 and 256 (group size 32, and 64 at
    D = 64 or 128 at D = 256) against the float64 oracle."""
    G = (64 if D == 64 else 128) if big_g else 32
    out, ref = decode_both(D, G, bits, B, hq, hkv, S_q, n_res, seed=900 + D + G + bits + S_q + hq)
    err = np.max(np.abs(out - ref))
    assert err <= TOL, err


@pytest.mark.parametrize("D", [64, 256])
def test_decode_head_dims_batched_and_noalloc(D):
    """A batch of 8 sequences x 2048 tokens (4 query heads per KV head), and
    the no-alloc entry point on a split plan."""
    out, ref = decode_both(D, 32, 4, 8, 32, 8, 2016, 32, seed=950 + D)
    assert np.max(np.abs(out - ref)) <= TOL
    out, ref = decode_both(D, 32, 4, 1, 32, 8, 4032, 64, seed=960 + D, noalloc=True)
    assert np.max(np.abs(out - ref)) <= TOL


def test_decode_rejects_unsupported_head_dim_pairs():
    """G > D is refused on the host: UNSUPPORTED, nothing launched."""
    D, G = 64, 128
    ks = kv.KiviStore(0, 8, 128, D, G, 4, device=DEV)
    vs = kv.KiviStore(1, 8, 128, D, G, 4, device=DEV)
    q = torch.zeros((1, 32, D), dtype=torch.float16, device=DEV)
    res = torch.zeros((8, 16, D), dtype=torch.float16, device=DEV)
    out = torch.full((1, 32, D), 7.0, dtype=torch.float32, device=DEV)
    with pytest.raises(kv.KiviError) as e:
        kv.kivi_decode_attend(q, ks, vs, 64, res, res, 16, 8, 0.1, out=out)
    assert e.value.status == 2
    assert bool((out == 7.0).all())
