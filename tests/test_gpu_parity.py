"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar: packed codes, scales and zeros bit-exact; dequantized fp16 bit-exact;
decode-attend max-abs error <= 2e-3 against the float64 oracle."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def assert_store_equal(gpu: kv.KiviStore, ref: oracle.Store, what=""):
    assert np.array_equal(host(gpu.codes), ref.codes), "packed codes differ " + what
    assert np.array_equal(host(gpu.scale).view(np.uint32), ref.scale.view(np.uint32)), "scales differ " + what
    assert np.array_equal(host(gpu.zero).view(np.uint16), ref.zero.view(np.uint16)), "zeros differ " + what


def flush_both(axis, x, R, G=32, bits=4, s_cap=None, fused_with=None):
    """GPU flush (single-axis call) and oracle flush of x [BH, S, D]."""
    BH, S, D = x.shape
    n = kv.kivi_flush_count(S, R, G)
    s_cap = s_cap or max(G, -(-n // G) * G)
    gs = kv.KiviStore(axis, BH, s_cap, D, G, bits, device=DEV)
    fn = kv.kivi_flush_keys if axis == 0 else kv.kivi_flush_values
    assert fn(dev(x), R, gs) == n
    rs = oracle.Store(axis, BH, s_cap, D, G, bits)
    if n:
        oracle.flush(axis, x, n, rs)
    return n, gs, rs


# ---------------------------------------------------------------------------
# flush + dequant on the workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "qwen8b", "long2bit"])
def test_flush_and_dequant_workloads(name):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.prefill_inputs(w)
    for axis, x in ((0, k), (1, v)):
        n, gs, rs = flush_both(axis, x, w.R, w.G, w.bits)
        assert n == oracle.flush_count(w.S, w.R, w.G)
        assert_store_equal(gs, rs, "%s axis %d" % (name, axis))
        d = host(kv.kivi_dequant(gs, n))
        assert np.array_equal(d.view(np.uint16), oracle.dequant(rs, n).view(np.uint16))


@pytest.mark.parametrize("name", ["tiny", "qwen8b", "long2bit"])
def test_fused_kv_flush_equals_separate(name):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.prefill_inputs(w)
    n = kv.kivi_flush_count(w.S, w.R, w.G)
    ks = kv.KiviStore(0, w.BH, n, w.D, w.G, w.bits, device=DEV)
    vs = kv.KiviStore(1, w.BH, n, w.D, w.G, w.bits, device=DEV)
    assert kv.kivi_flush_kv(dev(k), dev(v), w.R, ks, vs) == n
    assert_store_equal(ks, oracle.flush(0, k, n, oracle.Store(0, w.BH, n, w.D, w.G, w.bits)))
    assert_store_equal(vs, oracle.flush(1, v, n, oracle.Store(1, w.BH, n, w.D, w.G, w.bits)))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_flush_ragged_sweep(bits, axis):
    """residual_length 0 flushes every token, so S gives ragged last key groups."""
    rng = np.random.default_rng(40 + bits + axis)
    ch = np.array([3, 64, 65, 127])
    for S in [1, 2, 31, 32, 33, 63, 95, 100, 129, 255, 300]:
        BH = int(rng.integers(1, 6))
        x = synth.keys(rng, (BH, S), 128, ch, 10.0) if axis == 0 else synth.normal(rng, (BH, S, 128))
        n, gs, rs = flush_both(axis, x, 0, 32, bits)
        assert n == S
        assert_store_equal(gs, rs, "S=%d" % S)
        d = host(kv.kivi_dequant(gs, S))
        assert np.array_equal(d.view(np.uint16), oracle.dequant(rs, S).view(np.uint16)), S


def adversarial(rng, BH, S):
    x = synth.normal(rng, (BH, S, 128))
    x[0, :, 0] = np.float16(3.0)                          # max == min key group
    x[0, 5, :] = np.float16(-2.0)                         # max == min value row
    x[0, :32, 1] = (np.arange(32) % 16 * 0.5).astype(np.float16)   # exact grid, ties at .5 steps
    x[0, 6, :] = (np.arange(128) % 4 * 0.25).astype(np.float16)
    x[0, 7, :32] = np.float16(0.0)
    x[0, 7, 0] = np.float16(-0.0)                         # -0 minimum
    x[1 % BH, :, 2] = np.float16(65504.0)
    x[1 % BH, ::2, 2] = np.float16(-65504.0)              # full fp16 range
    x[1 % BH, 9, :] = np.float16(6e-8)                    # subnormals
    x[1 % BH, 9, ::3] = np.float16(-6e-8)
    x[1 % BH, 10, :] = (rng.integers(-2, 3, 128) * 2.0 ** -24).astype(np.float16)
    x[0, 40:72, 3] = (np.arange(32) * 1.5 - 3).astype(np.float16)
    # exact half-integer quotients: groups spanning [0, 15] on a 0.5 grid give
    # scale 1 (4-bit) or 5 (2-bit), so x = k + 0.5 (4-bit) or 2.5, 7.5, 12.5
    # (2-bit) round half to even
    x[0, 11, :] = (np.arange(128) % 31 * 0.5).astype(np.float16)
    x[0, :32, 4] = (np.arange(32) % 31 * 0.5).astype(np.float16)
    return x


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_flush_adversarial(bits, axis):
    rng = np.random.default_rng(77)
    x = adversarial(rng, 3, 96)
    n, gs, rs = flush_both(axis, x, 0, 32, bits)
    assert_store_equal(gs, rs)
    assert np.array_equal(host(kv.kivi_dequant(gs, n)).view(np.uint16), oracle.dequant(rs, n).view(np.uint16))


@pytest.mark.parametrize("G", [64, 128])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_flush_dequant_group_sizes(G, bits, axis):
    """Group sizes 64 and 128: ragged lengths (residual_length 0 flushes every
    token), residual windows, and the adversarial rows; codes, scales, zeros
    and dequantized fp16 bit-exact against the oracle."""
    rng = np.random.default_rng(300 + G + bits + axis)
    ch = np.array([3, 64, 65, 127])
    for S, R in [(1, 0), (63, 0), (64, 0), (129, 0), (300, 0), (700, 128), (2238, 128)]:
        BH = int(rng.integers(1, 5))
        x = synth.keys(rng, (BH, S), 128, ch, 10.0) if axis == 0 else synth.normal(rng, (BH, S, 128))
        n, gs, rs = flush_both(axis, x, R, G, bits)
        assert n == oracle.flush_count(S, R, G)
        assert_store_equal(gs, rs, "G=%d S=%d" % (G, S))
        if n:
            d = host(kv.kivi_dequant(gs, n))
            assert np.array_equal(d.view(np.uint16), oracle.dequant(rs, n).view(np.uint16)), (G, S)
    x = adversarial(rng, 3, 2 * G + 17)
    n, gs, rs = flush_both(axis, x, 0, G, bits)
    assert_store_equal(gs, rs, "adversarial G=%d" % G)
    assert np.array_equal(host(kv.kivi_dequant(gs, n)).view(np.uint16), oracle.dequant(rs, n).view(np.uint16))


@pytest.mark.parametrize("G", [64, 128])
def test_fused_kv_flush_and_dequant_group_sizes(G):
    w = synth.WORKLOADS["qwen8b"]
    k, v, _ = synth.prefill_inputs(w)
    n = kv.kivi_flush_count(w.S, w.R, G)
    ks = kv.KiviStore(0, w.BH, n, w.D, G, w.bits, device=DEV)
    vs = kv.KiviStore(1, w.BH, n, w.D, G, w.bits, device=DEV)
    assert kv.kivi_flush_kv(dev(k), dev(v), w.R, ks, vs) == n
    rk = oracle.flush(0, k, n, oracle.Store(0, w.BH, n, w.D, G, w.bits))
    rv = oracle.flush(1, v, n, oracle.Store(1, w.BH, n, w.D, G, w.bits))
    assert_store_equal(ks, rk)
    assert_store_equal(vs, rv)
    kd, vd = kv.kivi_dequant_kv(ks, vs, n)
    assert np.array_equal(host(kd).view(np.uint16), oracle.dequant(rk, n).view(np.uint16))
    assert np.array_equal(host(vd).view(np.uint16), oracle.dequant(rv, n).view(np.uint16))


@pytest.mark.parametrize("axis", [0, 1])
def test_flush_into_offset_of_larger_cache(axis):
    """Flush a strided view (head stride 300 tokens) at store offset 64."""
    rng = np.random.default_rng(5)
    big = synth.normal(rng, (4, 300, 128))
    x = dev(big)[:, 40:, :]  # view: tokens 40.., head stride 300
    gs = kv.KiviStore(axis, 4, 256, device=DEV)
    fn = kv.kivi_flush_keys if axis == 0 else kv.kivi_flush_values
    n = fn(x, 32, gs, s_off=64, n_tokens=200)  # flush_count(200, 32, 32) = 160
    assert n == 160
    rs = oracle.Store(axis, 4, 256, 128, 32, 4)
    oracle.flush(axis, big, 160, rs, s_off=64, t0=40)
    assert_store_equal(gs, rs)


# ---------------------------------------------------------------------------
# residual window
# ---------------------------------------------------------------------------

def test_residual_append_and_compact():
    rng = np.random.default_rng(8)
    res = synth.normal(rng, (6, 160, 128))
    src = synth.normal(rng, (6, 50, 128))
    g_res = dev(res)
    ref = res.copy()
    assert kv.kivi_residual_append(dev(src), g_res, 100, n_new=37) == 137
    oracle.residual_append(ref, 100, src, 37)
    assert np.array_equal(host(g_res), ref)
    for n_res, n_drop in ((137, 32), (105, 100), (5, 2), (160, 1)):
        g = dev(ref)
        kv.kivi_residual_compact(g, n_res, n_drop)
        r2 = ref.copy()
        oracle.residual_compact(r2, n_res, n_drop)
        assert np.array_equal(host(g), r2), (n_res, n_drop)


# ---------------------------------------------------------------------------
# decode-attend
# ---------------------------------------------------------------------------

def decode_case(w, S_q, n_res, k, v, q, res_k=None, res_v=None, workspace=None):
    BH = w.BH
    s_cap = max(w.G, -(-S_q // w.G) * w.G)
    gk = kv.KiviStore(0, BH, s_cap, w.D, w.G, w.bits, device=DEV)
    gv = kv.KiviStore(1, BH, s_cap, w.D, w.G, w.bits, device=DEV)
    rk = oracle.Store(0, BH, s_cap, w.D, w.G, w.bits)
    rv = oracle.Store(1, BH, s_cap, w.D, w.G, w.bits)
    if S_q:
        kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=S_q)
        oracle.flush(0, k, S_q, rk)
        oracle.flush(1, v, S_q, rv)
    kr = res_k if res_k is not None else k[:, S_q:S_q + n_res]
    vr = res_v if res_v is not None else v[:, S_q:S_q + n_res]
    kr = np.ascontiguousarray(kr)
    vr = np.ascontiguousarray(vr)
    out = kv.kivi_decode_attend(dev(q), gk, gv, S_q, dev(kr), dev(vr), n_res, w.Hkv, w.sm_scale,
                                workspace=workspace)
    ref = oracle.decode_attend(q, rk, rv, S_q, kr, vr, n_res, w.Hkv, w.sm_scale)
    return host(out).astype(np.float64), ref


@pytest.mark.parametrize("name", ["tiny", "qwen8b", "long2bit"])
def test_decode_prefill_workloads(name):
    w = synth.WORKLOADS[name]
    k, v, q = synth.prefill_inputs(w)
    n = kv.kivi_flush_count(w.S, w.R, w.G)
    out, ref = decode_case(w, n, w.S - n, k, v, q)
    err = np.max(np.abs(out - ref))
    assert err <= TOL, err


@pytest.mark.parametrize("hq", [32, 64])
def test_decode_batched_workload_sampled(hq):
    """Batched decode (32 sequences x 4096 cached tokens; 4 query heads per KV
    head as configured, and 8, which runs in two sub-groups of 4 heads); the
    oracle checks a sample of 4 sequences, the GPU runs the full batch and is
    sliced."""
    w = dataclasses.replace(synth.WORKLOADS["batched"], Hq=hq)
    rng = np.random.default_rng(w.seed)
    ch = synth.outlier_channels(w)
    k = synth.keys(rng, (w.BH, w.S_q + w.n_res), w.D, ch, w.outlier_scale)
    v = synth.normal(rng, (w.BH, w.S_q + w.n_res, w.D))
    q = synth.normal(rng, (w.B, w.Hq, w.D))
    s_cap = w.S_q
    gk = kv.KiviStore(0, w.BH, s_cap, device=DEV)
    gv = kv.KiviStore(1, w.BH, s_cap, device=DEV)
    kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=w.S_q)
    kr = np.ascontiguousarray(k[:, w.S_q:])
    vr = np.ascontiguousarray(v[:, w.S_q:])
    out = host(kv.kivi_decode_attend(dev(q), gk, gv, w.S_q, dev(kr), dev(vr), w.n_res, w.Hkv, w.sm_scale))
    for b in (0, 7, 19, 31):
        sl = slice(b * w.Hkv, (b + 1) * w.Hkv)
        rk = oracle.flush(0, k[sl].copy(), w.S_q, oracle.Store(0, w.Hkv, s_cap, 128, 32, 4))
        rv = oracle.flush(1, v[sl].copy(), w.S_q, oracle.Store(1, w.Hkv, s_cap, 128, 32, 4))
        ref = oracle.decode_attend(q[b:b + 1], rk, rv, w.S_q, kr[sl].copy(), vr[sl].copy(), w.n_res,
                                   w.Hkv, w.sm_scale)
        err = np.max(np.abs(out[b:b + 1] - ref))
        assert err <= TOL, (b, err)


@pytest.mark.parametrize("S_q,n_res", [(0, 1), (0, 37), (32, 0), (33, 0), (64, 5), (77, 31),
                                       (1000, 200), (4096, 0), (96, 128)])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (24, 8), (32, 8), (40, 8), (12, 2), (28, 4), (16, 2),
                                     (18, 2), (32, 1)])
def test_decode_edge_shapes(S_q, n_res, bits, hq, hkv):
    B = 2
    w = synth.Workload("edge", B=B, Hkv=hkv, Hq=hq, D=128, S=S_q + n_res, bits=bits, G=32, R=0,
                       n_outlier=4, outlier_scale=8.0, seed=S_q * 7 + n_res)
    rng = np.random.default_rng(w.seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
    v = synth.normal(rng, (w.BH, S_q + n_res, 128))
    q = synth.normal(rng, (B, hq, 128))
    out, ref = decode_case(w, S_q, n_res, k, v, q)
    err = np.max(np.abs(out - ref))
    assert err <= TOL, err


@pytest.mark.parametrize("B,S_q,n_res,bits", [
    (1, 1472, 64, 4),    # warp pairs, 13 splits, fewer CTAs than SMs: workspace merge
    (4, 960, 64, 4),     # warp pairs, 9 splits over 288 CTAs: cluster merge where resident
    (8, 960, 64, 2),     # the same, 2-bit, 576 CTAs
    (1, 3008, 64, 4),    # one warp per tile, 13 splits, 104 CTAs: workspace merge
    (4, 4032, 64, 4),    # one warp per tile, 9 splits over 288 CTAs: cluster merge
    (16, 1920, 128, 2),  # one warp per tile, 4 splits over 512 CTAs: cluster merge
    (16, 1408, 128, 4),  # 2-warp CTAs, 9 splits over 1152 CTAs
    (16, 896, 128, 2),   # 2-warp CTAs, 2-bit
    (8, 8064, 128, 4),   # 2-warp CTAs, 19 splits: workspace merge
])
def test_decode_merge_paths(B, S_q, n_res, bits):
    """Shapes on both sides of the grid-size rule that picks the split merge
    (cluster or workspace ticket) for each decode kernel, and plans of 2-, 4-
    and 8-warp CTAs; every output is checked against the oracle."""
    w = synth.Workload("merge", B=B, Hkv=8, Hq=32, D=128, S=S_q + n_res, bits=bits, G=32, R=0,
                       n_outlier=4, outlier_scale=8.0, seed=B * 31 + S_q % 97)
    rng = np.random.default_rng(w.seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
    v = synth.normal(rng, (w.BH, S_q + n_res, 128))
    q = synth.normal(rng, (B, 32, 128))
    out, ref = decode_case(w, S_q, n_res, k, v, q)
    err = np.max(np.abs(out - ref))
    assert err <= TOL, err


@pytest.mark.parametrize("B,Hq,S_q,n_res,hs", [
    (16, 32, 1408, 128, True),   # 2-warp CTAs, fp16 scales
    (8, 64, 1408, 128, False),   # 2-warp CTAs, sub-groups of 4 of 8 heads per KV head
    (16, 8, 1408, 128, False),   # 2-warp CTAs, one head per KV head
])
def test_decode_two_warp_plans(B, Hq, S_q, n_res, hs):
    """Plans of 2-warp CTAs for other scale storage and head groups, against
    the oracle."""
    assert kv.kivi_decode_plan_info(B, Hq, 8, S_q, n_res, 128, 32, 4, hs)["warps_per_cta"] == 2
    w = synth.Workload("w2", B=B, Hkv=8, Hq=Hq, D=128, S=S_q + n_res, bits=4, G=32, R=0, n_outlier=4,
                       outlier_scale=8.0, seed=B + Hq)
    rng = np.random.default_rng(w.seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
    v = synth.normal(rng, (w.BH, S_q + n_res, 128))
    q = synth.normal(rng, (B, Hq, 128))
    gk = kv.KiviStore(0, w.BH, S_q, 128, 32, 4, device=DEV, scale_f16=hs)
    gv = kv.KiviStore(1, w.BH, S_q, 128, 32, 4, device=DEV, scale_f16=hs)
    kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=S_q)
    rk = oracle.Store(0, w.BH, S_q, 128, 32, 4, scale_f16=hs)
    rv = oracle.Store(1, w.BH, S_q, 128, 32, 4, scale_f16=hs)
    oracle.flush(0, k, S_q, rk)
    oracle.flush(1, v, S_q, rv)
    kr, vr = np.ascontiguousarray(k[:, S_q:]), np.ascontiguousarray(v[:, S_q:])
    ref = oracle.decode_attend(q, rk, rv, S_q, kr, vr, n_res, 8, w.sm_scale)
    out = host(kv.kivi_decode_attend(dev(q), gk, gv, S_q, dev(kr), dev(vr), n_res, 8, w.sm_scale))
    assert np.max(np.abs(out - ref)) <= TOL


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("hq,hkv", [(16, 2), (6, 2)])
def test_decode_subgroups_many_splits(hq, hkv, bits):
    """Groups of 8 or 3 query heads per KV head over a long cache: sub-groups of
    up to 4 heads, each a head group with more splits than a cluster holds
    (merged through its own ticket counter)."""
    S_q, n_res = 16384, 100
    w = synth.Workload("subgroups", B=1, Hkv=hkv, Hq=hq, D=128, S=S_q + n_res, bits=bits, G=32, R=0,
                       n_outlier=4, outlier_scale=8.0, seed=77 + hq)
    rng = np.random.default_rng(w.seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
    v = synth.normal(rng, (w.BH, S_q + n_res, 128))
    q = synth.normal(rng, (1, hq, 128))
    out, ref = decode_case(w, S_q, n_res, k, v, q)
    assert np.max(np.abs(out - ref)) <= TOL


@pytest.mark.parametrize("G", [64, 128])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("B,hq,hkv,S_q,n_res", [
    (2, 8, 8, 70, 9),        # ragged last key group; a tile of 6 valid tokens
    (2, 32, 8, 4096, 37),    # 4 heads per KV head, several splits per head
    (1, 24, 8, 1000, 200),   # 3 heads per KV head (sub-group kernel), ragged store
    (1, 16, 2, 16384, 100),  # sub-groups of a long cache: more splits than a cluster holds
    (3, 4, 4, 64, 0),        # one key group, store only
])
def test_decode_group_sizes(G, bits, B, hq, hkv, S_q, n_res):
    """The fused decode over stores of group size 64 and 128: a key group spans
    2 or 4 of the decode's 32-token tiles and a token has 2 or 1 value groups."""
    w = synth.Workload("groups", B=B, Hkv=hkv, Hq=hq, D=128, S=S_q + n_res, bits=bits, G=G, R=0,
                       n_outlier=4, outlier_scale=8.0, seed=1000 + G + S_q + hq)
    rng = np.random.default_rng(w.seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
    v = synth.normal(rng, (w.BH, S_q + n_res, 128))
    q = synth.normal(rng, (B, hq, 128))
    out, ref = decode_case(w, S_q, n_res, k, v, q)
    err = np.max(np.abs(out - ref))
    assert err <= TOL, err


def test_decode_one_workspace_across_sizes():
    """One workspace serves calls of different sizes in turn: after every call
    the merge counters at its start are zero again, and every call matches the
    oracle (counters left non-zero would make a later merge fire early or
    never)."""
    cases = [(1, 8, 32, 2080, 158, 4), (3, 8, 32, 1000, 40, 2), (2, 4, 32, 4096, 16, 4), (1, 8, 64, 700, 3, 4)]
    need = max(kv.kivi_decode_workspace_size(B, hq, hkv, S_q, n_res) for B, hkv, hq, S_q, n_res, _ in cases)
    ws = kv.kivi_decode_workspace(need, DEV)
    for i, (B, hkv, hq, S_q, n_res, bits) in enumerate(cases + cases[:1]):
        assert kv.kivi_decode_workspace_size(B, hq, hkv, S_q, n_res) > 0  # all are split plans
        w = synth.Workload("ws", B=B, Hkv=hkv, Hq=hq, D=128, S=S_q + n_res, bits=bits, G=32, R=0,
                           n_outlier=4, outlier_scale=8.0, seed=500 + i)
        rng = np.random.default_rng(w.seed)
        k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
        v = synth.normal(rng, (w.BH, S_q + n_res, 128))
        q = synth.normal(rng, (B, hq, 128))
        out, ref = decode_case(w, S_q, n_res, k, v, q, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws[:32768])) == 0, i
        err = np.max(np.abs(out - ref))
        assert err <= TOL, (i, err)


@pytest.mark.parametrize("S_kv", [128, 512, 2048, 8192, 16384])
def test_decode_stream_sweep_sampled(S_kv):
    """The streaming workload's decode sweep at B=16 (cache of S_kv tokens with
    a 128-token residual window); the oracle checks sequences 0 and 15."""
    w = synth.WORKLOADS["stream"]
    rng = np.random.default_rng(1000 + S_kv)
    n_res = min(w.R, S_kv)
    S_q = S_kv - n_res
    ch = synth.outlier_channels(w)
    k = synth.keys(rng, (w.BH, S_kv), w.D, ch, w.outlier_scale)
    v = synth.normal(rng, (w.BH, S_kv, w.D))
    q = synth.normal(rng, (w.B, w.Hq, w.D))
    s_cap = max(32, S_q)
    gk = kv.KiviStore(0, w.BH, s_cap, device=DEV)
    gv = kv.KiviStore(1, w.BH, s_cap, device=DEV)
    if S_q:
        kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=S_q)
    kr = np.ascontiguousarray(k[:, S_q:])
    vr = np.ascontiguousarray(v[:, S_q:])
    out = host(kv.kivi_decode_attend(dev(q), gk, gv, S_q, dev(kr), dev(vr), n_res, w.Hkv, w.sm_scale))
    for b in (0, 15):
        sl = slice(b * w.Hkv, (b + 1) * w.Hkv)
        rk = oracle.Store(0, w.Hkv, s_cap, 128, 32, 4)
        rv = oracle.Store(1, w.Hkv, s_cap, 128, 32, 4)
        if S_q:
            oracle.flush(0, k[sl].copy(), S_q, rk)
            oracle.flush(1, v[sl].copy(), S_q, rv)
        ref = oracle.decode_attend(q[b:b + 1], rk, rv, S_q, kr[sl].copy(), vr[sl].copy(), n_res,
                                   w.Hkv, w.sm_scale)
        assert np.max(np.abs(out[b:b + 1] - ref)) <= TOL


def test_two_pass_decode_once_equals_fused():
    """The two-pass "decode-once" composition (dequantize the store, then the
    decode over an all-fp16 cache: S_q = 0) gives the fused decode's result
    within the decode tolerance, and both match the oracle."""
    w = synth.Workload("twopass", B=2, Hkv=8, Hq=32, D=128, S=1000 + 40, bits=4, G=32, R=0, n_outlier=4,
                       outlier_scale=8.0, seed=61)
    rng = np.random.default_rng(w.seed)
    S_q, n_res = 992, 48
    k = synth.keys(rng, (w.BH, S_q + n_res), 128, synth.outlier_channels(w), 8.0)
    v = synth.normal(rng, (w.BH, S_q + n_res, 128))
    q = synth.normal(rng, (w.B, w.Hq, 128))
    fused, ref = decode_case(w, S_q, n_res, k, v, q)
    gk = kv.KiviStore(0, w.BH, S_q, device=DEV)
    gv = kv.KiviStore(1, w.BH, S_q, device=DEV)
    kv.kivi_flush_kv(dev(k), dev(v), 0, gk, gv, n_tokens=S_q)
    kd, vd = kv.kivi_dequant_kv(gk, gv, S_q)
    kfull = torch.cat([kd, dev(k[:, S_q:])], dim=1)
    vfull = torch.cat([vd, dev(v[:, S_q:])], dim=1)
    two = host(kv.kivi_decode_attend(dev(q), gk, gv, 0, kfull, vfull, S_q + n_res, w.Hkv, w.sm_scale))
    assert np.max(np.abs(two - ref)) <= TOL
    assert np.max(np.abs(two - fused)) <= TOL


def test_decode_workspace_too_small_is_rejected():
    w = synth.WORKLOADS["qwen8b"]
    q = torch.zeros((1, 32, 128), dtype=torch.float16, device=DEV)
    gk = kv.KiviStore(0, 8, 2080, device=DEV)
    gv = kv.KiviStore(1, 8, 2080, device=DEV)
    kr = torch.zeros((8, 160, 128), dtype=torch.float16, device=DEV)
    need = kv.kivi_decode_workspace_size(1, 32, 8, 2080, 158)
    assert need > 0
    ws = torch.zeros(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(kv.KiviError) as e:
        kv.kivi_decode_attend(q, gk, gv, 2080, kr, kr, 158, 8, w.sm_scale, workspace=ws)
    assert e.value.status == 3


def test_many_sequence_lengths_one_build():
    """55 sequence lengths through flush and decode with no per-length
    specialisation (sequence length is a runtime argument, never compiled in)."""
    rng = np.random.default_rng(55)
    w = synth.Workload("len", B=1, Hkv=2, Hq=8, D=128, S=0, bits=4, G=32, R=32, n_outlier=4,
                       outlier_scale=8.0, seed=1)
    for i, S in enumerate(range(33, 33 + 55 * 7, 7)):
        k = synth.keys(rng, (2, S), 128, np.array([1, 2, 3, 4]), 8.0)
        v = synth.normal(rng, (2, S, 128))
        q = synth.normal(rng, (1, 8, 128))
        n = kv.kivi_flush_count(S, 32, 32)
        out, ref = decode_case(w, n, S - n, k, v, q)
        assert np.max(np.abs(out - ref)) <= TOL, S


@pytest.mark.parametrize("name", ["qwen8b", "long2bit"])
def test_dequant_kv_equals_oracle(name):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.prefill_inputs(w)
    n = kv.kivi_flush_count(w.S, w.R, w.G)
    ks = kv.KiviStore(0, w.BH, n, w.D, w.G, w.bits, device=DEV)
    vs = kv.KiviStore(1, w.BH, n, w.D, w.G, w.bits, device=DEV)
    kv.kivi_flush_kv(dev(k), dev(v), w.R, ks, vs)
    kd, vd = kv.kivi_dequant_kv(ks, vs, n)
    rk = oracle.flush(0, k, n, oracle.Store(0, w.BH, n, w.D, w.G, w.bits))
    rv = oracle.flush(1, v, n, oracle.Store(1, w.BH, n, w.D, w.G, w.bits))
    assert np.array_equal(host(kd).view(np.uint16), oracle.dequant(rk, n).view(np.uint16))
    assert np.array_equal(host(vd).view(np.uint16), oracle.dequant(rv, n).view(np.uint16))
    # ragged S through the fused call
    kd2, vd2 = kv.kivi_dequant_kv(ks, vs, n - 13)
    assert np.array_equal(host(kd2).view(np.uint16), oracle.dequant(rk, n - 13).view(np.uint16))
    assert np.array_equal(host(vd2).view(np.uint16), oracle.dequant(rv, n - 13).view(np.uint16))


def test_residual_kv_append_and_compact():
    rng = np.random.default_rng(18)
    kres = synth.normal(rng, (5, 160, 128))
    vres = synth.normal(rng, (5, 160, 128))
    ksrc = synth.normal(rng, (5, 70, 128))
    vsrc = synth.normal(rng, (5, 70, 128))
    gk, gv = dev(kres), dev(vres)
    assert kv.kivi_residual_append_kv(dev(ksrc), dev(vsrc), gk, gv, 90, n_new=70) == 160
    oracle.residual_append(kres, 90, ksrc, 70)
    oracle.residual_append(vres, 90, vsrc, 70)
    assert np.array_equal(host(gk), kres) and np.array_equal(host(gv), vres)
    assert kv.kivi_residual_compact_kv(gk, gv, 160, 32) == 128
    oracle.residual_compact(kres, 160, 32)
    oracle.residual_compact(vres, 160, 32)
    assert np.array_equal(host(gk), kres) and np.array_equal(host(gv), vres)


# ---------------------------------------------------------------------------
# maximum sizes: more heads than one grid dimension holds, more (batch, KV
# head) pairs than the decode has merge counters
# ---------------------------------------------------------------------------

def test_flush_dequant_fake_quant_beyond_65535_heads():
    """BH = 65543 heads of one 32-token group each: the launches cut the heads
    into slices of at most 65535 (grid y). Checked against the oracle on a
    sample of heads on both sides of each cut (the oracle runs per head)."""
    BH, S = 65535 + 8, 32
    gen = torch.Generator(device=DEV)
    gen.manual_seed(11)
    x = torch.randn((BH, S, 128), generator=gen, device=DEV).to(torch.float16)
    sample = [0, 1, 65533, 65534, 65535, 65536, BH - 1]
    xs = host(x[sample])
    for axis in (0, 1):
        gs = kv.KiviStore(axis, BH, S, device=DEV)
        fn = kv.kivi_flush_keys if axis == 0 else kv.kivi_flush_values
        assert fn(x, 0, gs) == S
        rs = oracle.Store(axis, len(sample), S, 128, 32, 4)
        oracle.flush(axis, xs, S, rs)
        assert np.array_equal(host(gs.codes[sample]), rs.codes)
        assert np.array_equal(host(gs.scale[sample]).view(np.uint32), rs.scale.view(np.uint32))
        d = host(kv.kivi_dequant(gs, S)[sample])
        assert np.array_equal(d.view(np.uint16), oracle.dequant(rs, S).view(np.uint16))
        ffn = kv.kivi_fake_quant_keys if axis == 0 else kv.kivi_fake_quant_values
        out, n = ffn(x, 0)
        assert n == S
        assert np.array_equal(host(out[sample]).view(np.uint16), d.view(np.uint16))
        del gs, out


def test_decode_beyond_merge_counters():
    """B * Hkv = 8800 > 8192 pairs: the plan gives every pair one split (no
    merge counters). Sampled sequences are checked against the oracle."""
    B, Hkv, Hq, S_q, n_res = 1100, 8, 32, 64, 5
    assert kv.kivi_decode_workspace_size(B, Hq, Hkv, S_q, n_res) == 0
    w = synth.Workload("wide", B=B, Hkv=Hkv, Hq=Hq, D=128, S=S_q + n_res, bits=4, G=32, R=0, n_outlier=4,
                       outlier_scale=8.0, seed=21)
    k, v, q = synth.prefill_inputs_torch(w, 3, DEV)
    gk = kv.KiviStore(0, w.BH, S_q, device=DEV)
    gv = kv.KiviStore(1, w.BH, S_q, device=DEV)
    kv.kivi_flush_kv(k, v, 0, gk, gv, n_tokens=S_q)
    out = host(kv.kivi_decode_attend(q, gk, gv, S_q, k[:, S_q:], v[:, S_q:], n_res, Hkv, w.sm_scale))
    kh, vh, qh = host(k), host(v), host(q)
    for b in (0, 549, 1099):
        sl = slice(b * Hkv, (b + 1) * Hkv)
        rk = oracle.flush(0, kh[sl].copy(), S_q, oracle.Store(0, Hkv, S_q, 128, 32, 4))
        rv = oracle.flush(1, vh[sl].copy(), S_q, oracle.Store(1, Hkv, S_q, 128, 32, 4))
        ref = oracle.decode_attend(qh[b:b + 1], rk, rv, S_q, np.ascontiguousarray(kh[sl, S_q:]),
                                   np.ascontiguousarray(vh[sl, S_q:]), n_res, Hkv, w.sm_scale)
        assert np.max(np.abs(out[b:b + 1] - ref)) <= TOL, b
