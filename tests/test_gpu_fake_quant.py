"""GPU parity of the fake quantization (the pages' kernels write the
quantize-then-dequantize fp16 tensor): for the tokens a flush would quantize,
the output must equal, bit for bit, the oracle's dequantization of the
oracle's flush of the same input; the remaining tokens are copied unchanged."""
import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def oracle_fake(axis, x, R, G=32, bits=4):
    """Oracle: dequant(flush(x)) for the flushed tokens, x itself after them."""
    BH, S, D = x.shape
    n = oracle.flush_count(S, R, G)
    out = x.astype(np.float16).copy()
    if n:
        rs = oracle.Store(axis, BH, -(-n // G) * G, D, G, bits)
        oracle.flush(axis, x, n, rs)
        out[:, :n] = oracle.dequant(rs, n)
    return out, n


def same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint16), np.asarray(b).view(np.uint16))


@pytest.mark.parametrize("name", ["tiny", "qwen8b", "long2bit"])
def test_fake_quant_workloads(name):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.prefill_inputs(w)
    for axis, x in ((0, k), (1, v)):
        fn = kv.kivi_fake_quant_keys if axis == 0 else kv.kivi_fake_quant_values
        out, n = fn(dev(x), w.R, bits=w.bits)
        ref, n_ref = oracle_fake(axis, x, w.R, bits=w.bits)
        assert n == n_ref
        assert same(host(out), ref), (name, axis)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_fake_quant_adversarial_ragged(bits, axis):
    """residual_length 0 (a ragged last key group), max == min groups, exact
    ties, -0, the full fp16 range and subnormals."""
    from test_gpu_parity import adversarial
    rng = np.random.default_rng(78)
    x = adversarial(rng, 3, 96)
    x = np.concatenate([x, synth.normal(rng, (3, 9, 128))], axis=1)  # S = 105: ragged at R = 0
    fn = kv.kivi_fake_quant_keys if axis == 0 else kv.kivi_fake_quant_values
    out, n = fn(dev(x), 0, bits=bits)
    ref, n_ref = oracle_fake(axis, x, 0, bits=bits)
    assert n == n_ref == 105
    assert same(host(out), ref)


def test_fake_quant_kv_strided_and_in_place():
    rng = np.random.default_rng(9)
    w = synth.WORKLOADS["qwen8b"]
    ch = synth.outlier_channels(w)
    big_k = synth.keys(rng, (8, 2400), 128, ch, 8.0)
    big_v = synth.normal(rng, (8, 2400, 128))
    S, R = 2238, 128
    k = dev(big_k)[:, 100:100 + S]  # views with a head stride of 2400 tokens
    v = dev(big_v)[:, 100:100 + S]
    kout = torch.full((8, 2300, 128), float("nan"), dtype=torch.float16, device=DEV)[:, :S]
    vout = torch.full((8, 2300, 128), float("nan"), dtype=torch.float16, device=DEV)[:, :S]
    _, _, n = kv.kivi_fake_quant_kv(k, v, R, kout=kout, vout=vout)
    rk, n_ref = oracle_fake(0, big_k[:, 100:100 + S], R)
    rv, _ = oracle_fake(1, big_v[:, 100:100 + S], R)
    assert n == n_ref == 2080
    assert same(host(kout), rk) and same(host(vout), rv)
    # in place: the output is the input view itself
    kv.kivi_fake_quant_kv(k, v, R, kout=k, vout=v)
    assert same(host(k), rk) and same(host(v), rv)
    # the tokens outside the views are untouched
    assert same(host(dev(big_k))[:, :100], big_k[:, :100])


@pytest.mark.parametrize("S,R", [(0, 128), (100, 128), (159, 128), (160, 128), (33, 0), (1, 0)])
def test_fake_quant_short_inputs(S, R):
    rng = np.random.default_rng(S + R)
    x = synth.normal(rng, (2, S, 128))
    for axis in (0, 1):
        fn = kv.kivi_fake_quant_keys if axis == 0 else kv.kivi_fake_quant_values
        out, n = fn(dev(x), R)
        ref, n_ref = oracle_fake(axis, x, R)
        assert n == n_ref
        assert same(host(out), ref), (S, R, axis)


@pytest.mark.parametrize("G", [64, 128])
@pytest.mark.parametrize("bits", [2, 4])
def test_fake_quant_group_sizes(G, bits):
    rng = np.random.default_rng(90 + G + bits)
    for S, R in [(100, 0), (700, 128)]:
        k = synth.keys(rng, (3, S), 128, np.array([3, 64, 65, 127]), 10.0)
        v = synth.normal(rng, (3, S, 128))
        for axis, x in ((0, k), (1, v)):
            fn = kv.kivi_fake_quant_keys if axis == 0 else kv.kivi_fake_quant_values
            out, n = fn(dev(x), R, G=G, bits=bits)
            ref, n_ref = oracle_fake(axis, x, R, G, bits)
            assert n == n_ref
            assert same(host(out), ref), (G, bits, S, axis)
