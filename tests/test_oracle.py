"""Pins for the CPU oracle: each test ties it to something other than itself --
values the pages print, hand-worked groups, closed forms, invariants, library
routines (numpy's fp16, torch's float64 attention) and brute force."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from kivi_kv_cache_gb300 import synth


# ---------------------------------------------------------------------------
# fp16 conversions against numpy's IEEE binary16
# ---------------------------------------------------------------------------

def test_half_to_float_all_65536_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_float(bits.view(np.float16))
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_round_trip_and_ties():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    finite = np.isfinite(h)
    f = h[finite].astype(np.float32)
    assert np.array_equal(oracle.float_to_half(f).view(np.uint16), h[finite].view(np.uint16))
    # exact midpoints between consecutive positive fp16 values: ties to even
    pos = np.arange(0, 0x7bff, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    exact = mid.astype(np.float64) == (pos[:-1] + pos[1:]) / 2
    ref = mid[exact].astype(np.float16)
    assert np.array_equal(oracle.float_to_half(mid[exact]).view(np.uint16), ref.view(np.uint16))
    assert np.array_equal(oracle.float_to_half(-mid[exact]).view(np.uint16), (-ref).view(np.uint16))


def test_float_to_half_random_and_edges():
    rng = np.random.default_rng(0)
    e = rng.uniform(-30, 17, size=400_000)
    f = (rng.choice([-1.0, 1.0], size=e.size) * rng.uniform(1, 2, size=e.size) * 2.0 ** e).astype(np.float32)
    edges = np.array([0.0, -0.0, 65504, 65519.996, 65520, 65536, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                      3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, np.inf, -np.inf,
                      6.1e-5, 5.96e-8], np.float32)
    f = np.concatenate([f, edges])
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16)
    assert np.array_equal(oracle.float_to_half(f).view(np.uint16), ref.view(np.uint16))


# ---------------------------------------------------------------------------
# hand-worked groups and flushes
# ---------------------------------------------------------------------------

def _floats(s):
    return [float(v) for v in s.split()]


@pytest.mark.parametrize("line", read_golden("quant_groups.txt"))
def test_golden_group(line):
    name, bits, x, codes, scale, zero, recon = [p.strip() for p in line.split(";")]
    bits = int(bits)
    x = np.array(_floats(x), np.float32)
    c, s, z = oracle.quantize_group(x, bits)
    assert c.tolist() == [int(v) for v in codes.split()], name
    assert s == np.float32(float(scale)) and z == np.float32(float(zero)), name
    assert np.signbit(z) == np.signbit(np.float32(float(zero))), name
    assert np.signbit(s) == np.signbit(np.float32(float(scale))), name
    # the recon of the same group through the key store path
    G = x.size
    store = oracle.Store(0, 1, G, 4 if bits == 2 else 2, G, bits)
    xs = np.repeat(x.astype(np.float16)[None, :, None], store.D, axis=2)
    oracle.flush(0, xs, G, store)
    r = oracle.recon_f32(store, G)[0, :, 0]
    assert r.tolist() == _floats(recon), name


@pytest.mark.parametrize("line", read_golden("quant_groups_scale_f16.txt"))
def test_golden_group_scale_f16(line):
    """The fp16-scale storage option on hand-worked groups: the rounding of
    the scale to fp16 changes codes (one_fifteenth, one_third), can zero the
    scale (underflow) and can engage the clip (clamp)."""
    name, bits, x, codes, scale, zero, recon = [p.strip() for p in line.split(";")]
    bits = int(bits)
    x = np.array(_floats(x), np.float32)
    c, s, z = oracle.quantize_group(x, bits | oracle.SCALE_F16)
    assert c.tolist() == [int(v) for v in codes.split()], name
    assert s == np.float32(float(scale)) and z == np.float32(float(zero)), name
    # through the key store: the stored scale is the fp16 value, and the
    # reconstruction uses it
    G = x.size
    store = oracle.Store(0, 1, G, 4 if bits == 2 else 2, G, bits, scale_f16=True)
    xs = np.repeat(x.astype(np.float16)[None, :, None], store.D, axis=2)
    oracle.flush(0, xs, G, store)
    assert store.scale.dtype == np.float16
    assert float(store.scale[0, 0, 0]) == float(scale), name
    assert oracle.recon_f32(store, G)[0, :, 0].tolist() == _floats(recon), name
    # and through the value store (one group per token row)
    vstore = oracle.Store(1, 1, G, G, G, bits, scale_f16=True)
    oracle.flush(1, x.astype(np.float16)[None, None, :], 1, vstore)
    assert float(vstore.scale[0, 0, 0]) == float(scale), name
    assert oracle.recon_f32(vstore, 1)[0, 0].tolist() == _floats(recon), name


def test_scale_f16_store_matches_rounded_fp32_scale():
    """On random data the fp16-scale store holds exactly the fp16 rounding of
    the fp32-scale store's scales (numpy's binary16 conversion), every code is
    within [0, 2^bits - 1], and codes differ from the fp32-scale codes only
    where the rounded scale moved a quotient across a rounding boundary."""
    rng = np.random.default_rng(71)
    for axis in (0, 1):
        for bits in (2, 4):
            x = synth.normal(rng, (3, 96, 64)) * np.float16(3)
            a = oracle.flush(axis, x, 96, oracle.Store(axis, 3, 96, 64, 32, bits))
            b = oracle.flush(axis, x, 96, oracle.Store(axis, 3, 96, 64, 32, bits, scale_f16=True))
            assert np.array_equal(b.scale.view(np.uint16), a.scale.astype(np.float16).view(np.uint16))
            assert np.array_equal(b.zero.view(np.uint16), a.zero.view(np.uint16))
            ca = np.stack([oracle.unpack_codes(r, 64, bits) for r in a.codes.reshape(-1, 64 * bits // 8)])
            cb = np.stack([oracle.unpack_codes(r, 64, bits) for r in b.codes.reshape(-1, 64 * bits // 8)])
            assert cb.max() <= 2 ** bits - 1
            assert 0 < np.count_nonzero(ca != cb) < ca.size // 20  # some, never many, codes move
            assert np.max(np.abs(ca.astype(int) - cb.astype(int))) == 1
            # the reconstruction error stays within half a stored step (plus rounding)
            r = oracle.recon_f32(b, 96)
            s = b.scale.astype(np.float32)
            step = np.repeat(s, 32, axis=1) if axis == 0 else np.repeat(s, 32, axis=2)
            assert np.all(np.abs(r - x.astype(np.float32)) <= step * 0.5 * (1 + 2 ** -9) + 1e-6)


def test_scale_f16_decode_matches_brute_force():
    """Attention over fp16-scale stores of 2 KV heads equals float64 softmax
    attention written out here over the stores' fp32 reconstructions (each
    head's scales must be read at its own offset)."""
    rng = np.random.default_rng(72)
    B, Hkv, Hq, D, S_q, n_res = 1, 2, 4, 64, 64, 5
    k = synth.normal(rng, (B * Hkv, S_q + n_res, D))
    v = synth.normal(rng, (B * Hkv, S_q + n_res, D))
    q = synth.normal(rng, (B, Hq, D))
    rk = oracle.flush(0, k, S_q, oracle.Store(0, B * Hkv, S_q, D, 32, 4, scale_f16=True))
    rv = oracle.flush(1, v, S_q, oracle.Store(1, B * Hkv, S_q, D, 32, 4, scale_f16=True))
    kr, vr = np.ascontiguousarray(k[:, S_q:]), np.ascontiguousarray(v[:, S_q:])
    out = oracle.decode_attend(q, rk, rv, S_q, kr, vr, n_res, Hkv, 0.125)
    K = np.concatenate([oracle.recon_f32(rk, S_q), kr.astype(np.float32)], axis=1).astype(np.float64)
    V = np.concatenate([oracle.recon_f32(rv, S_q), vr.astype(np.float32)], axis=1).astype(np.float64)
    for h in range(Hq):
        hk = h // (Hq // Hkv)
        sc = 0.125 * (K[hk] @ q[0, h].astype(np.float64))
        p = np.exp(sc - sc.max())
        ref = (p / p.sum()) @ V[hk]
        assert np.max(np.abs(out[0, h] - ref)) < 1e-12


def _parse_table(name):
    rows = {}
    for ln in read_golden(name):
        key, *vals = ln.split()
        rows.setdefault(key, []).append(vals)
    return rows


def test_golden_key_flush_ragged():
    t = _parse_table("key_flush_ragged.txt")
    x = np.array([[float(v) for v in r] for r in t["x"]], np.float16)[None]
    n_flush = oracle.flush_count(5, 0, 4)
    assert n_flush == 5
    store = oracle.Store(0, 1, 8, 4, 4, 2)
    oracle.flush(0, x, n_flush, store)
    packed = [int(v, 16) for v in t["packed"][0]]
    assert store.codes[0, :5, 0].tolist() == packed
    codes = np.array([[int(v) for v in r] for r in t["codes"]])
    assert np.array_equal(np.stack([oracle.unpack_codes(store.codes[0, s], 4, 2) for s in range(5)]), codes)
    assert store.scale[0].tolist() == [[float(v) for v in r] for r in t["scale"]]
    assert store.zero[0].astype(np.float32).tolist() == [[float(v) for v in r] for r in t["zero"]]
    assert oracle.recon_f32(store, 5)[0].tolist() == [[float(v) for v in r] for r in t["recon"]]


def test_golden_value_flush():
    t = _parse_table("value_flush.txt")
    x = np.array([[float(v) for v in r] for r in t["x"]], np.float16)[None]
    store = oracle.Store(1, 1, 4, 8, 4, 2)
    oracle.flush(1, x, 2, store)
    assert store.codes[0, :2].reshape(-1).tolist() == [int(v, 16) for v in t["packed"][0]]
    assert store.scale[0, :2].tolist() == [[float(v) for v in r] for r in t["scale"]]
    assert store.zero[0, :2].astype(np.float32).tolist() == [[float(v) for v in r] for r in t["zero"]]
    assert oracle.recon_f32(store, 2)[0].tolist() == [[float(v) for v in r] for r in t["recon"]]
    # the fp16 dequant of exactly representable recon values is the same
    assert oracle.dequant(store, 2)[0].astype(np.float32).tolist() == [[float(v) for v in r] for r in t["recon"]]


@pytest.mark.parametrize("line", read_golden("packing.txt"))
def test_golden_packing(line):
    bits, codes, packed = [p.strip() for p in line.split(";")]
    bits = int(bits)
    codes = [int(v) for v in codes.split()]
    packed = [int(v, 16) for v in packed.split()]
    assert oracle.pack_codes(codes, bits).tolist() == packed
    assert oracle.unpack_codes(packed, len(codes), bits).tolist() == codes


# ---------------------------------------------------------------------------
# flush rule against the counts the pages print
# ---------------------------------------------------------------------------

R, G, CHUNK = 32, 32, 2048


def _prefill(n_res, prompt):
    """Feed a prompt in 2048-token chunks while more than 2048 remain, then the
    rest; return (n_res, tokens flushed, flush events)."""
    flushed = events = 0
    remaining = prompt
    while remaining > 0:
        piece = CHUNK if remaining > CHUNK else remaining
        remaining -= piece
        n_res += piece
        n = oracle.flush_count(n_res, R, G)
        if n:
            flushed += n
            events += 1
            n_res -= n
    return n_res, flushed, events


def _decode(n_res, appended):
    events = 0
    for _ in range(appended):
        n_res += 1
        n = oracle.flush_count(n_res, R, G)
        if n:
            assert n == G
            events += 1
            n_res -= n
        assert R <= n_res < R + G or n_res < R
    return n_res, events


@pytest.mark.parametrize("line", read_golden("flush_counts.txt"))
def test_flush_rule_matches_pages(line):
    kind, *vals = [p.strip() for p in line.split(";")]
    vals = [int(v) for v in vals]
    if kind == "prefill":
        prompt, flushed = vals
        assert _prefill(0, prompt)[1] == flushed
    elif kind == "calls":
        prompt, new, calls = vals
        n_res, _, ev = _prefill(0, prompt)
        _, ev2 = _decode(n_res, new)
        assert 2 * (ev + ev2) == calls
    else:
        start, appended, events = vals
        assert _decode(start, appended)[1] == events


def test_flush_count_closed_form():
    for n_res in range(0, 400):
        for r in (0, 32, 128):
            for g in (32, 64):
                n = oracle.flush_count(n_res, r, g)
                if r == 0:
                    assert n == n_res
                else:
                    assert n % g == 0 and 0 <= n_res - n
                    assert n == 0 or (r <= n_res - n < r + g)
                    assert n != 0 or n_res < r + g


# ---------------------------------------------------------------------------
# invariants and an independent restatement with torch fp32 ops
# ---------------------------------------------------------------------------

def _unpack_np(packed, bits):
    """Independent numpy unpack: element i at bit offset i*bits, low bits first."""
    per = 8 // bits
    mask = (1 << bits) - 1
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * per,), np.uint8)
    for k in range(per):
        out[..., k::per] = (packed >> (k * bits)) & mask
    return out


def torch_eight_ops(x16: np.ndarray, G: int, bits: int, axis: int):
    """The reference's array-op path restated with torch fp32 CPU ops: expose
    the group axis (edge-replicate pad), min, max, subtract, divide, round
    (half-to-even), clip, multiply, add. Returns (codes, scale, zero, recon)
    shaped like x (scale/zero per group)."""
    x = torch.from_numpy(x16.astype(np.float32))
    BH, S, D = x.shape
    L = float((1 << bits) - 1)
    if axis == 0:
        ng = -(-S // G)
        pad = ng * G - S
        if pad:
            x = torch.cat([x, x[:, -1:, :].expand(BH, pad, D)], dim=1)
        xg = x.reshape(BH, ng, G, D)
        mn = xg.amin(dim=2, keepdim=True)
        mx = xg.amax(dim=2, keepdim=True)
    else:
        xg = x.reshape(BH, S, D // G, G)
        mn = xg.amin(dim=3, keepdim=True)
        mx = xg.amax(dim=3, keepdim=True)
    mn = mn + 0.0
    mx = mx + 0.0
    s = (mx - mn) / L
    q = torch.round((xg - mn) / s).clamp(0, L)
    q = torch.where(s == 0, torch.zeros_like(q), q)
    prod = q * s
    recon = prod + mn
    if axis == 0:
        codes = q.reshape(BH, -1, D)[:, :S].to(torch.uint8)
        recon = recon.reshape(BH, -1, D)[:, :S]
        s, mn = s[:, :, 0, :], mn[:, :, 0, :]
    else:
        codes = q.reshape(BH, S, D).to(torch.uint8)
        recon = recon.reshape(BH, S, D)
        s, mn = s[..., 0], mn[..., 0]
    return codes.numpy(), s.numpy(), mn.numpy(), recon.numpy()


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("S", [64, 77, 256])
def test_oracle_matches_torch_eight_ops(axis, bits, S):
    w = synth.WORKLOADS["tiny"]
    rng = np.random.default_rng(100 + S + bits + 7 * axis)
    ch = synth.outlier_channels(w)
    x = synth.keys(rng, (3, S), 128, ch, 10.0) if axis == 0 else synth.normal(rng, (3, S, 128))
    # plant exact ties: a grid-aligned token row / channel run
    x[0, 0, :] = np.float16(0.0)
    x[0, 1, :] = np.float16(1.5)
    x[0, 2, :] = np.float16(0.75)
    x[1, :, 5] = np.float16(2.0)  # a constant key group (max == min)
    G = 32
    s_cap = -(-S // G) * G
    store = oracle.Store(axis, 3, s_cap, 128, G, bits)
    n = S if axis == 0 else S
    oracle.flush(axis, x, n, store)
    codes, s, z, recon = torch_eight_ops(x, G, bits, axis)
    ours = _unpack_np(store.codes[:, :S], bits)
    assert np.array_equal(ours, codes)
    if axis == 0:
        ng = -(-S // G)
        assert np.array_equal(store.scale[:, :ng].view(np.uint32), s.astype(np.float32).view(np.uint32))
        assert np.array_equal(store.zero[:, :ng].astype(np.float32), z)
    else:
        assert np.array_equal(store.scale[:, :S].view(np.uint32), s.astype(np.float32).view(np.uint32))
        assert np.array_equal(store.zero[:, :S].astype(np.float32), z)
    r = oracle.recon_f32(store, S)
    assert np.array_equal(r.view(np.uint32), recon.astype(np.float32).view(np.uint32))
    d16 = oracle.dequant(store, S)
    assert np.array_equal(d16.view(np.uint16), recon.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_invariants(bits):
    rng = np.random.default_rng(7 + bits)
    L = (1 << bits) - 1
    for trial in range(300):
        n = int(rng.integers(1, 65))
        x = (rng.standard_normal(n) * 10 ** rng.uniform(-3, 3)).astype(np.float16).astype(np.float32)
        c, s, z = oracle.quantize_group(x, bits)
        assert c.min() >= 0 and c.max() <= L
        assert z == x.min()
        if x.max() > x.min():
            assert c[np.argmin(x)] == 0 and c[np.argmax(x)] == L
            recon = c.astype(np.float32) * np.float32(s)
            recon = recon + np.float32(z)
            ulp32 = np.spacing(np.abs(x).max().astype(np.float32))
            assert np.all(np.abs(recon - x) <= s / 2 + 4 * ulp32)
        else:
            assert s == 0 and np.all(c == 0)


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_invariants_scale_f16(bits):
    """The fp16-scale option on random groups over six decades of magnitude:
    the scale is numpy's binary16 rounding of the fp32-scale quantizer's scale;
    codes stay in [0, 2^bits - 1]; whenever that scale is a normal fp16 number
    the minimum codes to 0, the maximum to 2^bits - 1, and every
    reconstruction lies within half a stored step (plus rounding)."""
    rng = np.random.default_rng(17 + bits)
    L = (1 << bits) - 1
    normal = 0
    for trial in range(300):
        n = int(rng.integers(1, 65))
        x = (rng.standard_normal(n) * 10 ** rng.uniform(-6, 3)).astype(np.float16).astype(np.float32)
        c32, s32, _ = oracle.quantize_group(x, bits)
        c, s, z = oracle.quantize_group(x, bits | oracle.SCALE_F16)
        assert s == np.float32(np.float16(s32))
        assert c.min() >= 0 and c.max() <= L and z == x.min()
        if s >= 2.0 ** -14:
            normal += 1
            assert c[np.argmin(x)] == 0 and c[np.argmax(x)] == L
            recon = c.astype(np.float32) * np.float32(s) + np.float32(z)
            ulp32 = np.spacing(np.abs(x).max().astype(np.float32))
            assert np.all(np.abs(recon - x) <= s / 2 + 4 * ulp32)
            assert np.max(np.abs(c.astype(int) - c32.astype(int))) <= 1
        elif s == 0:
            assert np.all(c == 0)
    assert normal > 150


def test_grid_values_round_trip():
    # values on min + k*scale with dyadic scale are reproduced exactly
    rng = np.random.default_rng(3)
    for bits in (2, 4):
        L = (1 << bits) - 1
        for _ in range(100):
            z = float(rng.integers(-64, 64)) / 4
            s = 2.0 ** int(rng.integers(-4, 3))
            k = rng.integers(0, L + 1, size=32)
            k[0], k[1] = 0, L
            x = (z + k * s).astype(np.float32)
            c, s2, z2 = oracle.quantize_group(x, bits)
            assert s2 == s and z2 == z and np.array_equal(c, k)


def test_pack_unpack_round_trip():
    rng = np.random.default_rng(5)
    for bits in (2, 4):
        c = rng.integers(0, 1 << bits, size=128).astype(np.uint8)
        p = oracle.pack_codes(c, bits)
        assert np.array_equal(oracle.unpack_codes(p, 128, bits), c)
        assert np.array_equal(_unpack_np(p[None], bits)[0], c)


def test_residual_append_compact_match_slicing():
    rng = np.random.default_rng(9)
    res = synth.normal(rng, (3, 40, 8))
    ref = res.copy()
    src = synth.normal(rng, (3, 10, 8))
    oracle.residual_append(res, 20, src, 6)
    ref[:, 20:26] = src[:, :6]
    assert np.array_equal(res, ref)
    oracle.residual_compact(res, 26, 16)
    ref2 = ref.copy()
    ref2[:, :10] = ref[:, 16:26]
    assert np.array_equal(res, ref2)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _case(B=2, Hkv=2, Hq=8, D=64, S_q=96, n_res=20, bits=4, G=32, seed=0):
    rng = np.random.default_rng(seed)
    BH = B * Hkv
    ch = np.array([3, 5]) if D < 32 else np.array([3, 17])
    k = synth.keys(rng, (BH, S_q), D, ch, 8.0)
    v = synth.normal(rng, (BH, S_q, D))
    s_cap = -(-max(S_q, 1) // G) * G
    ks = oracle.Store(0, BH, s_cap, D, G, bits)
    vs = oracle.Store(1, BH, s_cap, D, G, bits)
    if S_q:
        oracle.flush(0, k, S_q, ks)
        oracle.flush(1, v, S_q, vs)
    kr = synth.keys(rng, (BH, n_res + 3), D, ch, 8.0)
    vr = synth.normal(rng, (BH, n_res + 3, D))
    q = synth.normal(rng, (B, Hq, D))
    return q, k, v, ks, vs, kr, vr


@pytest.mark.parametrize("S_q,n_res,bits", [(96, 20, 4), (77, 0, 2), (0, 9, 4), (64, 1, 2)])
def test_attention_matches_torch_sdpa_float64(S_q, n_res, bits):
    B, Hkv, Hq, D, G = 2, 2, 8, 64, 32
    q, k, v, ks, vs, kr, vr = _case(B, Hkv, Hq, D, S_q, n_res, bits, G, seed=S_q + n_res)
    sm = 1 / math.sqrt(D)
    out = oracle.decode_attend(q, ks, vs, S_q, kr, vr, n_res, Hkv, sm)
    # K, V from the independent torch restatement of the quantizer
    if S_q:
        kh = torch_eight_ops(k, G, bits, 0)[3].astype(np.float64)
        vh = torch_eight_ops(v, G, bits, 1)[3].astype(np.float64)
    else:
        kh = np.zeros((B * Hkv, 0, D))
        vh = np.zeros((B * Hkv, 0, D))
    K = np.concatenate([kh, kr[:, :n_res].astype(np.float64)], 1).reshape(B, Hkv, -1, D)
    V = np.concatenate([vh, vr[:, :n_res].astype(np.float64)], 1).reshape(B, Hkv, -1, D)
    K = torch.from_numpy(K).repeat_interleave(Hq // Hkv, dim=1)
    V = torch.from_numpy(V).repeat_interleave(Hq // Hkv, dim=1)
    Q = torch.from_numpy(q.astype(np.float64))[:, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=sm)[:, :, 0, :].numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_attention_brute_force_tiny():
    # D=8, G=4, bits=2, one group of 4 store tokens and 2 residual tokens, GQA 2:1
    q, k, v, ks, vs, kr, vr = _case(B=1, Hkv=1, Hq=2, D=8, S_q=4, n_res=2, bits=2, G=4, seed=11)
    out = oracle.decode_attend(q, ks, vs, 4, kr, vr, 2, 1, 0.3)
    K = [list(map(float, r)) for r in oracle.recon_f32(ks, 4)[0]] + [list(map(float, r)) for r in kr[0, :2]]
    V = [list(map(float, r)) for r in oracle.recon_f32(vs, 4)[0]] + [list(map(float, r)) for r in vr[0, :2]]
    for h in range(2):
        qh = [float(a) for a in q[0, h]]
        sc = [0.3 * sum(qh[d] * K[t][d] for d in range(8)) for t in range(6)]
        m = max(sc)
        p = [math.exp(s - m) for s in sc]
        den = sum(p)
        ref = [sum(p[t] * V[t][d] for t in range(6)) / den for d in range(8)]
        assert np.allclose(out[0, h], ref, rtol=0, atol=1e-13)


def test_attention_special_cases():
    q, k, v, ks, vs, kr, vr = _case(B=1, Hkv=2, Hq=4, D=64, S_q=0, n_res=5, seed=3)
    assert kr.shape[1] >= 5
    # one cached token: the output is that token's value row
    out = oracle.decode_attend(q, ks, vs, 0, kr, vr, 1, 2, 0.125)
    assert np.array_equal(out[0, :2], np.repeat(vr[0:1, 0].astype(np.float64), 2, 0))
    assert np.array_equal(out[0, 2:], np.repeat(vr[1:2, 0].astype(np.float64), 2, 0))
    # identical keys: uniform weights, the output is the mean of the value rows
    kr2 = np.repeat(kr[:, :1], kr.shape[1], axis=1).copy()
    out = oracle.decode_attend(q, ks, vs, 0, kr2, vr, 5, 2, 0.125)
    assert np.allclose(out[0, 0], vr[0, :5].astype(np.float64).mean(0), atol=1e-14)
    assert np.allclose(out[0, 3], vr[1, :5].astype(np.float64).mean(0), atol=1e-14)
    # one dominant logit selects its value row
    kr3 = np.zeros_like(kr)
    kr3[:, 2, :] = np.float16(4.0)
    q3 = np.ones_like(q)
    out = oracle.decode_attend(q3, ks, vs, 0, kr3, vr, 5, 2, 1.0)
    assert np.allclose(out[0, 1], vr[0, 2].astype(np.float64), atol=1e-12)


def test_attention_gqa_head_mapping():
    # each KV head carries a constant value row equal to its index; query head
    # h must read KV head h // (Hq / Hkv)
    B, Hkv, Hq, D = 2, 4, 8, 32
    rng = np.random.default_rng(1)
    kr = synth.normal(rng, (B * Hkv, 3, D))
    vr = np.zeros((B * Hkv, 3, D), np.float16)
    for bh in range(B * Hkv):
        vr[bh] = bh
    q = synth.normal(rng, (B, Hq, D))
    ks = oracle.Store(0, B * Hkv, 32, D, 32, 4)
    vs = oracle.Store(1, B * Hkv, 32, D, 32, 4)
    out = oracle.decode_attend(q, ks, vs, 0, kr, vr, 3, Hkv, 0.2)
    for b in range(B):
        for h in range(Hq):
            assert np.allclose(out[b, h], b * Hkv + h // (Hq // Hkv))


def test_quotient_is_ieee_division_not_reciprocal_multiply():
    """Groups where rint(a / s) and rint(a * (1 / s)) disagree (found with
    numpy's IEEE float32 ops): the oracle must follow the division."""
    rng = np.random.default_rng(21)
    found = 0
    for bits in (2, 4):
        L = np.float32((1 << bits) - 1)
        x = (rng.standard_normal((200_000, 32)) * 3).astype(np.float16).astype(np.float32)
        mn = x.min(1, keepdims=True) + np.float32(0)
        s = (x.max(1, keepdims=True) - mn) / L
        a = x - mn
        div = np.rint(a / s)
        rec = np.rint(a * (np.float32(1) / s))
        rows = np.nonzero((div != rec).any(1))[0][:20]
        for r in rows:
            c, _, _ = oracle.quantize_group(x[r], bits)
            assert np.array_equal(c, np.clip(div[r], 0, L).astype(np.uint8))
            found += 1
    assert found >= 5


@pytest.mark.parametrize("axis", [0, 1])
def test_flush_in_pieces_equals_one_shot(axis):
    """Flushing [0, 64) then [64, 128) at store offset 64 (reading x with a head
    stride of 160 tokens) gives the same store as one flush of [0, 128)."""
    rng = np.random.default_rng(31 + axis)
    x = synth.keys(rng, (3, 160), 128, np.array([1, 50]), 8.0)
    one = oracle.Store(axis, 3, 128, 128, 32, 4)
    oracle.flush(axis, x, 128, one)
    two = oracle.Store(axis, 3, 128, 128, 32, 4)
    oracle.flush(axis, x, 64, two, s_off=0, t0=0)
    oracle.flush(axis, x, 64, two, s_off=64, t0=64)
    for a, b in ((one.codes, two.codes), (one.scale, two.scale), (one.zero, two.zero)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    # and the pieces really came from the right tokens
    assert np.array_equal(oracle.recon_f32(one, 128), torch_eight_ops(x[:, :128].copy(), 32, 4, axis)[3])
