"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/kivi.h declares, computes the flush plan like the
oracle, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kivi.h")
OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, ALIGN = range(6)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(kivi_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return kv.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 11, names
    raw = ctypes.CDLL(kv.library_path)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing


def test_status_strings_and_version(L):
    for s, name in enumerate(["KIVI_OK", "KIVI_ERR_INVALID_ARG", "KIVI_ERR_UNSUPPORTED",
                              "KIVI_ERR_WORKSPACE", "KIVI_ERR_CUDA", "KIVI_ERR_ALIGNMENT"]):
        assert kv.kivi_status_string(s) == name
    assert kv.kivi_status_string(99) == "KIVI_ERR_UNKNOWN"
    assert kv.kivi_version() >= 100


def test_flush_count_matches_oracle(L):
    for n_res in range(0, 300):
        for r in (0, 1, 32, 128):
            for g in (32, 64):
                assert kv.kivi_flush_count(n_res, r, g) == oracle.flush_count(n_res, r, g)
    assert kv.kivi_flush_count(-1, 32, 32) == -1
    assert kv.kivi_flush_count(5, 32, 0) == -1


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced

# Every call below with FAKE pointers must be rejected by the host-side checks.
# They run only where no GPU is visible, so that a bug in those checks can
# never launch a kernel on a bogus address.
no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="fake-pointer validation tests run only without a GPU")


def flush(L, name="kivi_flush_keys", x=FAKE, BH=8, S=256, stride=256, D=128, G=32, bits=4, R=128,
          codes=FAKE, scale=FAKE, zero=FAKE, s_off=0, s_cap=256):
    n = ctypes.c_int(-7)
    st = getattr(L, name)(x, BH, S, stride, D, G, bits, R, codes, scale, zero, s_off, s_cap,
                          ctypes.byref(n), None)
    return st, n.value


@no_gpu
@pytest.mark.parametrize("name", ["kivi_flush_keys", "kivi_flush_values"])
def test_flush_rejects_bad_arguments_without_launching(L, name):
    assert flush(L, name, bits=3)[0] == UNSUPPORTED
    assert flush(L, name, bits=3 | 0x100)[0] == UNSUPPORTED   # KIVI_SCALE_F16 with a bad width
    assert flush(L, name, bits=4 | 0x200)[0] == UNSUPPORTED   # an unknown option bit
    assert flush(L, name, bits=4 | 0x100, zero=FAKE + 2)[0] == ALIGN  # the option passes the checks
    assert flush(L, name, D=96)[0] == UNSUPPORTED
    assert flush(L, name, D=512)[0] == UNSUPPORTED
    assert flush(L, name, D=64, G=128)[0] == UNSUPPORTED  # a value group would outgrow the row
    assert flush(L, name, G=16)[0] == UNSUPPORTED
    assert flush(L, name, G=256)[0] == UNSUPPORTED
    assert flush(L, name, G=96)[0] == UNSUPPORTED
    assert flush(L, name, G=64, s_cap=288)[0] == INVALID     # not a multiple of G
    assert flush(L, name, BH=0)[0] == INVALID
    assert flush(L, name, S=-1)[0] == INVALID
    assert flush(L, name, stride=100)[0] == INVALID          # head stride < S
    assert flush(L, name, s_cap=100)[0] == INVALID           # not a multiple of G
    assert flush(L, name, s_off=160)[0] == INVALID           # 160 + 128 > 256
    assert flush(L, name, x=None)[0] == INVALID
    assert flush(L, name, codes=FAKE + 4)[0] == ALIGN
    assert flush(L, name, zero=FAKE + 2)[0] == ALIGN
    # nothing to flush: OK, n_flushed = 0, no launch and no pointer needed
    assert flush(L, name, S=100, x=None, codes=None, scale=None, zero=None) == (OK, 0)


@no_gpu
def test_key_flush_needs_group_aligned_offset(L):
    assert flush(L, "kivi_flush_keys", s_off=16, s_cap=512)[0] == INVALID


@no_gpu
def test_dequant_rejects_bad_arguments(L):
    f = L.kivi_dequant
    assert f(0, FAKE, FAKE, FAKE, 8, 300, 128, 32, 4, 256, FAKE, None) == INVALID  # S > s_cap
    assert f(2, FAKE, FAKE, FAKE, 8, 64, 128, 32, 4, 256, FAKE, None) == INVALID   # bad axis
    assert f(0, FAKE, FAKE, FAKE, 8, 64, 128, 32, 5, 256, FAKE, None) == UNSUPPORTED
    assert f(0, FAKE, FAKE, FAKE + 8, 8, 64, 128, 32, 4, 256, FAKE, None) == ALIGN
    assert f(1, None, FAKE, FAKE, 8, 64, 128, 32, 4, 256, FAKE, None) == INVALID
    assert f(1, None, None, None, 8, 0, 128, 32, 4, 256, None, None) == OK         # empty


@no_gpu
def test_residual_rejects_bad_arguments(L):
    assert L.kivi_residual_append(FAKE, 4, 4, FAKE, 8, 160, 128, 158, None) == INVALID  # overflow
    assert L.kivi_residual_append(FAKE, 2, 4, FAKE, 8, 160, 128, 0, None) == INVALID    # stride < n_new
    assert L.kivi_residual_append(FAKE, 4, 4, FAKE, 8, 160, 96, 0, None) == UNSUPPORTED  # D in {64, 128, 256}
    assert L.kivi_residual_append(FAKE + 2, 4, 4, FAKE, 8, 160, 128, 0, None) == ALIGN
    assert L.kivi_residual_append(None, 4, 0, None, 8, 160, 128, 0, None) == OK
    assert L.kivi_residual_compact(FAKE, 8, 160, 128, 100, 101, None) == INVALID
    assert L.kivi_residual_compact(FAKE, 8, 160, 128, 161, 1, None) == INVALID
    assert L.kivi_residual_compact(FAKE, 8, 160, 128, 100, 0, None) == OK
    assert L.kivi_residual_compact(FAKE, 8, 160, 128, 100, 100, None) == OK


def decode(L, q=FAKE, S_q=2080, s_cap=2080, n_res=158, res_cap=160, B=1, Hq=32, Hkv=8, D=128,
           G=32, bits=4, ws=FAKE, wbytes=1 << 30, sm=0.088, out=FAKE):
    return L.kivi_decode_attend(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, S_q, s_cap, FAKE, FAKE, n_res,
                                res_cap, B, Hq, Hkv, D, G, bits, sm, out, ws, wbytes, None)


@no_gpu
def test_decode_rejects_bad_arguments(L):
    assert decode(L, Hq=12) == INVALID               # 12 / 8 is not an integer
    assert decode(L, G=16) == UNSUPPORTED            # group sizes 32, 64, 128
    assert decode(L, D=96) == UNSUPPORTED            # head dims 64, 128, 256
    assert decode(L, D=64, G=128, S_q=2048, s_cap=2048) == UNSUPPORTED  # G > D
    assert decode(L, D=256, ws=None) == WORKSPACE    # D = 256 passes the checks
    assert decode(L, bits=4 | 0x100, ws=None) == WORKSPACE  # fp16 scales pass the checks
    assert decode(L, bits=4 | 0x400) == UNSUPPORTED
    assert decode(L, G=64) == INVALID                # s_cap 2080 is not a multiple of 64
    assert decode(L, G=128, S_q=2048, s_cap=2048, ws=None) == WORKSPACE  # G = 128 passes the checks
    assert decode(L, Hq=520) == UNSUPPORTED          # 65 query heads per KV head
    assert decode(L, Hq=1024) == UNSUPPORTED         # 128 query heads per KV head
    assert decode(L, S_q=0, n_res=0) == INVALID
    assert decode(L, S_q=3000) == INVALID            # S_q > s_cap
    assert decode(L, n_res=200) == INVALID           # n_res > res_cap
    assert decode(L, q=None) == INVALID
    assert decode(L, out=FAKE + 4) == ALIGN
    assert decode(L, sm=float("inf")) == INVALID
    assert decode(L, ws=None) == WORKSPACE
    need = L.kivi_decode_workspace_size(1, 32, 8, 2080, 158, 128)
    assert need > 0
    assert decode(L, wbytes=need - 1) == WORKSPACE


@no_gpu
def test_fake_quant_argument_checks(L):
    n = ctypes.c_int(-7)
    fk = L.kivi_fake_quant_keys
    assert fk(FAKE, 8, 256, 256, 96, 32, 4, 128, FAKE + 4096, 256, ctypes.byref(n), None) == UNSUPPORTED
    assert fk(FAKE, 8, 256, 256, 128, 32, 3, 128, FAKE + 4096, 256, ctypes.byref(n), None) == UNSUPPORTED
    assert fk(FAKE, 8, 256, 200, 128, 32, 4, 128, FAKE + 4096, 256, ctypes.byref(n), None) == INVALID  # stride < S
    assert fk(FAKE, 8, 256, 256, 128, 32, 4, 128, FAKE + 4096, 255, ctypes.byref(n), None) == INVALID
    assert fk(FAKE, 8, 256, 256, 128, 32, 4, -1, FAKE + 4096, 256, ctypes.byref(n), None) == INVALID
    assert fk(None, 8, 256, 256, 128, 32, 4, 128, FAKE + 4096, 256, ctypes.byref(n), None) == INVALID
    assert fk(FAKE, 8, 256, 256, 128, 32, 4, 128, None, 256, ctypes.byref(n), None) == INVALID
    assert fk(FAKE, 8, 256, 256, 128, 32, 4, 128, FAKE, 300, ctypes.byref(n), None) == INVALID  # in place, other stride
    assert fk(FAKE + 8, 8, 256, 256, 128, 32, 4, 128, FAKE + 4096, 256, ctypes.byref(n), None) == ALIGN
    # nothing to do: S == 0 reports n = 0 without touching the device
    assert fk(None, 8, 0, 0, 128, 32, 4, 128, None, 0, ctypes.byref(n), None) == OK and n.value == 0
    assert L.kivi_fake_quant_kv(FAKE, None, 8, 256, 256, 128, 32, 4, 128, FAKE + 4096, FAKE + 8192, 256,
                                ctypes.byref(n), None) == INVALID


def test_wait_timeouts_rejects_null(L):
    assert L.kivi_wait_timeouts(None, 0) == INVALID


@no_gpu
def test_workspace_init_rejects_null(L):
    assert L.kivi_decode_workspace_init(None, 0, None) == OK      # nothing to zero
    assert L.kivi_decode_workspace_init(None, 1024, None) == INVALID


def test_workspace_size(L):
    assert L.kivi_decode_workspace_size(1, 32, 8, 0, 0, 128) == 0
    assert L.kivi_decode_workspace_size(1, 32, 8, 64, 0, 96) == 0      # unsupported head dim
    # the partials hold D floats per split: a wider head needs a larger workspace
    w64, w128, w256 = (L.kivi_decode_workspace_size(1, 32, 8, 4096, 64, d) for d in (64, 128, 256))
    assert 32768 < w64 < w128 < w256
    small = L.kivi_decode_workspace_size(1, 32, 8, 2080, 158, 128)
    big = L.kivi_decode_workspace_size(1, 32, 8, 32640, 128, 128)
    assert 0 < small <= big
    # a single 32-token tile needs no split and no workspace
    assert L.kivi_decode_workspace_size(1, 32, 8, 32, 0, 128) == 0
    # a split plan's workspace starts with the fixed merge-counter block
    assert small > 32768
    # more (batch, KV head) pairs than merge counters: one split each, no workspace
    assert L.kivi_decode_workspace_size(2048, 32, 8, 32640, 128, 128) == 0


@no_gpu
def test_every_plan_fits_the_noalloc_scratch(L):
    """Without a device the planner sizes for 152 SMs (a GB300). Its split
    count keeps the partials near one per planned warp, so over a wide grid of
    shapes (group sizes 1 to 64, sub-groups included) no workspace exceeds
    the 8 MiB library-owned scratch of kivi_decode_attend_noalloc, at any
    supported head dim (the partials hold D floats per split)."""
    worst = {64: 0, 128: 0, 256: 0}
    for hkv in (1, 2, 8, 32):
        for gq in (1, 2, 3, 4, 6, 8, 12, 32, 64):
            for B in (1, 3, 16, 64, 256):
                for S in (32, 100, 1024, 4096, 32768, 131072):
                    for n_res in (0, 37):
                        for D in worst:
                            worst[D] = max(worst[D], L.kivi_decode_workspace_size(B, hkv * gq, hkv, S, n_res, D))
    assert 3 << 20 < worst[128] <= 4 * 1024 * 1024
    assert worst[64] < worst[128] < worst[256]
    assert 6 << 20 < worst[256] <= 8 * 1024 * 1024


def test_decode_plan_rules(L):
    """The decode's split plan (kivi_decode_plan_info; planned for 152 SMs
    without a device) follows its rules on a grid of shapes: splits cover the
    tiles without an empty split, the warp-pair kernel only for group size 32,
    head dim 128, fp32 scales and 1, 2 or 4 heads per KV head, query
    sub-groups of 4, one split per head group beyond the merge counters, and
    a workspace at least as large as the plan's partials."""
    seen_pair = seen_mma = seen_one_split = 0
    for B in (1, 4, 32, 256, 2048):
        for hkv, gq in ((8, 4), (8, 1), (2, 8), (8, 3), (1, 12)):
            for S_q, n_res in ((0, 37), (2080, 158), (4032, 64), (16256, 128)):
                for D, G, hs in ((128, 32, False), (128, 64, False), (64, 32, False), (256, 128, False),
                                 (128, 32, True)):
                    p = kv.kivi_decode_plan_info(B, hkv * gq, hkv, S_q, n_res, D, G, 4, hs)
                    assert p["n_tiles"] == -(-S_q // 32) + -(-n_res // 16)
                    # the kernels spread a head group's tiles evenly over its splits: none is empty
                    assert p["n_split"] * p["tiles_per_split"] >= p["n_tiles"]
                    assert 1 <= p["n_split"] <= p["n_tiles"]
                    assert p["q_sub"] == (1 if gq in (1, 2, 4) else -(-gq // 4))
                    if p["pair_kernel"]:
                        seen_pair += 1
                        assert (D, G, hs) == (128, 32, False) and gq in (1, 2, 4)
                        assert p["warps_per_cta"] == 8
                    else:
                        seen_mma += 1
                        assert p["warps_per_cta"] in ((2, 4, 8) if D == 128 else (4, 8))
                    if B * hkv * p["q_sub"] > 8192:
                        seen_one_split += 1
                        assert p["n_split"] == 1  # more head groups than merge counters: one split each
                    ws = L.kivi_decode_workspace_size(B, hkv * gq, hkv, S_q, n_res, D)
                    if p["n_split"] > 1:
                        assert ws >= 32768 + B * hkv * gq * p["n_split"] * (D + 2) * 4
    assert seen_pair and seen_mma and seen_one_split
    # balance: a one-warp-per-tile grid between one CTA per SM and one wave
    # (8-warp CTAs, two per SM on 152 SMs) fills every SM's slots
    for S_q, bits in ((16256, 4), (32640, 2), (8064, 4)):
        p = kv.kivi_decode_plan_info(1, 32, 8, S_q, 128, bits=bits)
        assert p["pair_kernel"] == 0 and p["warps_per_cta"] == 8
        assert 8 * p["n_split"] == 2 * 152, (S_q, p)
    # short warp runs at B=16: 2-warp CTAs, 8 per SM, one wave, shorter runs
    # than the 4-warp plan (which spilled past one wave or left longer runs)
    for S_q, n_res in ((1408, 128), (2944, 128), (3968, 128), (896, 128)):
        p = kv.kivi_decode_plan_info(16, 32, 8, S_q, n_res)
        assert p["warps_per_cta"] == 2 and 16 * 8 * p["n_split"] <= 8 * 152, (S_q, p)
        assert p["tiles_per_warp"] <= 8
    for S_q, n_res in ((1920, 128), (3456, 128)):  # one wave, runs nearly as short already: unchanged
        assert kv.kivi_decode_plan_info(16, 32, 8, S_q, n_res)["warps_per_cta"] == 4
    assert kv.kivi_decode_plan_info(32, 32, 8, 4032, 64)["warps_per_cta"] == 4  # long runs: unchanged
    for B, S_q in ((1, 65408), (2, 32640), (6, 2944)):  # a 2-warp plan would need more than 24 splits
        p = kv.kivi_decode_plan_info(B, 32, 8, S_q, 128)
        assert p["warps_per_cta"] != 2 or p["n_split"] <= 24, (B, S_q, p)
    # the qwen8b decode takes the warp-pair kernel; stores of another group
    # size or head dim, or with fp16 scales, the one-warp-per-tile kernel
    assert kv.kivi_decode_plan_info(1, 32, 8, 2080, 158)["pair_kernel"] == 1
    for kw in ({"G": 64}, {"D": 64}, {"scale_f16": True}):
        assert kv.kivi_decode_plan_info(1, 32, 8, 2080, 158, **kw)["pair_kernel"] == 0
    with pytest.raises(kv.KiviError):
        kv.kivi_decode_plan_info(1, 12, 8, 2080, 158)          # 12 / 8 heads
    with pytest.raises(kv.KiviError):
        kv.kivi_decode_plan_info(1, 32, 8, 2080, 158, D=64, G=128)


def fake_cache(**kw):
    """A kivi_cache struct over never-dereferenced 16-byte aligned addresses."""
    c = kv._CacheStruct(8, 128, 32, 4, 128, 256, 160, *([FAKE] * 8), 0, 0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@no_gpu
def test_cache_rejects_bad_arguments_without_launching(L):
    """Every check of kivi_cache_prefill / _append / _decode runs before the
    first launch and leaves the counters unchanged: geometry, buffers,
    counters, and room in the stores for every flush the call would make."""
    n = ctypes.c_int(-7)

    def prefill(c, S=200, stride=None, k=FAKE, v=FAKE):
        return L.kivi_cache_prefill(ctypes.byref(c), k, v, S if stride is None else stride, S, ctypes.byref(n), None)

    def append(c, n_new=1, k=FAKE, v=FAKE, stride=None):
        return L.kivi_cache_append(ctypes.byref(c), k, v, n_new if stride is None else stride, n_new,
                                   ctypes.byref(n), None)

    assert prefill(fake_cache(res_cap=159)) == INVALID            # window < R + G
    assert prefill(fake_cache(D=96)) == UNSUPPORTED
    assert prefill(fake_cache(bits=3)) == UNSUPPORTED
    assert prefill(fake_cache(group_size=0)) == INVALID
    assert prefill(fake_cache(s_cap=250)) == INVALID              # not a multiple of G
    assert prefill(fake_cache(S_q=288)) == INVALID                # S_q > s_cap
    assert prefill(fake_cache(n_res=161)) == INVALID              # n_res > res_cap
    assert prefill(fake_cache(res_off=-1)) == INVALID             # window start before the buffer
    assert prefill(fake_cache(res_off=100, n_res=61)) == INVALID  # window past the buffer's end
    assert prefill(fake_cache(k_res=None)) == INVALID
    assert prefill(fake_cache(vzero=FAKE + 2)) == ALIGN
    assert prefill(fake_cache(), k=FAKE + 8) == ALIGN
    assert prefill(fake_cache(), k=None) == INVALID
    assert prefill(fake_cache(), stride=100) == INVALID           # head stride < S
    c = fake_cache(n_res=5)
    assert prefill(c) == INVALID and (c.S_q, c.n_res) == (0, 5)   # windows not empty
    c = fake_cache(S_q=224)
    assert prefill(c, S=300) == INVALID and c.S_q == 224          # flush of 160 overruns the store
    assert prefill(fake_cache(), S=0) == OK                       # nothing to do
    # append: a full store cannot take the flush the 160th window token triggers
    c = fake_cache(S_q=256, n_res=159)
    assert append(c) == INVALID and (c.S_q, c.n_res) == (256, 159)
    c = fake_cache(S_q=250, s_cap=512, n_res=159)                 # ragged store end: no further key flush
    assert append(c) == INVALID and (c.S_q, c.n_res) == (250, 159)
    # pieces: 340 tokens through a 160-token window would flush 288 tokens into a 256-token store
    c = fake_cache(S_q=0, n_res=100)
    assert append(c, n_new=340) == INVALID and (c.S_q, c.n_res) == (0, 100)
    assert append(fake_cache(), n_new=2, stride=1) == INVALID     # head stride < n_new
    assert append(fake_cache(), v=None) == INVALID
    assert append(fake_cache(), k=FAKE + 4) == ALIGN
    assert append(fake_cache(), n_new=0, k=None, v=None) == OK
    # decode: B * Hkv must be the cache's BH
    c = fake_cache(S_q=256, n_res=150)
    assert L.kivi_cache_decode(ctypes.byref(c), FAKE, 2, 32, 8, 0.088, FAKE, FAKE, 1 << 30, None) == INVALID
    assert L.kivi_cache_decode(ctypes.byref(c), FAKE, 1, 32, 8, 0.088, FAKE, None, 0, None) == WORKSPACE
    assert L.kivi_cache_decode(None, FAKE, 1, 32, 8, 0.088, FAKE, FAKE, 1 << 30, None) == INVALID
