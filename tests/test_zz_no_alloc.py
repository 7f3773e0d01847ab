"""kivi_decode_attend_noalloc: the decode for callers that cannot allocate
device memory when they decode (runtimes that pre-assign all of HBM, C callers
without an allocator of their own). It must give the same result as
kivi_decode_attend with a caller-provided workspace, call after call, while
using only the library's fixed 8 MiB device scratch.

This file is named so that pytest collects it last; it needs nothing from the
other test files and also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
SCRATCH_BYTES = 8 * 1024 * 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _decode_inputs(w, S_q, n_res, seed, scale_f16=False):
    rng = np.random.default_rng(seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), w.D, synth.outlier_channels(w), w.outlier_scale)
    v = synth.normal(rng, (w.BH, S_q + n_res, w.D))
    q = synth.normal(rng, (w.B, w.Hq, w.D))
    k, v, q = (torch.from_numpy(a).cuda() for a in (k, v, q))
    ks = kv.KiviStore(0, w.BH, S_q, w.D, w.G, w.bits, device="cuda", scale_f16=scale_f16)
    vs = kv.KiviStore(1, w.BH, S_q, w.D, w.G, w.bits, device="cuda", scale_f16=scale_f16)
    assert kv.kivi_flush_kv(k, v, 0, ks, vs, n_tokens=S_q) == S_q
    return q, ks, vs, k[:, S_q:], v[:, S_q:]


@pytest.mark.parametrize("name,S_q,n_res", [("qwen8b", 2080, 158), ("long2bit", 32640, 128),
                                            ("batched", 4032, 64)])
def test_noalloc_matches_workspace_entry_point_twice(name, S_q, n_res):
    w = synth.WORKLOADS[name]
    q, ks, vs, kr, vr = _decode_inputs(w, S_q, n_res, seed=w.seed + 17)
    need = kv.kivi_decode_workspace_size(w.B, w.Hq, w.Hkv, S_q, n_res, w.D)
    assert 0 < need <= SCRATCH_BYTES
    ref = kv.kivi_decode_attend(q, ks, vs, S_q, kr, vr, n_res, w.Hkv, w.sm_scale)
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        out = torch.full_like(ref, float("nan"))
        kv.kivi_decode_attend_noalloc(q, ks, vs, S_q, kr, vr, n_res, w.Hkv, w.sm_scale, out=out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= TOL, err


@pytest.mark.parametrize("D,lo_mb", [(128, 3), (256, 6)])
def test_noalloc_largest_plan(D, lo_mb):
    """The largest workspace plan over a wide grid of shapes (256 sequences of
    one KV head with 12 query heads, three sub-groups of 4, over 1024 packed
    2-bit tokens: about 3.2 MB of partials at head dim 128, 6.4 MB at 256):
    the library-owned scratch holds it, and the result equals the workspace
    entry point's."""
    w = synth.Workload("widest", B=256, Hkv=1, Hq=12, D=D, S=1024, bits=2, G=32, R=0, n_outlier=4,
                       outlier_scale=8.0, seed=9)
    need = kv.kivi_decode_workspace_size(w.B, w.Hq, w.Hkv, 1024, 0, w.D)
    assert lo_mb << 20 < need <= SCRATCH_BYTES
    q, ks, vs, kr, vr = _decode_inputs(w, 1024, 0, seed=3)
    ref = kv.kivi_decode_attend(q, ks, vs, 1024, None, None, 0, w.Hkv, w.sm_scale)
    out = kv.kivi_decode_attend_noalloc(q, ks, vs, 1024, None, None, 0, w.Hkv, w.sm_scale)
    torch.cuda.synchronize()
    err = (out.double() - ref.double()).abs().max().item()
    assert err <= TOL, err


def test_noalloc_alternating_plans():
    """Back-to-back no-alloc calls whose plans use the shared scratch
    differently: an fp16-scale store of group size 64 read by 8 query heads
    per KV head (two sub-groups of 4 heads, each with its own merge counter
    and partials), then a 4-head fp32-scale store of group size 32 (the
    warp-pair kernel), then the first again. Each call must leave the
    counters it used at zero for the next, whatever its plan; every result
    equals kivi_decode_attend with a workspace of its own."""
    # 16384 tokens: 13 splits per head group over 416 CTAs, more than one
    # wave of clusters, so the splits merge through the scratch's counters
    wa = synth.Workload("gq8_g64_f16", B=2, Hkv=8, Hq=64, D=128, S=16384 + 100, bits=4, G=64, R=0, n_outlier=4,
                        outlier_scale=8.0, seed=21)
    wb = synth.WORKLOADS["qwen8b"]
    A = _decode_inputs(wa, 16384, 100, seed=5, scale_f16=True)
    Bc = _decode_inputs(wb, 2080, 158, seed=6)
    assert kv.kivi_decode_plan_info(wa.B, wa.Hq, wa.Hkv, 16384, 100, 128, 64, 4, True)["q_sub"] == 2
    assert kv.kivi_decode_plan_info(wb.B, wb.Hq, wb.Hkv, 2080, 158)["pair_kernel"] == 1
    cases = [(wa, A, 16384, 100), (wb, Bc, 2080, 158)]
    refs = [kv.kivi_decode_attend(x[0], x[1], x[2], S_q, x[3], x[4], n_res, w.Hkv, w.sm_scale)
            for w, x, S_q, n_res in cases]
    for w, x, S_q, n_res in cases:
        assert 0 < kv.kivi_decode_workspace_size(w.B, w.Hq, w.Hkv, S_q, n_res, w.D) <= SCRATCH_BYTES
    for i in (0, 1, 0, 1):
        w, x, S_q, n_res = cases[i]
        out = torch.full_like(refs[i], float("nan"))
        kv.kivi_decode_attend_noalloc(x[0], x[1], x[2], S_q, x[3], x[4], n_res, w.Hkv, w.sm_scale, out=out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        err = (out.double() - refs[i].double()).abs().max().item()
        assert err <= TOL, (i, err)


def test_noalloc_two_warp_plan():
    """A plan of 2-warp CTAs (B=16, 1408 packed + 128 fp16 tokens: 9 splits
    per head group, 8 CTAs per SM) through the library-owned scratch, twice,
    equals the workspace entry point."""
    w = synth.Workload("w2", B=16, Hkv=8, Hq=32, D=128, S=1408 + 128, bits=4, G=32, R=0, n_outlier=4,
                       outlier_scale=8.0, seed=13)
    assert kv.kivi_decode_plan_info(16, 32, 8, 1408, 128)["warps_per_cta"] == 2
    q, ks, vs, kr, vr = _decode_inputs(w, 1408, 128, seed=8)
    ref = kv.kivi_decode_attend(q, ks, vs, 1408, kr, vr, 128, w.Hkv, w.sm_scale)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kv.kivi_decode_attend_noalloc(q, ks, vs, 1408, kr, vr, 128, w.Hkv, w.sm_scale, out=out)
        torch.cuda.synchronize()
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= TOL, err
