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


def _decode_inputs(w, S_q, n_res, seed):
    rng = np.random.default_rng(seed)
    k = synth.keys(rng, (w.BH, S_q + n_res), w.D, synth.outlier_channels(w), w.outlier_scale)
    v = synth.normal(rng, (w.BH, S_q + n_res, w.D))
    q = synth.normal(rng, (w.B, w.Hq, w.D))
    k, v, q = (torch.from_numpy(a).cuda() for a in (k, v, q))
    ks = kv.KiviStore(0, w.BH, S_q, w.D, w.G, w.bits, device="cuda")
    vs = kv.KiviStore(1, w.BH, S_q, w.D, w.G, w.bits, device="cuda")
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
