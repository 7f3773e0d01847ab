"""KIVI_DECODE_STORE_READY: the decode requests its first store tiles before
waiting for the preceding kernel on its stream. The arithmetic is unchanged,
so the outputs must be bit-identical to the plain decode's, and within 2e-3 of
the float64 oracle, whichever kernel and merge the plan takes. The graph case
launches decodes back to back (each one's early loads overlap the previous
decode's tail), the way a serving loop issues them."""
import numpy as np
import pytest
import torch

import oracle
import kivi_kv_cache_gb300 as kv
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _case(B, Hkv, Hq, S_q, n_res, bits, G=32, D=128, seed=0, scale_f16=False):
    w = synth.Workload("sr", B=B, Hkv=Hkv, Hq=Hq, D=D, S=S_q + n_res, bits=bits, G=G, R=0, n_outlier=4,
                       outlier_scale=8.0, seed=seed)
    k, v, q = synth.prefill_inputs(w)
    dev = torch.device("cuda")
    kt, vt = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    s_cap = max(G, -(-S_q // G) * G)
    ks = kv.KiviStore(0, w.BH, s_cap, D, G, bits, device=dev, scale_f16=scale_f16)
    vs = kv.KiviStore(1, w.BH, s_cap, D, G, bits, device=dev, scale_f16=scale_f16)
    if S_q:
        kv.kivi_flush_kv(kt, vt, 0, ks, vs, n_tokens=S_q)
    kr, vr = kt[:, S_q:].contiguous(), vt[:, S_q:].contiguous()
    return w, torch.from_numpy(q).to(dev), ks, vs, kr, vr, (k, v, q)


@pytest.mark.parametrize("B,Hkv,Hq,S_q,n_res,bits,G,D,hs", [
    (1, 8, 32, 2080, 158, 4, 32, 128, False),    # warp pairs
    (1, 8, 32, 16256, 128, 4, 32, 128, False),   # one warp per tile, balanced ticket merge
    (1, 8, 32, 32640, 128, 2, 32, 128, False),   # long 2-bit
    (4, 8, 32, 4032, 64, 4, 32, 128, False),     # cluster merge
    (2, 8, 64, 8192, 40, 4, 64, 128, True),      # two query sub-groups, G = 64, fp16 scales
    (1, 4, 4, 3000, 0, 2, 32, 256, False),       # head dim 256, store only
    (3, 2, 6, 96, 17, 4, 32, 64, False),         # head dim 64, a few tiles
])
def test_store_ready_is_bit_identical(B, Hkv, Hq, S_q, n_res, bits, G, D, hs):
    w, q, ks, vs, kr, vr, host = _case(B, Hkv, Hq, S_q, n_res, bits, G, D, seed=B + S_q % 97, scale_f16=hs)
    res = (kr, vr) if n_res else (None, None)
    plain = kv.kivi_decode_attend(q, ks, vs, S_q, res[0], res[1], n_res, Hkv, w.sm_scale)
    ready = kv.kivi_decode_attend(q, ks, vs, S_q, res[0], res[1], n_res, Hkv, w.sm_scale, store_ready=True)
    torch.cuda.synchronize()
    assert torch.equal(plain, ready)
    ok = oracle.Store(0, w.BH, ks.s_cap, D, G, bits, scale_f16=hs)
    ov = oracle.Store(1, w.BH, vs.s_cap, D, G, bits, scale_f16=hs)
    k, v, qh = host
    if S_q:
        oracle.flush(0, k, S_q, ok)
        oracle.flush(1, v, S_q, ov)
    kres = np.ascontiguousarray(k[:, S_q:]) if n_res else np.zeros((w.BH, 1, D), np.float16)
    vres = np.ascontiguousarray(v[:, S_q:]) if n_res else np.zeros((w.BH, 1, D), np.float16)
    ref = oracle.decode_attend(qh, ok, ov, S_q, kres, vres, n_res, Hkv, w.sm_scale)
    err = float(np.max(np.abs(ready.cpu().numpy().astype(np.float64) - ref)))
    assert err <= TOL, err


def test_store_ready_back_to_back_in_a_graph():
    """Eight decodes on four independent caches, captured in one CUDA graph
    with the option set (each decode's early store loads overlap the previous
    decode's tail); every output equals the plain eager decode's."""
    cases = [_case(1, 8, 32, 16256, 128, 4, seed=30 + i) for i in range(2)]
    cases += [_case(1, 8, 32, 4064, 32, 4, seed=40 + i) for i in range(2)]
    dev = torch.device("cuda")
    refs, outs, wss = [], [], []
    for w, q, ks, vs, kr, vr, _ in cases:
        S_q, n_res = ks.s_cap, kr.shape[1]
        refs.append(kv.kivi_decode_attend(q, ks, vs, S_q, kr, vr, n_res, w.Hkv, w.sm_scale))
        outs.append(torch.full_like(refs[-1], float("nan")))
        wss.append(kv.kivi_decode_workspace(kv.kivi_decode_workspace_size(w.B, w.Hq, w.Hkv, S_q, n_res, w.D), dev))

    def run():
        for rep in range(2):
            for (w, q, ks, vs, kr, vr, _), out, ws in zip(cases, outs, wss):
                kv.kivi_decode_attend(q, ks, vs, ks.s_cap, kr, vr, kr.shape[1], w.Hkv, w.sm_scale, out=out,
                                      workspace=ws, store_ready=True)

    run()
    torch.cuda.synchronize()
    for o in outs:
        o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o, r)
