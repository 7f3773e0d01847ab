"""The documented usage example of the package (flush, dequant, decode), run as written and checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def test_readme_example():
    import __graft_entry__
    __graft_entry__.build()
    torch.manual_seed(0)
    # --- the usage example, as documented ---
    import kivi_kv_cache_gb300 as kv
    k = torch.randn(8, 2238, 128, device="cuda").half()       # [B*H_kv, S, D]
    v = torch.randn_like(k)
    n = kv.kivi_flush_count(2238, 128)                         # tokens the flush takes: 2080
    ks, vs = kv.KiviStore(0, 8, n, device="cuda"), kv.KiviStore(1, 8, n, device="cuda")
    kv.kivi_flush_kv(k, v, 128, ks, vs)                        # packed 4-bit store
    q = torch.randn(1, 32, 128, device="cuda").half()          # one query token, 32 heads
    out = kv.kivi_decode_attend(q, ks, vs, n, k[:, n:], v[:, n:], 2238 - n, 8, 128 ** -0.5)
    # --- check ---
    assert n == 2080
    kh, vh, qh = (t.cpu().numpy() for t in (k, v, q))
    rk = oracle.flush(0, kh, n, oracle.Store(0, 8, n, 128, 32, 4))
    rv = oracle.flush(1, vh, n, oracle.Store(1, 8, n, 128, 32, 4))
    assert np.array_equal(ks.codes.cpu().numpy(), rk.codes)
    ref = oracle.decode_attend(qh, rk, rv, n, np.ascontiguousarray(kh[:, n:]), np.ascontiguousarray(vh[:, n:]),
                               2238 - n, 8, 128 ** -0.5)
    assert np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)) <= 2e-3
