"""The flush stages its group-size-32, head-dim-128 items with bulk tensor
copies and bounds every wait for one; a wait that ran out would be counted
in kivi_wait_timeouts. After the flushes of the other test files (collected
before this one) and one more long flush here, the count is zero.

Named so that pytest collects it after the parity files; it also passes when
run alone in a fresh process."""
import numpy as np
import pytest
import torch

import kivi_kv_cache_gb300 as kv
import oracle
from kivi_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_no_bulk_copy_wait_ran_out():
    assert kv.kivi_wait_timeouts() == 0  # the flushes of the earlier test files
    rng = np.random.default_rng(11)
    BH, S, D = 16, 4096 + 7, 128  # ragged: the last key group holds 7 tokens
    k = torch.from_numpy(synth.normal(rng, (BH, S, D))).cuda()
    v = torch.from_numpy(synth.normal(rng, (BH, S, D))).cuda()
    ks = kv.KiviStore(0, BH, S + 25, D, 32, 2, device="cuda")
    vs = kv.KiviStore(1, BH, S + 25, D, 32, 2, device="cuda")
    assert kv.kivi_flush_kv(k, v, 0, ks, vs) == S
    torch.cuda.synchronize()
    assert kv.kivi_wait_timeouts(reset=True) == 0
    assert kv.kivi_wait_timeouts() == 0
    # and the codes of the ragged last group are the oracle's
    ref = oracle.flush(0, k[:2].cpu().numpy(), S, oracle.Store(0, 2, S + 25, D, 32, 2))
    assert np.array_equal(ks.codes[:2].cpu().numpy(), ref.codes)
