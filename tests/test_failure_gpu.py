"""The failure path on a GPU, without a fault: fa_selftest_wait_timeout runs
the pipeline kernels' bounded mbarrier wait on barriers nobody arrives on.
The wait gives up after its 2 s limit, records the timeout in the device
status word (code, role, site, block) and raises the CTA's abort flag, so
the second waiting warp returns promptly; the host reads FA_ERR_TIMEOUT
through fa_check_status, the word is cleared, and the context still runs
attention."""
import time

import pytest
import torch

from exact_attention_forward_fa_gb300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(gpu_lib):
    fa = gpu_lib
    assert fa.fa_check_status() == fa.FA_OK              # start clean
    res = torch.zeros(2, dtype=torch.int32, device="cuda")
    t0 = time.time()
    assert fa.fa_selftest_wait_timeout(res) == fa.FA_OK
    assert fa.fa_check_status() == fa.FA_ERR_TIMEOUT
    elapsed = time.time() - t0
    assert 1.5 < elapsed < 30.0, elapsed                # one 2 s limit, not two in a row
    assert res.cpu().tolist() == [1, 1]                 # both waits returned false
    code, role, site, block = fa.fa_status_detail()
    assert (code, role, block) == (1, 7, 0) and site in (1, 2)
    assert fa.fa_check_status() == fa.FA_OK              # the word was cleared
    # the context is usable: a normal forward still runs and checks clean
    q, k, v = (x.cuda() for x in synth.qkv(1, 2, 256, 128, seed=5))
    o, lse = fa.attention(q, k, v)
    assert fa.fa_check_status() == fa.FA_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
