"""The failure path on the device: a pipeline wait that nothing completes runs out
of time, the kernel reports FA_ERR_TIMEOUT through the status word and returns, and
the context stays usable. No fault, trap or hang is involved."""
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import inputs

from _util import compare

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from tiled_attention_06_gb300 import build
    build.build()
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_selftest_timeout(2000)  # 2 ms limit
    assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    assert "wait" in fa.fa_last_error_string()
    assert fa.fa_get_device_status() == fa.FA_OK
    q, k, v = inputs.prefill_inputs(1, 2, 130, 130, 64, torch.float16, seed=1)
    o = torch.empty_like(q, device="cuda")
    lse = torch.empty(1, 2, 130, device="cuda")
    fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), o, lse, 0.125, fa.FA_MASK_CAUSAL)
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention(q, k, v, 0.125, oracle.MASK_CAUSAL)
    compare(o, lse, ref_o, ref_l, "after timeout")
