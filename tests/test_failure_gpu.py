"""Failure detection without a GPU fault: a bounded wait that nothing
completes gives up after its limit, records FATTN_ERR_TIMEOUT in the device
error word and returns; the context stays usable afterwards."""
import pytest
import torch

import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert fattn.get_device_status() == 0            # clean before
    fattn.selftest_wait_timeout(2_000_000)            # 2 ms
    assert fattn.get_device_status() == 5             # FATTN_ERR_TIMEOUT, read and cleared
    assert fattn.get_device_status() == 0             # cleared
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 300, 128, "bf16", 5))
    o, lse = fattn.fwd(q, k, v, causal=True)          # the context still works
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and fattn.get_device_status() == 0


def test_selftest_rejects_bad_limits():
    with pytest.raises(fattn.FattnError):
        fattn.selftest_wait_timeout(0)
    with pytest.raises(fattn.FattnError):
        fattn.selftest_wait_timeout(2_000_000_000)
