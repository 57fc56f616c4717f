"""Failure detection on the GPU without a fault: a bounded wait that can never
complete gives up after its limit, the device error word records it, the
host reads RF_ERR_DEVICE_TIMEOUT, and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    import cascaded_reductions_loop_gb300 as rf
    assert rf.rf_get_device_status() == rf.RF_OK
    rf.rf_selftest_wait_timeout(2000)            # 2 ms limit
    assert rf.rf_get_device_status() == rf.RF_ERR_DEVICE_TIMEOUT
    assert rf.rf_get_device_status() == rf.RF_OK  # read-and-clear
    # the context still works: a normal call succeeds afterwards
    q = torch.randn(1, 1, 64, 64, device="cuda")
    o = torch.empty_like(q)
    rf.rf_attn_fwd(q, q, q, o, 0.125)
    assert rf.rf_get_device_status() == rf.RF_OK
    assert torch.isfinite(o).all()
