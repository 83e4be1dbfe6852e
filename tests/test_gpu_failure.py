"""Failure detection on the GPU without a fault: bounded waits that expire set
a status the host reads, and the context stays usable afterwards."""
import pytest
import torch

import moe_expert_layer_06_gb300 as m

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    m.moe_set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        m.moe_debug_expire_wait()
        assert m.moe_check_status() == m.MOE_ERR_DEVICE_TIMEOUT
        assert "wait" in m.last_error()
        assert m.moe_check_status() == m.MOE_OK  # read clears it
    finally:
        m.moe_set_wait_limit_ns(2_000_000_000)
    a = torch.arange(1000, device="cuda", dtype=torch.float32)
    assert float(a.sum().item()) == 499500.0
