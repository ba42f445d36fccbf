"""The error path of the pipelined kernels on a real GPU: a wait that runs out
of budget is reported by w4a8_device_error as W4A8_ERR_TIMEOUT, reading the
word clears it, and the context keeps working (no fault, no hang: the wait is
bounded and the kernel returns)."""
import pytest
import torch

from helpers import MoECase, assert_close, bf16_to_f64, ensure_built

pytestmark = pytest.mark.gpu

W4A8_ERR_TIMEOUT = 7


def test_wait_timeout_is_reported_and_the_context_survives():
    ensure_built()
    import w4a8_moe_gb300 as lib
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lib.w4a8_selftest_wait_timeout(ws)
    assert lib.w4a8_device_error(ws) == W4A8_ERR_TIMEOUT
    assert lib.w4a8_device_error(ws) == 0          # reading clears the word
    case = MoECase(16, 256, 512, 8, 2, 0, seed=5)  # the same context still computes correctly
    out = case.run_gpu()
    assert_close(bf16_to_f64(out), case.oracle_out(), "forward after a reported timeout")
