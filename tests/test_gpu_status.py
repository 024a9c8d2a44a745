"""Bounded waits report instead of hanging, and argument errors are caught on
the host before anything is launched."""
import pytest
import torch

from dense_fp32_gemm_gb300 import binding

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_status():
    s = torch.cuda.current_stream().cuda_stream
    assert binding.sgemm_poll_device_status(s) == (0, 0)
    assert binding.sgemm_diag_wait_timeout(2_000_000, s) == 0  # 2 ms limit
    st, detail = binding.sgemm_poll_device_status(s)
    assert st == binding.SGEMM_ERR_DEVICE_TIMEOUT and detail == 1
    # the status was cleared by the poll and the context is still usable
    assert binding.sgemm_poll_device_status(s) == (0, 0)
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


def test_invalid_arguments_leave_c_untouched():
    C = torch.full((64,), 5.0, device="cuda")
    p = C.data_ptr()
    cases = [
        ((-1, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 4), binding.SGEMM_ERR_INVALID_DIM),
        ((4, 4, 4, 1.0, p, 3, p, 4, 0.0, p, 4), binding.SGEMM_ERR_INVALID_LD),
        ((4, 4, 4, 1.0, p, 4, p, 3, 0.0, p, 4), binding.SGEMM_ERR_INVALID_LD),
        ((4, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 2), binding.SGEMM_ERR_INVALID_LD),
        ((4, 4, 4, 1.0, 0, 4, p, 4, 0.0, p, 4), binding.SGEMM_ERR_NULL_PTR),
        ((4, 4, 4, 1.0, p, 4, p, 4, 0.0, 0, 4), binding.SGEMM_ERR_NULL_PTR),
        ((4, 4, 4, 1.0, p + 2, 4, p, 4, 0.0, p, 4), binding.SGEMM_ERR_MISALIGNED),
    ]
    for args, want in cases:
        assert binding.sgemm(*args, None) == want
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)


def test_status_is_clean_after_normal_runs():
    A = torch.randn(300, 200, device="cuda")
    B = torch.randn(200, 500, device="cuda")
    C = torch.zeros(300, 500, device="cuda")
    for _ in range(3):
        binding.gemm(A, B, C, 1.0, 0.0)
    assert binding.sgemm_poll_device_status(torch.cuda.current_stream().cuda_stream) == (0, 0)
