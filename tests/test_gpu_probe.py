"""The TF32 tensor-core throughput probe (the 3xTF32 roofline's denominator)
returns a plausible rate: above what the 3xTF32 path itself reaches per TF32
product, below the nominal dense TF32 peak at the maximum clock."""
import pytest

from dense_fp32_gemm_gb300 import binding

pytestmark = pytest.mark.gpu


def test_tf32_mma_rate_is_plausible():
    st, tf = binding.sgemm_diag_tf32_mma_rate(20000)
    assert st == 0, binding.sgemm_status_string(st)
    # 152 SMs x 2.07 GHz x 4096 TF32 FLOP/clk/SM = 1289 TFLOP/s at most; the
    # 3xTF32 path's 16384^3 rate implies at least ~800 (three products each)
    assert 500.0 < tf < 1300.0, tf


def test_tf32_pair_mma_rate_is_plausible():
    # the two-SM form issues M = 256 MMAs over CTA pairs: per SM the same work
    st, tf = binding.sgemm_diag_tf32_pair_mma_rate(20000)
    assert st == 0, binding.sgemm_status_string(st)
    assert 500.0 < tf < 1300.0, tf
