"""CUDA path vs the oracle at the full workload sizes, in the launch
configuration the benchmark times (automatic tile choice, default stream):
sampled rows and elements against the oracle, and for integer inputs a
Freivalds identity that involves every element."""
import pytest

from dense_fp32_gemm_gb300.workloads import SWEEP_SIZES, WORKLOADS, integer_variant

import gpu_helpers as H

pytestmark = pytest.mark.gpu

NAMED = ["square4096", "edges8191x1000x777", "kdominant1024x1024x16384", "skinny16384x64x4096"]


@pytest.mark.parametrize("name", NAMED)
def test_named_real(name):
    H.check_sampled(WORKLOADS[name], rows=16, elements=2048)


@pytest.mark.parametrize("name", NAMED)
def test_named_integer_bit_exact(name):
    H.check_sampled(integer_variant(WORKLOADS[name]), rows=8, elements=1024)


@pytest.mark.parametrize("n", SWEEP_SIZES)
def test_sweep_integer_bit_exact(n):
    H.check_sampled(WORKLOADS[f"sweep{n}_int"], rows=4 if n >= 8192 else 16, elements=1024)


@pytest.mark.parametrize("n", SWEEP_SIZES)
def test_sweep_real(n):
    H.check_sampled(WORKLOADS[f"sweep{n}"], rows=2 if n >= 8192 else 8, elements=1024)
