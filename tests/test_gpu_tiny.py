"""The kernel for very small problems (M * N * K <= 2^25, row-major, one
matrix; tiny.cu) against the oracle: ragged tiles, K beyond one 256-wide
chunk, padded leading dimensions (NaN padding), unaligned pointers, beta == 0
with NaN in C, integer inputs bit-exact. A forced tile configuration bypasses
it."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload, make_inputs

import gpu_helpers as H

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, 128), (1, 1, 1), (1, 37, 5), (37, 1, 5), (33, 65, 17), (31, 31, 257),
          (100, 90, 600), (30, 40, 3000), (64, 64, 1024), (200, 300, 150), (257, 129, 100),
          (2, 2, 8000)]


@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes(shape, dist):
    M, N, K = shape
    assert M * N * K <= 1 << 25
    H.check_against_oracle(Workload("tiny", M, N, K, 1.25, -0.5, dist, 71))
    assert binding.sgemm_last_config().startswith("tiny_32x32")


@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 0, 0), (0, 3, 0), (0, 0, 2)])
def test_padded_and_unaligned(offsets):
    w = Workload("tinypad", 70, 90, 333, 0.5, 3.0, "int3", 72, lda=335, ldb=93, ldc=97)
    H.check_against_oracle(w, offsets=offsets)
    assert binding.sgemm_last_config().startswith("tiny_32x32")
    H.check_against_oracle(w.with_(dist="normal"), offsets=offsets)


def test_vector_form_when_aligned():
    H.check_against_oracle(Workload("tinyvec", 96, 64, 256, 1.0, 1.0, "int3", 73))
    assert "vec128" in binding.sgemm_last_config()
    H.check_against_oracle(Workload("tinyscalar", 96, 64, 255, 1.0, 1.0, "int3", 73))
    assert "scalar" in binding.sgemm_last_config()


def test_beta_zero_does_not_read_c():
    w = Workload("tinybeta0", 60, 70, 80, 1.0, 0.0, "uniform", 74)
    A, B, _ = make_inputs(w)
    out = H.run_cuda(w, A, B, torch.full((w.M * w.LDC,), float("nan")))
    ref, mag = H.oracle_full(w, A, B, None)
    H.assert_match(w, H.logical(out, w.M, w.N, w.LDC), ref, mag)


def test_forced_configuration_bypasses_the_tiny_kernel():
    w = Workload("tinyforced", 128, 128, 128, 1.0, 0.0, "int3", 75)
    H.check_against_oracle(w, config=0)
    assert not binding.sgemm_last_config().startswith("tiny")


def test_just_above_the_threshold_uses_the_persistent_kernel():
    w = Workload("tinyedge", 256, 256, 513, 1.0, 0.0, "int3", 76)  # 2^25 + 2^16
    H.check_against_oracle(w)
    assert not binding.sgemm_last_config().startswith("tiny")
