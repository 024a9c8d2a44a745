"""The pages' kernels 3, 7 and 8 (sgemm_ladder) against the oracle, element by
element: several tiles with ragged tails on every dimension, padded leading
dimensions (NaN padding), the 128-bit and the 4-byte access forms, unaligned
pointers, the degenerate cases, and the 4096 cube on sampled rows and
elements."""
import functools

import numpy as np
import pytest
import torch

from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import WORKLOADS, Workload, integer_variant, make_inputs

import gpu_helpers as H

pytestmark = pytest.mark.gpu

KERNELS = list(binding.LADDER_KERNELS)

SHAPES = [
    (128, 128, 128), (1, 1, 1), (7, 9, 3), (33, 65, 17), (257, 129, 100), (300, 520, 77),
    (129, 257, 1000), (64, 64, 4097), (1000, 40, 129), (2, 700, 33),
]


def ladder(kernel):
    return functools.partial(binding.sgemm_ladder, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes(kernel, dist, shape):
    M, N, K = shape
    w = Workload("ladder", M, N, K, 1.25, -0.5, dist, 21)
    H.check_against_oracle(w, fn=ladder(kernel))
    cfg = binding.sgemm_last_config()
    assert cfg.startswith(f"ladder_kernel{kernel} "), cfg


@pytest.mark.parametrize("kernel", KERNELS)
def test_vector_form_with_ragged_edges(kernel):
    # leading dimensions multiples of 4 and aligned pointers: the 128-bit
    # form, with N and K not multiples of 4 at the tile edges
    w = Workload("vec", 300, 202, 77, 0.5, 3.0, "int3", 22, lda=80, ldb=204, ldc=208)
    H.check_against_oracle(w, fn=ladder(kernel))
    if kernel != 3:
        assert "vec128" in binding.sgemm_last_config()
    H.check_against_oracle(w.with_(dist="normal"), fn=ladder(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
def test_scalar_form_padded(kernel):
    # lda not a multiple of 4: the 4-byte form; padding holds NaN
    w = Workload("padded", 301, 203, 777, 1.25, -0.5, "normal", 2, lda=779, ldb=207, ldc=210)
    H.check_against_oracle(w, fn=ladder(kernel))
    if kernel != 3:
        assert "scalar" in binding.sgemm_last_config()
    H.check_against_oracle(w.with_(dist="int3"), fn=ladder(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 3)])
def test_unaligned_pointers(kernel, offsets):
    w = Workload("unaligned", 190, 260, 150, 0.5, 3.0, "int3", 6)
    H.check_against_oracle(w, offsets=offsets, fn=ladder(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
def test_beta_zero_does_not_read_c(kernel):
    w = Workload("beta0", 140, 300, 50, 1.0, 0.0, "uniform", 9)
    A, B, _ = make_inputs(w)
    Cnan = torch.full((w.M * w.LDC,), float("nan"))
    out = H.run_cuda(w, A, B, Cnan, fn=ladder(kernel))
    ref, mag = H.oracle_full(w, A, B, None)
    H.assert_match(w, H.logical(out, w.M, w.N, w.LDC), ref, mag)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_alpha_zero_never_reads_ab(kernel, beta):
    w = Workload("alpha0", 70, 90, 33, 0.0, beta, "int3", 10)
    _, _, C = make_inputs(w)
    nanA = torch.full((w.M * w.LDA,), float("nan"))
    nanB = torch.full((w.K * w.LDB,), float("nan"))
    out = H.run_cuda(w, nanA, nanB, C, fn=ladder(kernel))
    got = H.logical(out, w.M, w.N, w.LDC).astype(np.float64)
    want = beta * C.numpy().astype(np.float64).reshape(w.M, w.N) if beta != 0 else np.zeros((w.M, w.N))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kernel", KERNELS)
def test_k_zero_and_empty(kernel):
    w = Workload("k0", 40, 50, 0, 2.0, 3.0, "int3", 11)
    C = torch.randint(-3, 4, (w.M * w.N,), generator=torch.Generator().manual_seed(3)).float()
    out = H.run_cuda(w, torch.zeros(1), torch.zeros(w.LDB), C, fn=ladder(kernel))
    assert np.array_equal(out[: w.M * w.N].astype(np.float64), 3.0 * C.numpy().astype(np.float64))
    for M, N in ((0, 5), (5, 0)):
        Cd = torch.full((32,), 7.0, device="cuda")
        st = binding.sgemm_ladder(kernel, M, N, 3, 1.0, Cd.data_ptr(), 3, Cd.data_ptr(), max(N, 1),
                                  0.0, Cd.data_ptr(), max(N, 1), None)
        torch.cuda.synchronize()
        assert st == 0 and torch.all(Cd == 7.0)


@pytest.mark.parametrize("kernel", KERNELS)
def test_square4096_sampled(kernel):
    # the pages' measurement size, alpha 0.5 and beta 3
    H.check_sampled(WORKLOADS["square4096"], rows=8, elements=1024, fn=ladder(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
def test_square4096_integer_every_element(kernel):
    # integer inputs: bit-exact on the samples, Freivalds over every element
    H.check_sampled(integer_variant(WORKLOADS["square4096"]), rows=4, elements=1024,
                    fn=ladder(kernel))
