"""CUDA path vs the oracle, element by element, on sizes the oracle finishes
in seconds: several tiles, ragged tails on every dimension, padded leading
dimensions (padding holds NaN), unaligned pointers, every compiled tile
configuration, and the degenerate cases."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import WORKLOADS, Workload, make_inputs

import gpu_helpers as H
from conftest import compiled_config_count

pytestmark = pytest.mark.gpu

CONFIGS = list(range(compiled_config_count()))

SHAPES = [
    (128, 128, 128), (1, 1, 1), (1, 300, 5), (300, 1, 5), (7, 9, 3), (33, 65, 17),
    (257, 129, 100), (300, 520, 77), (129, 257, 1000), (513, 1031, 40), (64, 64, 4097),
    (200, 64, 300), (1000, 40, 129), (2, 700, 2049),
]


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes_all_configs(shape, dist, config):
    M, N, K = shape
    w = Workload("shape", M, N, K, 1.25, -0.5, dist, 5)
    H.check_against_oracle(w, config=config)


@pytest.mark.parametrize("name", ["square128", "square128_int"])
def test_square128(name):
    H.check_against_oracle(WORKLOADS[name])


@pytest.mark.parametrize("config", CONFIGS)
def test_padded_leading_dimensions(config):
    # lda not a multiple of 4 (rows of A are not 16-byte strided), ldb and ldc
    # padded; padding holds NaN and must neither be read nor written
    w = Workload("padded", 301, 203, 777, 1.25, -0.5, "normal", 2, lda=779, ldb=207, ldc=210)
    H.check_against_oracle(w, config=config)
    wi = w.with_(dist="int3")
    H.check_against_oracle(wi, config=config)


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_unaligned_pointers(config, offsets):
    # B off its 16-byte boundary disables TMA; C off it disables 128-bit stores
    w = Workload("unaligned", 190, 260, 150, 0.5, 3.0, "int3", 6)
    H.check_against_oracle(w, offsets=offsets, config=config)
    H.check_against_oracle(w.with_(dist="uniform"), offsets=offsets, config=config)


@pytest.mark.parametrize("config", CONFIGS)
def test_odd_ldb_uses_copy_path(config):
    w = Workload("oddldb", 150, 97, 131, 1.0, 1.0, "int3", 8, ldb=99)
    H.check_against_oracle(w, config=config)


def test_beta_zero_does_not_read_c():
    w = Workload("beta0", 140, 300, 50, 1.0, 0.0, "uniform", 9)
    A, B, _ = make_inputs(w)
    Cnan = torch.full((w.M * w.LDC,), float("nan"))
    out = H.run_cuda(w, A, B, Cnan)
    ref, mag = H.oracle_full(w, A, B, None)
    H.assert_match(w, H.logical(out, w.M, w.N, w.LDC), ref, mag)


@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_alpha_zero_scales_c_without_reading_ab(beta):
    w = Workload("alpha0", 70, 90, 33, 0.0, beta, "int3", 10)
    _, _, C = make_inputs(w)
    nanA = torch.full((w.M * w.LDA,), float("nan"))
    nanB = torch.full((w.K * w.LDB,), float("nan"))
    out = H.run_cuda(w, nanA, nanB, C)
    got = H.logical(out, w.M, w.N, w.LDC).astype(np.float64)
    want = beta * C.numpy().astype(np.float64).reshape(w.M, w.N) if beta != 0 else np.zeros((w.M, w.N))
    assert np.array_equal(got, want)


def test_k_zero_scales_c():
    w = Workload("k0", 40, 50, 0, 2.0, 3.0, "int3", 11)
    A = torch.zeros(0)
    B = torch.zeros(0)
    C = torch.randint(-3, 4, (w.M * w.N,), generator=torch.Generator().manual_seed(3)).float()
    out = H.run_cuda(w, torch.zeros(1), torch.zeros(w.LDB), C)
    assert np.array_equal(out[: w.M * w.N].astype(np.float64), 3.0 * C.numpy().astype(np.float64))


def test_empty_m_or_n_is_a_no_op():
    for M, N in ((0, 5), (5, 0)):
        C = torch.full((32,), 7.0, device="cuda")
        st = binding.sgemm(M, N, 3, 1.0, C.data_ptr(), 3, C.data_ptr(), max(N, 1), 0.0,
                           C.data_ptr(), max(N, 1), None)
        torch.cuda.synchronize()
        assert st == 0 and torch.all(C == 7.0)


def test_repeat_calls_are_bitwise_deterministic():
    # the split-K fix-up adds partials in a fixed order
    w = Workload("det", 512, 512, 8192, 1.0, 0.0, "uniform", 12)
    A, B, C = make_inputs(w)
    first = H.run_cuda(w, A, B, C)
    for _ in range(3):
        again = H.run_cuda(w, A, B, C)
        assert np.array_equal(first, again)


def test_split_schedule_parity():
    # few tiles and a long K: the persistent grid splits every tile along K
    w = Workload("split", 256, 512, 9000, 1.0, 1.0, "int3", 13)
    for cfg in CONFIGS:
        H.check_against_oracle(w, config=cfg)
        H.check_against_oracle(w.with_(dist="uniform"), config=cfg)
    assert "split=" in binding.sgemm_last_config()
