"""The opt-in tensor-core path (sgemm_3xtf32) against the oracle: the same
bar as the FFMA path -- bit-exact on integer inputs, the FP32 tolerance
|C - C_ref| <= 1e-5 * (|alpha| sum |a||b| + |beta| |c|) + 1e-30 on real inputs --
on small shapes element by element and on the full workloads by sampling.
Every test runs in both kernel forms: CTA pairs with two-SM MMAs (the
default) and single CTAs."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import SWEEP_SIZES, WORKLOADS, Workload, integer_variant, make_inputs

import gpu_helpers as H

pytestmark = pytest.mark.gpu
X3 = binding.sgemm_3xtf32


FORM_TEXT = {binding.SGEMM_X3_PAIR: "cluster=2 pair=2sm",
             binding.SGEMM_X3_SINGLE: "cluster=1 "}


@pytest.fixture(autouse=True, params=binding.X3_FORMS, ids=["pair2sm", "single"])
def kernel_form(request):
    prev = binding.sgemm_3xtf32_set_kernel_form(request.param)
    yield request.param
    binding.sgemm_3xtf32_set_kernel_form(prev)


def test_kernel_form_is_reported(kernel_form):
    # two waves of whole tile pairs: the pair forms run when selected
    w = Workload("x3form", 128 * 2 * 76 * 2, 256, 64, 1.0, 0.0, "int3", 36)
    H.check_sampled(w, rows=64, elements=4096, fn=X3)
    assert FORM_TEXT[kernel_form] in binding.sgemm_last_config()
    # every tile split along K: single CTAs either way
    H.check_against_oracle(Workload("x3split", 300, 520, 4000, 1.0, 0.0, "int3", 37), fn=X3)
    assert "cluster=1 " in binding.sgemm_last_config()

SHAPES = [(128, 256, 32), (1, 1, 1), (7, 9, 3), (33, 65, 17), (257, 129, 100), (300, 520, 77),
          (129, 257, 1000), (513, 1031, 40), (64, 64, 4097), (2, 700, 2049), (1000, 40, 129)]


@pytest.mark.parametrize("dist", ["int3", "uniform", "normal"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes(shape, dist):
    M, N, K = shape
    H.check_against_oracle(Workload("x3", M, N, K, 1.25, -0.5, dist, 31), fn=X3)


@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_unaligned_and_padded(offsets):
    w = Workload("x3pad", 301, 203, 777, 1.25, -0.5, "normal", 32, lda=779, ldb=207, ldc=210)
    H.check_against_oracle(w, offsets=offsets, fn=X3)
    H.check_against_oracle(w.with_(dist="int3"), offsets=offsets, fn=X3)


def test_beta_zero_does_not_read_c():
    w = Workload("x3beta0", 140, 300, 50, 1.0, 0.0, "uniform", 33)
    A, B, _ = make_inputs(w)
    out = H.run_cuda(w, A, B, torch.full((w.M * w.LDC,), float("nan")), fn=X3)
    ref, mag = H.oracle_full(w, A, B, None)
    H.assert_match(w, H.logical(out, w.M, w.N, w.LDC), ref, mag)


def test_alpha_zero_scales_c():
    w = Workload("x3alpha0", 70, 90, 33, 0.0, -0.5, "int3", 34)
    _, _, C = make_inputs(w)
    out = H.run_cuda(w, torch.full((w.M * w.LDA,), float("nan")),
                     torch.full((w.K * w.LDB,), float("nan")), C, fn=X3)
    assert np.array_equal(H.logical(out, w.M, w.N, w.LDC).astype(np.float64),
                          -0.5 * C.numpy().astype(np.float64).reshape(w.M, w.N))


def test_repeat_calls_are_bitwise_deterministic():
    w = Workload("x3det", 300, 700, 3000, 1.0, 0.0, "uniform", 35)
    A, B, C = make_inputs(w)
    first = H.run_cuda(w, A, B, C, fn=X3)
    assert np.array_equal(first, H.run_cuda(w, A, B, C, fn=X3))


NAMED = ["square4096", "edges8191x1000x777", "kdominant1024x1024x16384", "skinny16384x64x4096"]


@pytest.mark.parametrize("name", NAMED)
def test_named_real(name):
    H.check_sampled(WORKLOADS[name], rows=8, elements=1024, fn=X3)


@pytest.mark.parametrize("name", NAMED)
def test_named_integer_bit_exact(name):
    H.check_sampled(integer_variant(WORKLOADS[name]), rows=4, elements=512, fn=X3)


@pytest.mark.parametrize("n", [s for s in SWEEP_SIZES if s <= 8192])
def test_sweep_integer_bit_exact(n):
    H.check_sampled(WORKLOADS[f"sweep{n}_int"], rows=4, elements=512, fn=X3)


@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape, width", [((6000, 100, 1100), 128), ((3000, 300, 777), 128),
                                          ((4100, 127, 2049), 128), ((5000, 1000, 200), 128),
                                          ((3000, 64, 1100), 64), ((700, 33, 3000), 64)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_narrow_tiles_ragged_and_misaligned(shape, width, dist):
    # the 64- and 128-wide tiles (A's parts in tensor memory) on a ragged last
    # tile row, tile column and k-slice; K-split tiles everywhere, and whole
    # tiles too at 5000 x 1000 x 200 (two waves of 128-wide tiles). First with
    # every pointer off 16 bytes and padded leading dimensions (A then copied,
    # C by scalar accesses) and beta = 0, then aligned with beta != 0
    M, N, K = shape
    for beta, offsets, pads in ((0.0, (1, 2, 3), (1, 2, 3)), (-0.5, (0, 0, 0), (4, 0, 4))):
        w = Workload("x3narrow", M, N, K, 1.25, beta, dist, 43, lda=K + pads[0], ldb=N + pads[1],
                     ldc=N + pads[2])
        H.check_against_oracle(w, offsets=offsets, fn=X3)
        assert f"3xtf32_tcgen05_128x{width}x32" in binding.sgemm_last_config(), (shape, beta)


def test_slice_width_follows_k(kernel_form):
    # single CTAs with 256-wide tiles (40 x 6 of them, more than 48 slices of
    # 32 per CTA; 120 tile pairs, fewer than two waves of the 76 clusters, so
    # the pair form falls back): BK = 32 (two stages) below K = 1024, BK = 16
    # (four stages) from there
    H.check_sampled(Workload("x3k", 5000, 1300, 1023, 1.0, 0.5, "int3", 38), rows=8, elements=1024,
                    fn=X3)
    assert "128x256x32_s2" in binding.sgemm_last_config()
    H.check_sampled(Workload("x3k", 5000, 1300, 1024, 1.0, 0.5, "int3", 38), rows=8, elements=1024,
                    fn=X3)
    assert "128x256x16_s4" in binding.sgemm_last_config()
    # little 256-wide work: 128-wide tiles, BK = 32 at any K (four stages:
    # A's parts sit in tensor memory); few 128-wide tiles: 64-wide tiles, six
    # stages
    for K in (1023, 1024):
        H.check_sampled(Workload("x3k", 2000, 300, K, 1.0, 0.5, "int3", 38), rows=16, elements=2048,
                        fn=X3)
        assert "128x128x32_s4" in binding.sgemm_last_config()
        H.check_against_oracle(Workload("x3k", 200, 300, K, 1.0, 0.5, "int3", 38), fn=X3)
        assert "128x64x32_s6" in binding.sgemm_last_config()
    # whole waves of tile pairs at K = 1024: the two-SM form keeps BK = 32
    # (three stages of half B tiles), single CTAs take BK = 16
    H.check_sampled(Workload("x3k2", 128 * 2 * 76 * 2, 256, 1024, 1.0, 0.5, "int3", 39),
                    rows=32, elements=2048, fn=X3)
    want = {binding.SGEMM_X3_PAIR: "128x256x32_s3", binding.SGEMM_X3_SINGLE: "128x256x16_s4"}[kernel_form]
    assert want in binding.sgemm_last_config()


@pytest.mark.parametrize("dist", ["int3", "uniform"])
def test_pair_size_with_ragged_edges(dist, kernel_form):
    # 305 tile rows (the last pair's odd CTA lies below M), a ragged second tile
    # column and a ragged last k-slice, with whole waves of tile pairs, so the
    # pair forms run: Freivalds over every element (integer inputs), sampled
    # rows, and the last 90 rows (the ragged last tile row) against the oracle
    w = Workload("x3pairedge", 128 * 304 + 88, 300, 1100, 1.25, -0.5, dist, 41)
    A, B, C = make_inputs(w)
    out = H.run_cuda(w, A, B, C, fn=X3)
    assert FORM_TEXT[kernel_form] in binding.sgemm_last_config()
    gpu = H.logical(out, w.M, w.N, w.LDC)
    lo = w.M - 90
    ref, mag = oracle.sgemm_rows(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB, w.beta,
                                 C.numpy(), w.LDC, lo, w.M)
    H.assert_match(w, gpu[lo:], ref, mag, what="last rows")
    H.check_sampled(w, rows=32, elements=2048, fn=X3)
