"""The FP32 acceptance bound has teeth (no GPU needed).

The parity tests accept a real-input result when every element satisfies
|C - C_ref| <= 1e-5 * (|alpha| sum_k |a_ik b_kj| + |beta| |c_ij|) + 1e-30.
These tests show, on the square-4096 workload's distribution and alpha/beta
(uniform[-1,1], alpha 0.5, beta 3) and its accumulation length K = 4096, that
the bound tells a correct FP32 result from the plausible wrong ones:

  * FP32 sequential accumulation and the 3xTF32 split (Ootomo and Yokota,
    2022: three TF32 products, the residual x residual term dropped) pass
    with a wide margin;
  * a single TF32 product (operands truncated or rounded to 10 mantissa bits,
    as a tensor core without the split computes), a 3xTF32 result missing
    either cross term, BF16-width operands, and one element moved by
    2e-5 of its bound all fail.

Every candidate is computed here in NumPy from its own definition; the
reference is the oracle.
"""
import math

import numpy as np
import pytest

import oracle

REL_TOL, ABS_FLOOR = 1e-5, 1e-30
M = N = 48
K = 4096
ALPHA, BETA = 0.5, 3.0


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(5)
    A = (rng.random((M, K), dtype=np.float32) * 2 - 1).astype(np.float32)
    B = (rng.random((K, N), dtype=np.float32) * 2 - 1).astype(np.float32)
    C = (rng.random((M, N), dtype=np.float32) * 2 - 1).astype(np.float32)
    ref, mag = oracle.sgemm_rows(M, N, K, ALPHA, A.reshape(-1), K, B.reshape(-1), N, BETA,
                                 C.reshape(-1), N)
    return A, B, C, ref, mag


def _mask(x, keep_mask):
    return (x.view(np.uint32) & np.uint32(keep_mask)).view(np.float32)


def _tf32_trunc(x):
    """Sign, exponent and the top 10 mantissa bits (the low 13 cleared)."""
    return _mask(x, 0xFFFFE000)


def _tf32_round(x):
    """Nearest TF32 value, ties away from zero (inputs here are far from overflow)."""
    return ((x.view(np.uint32) + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def _fail_fraction(result, ref, mag):
    ok = oracle.within_tolerance(result, ref, mag, REL_TOL, ABS_FLOOR)
    return 1.0 - float(ok.mean())


def _d(x):
    return x.astype(np.float64)


def test_fp32_sequential_accumulation_passes(case):
    A, B, C, ref, mag = case
    acc = np.zeros((M, N), np.float32)
    for k in range(K):  # one rounding per product and one per addition
        acc = (acc + np.outer(A[:, k], B[k, :])).astype(np.float32)
    res = (np.float32(ALPHA) * acc + np.float32(BETA) * C).astype(np.float64)
    assert _fail_fraction(res, ref, mag) == 0.0
    # with a margin: the worst element uses under a tenth of its bound
    assert np.max(np.abs(res - ref) / mag) < 0.1 * REL_TOL


def test_correctly_rounded_result_passes(case):
    _, _, _, ref, mag = case
    res = ref.astype(np.float32).astype(np.float64)
    assert _fail_fraction(res, ref, mag) == 0.0


def test_three_tf32_products_pass(case):
    A, B, C, ref, mag = case
    Ah, Bh = _tf32_trunc(A), _tf32_trunc(B)
    Al, Bl = _tf32_trunc(A - Ah), _tf32_trunc(B - Bh)
    res = ALPHA * (_d(Ah) @ _d(Bh) + _d(Ah) @ _d(Bl) + _d(Al) @ _d(Bh)) + BETA * _d(C)
    assert _fail_fraction(res, ref, mag) == 0.0
    # the dropped terms are bounded by 3 * 2^-20 of sum |a||b|
    assert np.max(np.abs(res - ref) / mag) < 3 * 2.0 ** -20


@pytest.mark.parametrize("rounding", ["truncate", "nearest"])
def test_single_tf32_product_fails(case, rounding):
    A, B, C, ref, mag = case
    f = _tf32_trunc if rounding == "truncate" else _tf32_round
    res = ALPHA * (_d(f(A)) @ _d(f(B))) + BETA * _d(C)
    assert _fail_fraction(res, ref, mag) > 0.02


@pytest.mark.parametrize("dropped", ["hi*lo", "lo*hi"])
def test_three_tf32_missing_a_cross_term_fails(case, dropped):
    A, B, C, ref, mag = case
    Ah, Bh = _tf32_trunc(A), _tf32_trunc(B)
    Al, Bl = _tf32_trunc(A - Ah), _tf32_trunc(B - Bh)
    terms = _d(Ah) @ _d(Bh) + (_d(Al) @ _d(Bh) if dropped == "hi*lo" else _d(Ah) @ _d(Bl))
    res = ALPHA * terms + BETA * _d(C)
    assert _fail_fraction(res, ref, mag) > 0.05


def test_bf16_width_operands_fail(case):
    A, B, C, ref, mag = case
    res = ALPHA * (_d(_mask(A, 0xFFFF0000)) @ _d(_mask(B, 0xFFFF0000))) + BETA * _d(C)
    assert _fail_fraction(res, ref, mag) > 0.5


def test_one_element_off_by_twice_its_bound_fails(case):
    _, _, _, ref, mag = case
    res = ref.astype(np.float32).astype(np.float64)
    i, j = 17, 29
    res[i, j] = ref[i, j] + 2 * REL_TOL * mag[i, j]
    ok = oracle.within_tolerance(res, ref, mag, REL_TOL, ABS_FLOOR)
    assert not ok[i, j] and int((~ok).sum()) == 1
    # half the bound still passes
    res[i, j] = ref[i, j] + 0.5 * REL_TOL * mag[i, j]
    assert oracle.within_tolerance(res, ref, mag, REL_TOL, ABS_FLOOR).all()


def test_oracle_is_near_exact(case):
    """The oracle against the exact sum: math.fsum of the products (each
    product of two floats is exact in double) is the correctly rounded exact
    value, and the oracle stays within K * 2^-53 of sum |a||b| of it."""
    A, B, C, ref, mag = case
    rng = np.random.default_rng(6)
    for i, j in zip(rng.integers(0, M, 24), rng.integers(0, N, 24)):
        prods = _d(A[i, :]) * _d(B[:, j])
        exact = ALPHA * math.fsum(prods.tolist()) + BETA * float(C[i, j])
        assert abs(ref[i, j] - exact) <= (K + 2) * 2.0 ** -53 * mag[i, j]
