"""Pins that tie the CPU oracle to facts other than its own formula.

Each pin takes an oracle library handle (so the same pins can be run against
deliberately broken copies of the oracle) and returns a list of failure
messages; an empty list means the pin holds. The facts used:

  * special cases that reduce to something simpler: identity and permutation
    matrices, rank-1 operands, unit-basis matrices (GEMM is bilinear, so the
    4x4x4 unit-basis enumeration fixes the whole map at that size);
  * exhaustive enumeration of all 2x2 operands over {-1, 0, 1};
  * library routines on inputs where they are exact or where their error is
    bounded: numpy int64 matmul on integer data (exact), numpy float64 matmul
    on real data (within K * 2^-52 of the magnitude);
  * an independent outer-product formulation in Python integers;
  * structural facts: padding beyond the leading dimension is never read, C is
    not read when beta == 0, A and B are not read when alpha == 0, row ranges
    and element queries agree with the full result, and the magnitude term is
    sum |a||b| (checked where it has a closed form).
"""
from __future__ import annotations

import itertools

import numpy as np

import oracle

ALPHA_BETA = [(1.0, 0.0), (0.5, 3.0), (1.25, -0.5), (2.0, -1.0), (1.0, 1.0)]


def _run(lib, A2, B2, C2, alpha, beta, lda=None, ldb=None, ldc=None, pad=np.nan):
    """Call the oracle on 2-D operands, optionally embedding them in buffers
    with larger leading dimensions whose padding holds ``pad``."""
    M, K = A2.shape
    N = B2.shape[1]
    lda = lda or max(K, 1)
    ldb = ldb or max(N, 1)
    ldc = ldc or max(N, 1)

    def embed(x, ld):
        buf = np.full((x.shape[0], ld), pad, dtype=np.float32)
        buf[:, : x.shape[1]] = x
        return buf.reshape(-1)

    A = embed(np.asarray(A2, np.float32), lda)
    B = embed(np.asarray(B2, np.float32), ldb)
    C = None if C2 is None else embed(np.asarray(C2, np.float32), ldc)
    return oracle.sgemm_rows(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, library=lib, threads=1)


def _ints(rng, shape, lo=-3, hi=3):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


def pin_identity(lib):
    fails = []
    rng = np.random.default_rng(11)
    for n, m in ((5, 5), (7, 3), (1, 4)):
        B = _ints(rng, (n, m))
        C = _ints(rng, (n, m))
        for a, b in ALPHA_BETA:
            ref, _ = _run(lib, np.eye(n, dtype=np.float32), B, C, a, b)
            want = a * B.astype(np.float64) + (b * C.astype(np.float64) if b != 0 else 0.0)
            if not np.array_equal(ref, want):
                fails.append(f"identity n={n} m={m} alpha={a} beta={b}")
    return fails


def pin_permutation(lib):
    fails = []
    rng = np.random.default_rng(12)
    # A selects rows of B: A[i, sigma(i)] = 1  ->  (A B)[i, :] = B[sigma(i), :]
    M, K, N = 6, 9, 5
    sigma = rng.permutation(K)[:M]
    A = np.zeros((M, K), np.float32)
    A[np.arange(M), sigma] = 1
    B = _ints(rng, (K, N))
    ref, _ = _run(lib, A, B, None, 1.0, 0.0)
    if not np.array_equal(ref, B[sigma].astype(np.float64)):
        fails.append("row-selection permutation")
    # B selects columns of A: B[tau(j), j] = 1  ->  (A B)[:, j] = A[:, tau(j)]
    M, K, N = 4, 7, 7
    tau = rng.permutation(K)[:N]
    Bq = np.zeros((K, N), np.float32)
    Bq[tau, np.arange(N)] = 1
    A2 = _ints(rng, (M, K))
    ref, _ = _run(lib, A2, Bq, None, 1.0, 0.0)
    if not np.array_equal(ref, A2[:, tau].astype(np.float64)):
        fails.append("column-selection permutation")
    return fails


def pin_rank_one(lib):
    fails = []
    rng = np.random.default_rng(13)
    M, K, N = 5, 11, 6
    u = _ints(rng, (M,))
    v = _ints(rng, (N,))
    C = _ints(rng, (M, N))
    A = np.outer(u, np.ones(K)).astype(np.float32)      # A = u 1^T
    B = np.outer(np.ones(K), v).astype(np.float32)      # B = 1 v^T
    for a, b in ALPHA_BETA:
        ref, _ = _run(lib, A, B, C, a, b)
        want = a * K * np.outer(u, v).astype(np.float64) + (b * C if b != 0 else 0.0)
        if not np.array_equal(ref, want):
            fails.append(f"rank-1 u1^T 1v^T alpha={a} beta={b}")
    # A = u e_k^T, B = e_k' v^T: alpha * [k == k'] * u v^T + beta C
    for k, kp in ((2, 2), (3, 7), (10, 10), (0, 10)):
        A = np.zeros((M, K), np.float32)
        A[:, k] = u
        B = np.zeros((K, N), np.float32)
        B[kp, :] = v
        ref, _ = _run(lib, A, B, C, 1.25, -0.5)
        want = (1.25 * np.outer(u, v) if k == kp else 0.0) + (-0.5) * C.astype(np.float64)
        if not np.array_equal(ref, want):
            fails.append(f"rank-1 unit columns k={k} k'={kp}")
    return fails


def pin_unit_basis_4x4x4(lib):
    """Bilinearity: results on all pairs of unit-basis matrices fix the map."""
    fails = []
    n = 4
    rng = np.random.default_rng(14)
    C = _ints(rng, (n, n))
    for a, b in ((1.0, 0.0), (2.0, -1.0), (0.5, 3.0)):
        for i, k, kp, j in itertools.product(range(n), repeat=4):
            A = np.zeros((n, n), np.float32)
            A[i, k] = 1
            B = np.zeros((n, n), np.float32)
            B[kp, j] = 1
            ref, _ = _run(lib, A, B, C, a, b)
            want = (b * C.astype(np.float64)) if b != 0 else np.zeros((n, n))
            if k == kp:
                want[i, j] += a
            if not np.array_equal(ref, want):
                fails.append(f"unit basis E{i}{k} E{kp}{j} alpha={a} beta={b}")
                return fails
    return fails


def pin_exhaustive_2x2(lib):
    """All 3^4 x 3^4 pairs of 2x2 operands over {-1,0,1} against the expanded
    entries c_ij = a_i0 b_0j + a_i1 b_1j."""
    fails = []
    vals = (-1.0, 0.0, 1.0)
    mats = [np.array(t, np.float32).reshape(2, 2) for t in itertools.product(vals, repeat=4)]
    C = np.array([[2.0, -3.0], [1.0, 0.5]], np.float32)
    for A in mats:
        for B in mats:
            ref, _ = _run(lib, A, B, C, 2.0, -1.0)
            a00, a01, a10, a11 = (float(x) for x in A.reshape(-1))
            b00, b01, b10, b11 = (float(x) for x in B.reshape(-1))
            want = np.array([[a00 * b00 + a01 * b10, a00 * b01 + a01 * b11],
                             [a10 * b00 + a11 * b10, a10 * b01 + a11 * b11]])
            want = 2.0 * want - C.astype(np.float64)
            if not np.array_equal(ref, want):
                fails.append(f"exhaustive 2x2 A={A.tolist()} B={B.tolist()}")
                return fails
    return fails


def pin_integer_exact_vs_int64(lib):
    """Integer inputs: exact agreement with numpy's int64 matmul."""
    fails = []
    rng = np.random.default_rng(15)
    for (M, K, N) in ((37, 1000, 29), (3, 4096, 2), (64, 64, 64), (1, 1, 1)):
        A = _ints(rng, (M, K))
        B = _ints(rng, (K, N))
        C = _ints(rng, (M, N))
        exact = A.astype(np.int64) @ B.astype(np.int64)
        for a, b in ((1.0, 0.0), (0.5, 3.0), (1.25, -0.5)):
            ref, _ = _run(lib, A, B, C, a, b)
            want = a * exact.astype(np.float64) + (b * C.astype(np.float64) if b != 0 else 0.0)
            if not np.array_equal(ref, want):
                fails.append(f"int64 exact M={M} K={K} N={N} alpha={a} beta={b}")
    return fails


def pin_outer_product_form(lib):
    """C = sum_k outer(A[:, k], B[k, :]) in Python integers (a different
    formulation: a sum of rank-1 terms rather than row-by-column dots)."""
    fails = []
    rng = np.random.default_rng(16)
    M, K, N = 5, 8, 7
    A = _ints(rng, (M, K))
    B = _ints(rng, (K, N))
    acc = [[0] * N for _ in range(M)]
    for k in range(K):
        col = [int(A[i, k]) for i in range(M)]
        row = [int(B[k, j]) for j in range(N)]
        for i in range(M):
            for j in range(N):
                acc[i][j] += col[i] * row[j]
    ref, _ = _run(lib, A, B, None, 1.0, 0.0)
    if not np.array_equal(ref, np.array(acc, dtype=np.float64)):
        fails.append("outer-product formulation")
    return fails


def pin_real_vs_float64_matmul(lib):
    """Real inputs: agreement with numpy float64 matmul within the double
    rounding bound K * 2^-52 * sum|a||b| (both sides are near-exact)."""
    fails = []
    rng = np.random.default_rng(17)
    for (M, K, N) in ((33, 300, 41), (8, 2000, 5)):
        A = (rng.random((M, K), dtype=np.float32) * 2 - 1).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        C = rng.standard_normal((M, N)).astype(np.float32)
        ref, mag = _run(lib, A, B, C, 1.25, -0.5)
        want = 1.25 * (A.astype(np.float64) @ B.astype(np.float64)) - 0.5 * C.astype(np.float64)
        bound = (K + 4) * 2.0 ** -52 * mag + 1e-300
        if not np.all(np.abs(ref - want) <= bound):
            fails.append(f"float64 matmul agreement M={M} K={K} N={N}")
        absmag = 1.25 * (np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))) \
            + 0.5 * np.abs(C.astype(np.float64))
        if not np.all(np.abs(mag - absmag) <= (K + 4) * 2.0 ** -52 * absmag):
            fails.append(f"magnitude vs |A||B| matmul M={M} K={K} N={N}")
    return fails


def pin_magnitude_closed_form(lib):
    """Signs do not enter the magnitude: random +-1 operands give K exactly."""
    fails = []
    rng = np.random.default_rng(18)
    M, K, N = 4, 13, 3
    A = rng.choice([-1.0, 1.0], size=(M, K)).astype(np.float32)
    B = rng.choice([-1.0, 1.0], size=(K, N)).astype(np.float32)
    C = rng.choice([-2.0, 2.0], size=(M, N)).astype(np.float32)
    _, mag = _run(lib, A, B, C, -0.5, -3.0)
    if not np.array_equal(mag, np.full((M, N), 0.5 * K + 3.0 * 2.0)):
        fails.append("magnitude closed form")
    return fails


def pin_leading_dimensions(lib):
    """Padded leading dimensions (padding holds NaN) give the same result as
    the natural ones, and no NaN."""
    fails = []
    rng = np.random.default_rng(19)
    M, K, N = 9, 7, 5
    A = _ints(rng, (M, K))
    B = _ints(rng, (K, N))
    C = _ints(rng, (M, N))
    base, _ = _run(lib, A, B, C, 1.25, -0.5)
    for lda, ldb, ldc in ((K + 3, N, N), (K, N + 5, N), (K, N, N + 2), (K + 1, N + 2, N + 7)):
        ref, _ = _run(lib, A, B, C, 1.25, -0.5, lda=lda, ldb=ldb, ldc=ldc)
        if not np.array_equal(ref, base):
            fails.append(f"leading dimensions lda={lda} ldb={ldb} ldc={ldc}")
    return fails


def pin_beta_zero_and_alpha_zero(lib):
    fails = []
    rng = np.random.default_rng(20)
    M, K, N = 4, 6, 3
    A = _ints(rng, (M, K))
    B = _ints(rng, (K, N))
    Cnan = np.full((M, N), np.nan, np.float32)
    ref, mag = _run(lib, A, B, Cnan, 1.0, 0.0)
    if not (np.all(np.isfinite(ref)) and np.all(np.isfinite(mag))):
        fails.append("beta == 0 read C")
    C = _ints(rng, (M, N))
    ref, _ = _run(lib, np.full((M, K), np.nan, np.float32), np.full((K, N), np.nan, np.float32),
                  C, 0.0, -0.5)
    if not np.array_equal(ref, -0.5 * C.astype(np.float64)):
        fails.append("alpha == 0 read A or B")
    ref, _ = _run(lib, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), C, 2.0, 3.0)
    if not np.array_equal(ref, 3.0 * C.astype(np.float64)):
        fails.append("K == 0")
    return fails


def pin_rows_and_elements(lib):
    fails = []
    rng = np.random.default_rng(21)
    M, K, N = 23, 17, 19
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    C = rng.standard_normal((M, N)).astype(np.float32)
    full, fmag = _run(lib, A, B, C, 1.25, -0.5)
    Af, Bf, Cf = A.reshape(-1), B.reshape(-1), C.reshape(-1)
    part, pmag = oracle.sgemm_rows(M, N, K, 1.25, Af, K, Bf, N, -0.5, Cf, N, 5, 14,
                                   library=lib, threads=3)
    if not (np.array_equal(part, full[5:14]) and np.array_equal(pmag, fmag[5:14])):
        fails.append("row range")
    rows = rng.integers(0, M, 50)
    cols = rng.integers(0, N, 50)
    ev, em = oracle.sgemm_elements(M, N, K, 1.25, Af, K, Bf, N, -0.5, Cf, N, rows, cols,
                                   library=lib)
    if not (np.array_equal(ev, full[rows, cols]) and np.array_equal(em, fmag[rows, cols])):
        fails.append("element query")
    return fails


ALL_PINS = [
    pin_identity, pin_permutation, pin_rank_one, pin_unit_basis_4x4x4, pin_exhaustive_2x2,
    pin_integer_exact_vs_int64, pin_outer_product_form, pin_real_vs_float64_matmul,
    pin_magnitude_closed_form, pin_leading_dimensions, pin_beta_zero_and_alpha_zero,
    pin_rows_and_elements,
]


def run_all(lib):
    """All pin failures for an oracle library (empty when every pin holds).
    A pin that raises counts as failed."""
    fails = []
    for pin in ALL_PINS:
        try:
            fails.extend(pin(lib))
        except Exception as e:  # a broken oracle may reject its own output shape
            fails.append(f"{pin.__name__} raised {type(e).__name__}: {e}")
    return fails
