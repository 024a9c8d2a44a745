"""Maximum sizes: one operand of more than 2^31 elements (10.5 GB) at a time,
so every element offset beyond 2^31 has to be computed in 64 bits. The
matrices are counter-based integers in {-3..3} (workloads.hashed_int3),
generated on the device; the oracle regenerates only the sampled rows and
columns on the host and computes that block of C exactly. Rows near the end
(whose offsets exceed 2^31) are always sampled."""
import functools

import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import (hashed_int3_cols, hashed_int3_device,
                                             hashed_int3_rows)

pytestmark = pytest.mark.gpu

ALPHA, BETA = 1.25, -0.5    # integer inputs stay exact: |alpha * acc| < 2^24
SEEDS = (11, 12, 13)        # A, B, C
CASES = {
    "A_huge": (65536, 64, 40000),   # A: 65536 x 40000 = 2.62e9 elements
    "B_huge": (64, 65536, 40000),   # B: 40000 x 65536
    "C_huge": (65536, 40000, 8),    # C: 65536 x 40000
}


def _sample(n, count, seed):
    g = torch.Generator().manual_seed(seed)
    picks = torch.randint(0, n, (count,), generator=g).tolist()
    # the first and the last rows or columns, and a block near the end
    return sorted(set(picks + [0, n - 1, n - 2] + list(range(max(0, n - 70), n, 7))))


def _check(fn, M, N, K):
    sa, sb, sc = SEEDS
    dA = hashed_int3_device(sa, M, K)
    dB = hashed_int3_device(sb, K, N)
    dC = hashed_int3_device(sc, M, N)
    s = torch.cuda.current_stream()
    st = fn(M, N, K, ALPHA, dA.data_ptr(), K, dB.data_ptr(), N, BETA, dC.data_ptr(), N,
            s.cuda_stream)
    assert st == 0, binding.sgemm_status_string(st)
    torch.cuda.synchronize()
    assert binding.sgemm_poll_device_status(s.cuda_stream) == (0, 0)
    rows, cols = _sample(M, 24, M + 1), _sample(N, 24, N + 2)
    got = dC[torch.tensor(rows, device="cuda")][:, torch.tensor(cols, device="cuda")].cpu()
    del dA, dB, dC
    torch.cuda.empty_cache()
    A_sub = hashed_int3_rows(sa, K, rows)
    B_sub = hashed_int3_cols(sb, K, N, cols)
    C_sub = hashed_int3_rows(sc, N, rows)[:, cols].contiguous()
    ref, _ = oracle.sgemm_rows(len(rows), len(cols), K, ALPHA, A_sub.numpy().reshape(-1), K,
                               B_sub.numpy().reshape(-1), len(cols), BETA,
                               C_sub.numpy().reshape(-1), len(cols))
    g = got.numpy().astype(np.float64)
    bad = np.argwhere(g != ref)
    assert bad.size == 0, (f"{bad.shape[0]} of {g.size} sampled elements differ; first at row "
                           f"{rows[bad[0][0]]}, column {cols[bad[0][1]]}")


@pytest.mark.parametrize("case", list(CASES))
def test_sgemm_max_size(case):
    _check(binding.sgemm, *CASES[case])


@pytest.mark.parametrize("case", list(CASES))
def test_3xtf32_max_size(case):
    _check(binding.sgemm_3xtf32, *CASES[case])


@pytest.mark.parametrize("kernel", binding.LADDER_KERNELS)
def test_ladder_max_size(kernel):
    _check(functools.partial(binding.sgemm_ladder, kernel), *CASES["A_huge"])
