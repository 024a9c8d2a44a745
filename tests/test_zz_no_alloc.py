"""sgemm_noalloc: the entry point for callers that cannot allocate device
memory (graph capture, a memory pool that owns the device, latency-bound
loops). It must give the same results as sgemm() while allocating nothing.

Collected last on purpose (the file name sorts after every other test file),
so a run that stops at the first failure has already run everything else.
Passes alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import WORKLOADS, Workload, make_inputs, row_sample

import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _call(fn, w, dA, dB, C_host):
    dC = C_host.to("cuda")
    st = fn(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB, w.beta,
            dC.data_ptr(), w.LDC, torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.sgemm_status_string(st)
    torch.cuda.synchronize()
    return dC.cpu().numpy().reshape(w.M, w.LDC)[:, : w.N]


def _within(w, got, want, mag):
    ok = oracle.within_tolerance(got, want.astype(np.float64), mag, H.REL_TOL, H.ABS_FLOOR)
    return bool(ok.all())


# few tiles and a long K: every tile is split, so the partial-tile scratch is used
SPLIT = Workload("noalloc_split", 256, 512, 8192, 1.25, -0.5, "uniform", 21)
RAGGED = Workload("noalloc_ragged", 301, 203, 777, 1.25, -0.5, "normal", 22, lda=779, ldb=207, ldc=210)


@pytest.mark.parametrize("w", [SPLIT, RAGGED, WORKLOADS["square4096"], WORKLOADS["skinny16384x64x4096"]],
                         ids=lambda w: w.name)
def test_noalloc_matches_sgemm_twice(w):
    A, B, C = make_inputs(w)
    dA, dB = A.to("cuda"), B.to("cuda")
    ref = _call(binding.sgemm, w, dA, dB, C)          # existing entry point
    Cn = None if w.beta == 0 else C.numpy()
    if w.M * w.N * w.K <= (1 << 31):
        rows = list(range(w.M))
    else:
        rows = row_sample(w.M, 6, w.seed)
    mags = {}
    for i in rows:
        _, mag = oracle.sgemm_rows(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB,
                                   w.beta, Cn, w.LDC, i, i + 1)
        mags[i] = mag
    for _ in range(2):                                 # two calls in a row
        got = _call(binding.sgemm_noalloc, w, dA, dB, C)
        for i in rows:
            assert _within(w, got[i: i + 1], ref[i: i + 1], mags[i]), f"row {i}"
        # same kernel, same schedule: the whole result agrees with sgemm()
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_noalloc_follows_the_staged_a_switch(mode):
    # the same A load mode as sgemm() under every setting of sgemm_set_staged_a
    # (SPLIT: row-major, TMA-aligned, every tile split; SKINNY: 64 k-slices per CTA)
    prev = binding.sgemm_set_staged_a(mode)
    try:
        for w in (SPLIT, Workload("noalloc_skinny", 4096, 64, 4096, 1.0, 1.0, "uniform", 23)):
            A, B, C = make_inputs(w)
            dA, dB = A.to("cuda"), B.to("cuda")
            ref = _call(binding.sgemm, w, dA, dB, C)
            assert np.array_equal(_call(binding.sgemm_noalloc, w, dA, dB, C), ref), (mode, w.name)
    finally:
        binding.sgemm_set_staged_a(prev)


def test_noalloc_allocates_nothing():
    w = SPLIT
    A, B, C = make_inputs(w)
    dA, dB, dC = A.to("cuda"), B.to("cuda"), C.to("cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB, w.beta,
            dC.data_ptr(), w.LDC, s)
    assert binding.sgemm_noalloc(*args) == 0          # first call: per-device set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert binding.sgemm_noalloc(*args) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_argument_errors():
    C = torch.full((64,), 5.0, device="cuda")
    p = C.data_ptr()
    assert binding.sgemm_noalloc(-1, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 4, None) == binding.SGEMM_ERR_INVALID_DIM
    assert binding.sgemm_noalloc(4, 4, 4, 1.0, p, 3, p, 4, 0.0, p, 4, None) == binding.SGEMM_ERR_INVALID_LD
    assert binding.sgemm_noalloc(4, 4, 4, 1.0, p, 4, p, 4, 0.0, 0, 4, None) == binding.SGEMM_ERR_NULL_PTR
    # more C tiles than the 32-bit schedule numbers: refused on the host, as by
    # sgemm() (no operand is touched; the sizes only have to be consistent)
    big = 2**31 - 1
    assert binding.sgemm_noalloc(big, big, 1, 1.0, p, 1, p, big, 0.0, p, big, None) == binding.SGEMM_ERR_INVALID_DIM
    assert binding.sgemm(big, big, 1, 1.0, p, 1, p, big, 0.0, p, big, None) == binding.SGEMM_ERR_INVALID_DIM
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)


def test_noalloc_honours_the_wait_limit_and_reports_status():
    # a short (20 ms) limit on every wait still lets a split-K problem finish
    # normally, twice in a row, with the same bits as sgemm(); the status the
    # calls left in the fixed array reads clean
    w = SPLIT
    A, B, C = make_inputs(w)
    dA, dB = A.to("cuda"), B.to("cuda")
    ref = _call(binding.sgemm, w, dA, dB, C)
    s = torch.cuda.current_stream().cuda_stream
    prev = binding.sgemm_set_wait_timeout_ns(20_000_000)
    try:
        for _ in range(2):
            assert np.array_equal(_call(binding.sgemm_noalloc, w, dA, dB, C), ref)
        assert binding.sgemm_noalloc_poll_status(s) == (0, 0)
    finally:
        binding.sgemm_set_wait_timeout_ns(prev)
