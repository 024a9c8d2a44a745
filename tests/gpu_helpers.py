"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI on seeded inputs and compare with the oracle.

Comparison rules (stated as the acceptance bar of the library):
  * integer-valued inputs whose partial sums stay below 2^24: bit-exact, i.e.
    the FP32 result equals the oracle's exact value;
  * real inputs: |C_gpu - C_ref| <= 1e-5 * (|alpha| sum_k |a_ik b_kj| +
    |beta| |c_ij|) + 1e-30 for every element checked.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload, element_sample, make_inputs, row_sample

REL_TOL = 1e-5
ABS_FLOOR = 1e-30


GUARD = 64  # NaN floats after every device buffer (and before it when offset)


def device_buffer(host_flat: torch.Tensor, offset_floats: int = 0):
    """Copy a flat host buffer to the device, optionally starting
    `offset_floats` floats past a 256-byte aligned allocation (to exercise
    unaligned pointers), with GUARD NaN floats after it. Returns (storage
    tensor, view tensor)."""
    n = host_flat.numel()
    store = torch.empty(n + offset_floats + GUARD, dtype=torch.float32, device="cuda")
    store.fill_(float("nan"))
    view = store[offset_floats: offset_floats + n]
    view.copy_(host_flat)
    return store, view


def assert_guards_intact(store: torch.Tensor, offset_floats: int, n: int, what=""):
    """The NaN floats before and after a buffer's view were not written."""
    host = store.cpu().numpy()
    before, after = host[:offset_floats], host[offset_floats + n:]
    assert np.all(np.isnan(before)) and np.all(np.isnan(after)), f"{what}: a guard band was written"


def run_cuda(w: Workload, A, B, C, offsets=(0, 0, 0), config=None, stream=None, check_status=True,
             fn=None):
    """Run the CUDA path on host inputs (flat float32 tensors with the
    workload's leading dimensions) and return the device result copied back as
    a flat numpy array (M*ldc floats). `fn` is the C-ABI entry point
    (default: sgemm; sgemm_3xtf32 for the tensor-core path)."""
    fn = fn or binding.sgemm
    _, dA = device_buffer(A, offsets[0])
    _, dB = device_buffer(B, offsets[1])
    if C is None:
        C = torch.full((w.M * w.LDC,), float("nan"))
    storeC, dC = device_buffer(C, offsets[2])
    if config is not None:
        assert binding.sgemm_force_config(config) == 0
    try:
        s = stream if stream is not None else torch.cuda.current_stream()
        st = fn(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB,
                w.beta, dC.data_ptr(), w.LDC, s.cuda_stream)
        assert st == 0, f"sgemm returned {st}: {binding.sgemm_status_string(st)}"
        if check_status:
            pst, detail = binding.sgemm_poll_device_status(s.cuda_stream)
            assert pst == 0, f"device status {pst} detail {detail}"
        torch.cuda.synchronize()
    finally:
        if config is not None:
            binding.sgemm_force_config(-1)
    assert_guards_intact(storeC, offsets[2], C.numel(), what=f"{w.name} C")
    return dC.cpu().numpy()


def logical(flat: np.ndarray, rows: int, cols: int, ld: int) -> np.ndarray:
    return flat.reshape(rows, ld)[:, :cols] if rows > 0 else np.zeros((0, cols), flat.dtype)


def oracle_full(w: Workload, A, B, C):
    Cn = None if w.beta == 0 else C.numpy()
    return oracle.sgemm_rows(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB, w.beta,
                             Cn, w.LDC)


def assert_match(w: Workload, gpu2d: np.ndarray, ref: np.ndarray, mag: np.ndarray, what=""):
    """Bit-exact for integer inputs, the FP32 tolerance otherwise."""
    g = gpu2d.astype(np.float64)
    if w.dist == "int3":
        bad = ~(g == ref)
        kind = "bit-exact"
    else:
        bad = ~oracle.within_tolerance(g, ref, mag, REL_TOL, ABS_FLOOR)
        kind = "tolerance"
    if bad.any():
        idx = np.argwhere(bad)
        i, j = idx[0]
        raise AssertionError(
            f"{w.name} {what}: {int(bad.sum())} of {bad.size} elements fail the {kind} check; "
            f"first at ({i},{j}): gpu={g[i, j]!r} ref={ref[i, j]!r} mag={mag[i, j]!r}")


def check_against_oracle(w: Workload, offsets=(0, 0, 0), config=None, pad=float("nan"), fn=None):
    """Whole-result comparison (sizes the oracle finishes in seconds)."""
    A, B, C = make_inputs(w, pad_value=pad)
    out = run_cuda(w, A, B, C, offsets=offsets, config=config, fn=fn)
    ref, mag = oracle_full(w, A, B, C)
    gpu = logical(out, w.M, w.N, w.LDC)
    assert_match(w, gpu, ref, mag, what=f"config={config} offsets={offsets}")
    # padding columns of C are never written
    if w.LDC > w.N and w.M > 0:
        pad_out = out.reshape(w.M, w.LDC)[:, w.N:]
        pad_in = C.numpy().reshape(w.M, w.LDC)[:, w.N:]
        assert np.array_equal(pad_out, pad_in, equal_nan=True), "C padding was written"
    return gpu


def check_sampled(w: Workload, rows=32, elements=2048, config=None, fn=None):
    """Large sizes: oracle on sampled full rows and random elements; for
    integer inputs also a Freivalds check of every element,
    C x == alpha A (B x) + beta C_in x, exact in float64."""
    A, B, C = make_inputs(w)
    out = run_cuda(w, A, B, C, config=config, fn=fn)
    gpu = logical(out, w.M, w.N, w.LDC)
    Cn = None if w.beta == 0 else C.numpy()
    r = row_sample(w.M, rows, w.seed)
    for i in r:
        ref, mag = oracle.sgemm_rows(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB,
                                     w.beta, Cn, w.LDC, i, i + 1)
        assert_match(w, gpu[i: i + 1], ref, mag, what=f"row {i}")
    er, ec = element_sample(w.M, w.N, elements, w.seed)
    ref, mag = oracle.sgemm_elements(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB,
                                     w.beta, Cn, w.LDC, er, ec)
    assert_match(w, gpu[er, ec][None, :], ref[None, :], mag[None, :], what="elements")
    if w.dist == "int3":
        freivalds(w, A, B, C, gpu)
    return gpu


def freivalds(w: Workload, A, B, C, gpu, trials=2):
    """Every element participates: for random x in {-1, 0, 1}^N, the exact
    products of the integer inputs give C x exactly (all magnitudes < 2^53)."""
    gen = np.random.default_rng(7 + w.seed)
    Am = logical(A.numpy(), w.M, w.K, w.LDA)
    Bm = logical(B.numpy(), w.K, w.N, w.LDB)
    Cm = logical(C.numpy(), w.M, w.N, w.LDC) if w.beta != 0 else None
    for _ in range(trials):
        x = gen.integers(-1, 2, size=w.N).astype(np.float64)
        bx = Bm.astype(np.float64) @ x if w.K * w.N <= (1 << 26) else _chunked_matvec(Bm, x)
        abx = _chunked_matvec(Am, bx)
        want = w.alpha * abx
        if Cm is not None:
            want = want + w.beta * _chunked_matvec(Cm, x)
        got = _chunked_matvec(gpu, x)
        assert np.array_equal(got, want), f"{w.name}: Freivalds check failed"


def _chunked_matvec(M2, x, chunk=2048):
    out = np.empty(M2.shape[0], dtype=np.float64)
    for r0 in range(0, M2.shape[0], chunk):
        out[r0: r0 + chunk] = M2[r0: r0 + chunk].astype(np.float64) @ x
    return out
