"""CPU oracle for C = alpha*A*B + beta*C on row-major FP32 matrices.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package. The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two sides share no code.

The arithmetic lives in ``oracle_sgemm.c`` (plain C, FP64 triple loop, the
plain definition of the operation used by every kernel listing on the pages:
"Shared Memory Tiling", "Vectorized Memory Access: 128-bit Loads and Stores"
and "Warp Tiling: A Third Level of Tiling", each in its epilogue
``alpha * acc + beta * C``). This module only compiles that file, marshals
numpy arrays into it and splits rows across host threads (the sum for each
element is computed by one thread, in ascending k, so threading never changes
a result).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_sgemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_sgemm.so")

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source into a shared library (gcc -O2, IEEE double,
    no fast-math so that every double operation rounds as written)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle shared library and declare its two entry points."""
    lib = ctypes.CDLL(path)
    L, F, P = ctypes.c_long, ctypes.c_float, ctypes.c_void_p
    lib.oracle_sgemm_rows.restype = ctypes.c_int
    lib.oracle_sgemm_rows.argtypes = [L, L, L, F, P, L, P, L, F, P, L, L, L, P, P, L]
    lib.oracle_sgemm_elements.restype = ctypes.c_int
    lib.oracle_sgemm_elements.argtypes = [L, L, L, F, P, L, P, L, F, P, L, L, P, P, P, P]
    return lib


def lib() -> ctypes.CDLL:
    """The oracle library, compiled on first use if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                compile_library()
            _lib = load_library(_LIB_PATH)
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check_operand(x, name):
    if x.dtype != np.float32:
        raise TypeError(f"{name} must be float32, got {x.dtype}")
    if x.ndim != 1:
        raise ValueError(f"{name} must be passed as a flat buffer with an explicit leading dimension")
    if not x.flags["C_CONTIGUOUS"]:
        raise ValueError(f"{name} must be contiguous")


def sgemm_rows(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, row_begin=0, row_end=None,
               threads=None, library=None):
    """Reference rows [row_begin, row_end) of alpha*A*B + beta*C.

    A, B, C are flat float32 buffers holding row-major matrices with leading
    dimensions lda, ldb, ldc (C may be None when beta == 0: it is not read).
    Returns (ref, mag), both float64 arrays of shape (row_end-row_begin, N):
    the reference value and |alpha|*sum_k|a||b| + |beta||c|.
    """
    lib_ = library if library is not None else lib()
    row_end = M if row_end is None else row_end
    for x, nm in ((A, "A"), (B, "B")):
        _check_operand(x, nm)
    if C is not None:
        _check_operand(C, "C")
    rows = row_end - row_begin
    ref = np.empty((max(rows, 0), N), dtype=np.float64)
    mag = np.empty((max(rows, 0), N), dtype=np.float64)
    if rows <= 0 or N == 0:
        return ref, mag
    Cp = _ptr(C) if C is not None else None
    nthreads = threads if threads is not None else min(os.cpu_count() or 1, 16)
    nthreads = max(1, min(nthreads, rows))
    bounds = [row_begin + (rows * t) // nthreads for t in range(nthreads + 1)]

    def work(t):
        r0, r1 = bounds[t], bounds[t + 1]
        if r1 <= r0:
            return 0
        off = (r0 - row_begin) * N
        rp = ctypes.c_void_p(ref.ctypes.data + off * 8)
        mp = ctypes.c_void_p(mag.ctypes.data + off * 8)
        return lib_.oracle_sgemm_rows(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, Cp, ldc,
                                      r0, r1, rp, mp, N)

    if nthreads == 1:
        codes = [work(0)]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            codes = list(ex.map(work, range(nthreads)))
    if any(c != 0 for c in codes):
        raise ValueError("oracle_sgemm_rows rejected its arguments")
    return ref, mag


def sgemm_elements(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, rows, cols, library=None):
    """Reference values and magnitudes for the elements (rows[t], cols[t])."""
    lib_ = library if library is not None else lib()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    ref = np.empty(rows.shape[0], dtype=np.float64)
    mag = np.empty(rows.shape[0], dtype=np.float64)
    Cp = _ptr(C) if C is not None else None
    code = lib_.oracle_sgemm_elements(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, Cp, ldc,
                                      rows.shape[0], _ptr(rows), _ptr(cols), _ptr(ref), _ptr(mag))
    if code != 0:
        raise ValueError("oracle_sgemm_elements: index outside the result")
    return ref, mag


def sgemm(A2, B2, C2, alpha, beta, library=None, threads=None):
    """Convenience form on 2-D row-major float32 arrays (natural leading dims)."""
    M, K = A2.shape
    K2, N = B2.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    A = np.ascontiguousarray(A2, dtype=np.float32).reshape(-1)
    B = np.ascontiguousarray(B2, dtype=np.float32).reshape(-1)
    C = None if C2 is None else np.ascontiguousarray(C2, dtype=np.float32).reshape(-1)
    return sgemm_rows(M, N, K, alpha, A, max(K, 1), B, max(N, 1), beta, C, max(N, 1),
                      library=library, threads=threads)


def within_tolerance(gpu, ref, mag, rel=1e-5, floor=1e-30):
    """Elementwise test of |gpu - ref| <= rel * mag + floor (NaN fails)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    ok = err <= rel * mag + floor
    return np.logical_and(ok, np.isfinite(gpu))
