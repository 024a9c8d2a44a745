"""ctypes binding of libsgemm_gb300.so: the C ABI of include/sgemm_gb300.h
under the same names, plus a torch convenience that only marshals arguments
(device tensors -> pointers and leading dimensions, the current stream).

There is no fallback: if the CUDA library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

SGEMM_OK = 0
SGEMM_ERR_INVALID_DIM = -1
SGEMM_ERR_INVALID_LD = -2
SGEMM_ERR_NULL_PTR = -3
SGEMM_ERR_UNSUPPORTED_DEVICE = -4
SGEMM_ERR_LAUNCH = -5
SGEMM_ERR_DEVICE_TIMEOUT = -6
SGEMM_ERR_ALLOC = -7
SGEMM_ERR_MISALIGNED = -8
SGEMM_ERR_INVALID_VALUE = -9
SGEMM_ERR_NOALLOC_CAPACITY = -10
SGEMM_ERR_CAPTURE = -11

SGEMM_OP_N = 0
SGEMM_OP_T = 1

PARAM_NAMES = ("BM", "BN", "BK", "WM", "WN", "WNITER", "TM", "TN", "NT", "STAGES", "MINB", "KU", "ORDER")


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {sgemm_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    """The library to load: SGEMM_GB300_LIB if set (the tuner's candidate
    build), else the in-tree product library."""
    return os.environ.get("SGEMM_GB300_LIB") or _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(path)
            I, F, P, LL = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_longlong
            IP = ctypes.POINTER(ctypes.c_int)
            sig = {
                "sgemm": (I, [I, I, I, F, P, I, P, I, F, P, I, P]),
                "sgemm_status_string": (ctypes.c_char_p, [I]),
                "sgemm_last_config": (I, [ctypes.c_char_p, I]),
                "sgemm_poll_device_status": (I, [P, IP]),
                "sgemm_shutdown": (None, []),
                "sgemm_config_count": (I, []),
                "sgemm_config_info": (I, [I, ctypes.c_char_p, I, IP]),
                "sgemm_force_config": (I, [I]),
                "sgemm_set_staged_a": (I, [I]),
                "sgemm_cfg_check": (I, [IP, IP]),
                "sgemm_schedule_query": (I, [I, I, I, I, I, IP]),
                "sgemm_schedule_piece": (I, [IP, I, I, IP]),
                "sgemm_schedule_plan": (I, [I, I, I, I, I, I, I, IP, IP]),
                "sgemm_force_schedule": (I, [IP]),
                "sgemm_choose_policy": (I, [I, I, I, IP]),
                "sgemm_diag_wait_timeout": (I, [LL, P]),
                "sgemm_set_wait_timeout_ns": (LL, [LL]),
                "sgemm_noalloc": (I, [I, I, I, F, P, I, P, I, F, P, I, P]),
                "sgemm_noalloc_poll_status": (I, [P, IP]),
                "sgemm_choose_config": (I, [I, I, I, IP]),
                "sgemm_3xtf32": (I, [I, I, I, F, P, I, P, I, F, P, I, P]),
                "sgemm_ex": (I, [I, I, I, I, I, F, P, I, P, I, F, P, I, P]),
                "sgemm_host": (I, [I, I, I, F, P, I, P, I, F, P, I, P]),
                "sgemm_ladder": (I, [I, I, I, I, F, P, I, P, I, F, P, I, P]),
                "sgemm_3xtf32_set_kernel_form": (I, [I]),
                "sgemm_3xtf32_plan": (I, [I, I, I, I, I, I, IP]),
                "sgemm_host_set_pipeline": (I, [I, I, I, I]),
                "sgemm_config_layouts": (I, [I]),
                "sgemm_diag_tf32_mma_rate": (I, [I, ctypes.POINTER(ctypes.c_double)]),
                "sgemm_diag_tf32_pair_mma_rate": (I, [I, ctypes.POINTER(ctypes.c_double)]),
                "sgemm_strided_batched": (I, [I, I, I, I, I, F, P, I, LL, P, I, LL, F, P, I, LL,
                                              I, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _ints(n, values=None):
    arr = (ctypes.c_int * n)()
    if values is not None:
        for i, v in enumerate(values):
            arr[i] = int(v)
    return arr


# ---- the C ABI, same names ------------------------------------------------------
def sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Raw call: A, B, C are device addresses (ints), stream a cudaStream_t
    handle (int) or None. Returns the status code."""
    return lib().sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """C = alpha*A*B + beta*C on HOST matrices (addresses as ints), copies
    overlapped with the GEMM; C is final once `stream` is synchronised."""
    return lib().sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_host_set_pipeline(first: int, mid: int, last: int, panels: int) -> int:
    """K-chunk widths (first, middle, last) and the row panels of the last
    chunk for later sgemm_host calls; 0 picks the default. Returns a status."""
    return lib().sgemm_host_set_pipeline(first, mid, last, panels)


def sgemm_ex(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """C = alpha*op(A)*op(B) + beta*C (ops SGEMM_OP_N / SGEMM_OP_T)."""
    return lib().sgemm_ex(opA, opB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_strided_batched(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
                          ldc, strideC, batch, stream=None) -> int:
    """`batch` products C_i = alpha*op(A_i)*op(B_i) + beta*C_i, one launch."""
    return lib().sgemm_strided_batched(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                                       beta, C, ldc, strideC, batch, stream)


def sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Opt-in tensor-core path (three TF32 products per FP32 product), same
    arguments as sgemm(). Returns the status code."""
    return lib().sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_status_string(status: int) -> str:
    return lib().sgemm_status_string(status).decode()


def sgemm_last_config() -> str:
    buf = ctypes.create_string_buffer(256)
    lib().sgemm_last_config(buf, 256)
    return buf.value.decode()


def sgemm_poll_device_status(stream=None):
    """(status, device detail code)."""
    detail = ctypes.c_int(0)
    st = lib().sgemm_poll_device_status(stream, ctypes.byref(detail))
    return st, detail.value


def sgemm_shutdown() -> None:
    lib().sgemm_shutdown()


def sgemm_config_count() -> int:
    return lib().sgemm_config_count()


def sgemm_set_staged_a(on: int) -> int:
    """Row-major A through the staging ring and producer warp: 1 where allowed
    and each CTA runs at least 8 k-slices (default), 2 wherever allowed, 0
    never (the transposing copy). Returns the previous setting."""
    return lib().sgemm_set_staged_a(on)


def sgemm_config_info(cid: int):
    name = ctypes.create_string_buffer(128)
    params = _ints(13)
    st = lib().sgemm_config_info(cid, name, 128, params)
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_config_info")
    return name.value.decode(), dict(zip(PARAM_NAMES, list(params)))


def sgemm_diag_tf32_mma_rate(iters: int = 20000):
    """(status, TFLOP/s): the measured TF32 tensor-core throughput of the
    current device (synchronous, about 6 ms)."""
    v = ctypes.c_double(0.0)
    st = lib().sgemm_diag_tf32_mma_rate(iters, ctypes.byref(v))
    return st, v.value


def sgemm_diag_tf32_pair_mma_rate(iters: int = 20000):
    """(status, TFLOP/s): the same for two-SM (cta_group::2) MMAs issued by
    CTA pairs."""
    v = ctypes.c_double(0.0)
    st = lib().sgemm_diag_tf32_pair_mma_rate(iters, ctypes.byref(v))
    return st, v.value


def sgemm_config_layouts(cid: int) -> int:
    """1: configuration `cid` is built for every operand layout; 0: row-major
    operands only; negative: an error status."""
    return lib().sgemm_config_layouts(cid)


def sgemm_force_config(cid: int) -> int:
    return lib().sgemm_force_config(cid)


SHAPE_CLASSES = ("square_large", "square_small", "k_dominant", "skinny_n", "skinny_m", "tiny",
                 "square_mid")


def sgemm_choose_config(M, N, K):
    """(config id, shape class name) of the automatic choice."""
    cls = ctypes.c_int(-1)
    cid = lib().sgemm_choose_config(M, N, K, ctypes.byref(cls))
    if cid < 0:
        raise SgemmError(cid, "sgemm_choose_config")
    return cid, SHAPE_CLASSES[cls.value]


def sgemm_cfg_check(params):
    """(rule, derived): rule 0 = legal; derived = {WMITER, WSUBM, WSUBN,
    acc_per_thread, smem_bytes} for a legal tuple."""
    if isinstance(params, dict):
        params = [params[k] for k in PARAM_NAMES]
    p = _ints(13, params)
    d = _ints(5)
    rule = lib().sgemm_cfg_check(p, d)
    derived = dict(zip(("WMITER", "WSUBM", "WSUBN", "acc", "smem_bytes"), list(d))) if rule == 0 else None
    return rule, derived


SCHED_FIELDS = ("tiles_m", "tiles_n", "kiters", "grid", "dp_tiles", "sk_q", "sk_r", "group_m")
PIECE_FIELDS = ("tile", "kb", "ke", "tile_m", "tile_n", "contributors", "is_partial")


def sgemm_schedule_query(M, N, K, cid, capacity):
    out = _ints(8)
    st = lib().sgemm_schedule_query(M, N, K, cid, capacity, out)
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_schedule_query")
    return dict(zip(SCHED_FIELDS, list(out)))


SCHED_HYBRID, SCHED_HYBRID_TAIL, SCHED_DATA_PARALLEL, SCHED_STREAM_K, SCHED_SPLIT_K = 0, 1, 2, 3, 4
SCHED_MODES = (SCHED_HYBRID, SCHED_HYBRID_TAIL, SCHED_DATA_PARALLEL, SCHED_STREAM_K, SCHED_SPLIT_K)


def sgemm_schedule_plan(M, N, K, BM, BN, BK, capacity, policy):
    """The schedule for BM x BN x BK tiles under `policy` = (mode, group_m,
    min_units, splits), host arithmetic only; raises on an argument error."""
    out = _ints(8)
    st = lib().sgemm_schedule_plan(M, N, K, BM, BN, BK, capacity, _ints(4, policy), out)
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_schedule_plan")
    return dict(zip(SCHED_FIELDS, list(out)))


def sgemm_force_schedule(policy=None) -> int:
    """Force (mode, group_m, min_units, splits) on later calls; None restores
    the tuned per-class policy. Returns the status code."""
    return lib().sgemm_force_schedule(None if policy is None else _ints(4, policy))


def sgemm_choose_policy(M, N, K):
    """(status, (mode, group_m, min_units, splits)) that sgemm() takes by itself."""
    out = _ints(4)
    st = lib().sgemm_choose_policy(M, N, K, out)
    return st, tuple(out)


def sgemm_schedule_piece(sched: dict, b: int, i: int):
    """(number of pieces of CTA b, piece i as a dict)."""
    v = _ints(8, [sched[k] for k in SCHED_FIELDS])
    out = _ints(7)
    n = lib().sgemm_schedule_piece(v, b, i, out)
    if n < 0:
        raise SgemmError(n, "sgemm_schedule_piece")
    return n, dict(zip(PIECE_FIELDS, list(out)))


def sgemm_diag_wait_timeout(timeout_ns: int, stream=None) -> int:
    return lib().sgemm_diag_wait_timeout(timeout_ns, stream)


def sgemm_set_wait_timeout_ns(ns: int) -> int:
    return lib().sgemm_set_wait_timeout_ns(ns)


def sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Same call as sgemm() for callers that cannot allocate device memory:
    the kernel's scratch comes from a fixed buffer inside the library.
    Returns the status code."""
    return lib().sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_noalloc_poll_status(stream=None):
    """(status, device detail code) of the sgemm_noalloc calls on this device
    since the last poll; synchronises `stream` first."""
    detail = ctypes.c_int(0)
    st = lib().sgemm_noalloc_poll_status(stream, ctypes.byref(detail))
    return st, detail.value


def sgemm_ladder(kernel, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """One of the pages' kernels (3: shared-memory tiling, 7: vectorized
    block tiling, 8: warp tiling) on device matrices; same arguments and
    result as sgemm(). Returns the status code."""
    return lib().sgemm_ladder(kernel, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


LADDER_KERNELS = (3, 7, 8)


SGEMM_X3_SINGLE, SGEMM_X3_PAIR = 1, 2
X3_FORMS = (SGEMM_X3_PAIR, SGEMM_X3_SINGLE)


X3_PLAN_FIELDS = ("form", "bk", "stages", "ctas", "units", "dp_units", "split_units", "kiters",
                  "bn")


def sgemm_3xtf32_plan(M: int, N: int, K: int, form: int, pairs: int, sms: int):
    """(status, {field: value}) of the plan sgemm_3xtf32 follows (host only)."""
    out = _ints(len(X3_PLAN_FIELDS))
    st = lib().sgemm_3xtf32_plan(M, N, K, form, pairs, sms, out)
    return st, dict(zip(X3_PLAN_FIELDS, list(out)))


def sgemm_3xtf32_set_kernel_form(form: int) -> int:
    """SGEMM_X3_PAIR (default): CTA pairs with two-SM MMAs; SGEMM_X3_SINGLE: single
    CTAs. Returns the previous setting (or an error status)."""
    return lib().sgemm_3xtf32_set_kernel_form(form)


# ---- torch conveniences (marshalling only) ------------------------------------------
def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ld(t, name):
    if t.dim() != 2 or t.dtype.__repr__() != "torch.float32":
        raise ValueError(f"{name} must be a 2-D float32 tensor")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit stride along rows)")
    return max(t.stride(0), max(t.size(1), 1)) if t.size(0) > 1 else max(t.size(1), 1)


def gemm(A, B, C, alpha=1.0, beta=0.0, stream=None):
    """C <- alpha*A@B + beta*C on CUDA float32 tensors (row-major views with
    any row stride). Raises SgemmError on a non-zero status. Returns C."""
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch")
    for t, nm in ((A, "A"), (B, "B"), (C, "C")):
        if not t.is_cuda:
            raise ValueError(f"{nm} must be a CUDA tensor")
    st = sgemm(M, N, K, float(alpha), A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"),
               float(beta), C.data_ptr(), _ld(C, "C"), _stream_handle(stream))
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm")
    return C
