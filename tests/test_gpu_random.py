"""Seeded random cases against the oracle: shapes, padded leading dimensions,
pointer offsets, alpha and beta (zero included), input distributions,
operand forms, batch counts, forced tile configurations, and each entry point
(sgemm, sgemm_ex, sgemm_strided_batched, sgemm_3xtf32 in its three kernel forms,
sgemm_ladder, sgemm_noalloc, and sgemm_host on pinned or pageable host
memory). Every case is a fixed function of its index, so a failure
names a reproducible case. Padding holds NaN: a read outside an operand
shows up in the result."""
import numpy as np
import pytest
import torch

import oracle
from conftest import compiled_config_count
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload

import gpu_helpers as H

pytestmark = pytest.mark.gpu
N_, T_ = binding.SGEMM_OP_N, binding.SGEMM_OP_T
CASES = 420
ENTRIES = ["sgemm", "sgemm_ex", "batched", "tf32x3", "ladder", "noalloc", "host"]


def _case(i):
    r = np.random.default_rng(9000 + i)

    def dim():
        u = r.random()
        return int(r.integers(1, 33)) if u < 0.3 else int(r.integers(33, 700))
    M, N = dim(), dim()
    K = int(r.integers(1, 5000)) if r.random() < 0.25 else dim()
    entry = ENTRIES[i % len(ENTRIES)]
    return dict(
        entry=entry, M=M, N=N, K=K,
        alpha=float(r.choice([1.0, -0.75, 0.5, 2.5, 0.0], p=[0.3, 0.2, 0.2, 0.2, 0.1])),
        beta=float(r.choice([0.0, 1.0, -1.5, 3.0])),
        dist=str(r.choice(["int3", "uniform", "normal"])),
        pads=tuple(int(x) for x in r.integers(0, 6, 3)),
        offsets=tuple(int(x) for x in r.integers(0, 4, 3)),
        opA=int(r.integers(0, 2)) if entry in ("sgemm_ex", "batched") else N_,
        opB=int(r.integers(0, 2)) if entry in ("sgemm_ex", "batched") else N_,
        batch=int(r.integers(1, 4)) if entry == "batched" else 1,
        config=int(r.integers(-1, compiled_config_count())),
        # three equally likely draws over the two kernel forms (the draw keeps its
        # width so that every other field of every case stays as it was)
        x3form=(binding.SGEMM_X3_SINGLE, binding.SGEMM_X3_PAIR, binding.SGEMM_X3_SINGLE)[int(r.integers(0, 3))],
        kernel=int(r.choice(binding.LADDER_KERNELS)),
        seed=int(r.integers(0, 2**31 - 1)),
        pinned=bool(r.integers(0, 2)),
    )


def _draw(r, rows, cols, dist):
    if dist == "int3":
        return r.integers(-3, 4, (rows, cols)).astype(np.float32)
    if dist == "uniform":
        return (r.random((rows, cols), dtype=np.float32) * 2 - 1).astype(np.float32)
    return r.standard_normal((rows, cols), dtype=np.float32)


def _stored(x2d, op, pad):
    s = np.ascontiguousarray(x2d if op == N_ else x2d.T, dtype=np.float32)
    buf = np.full((s.shape[0], s.shape[1] + pad), np.nan, np.float32)
    buf[:, : s.shape[1]] = s
    return buf, s.shape[1] + pad


@pytest.mark.parametrize("i", range(CASES))
def test_random_case(i):
    c = _case(i)
    M, N, K, batch = c["M"], c["N"], c["K"], c["batch"]
    r = np.random.default_rng(c["seed"])
    mats = []
    for _ in range(batch):
        A2, B2, C2 = _draw(r, M, K, c["dist"]), _draw(r, K, N, c["dist"]), _draw(r, M, N, c["dist"])
        mats.append((A2, B2, C2))
    # stored operands, one matrix after another with a gap of NaN between them
    As, Bs, Cs = [], [], []
    for A2, B2, C2 in mats:
        a, lda = _stored(A2, c["opA"], c["pads"][0])
        b, ldb = _stored(B2, c["opB"], c["pads"][1])
        cc, ldc = _stored(C2, N_, c["pads"][2])
        As.append(a)
        Bs.append(b)
        Cs.append(cc)
    gap = 8
    sA, sB, sC = As[0].size + gap, Bs[0].size + gap, Cs[0].size + gap

    def flat(parts, stride):
        out = np.full(stride * len(parts), np.nan, np.float32)
        for j, p in enumerate(parts):
            out[j * stride: j * stride + p.size] = p.reshape(-1)
        return torch.from_numpy(out)
    e = c["entry"]
    if e == "host":
        def host_buffer(t, off):
            store = torch.full((t.numel() + off + 16,), float("nan"))
            if c["pinned"]:
                store = store.pin_memory()
            view = store[off: off + t.numel()]
            view.copy_(t)
            return store, view
        _, dA = host_buffer(flat(As, sA), c["offsets"][0])
        _, dB = host_buffer(flat(Bs, sB), c["offsets"][1])
        _, dC = host_buffer(flat(Cs, sC), c["offsets"][2])
    else:
        _, dA = H.device_buffer(flat(As, sA), c["offsets"][0])
        _, dB = H.device_buffer(flat(Bs, sB), c["offsets"][1])
        storeC, dC = H.device_buffer(flat(Cs, sC), c["offsets"][2])
    s = torch.cuda.current_stream().cuda_stream
    pA, pB, pC = dA.data_ptr(), dB.data_ptr(), dC.data_ptr()
    alpha, beta = c["alpha"], c["beta"]
    if e in ("sgemm", "sgemm_ex", "batched"):
        assert binding.sgemm_force_config(c["config"]) == 0
    prev_form = binding.sgemm_3xtf32_set_kernel_form(c["x3form"])
    try:
        if e == "sgemm":
            st = binding.sgemm(M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc, s)
        elif e == "sgemm_ex":
            st = binding.sgemm_ex(c["opA"], c["opB"], M, N, K, alpha, pA, lda, pB, ldb, beta, pC,
                                  ldc, s)
        elif e == "batched":
            st = binding.sgemm_strided_batched(c["opA"], c["opB"], M, N, K, alpha, pA, lda, sA, pB,
                                               ldb, sB, beta, pC, ldc, sC, batch, s)
        elif e == "tf32x3":
            st = binding.sgemm_3xtf32(M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc, s)
        elif e == "noalloc":
            st = binding.sgemm_noalloc(M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc, s)
        elif e == "host":
            st = binding.sgemm_host(M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc, s)
        else:
            st = binding.sgemm_ladder(c["kernel"], M, N, K, alpha, pA, lda, pB, ldb, beta, pC, ldc,
                                      s)
        assert st == 0, f"case {c}: {binding.sgemm_status_string(st)}"
        torch.cuda.synchronize()
        if e != "noalloc":  # its status lives in its own buffer
            assert binding.sgemm_poll_device_status(s) == (0, 0)
    finally:
        binding.sgemm_force_config(-1)
        binding.sgemm_3xtf32_set_kernel_form(prev_form)
    if e != "host":
        H.assert_guards_intact(storeC, c["offsets"][2], dC.numel(), what=f"case {c}")
    out = dC.cpu().numpy() if e != "host" else dC.numpy()
    w = Workload(f"random{i}", M, N, K, alpha, beta, c["dist"], c["seed"])
    for j, (A2, B2, C2) in enumerate(mats):
        got = out[j * sC: j * sC + Cs[j].size].reshape(M, ldc)
        ref, mag = oracle.sgemm(A2, B2, None if beta == 0 else C2, alpha, beta)
        H.assert_match(w, got[:, :N], ref, mag, what=f"case {c} matrix {j}")
        if c["pads"][2]:
            assert np.all(np.isnan(got[:, N:])), f"case {c}: C padding was written"
        if j + 1 < batch:
            between = out[j * sC + Cs[j].size: (j + 1) * sC]
            assert np.all(np.isnan(between)), f"case {c}: the gap after matrix {j} was written"
