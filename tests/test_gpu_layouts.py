"""Transposed operands (sgemm_ex) and strided batches (sgemm_strided_batched)
against the oracle. The oracle always takes the logical row-major op(A)
(M x K) and op(B) (K x N); the GPU gets the stored matrices: A^T stored K x M
for op(A) = T and B^T stored N x K for op(B) = T. Padding between rows and
between the matrices of a batch holds NaN, so a read outside an operand shows
up as NaN."""
import numpy as np
import pytest
import torch

import oracle
from conftest import compiled_config_count
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload, make_inputs

import gpu_helpers as H

pytestmark = pytest.mark.gpu
N_, T_ = binding.SGEMM_OP_N, binding.SGEMM_OP_T
ALL_LAYOUT_CONFIGS = [i for i in range(compiled_config_count())]


def _stored(x2d, op, ld_pad):
    """Row-major storage of the operand whose logical form is x2d."""
    s = x2d if op == N_ else x2d.T
    s = np.ascontiguousarray(s, dtype=np.float32)
    buf = np.full((s.shape[0], s.shape[1] + ld_pad), np.nan, np.float32)
    buf[:, : s.shape[1]] = s
    return buf.reshape(-1), s.shape[1] + ld_pad


def _run_ex(w, opA, opB, offsets=(0, 0, 0), ld_pad=(0, 0, 0), config=None):
    A, B, C = make_inputs(w)
    A2 = A.numpy().reshape(w.M, w.LDA)[:, : w.K]
    B2 = B.numpy().reshape(w.K, w.LDB)[:, : w.N]
    Af, lda = _stored(A2, opA, ld_pad[0])
    Bf, ldb = _stored(B2, opB, ld_pad[1])
    Cf = np.full((w.M, w.N + ld_pad[2]), np.nan, np.float32)
    Cf[:, : w.N] = C.numpy().reshape(w.M, w.LDC)[:, : w.N]
    ldc = w.N + ld_pad[2]
    _, dA = H.device_buffer(torch.from_numpy(Af), offsets[0])
    _, dB = H.device_buffer(torch.from_numpy(Bf), offsets[1])
    storeC, dC = H.device_buffer(torch.from_numpy(Cf.reshape(-1)), offsets[2])
    if config is not None:
        binding.sgemm_force_config(config)
    try:
        s = torch.cuda.current_stream().cuda_stream
        st = binding.sgemm_ex(opA, opB, w.M, w.N, w.K, w.alpha, dA.data_ptr(), lda, dB.data_ptr(),
                              ldb, w.beta, dC.data_ptr(), ldc, s)
        assert st == 0, binding.sgemm_status_string(st)
        assert binding.sgemm_poll_device_status(s) == (0, 0)
        torch.cuda.synchronize()
    finally:
        binding.sgemm_force_config(-1)
    H.assert_guards_intact(storeC, offsets[2], Cf.size, what="sgemm_ex C")
    got = dC.cpu().numpy().reshape(w.M, ldc)
    ref, mag = oracle.sgemm(A2, B2, None if w.beta == 0 else C.numpy().reshape(w.M, w.LDC)[:, : w.N],
                            w.alpha, w.beta)
    H.assert_match(w, got[:, : w.N], ref, mag, what=f"op {opA}{opB} cfg {config}")
    if ld_pad[2]:
        assert np.all(np.isnan(got[:, w.N:])), "C padding was written"
    return binding.sgemm_last_config()


OPS = [(N_, N_), (N_, T_), (T_, N_), (T_, T_)]


@pytest.mark.parametrize("ops", OPS, ids=["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape", [(257, 129, 100), (300, 520, 77), (64, 700, 1025), (1000, 40, 129),
                                   (7, 9, 3), (129, 257, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_ops(shape, dist, ops):
    M, N, K = shape
    _run_ex(Workload("ops", M, N, K, 1.25, -0.5, dist, 41), *ops)


@pytest.mark.parametrize("ops", OPS[1:], ids=["NT", "TN", "TT"])
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (1, 1, 1)])
def test_ops_unaligned_and_padded(ops, offsets):
    w = Workload("opsu", 301, 203, 777, 1.25, -0.5, "int3", 42)
    cfg = _run_ex(w, *ops, offsets=offsets, ld_pad=(3, 5, 2))
    if ops[0] == T_ and offsets[0] % 4:
        assert "a=cp" in cfg       # A^T not 16-byte aligned: plain copies, not TMA
    _run_ex(w.with_(dist="normal"), *ops, offsets=offsets, ld_pad=(3, 5, 2))


def test_ops_transposed_a_uses_tma_when_aligned():
    cfg = _run_ex(Workload("tma", 512, 512, 512, 1.0, 0.0, "int3", 43), T_, N_)
    assert "a=tma" in cfg and "b=tma" in cfg
    cfg = _run_ex(Workload("colT", 512, 512, 512, 1.0, 0.0, "int3", 43), N_, T_)
    assert "b=colT" in cfg


@pytest.mark.parametrize("config", ALL_LAYOUT_CONFIGS)
def test_ops_every_config(config):
    name, _ = binding.sgemm_config_info(config)
    w = Workload("opscfg", 200, 264, 300, 0.5, 3.0, "int3", 44)
    for ops in OPS:
        cfg = _run_ex(w, *ops, config=config)
        if ops == (N_, N_):
            assert cfg.startswith(name)


def test_column_major_identity():
    # a column-major M x N product is the row-major N x M product with the
    # operands swapped: C^T = B^T A^T
    M, N, K = 150, 90, 70
    g = np.random.default_rng(45)
    A = g.integers(-3, 4, (M, K)).astype(np.float32)   # logical column-major A
    B = g.integers(-3, 4, (K, N)).astype(np.float32)
    A_cm = A.ravel(order="F").copy()                    # column-major storage, lda = M
    B_cm = B.ravel(order="F").copy()                    # ldb = K
    dA, dB = torch.from_numpy(A_cm).cuda(), torch.from_numpy(B_cm).cuda()
    dC = torch.zeros(M * N, device="cuda")
    # row-major view: B_cm is B^T stored N x K (ld K), A_cm is A^T stored K x M (ld M)
    st = binding.sgemm_ex(N_, N_, N, M, K, 1.0, dB.data_ptr(), K, dA.data_ptr(), M, 0.0,
                          dC.data_ptr(), M, None)
    torch.cuda.synchronize()
    assert st == 0
    C_cm = dC.cpu().numpy().reshape(N, M).T               # column-major result
    assert np.array_equal(C_cm, A.astype(np.int64) @ B.astype(np.int64))


def _batched_case(batch, M, N, K, opA, opB, gap, alpha, beta, dist, seed):
    ws = [Workload("bat", M, N, K, alpha, beta, dist, seed + i) for i in range(batch)]
    logical = [make_inputs(w) for w in ws]
    A2 = [x[0].numpy().reshape(M, K) for x in logical]
    B2 = [x[1].numpy().reshape(K, N) for x in logical]
    C2 = [x[2].numpy().reshape(M, N) for x in logical]
    As = [np.ascontiguousarray(a if opA == N_ else a.T) for a in A2]
    Bs = [np.ascontiguousarray(b if opB == N_ else b.T) for b in B2]
    lda, ldb, ldc = As[0].shape[1], Bs[0].shape[1], N
    sA, sB, sC = As[0].size + gap, Bs[0].size + gap, M * N + gap

    def pack(mats, stride):
        buf = np.full(stride * batch, np.nan, np.float32)
        for i, m in enumerate(mats):
            buf[i * stride: i * stride + m.size] = m.reshape(-1)
        return torch.from_numpy(buf).cuda()
    dA, dB, dC = pack(As, sA), pack(Bs, sB), pack(C2, sC)
    s = torch.cuda.current_stream().cuda_stream
    st = binding.sgemm_strided_batched(opA, opB, M, N, K, alpha, dA.data_ptr(), lda, sA,
                                       dB.data_ptr(), ldb, sB, beta, dC.data_ptr(), ldc, sC,
                                       batch, s)
    assert st == 0, binding.sgemm_status_string(st)
    assert binding.sgemm_poll_device_status(s) == (0, 0)
    out = dC.cpu().numpy()
    for i in range(batch):
        got = out[i * sC: i * sC + M * N].reshape(M, N)
        ref, mag = oracle.sgemm(A2[i], B2[i], None if beta == 0 else C2[i], alpha, beta)
        H.assert_match(ws[i], got, ref, mag, what=f"batch {i}")
        if gap:
            assert np.all(np.isnan(out[i * sC + M * N: (i + 1) * sC])), "gap written"
    return binding.sgemm_last_config()


@pytest.mark.parametrize("ops", OPS, ids=["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("gap", [0, 12, 3])
def test_strided_batched(ops, gap):
    cfg = _batched_case(5, 130, 200, 96, *ops, gap, 1.25, -0.5, "int3", 50)
    assert "batched" in cfg
    _batched_case(3, 257, 129, 300, *ops, gap, 0.5, 3.0, "uniform", 60)


def test_batched_split_schedule():
    # few tiles per matrix and a long K: the batch's tiles are split along K
    _batched_case(3, 128, 256, 6000, N_, N_, 4, 1.0, 1.0, "int3", 70)


def test_batched_edge_cases():
    C = torch.full((64,), 5.0, device="cuda")
    p = C.data_ptr()
    assert binding.sgemm_strided_batched(N_, N_, 4, 4, 4, 1.0, p, 4, 16, p, 4, 16, 0.0, p, 4, 16,
                                         0, None) == 0                    # empty batch
    assert binding.sgemm_strided_batched(N_, N_, 4, 4, 4, 1.0, p, 4, -1, p, 4, 16, 0.0, p, 4, 16,
                                         2, None) == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_ex(2, N_, 4, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 4, None) == \
        binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_ex(T_, N_, 8, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 4, None) == \
        binding.SGEMM_ERR_INVALID_LD                                      # lda < M for op T
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)
    # alpha == 0 scales every C_i by beta
    Cb = torch.arange(48, dtype=torch.float32, device="cuda")
    assert binding.sgemm_strided_batched(N_, N_, 2, 3, 5, 0.0, 0, 5, 0, 0, 3, 0, 2.0, Cb.data_ptr(),
                                         3, 16, 3, None) == 0
    torch.cuda.synchronize()
    ref = torch.arange(48, dtype=torch.float32)
    for i in range(3):
        ref[i * 16: i * 16 + 6] *= 2
    assert torch.equal(Cb.cpu(), ref)
