"""Row-major A through the staging ring (ALoad kARowStg: a TMA box per
k-slice as A is stored, transposed into As[k][m] by an extra producer warp)
against the oracle: every compiled configuration built with it, on shapes
with a ragged last tile row, column and k-slice, single and batched. The
variant fills the same As[k][m] as the transposing copy and the FMA warps run
the same loop, so switching it off must give bit-identical results; an A that
TMA cannot address (lda not a multiple of 4, or a pointer off 16 bytes) falls
back to the copy."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload, make_inputs

import gpu_helpers as H
import oracle

pytestmark = pytest.mark.gpu


def _round_1k(floats):
    return (floats + 255) // 256 * 256


def _staged_eligible(p):
    """tile_config.hpp's stg_eligible, restated for the test."""
    BM, BN, BK, NT, ST, MINB = p["BM"], p["BN"], p["BK"], p["NT"], p["STAGES"], p["MINB"]
    acc = (BM * BN) // NT

    def smem(st):
        return (1024 + st * (_round_1k(BK * (BM + 4)) + _round_1k(BK * (BN + 4))) * 4
                + 2 * BM * BK * 4 + st * 24 + 16 + 16)

    def fits(st):
        return smem(st) <= 227 * 1024 and MINB * (smem(st) + 1024) <= 228 * 1024
    while ST > 3 and not fits(ST):
        ST -= 1
    return (BK == 32 and BM % 32 == 0 and BM <= 256 and fits(ST) and acc <= 64
            and (NT + 32) * MINB * 200 <= 65536)


ELIGIBLE = [i for i in range(binding.sgemm_config_count())
            if _staged_eligible(binding.sgemm_config_info(i)[1])]


@pytest.fixture
def staged():
    # wherever allowed, whatever the size (the default also wants >= 8 k-slices per CTA)
    prev = binding.sgemm_set_staged_a(2)
    yield
    binding.sgemm_set_staged_a(prev)


def test_some_configuration_is_built_with_it():
    assert ELIGIBLE, "no compiled configuration is built with the staged-A variant"


def test_only_eligible_configurations_take_it(staged):
    w = Workload("stgsel", 200, 136, 96, 1.0, 0.0, "int3", 60)
    A, B, C = make_inputs(w)
    for cid in range(binding.sgemm_config_count()):
        H.run_cuda(w, A, B, C, config=cid)
        assert ("a=stg" in binding.sgemm_last_config()) == (cid in ELIGIBLE), cid


@pytest.mark.parametrize("config", ELIGIBLE)
@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape", [(300, 200, 777), (1000, 320, 96), (257, 129, 33), (64, 64, 4100),
                                   (520, 64, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_matches_oracle_and_the_copy_path(config, dist, shape, staged):
    M, N, K = shape
    # lda and ldb multiples of 4 (B by TMA), ldc = N (ragged rows of C)
    w = Workload("stg", M, N, K, 1.25, -0.5, dist, 61, lda=K + (-K) % 4 + 4, ldb=N + (-N) % 4)
    A, B, C = make_inputs(w)
    got = H.run_cuda(w, A, B, C, config=config)
    # lda, ldb multiples of 4 and the buffers 256-byte aligned: the staged variant
    assert "a=stg" in binding.sgemm_last_config()
    ref, mag = H.oracle_full(w, A, B, C)
    H.assert_match(w, H.logical(got, w.M, w.N, w.LDC), ref, mag, what=f"cfg {config} staged")
    assert binding.sgemm_set_staged_a(0) == 2
    try:
        got_copy = H.run_cuda(w, A, B, C, config=config)
        assert "a=rowT" in binding.sgemm_last_config()
    finally:
        binding.sgemm_set_staged_a(2)
    assert np.array_equal(got, got_copy, equal_nan=True)


@pytest.mark.parametrize("shape", [(1, 64, 1), (5, 7, 5), (255, 33, 31), (257, 100, 32), (64, 1, 65),
                                   (300, 64, 8), (1, 300, 100)], ids=lambda s: "x".join(map(str, s)))
def test_edge_shapes(shape, staged):
    # K below one slice, single rows and columns, ragged tiles: TMA fills what
    # lies outside A with zeros, and the result is exact on integers
    M, N, K = shape
    for cid in ELIGIBLE:
        w = Workload("stgedge", M, N, K, 1.0, 1.0, "int3", 67, lda=K + (-K) % 4,
                     ldb=N + (-N) % 4)
        A, B, C = make_inputs(w)
        got = H.run_cuda(w, A, B, C, config=cid)
        assert "a=stg" in binding.sgemm_last_config(), (cid, shape)
        ref, mag = H.oracle_full(w, A, B, C)
        H.assert_match(w, H.logical(got, w.M, w.N, w.LDC), ref, mag, what=f"cfg {cid} {shape}")


def _last_with(w, cid, offsets):
    A, B, C = make_inputs(w)
    H.run_cuda(w, A, B, C, offsets=offsets, config=cid)
    return binding.sgemm_last_config()


def test_path_is_reported_and_falls_back(staged):
    if not ELIGIBLE:
        pytest.skip("no configuration is built with the staged-A variant")
    cid = ELIGIBLE[0]
    w = Workload("stgrep", 500, 300, 640, 1.0, 0.0, "int3", 62)
    H.check_against_oracle(w, config=cid)
    assert "a=stg" in _last_with(w, cid, offsets=(0, 0, 0))
    # lda not a multiple of 4, or A off 16 bytes: the transposing copy
    w2 = Workload("stgodd", 500, 300, 641, 1.0, 0.0, "int3", 63)
    H.check_against_oracle(w2, config=cid)
    assert "a=rowT" in _last_with(w2, cid, offsets=(0, 0, 0))
    H.check_against_oracle(w, offsets=(1, 0, 0), config=cid)
    assert "a=rowT" in _last_with(w, cid, offsets=(1, 0, 0))
    # B not TMA-aligned: B by copy, so A by copy too
    H.check_against_oracle(w, offsets=(0, 1, 0), config=cid)
    assert "a=rowT b=cp" in _last_with(w, cid, offsets=(0, 1, 0))


@pytest.mark.parametrize("dist", ["int3", "uniform"])
def test_strided_batched(dist, staged):
    if not ELIGIBLE:
        pytest.skip("no configuration is built with the staged-A variant")
    M, N, K, batch = 300, 260, 500, 3
    g = torch.Generator().manual_seed(64)

    def draw(n):
        if dist == "int3":
            return torch.randint(-3, 4, (n,), generator=g).float()
        return torch.rand(n, generator=g) * 2 - 1
    lda, sA, sB, sC = K + 4, (K + 4) * M + 8, K * N + 4, M * N + 12
    A = draw(sA * batch).cuda()
    B = draw(sB * batch).cuda()
    C = draw(sC * batch).cuda()
    outs = []
    for on in (2, 0):
        binding.sgemm_set_staged_a(on)
        binding.sgemm_force_config(ELIGIBLE[0])
        try:
            Cw = C.clone()
            st = binding.sgemm_strided_batched(0, 0, M, N, K, 0.5, A.data_ptr(), lda, sA, B.data_ptr(), N, sB,
                                               2.0, Cw.data_ptr(), N, sC, batch,
                                               torch.cuda.current_stream().cuda_stream)
            assert st == 0
            torch.cuda.synchronize()
            assert ("a=stg" in binding.sgemm_last_config()) == bool(on)
            outs.append(Cw.cpu())
        finally:
            binding.sgemm_force_config(-1)
            binding.sgemm_set_staged_a(2)
    assert torch.equal(outs[0], outs[1])
    Ah, Bh, Ch = A.cpu().numpy(), B.cpu().numpy(), C.cpu().numpy()
    for b in range(batch):
        a = Ah[b * sA: b * sA + M * lda].reshape(M, lda)[:, :K]
        bb = Bh[b * sB: b * sB + K * N].reshape(K, N)
        c = Ch[b * sC: b * sC + M * N].reshape(M, N)
        ref, mag = oracle.sgemm(a, bb, c, 0.5, 2.0)
        got = outs[0].numpy()[b * sC: b * sC + M * N].reshape(M, N).astype(np.float64)
        if dist == "int3":
            assert np.array_equal(got, ref), b
        else:
            assert oracle.within_tolerance(got, ref, mag, H.REL_TOL, H.ABS_FLOOR).all(), b


def test_default_wants_enough_k_slices_per_cta():
    if not ELIGIBLE:
        pytest.skip("no configuration is built with the staged-A variant")
    prev = binding.sgemm_set_staged_a(1)
    try:
        cid = ELIGIBLE[0]
        BK = binding.sgemm_config_info(cid)[1]["BK"]
        # a handful of k-slices in all: the transposing copy
        few = Workload("stgfew", 256, 256, 2 * BK, 1.0, 0.0, "int3", 65)
        assert "a=rowT" in _last_with(few, cid, offsets=(0, 0, 0))
        # 8 tiles of up to 256 x 256 with 320 k-slices each: more than 8 per CTA
        # even on 304 CTAs, so staged
        many = Workload("stgmany", 512, 256, 320 * BK, 1.0, 0.0, "int3", 66)
        H.check_against_oracle(many, config=cid)
        assert "a=stg" in _last_with(many, cid, offsets=(0, 0, 0))
    finally:
        binding.sgemm_set_staged_a(prev)


def test_switch_arguments():
    for bad in (-1, 3):
        assert binding.sgemm_set_staged_a(bad) == binding.SGEMM_ERR_INVALID_VALUE
    prev = binding.sgemm_set_staged_a(0)
    assert binding.sgemm_set_staged_a(prev) == 0
