"""sgemm_host: the GEMM on host matrices with copies overlapped with the
multiplication, against the oracle (bit-exact on integer inputs, the FP32
tolerance on real inputs)."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload, make_inputs

import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _host_call(w, pinned=True, pad=(0, 0, 0), stream=None):
    A, B, C = make_inputs(w)
    A2 = A.numpy().reshape(w.M, w.LDA)[:, : w.K]
    B2 = B.numpy().reshape(w.K, w.LDB)[:, : w.N]
    C2 = C.numpy().reshape(w.M, w.LDC)[:, : w.N]

    def host(x2, p):
        buf = torch.full((x2.shape[0], x2.shape[1] + p), float("nan"))
        buf[:, : x2.shape[1]] = torch.from_numpy(np.ascontiguousarray(x2))
        return buf.pin_memory() if pinned else buf
    hA, hB, hC = host(A2, pad[0]), host(B2, pad[1]), host(C2, pad[2])
    s = stream if stream is not None else torch.cuda.current_stream()
    st = binding.sgemm_host(w.M, w.N, w.K, w.alpha, hA.data_ptr(), hA.shape[1], hB.data_ptr(),
                            hB.shape[1], w.beta, hC.data_ptr(), hC.shape[1], s.cuda_stream)
    assert st == 0, binding.sgemm_status_string(st)
    s.synchronize()
    assert binding.sgemm_poll_device_status(s.cuda_stream) == (0, 0)
    got = hC.numpy()
    ref, mag = oracle.sgemm(A2, B2, None if w.beta == 0 else C2, w.alpha, w.beta)
    H.assert_match(w, got[:, : w.N], ref, mag, what="sgemm_host")
    if pad[2]:
        assert np.all(np.isnan(got[:, w.N:])), "C padding was written"


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("dist", ["int3", "uniform"])
@pytest.mark.parametrize("shape", [(300, 520, 77), (257, 129, 3000), (64, 700, 5000),
                                   (1000, 40, 2049), (7, 9, 3)], ids=lambda s: "x".join(map(str, s)))
def test_host_matches_oracle(shape, dist, pinned):
    M, N, K = shape
    _host_call(Workload("host", M, N, K, 1.25, -0.5, dist, 81), pinned=pinned)


def test_host_beta_zero_padded_and_growing_buffers():
    _host_call(Workload("host0", 128, 96, 64, 1.0, 0.0, "int3", 82), pad=(3, 1, 2))
    _host_call(Workload("host1", 600, 700, 4100, 0.5, 3.0, "int3", 83), pad=(0, 4, 1))
    _host_call(Workload("host2", 90, 80, 70, 2.0, 1.0, "normal", 84))


def test_host_alpha_zero_and_other_stream():
    _host_call(Workload("host3", 70, 90, 33, 0.0, -0.5, "int3", 85))
    s = torch.cuda.Stream()
    _host_call(Workload("host4", 200, 300, 2100, 1.25, -0.5, "int3", 86), stream=s)


def test_host_full_size_integer():
    w = Workload("hostbig", 4096, 4096, 4096, 0.5, 3.0, "int3", 87)
    A, B, C = make_inputs(w)
    hA, hB, hC = A.pin_memory(), B.pin_memory(), C.clone().pin_memory()
    s = torch.cuda.current_stream()
    assert binding.sgemm_host(w.M, w.N, w.K, w.alpha, hA.data_ptr(), w.K, hB.data_ptr(), w.N,
                              w.beta, hC.data_ptr(), w.N, s.cuda_stream) == 0
    s.synchronize()
    H.freivalds(w, A, B, C, hC.numpy().reshape(w.M, w.N))


@pytest.mark.parametrize("pipeline", [(128, 512, 256, 8), (0, 4096, 0, 1), (256, 1024, 512, 2),
                                      (64, 64, 64, 3), (32, 0, 0, 8), (64, 0, 512, 3), (2048, 0, 0, 2)],
                         ids=lambda p: "-".join(map(str, p)))
def test_host_pipeline_settings(pipeline):
    # any chunking of K (equal middle chunks, or geometric growth when mid is
    # 0) and any panel count give the same (exact) result
    assert binding.sgemm_host_set_pipeline(*pipeline) == 0
    try:
        _host_call(Workload("hostpipe", 2100, 300, 3000, 1.25, -0.5, "int3", 88))
        _host_call(Workload("hostpipe", 2100, 300, 3000, 1.25, -0.5, "uniform", 89))
    finally:
        assert binding.sgemm_host_set_pipeline(0, 0, 0, 0) == 0
