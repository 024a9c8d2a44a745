"""The GEMM entry points captured into a CUDA graph and replayed on fresh
inputs, against the oracle each time. A split-K schedule publishes partial
tiles behind flags; a replay reuses the captured arguments, so this checks
that no replay can see an earlier replay's flags."""
import functools

import numpy as np
import pytest
import torch

from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload, make_inputs

import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _args(w, dA, dB, dC, stream):
    return (w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.LDA, dB.data_ptr(), w.LDB, w.beta,
            dC.data_ptr(), w.LDC, stream.cuda_stream)


def _replay_and_check(fn, w, replays=3):
    A, B, C = make_inputs(w)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    # outside the capture: device set-up and the stream's workspace
    assert fn(*_args(w, dA, dB, dC, s)) == 0
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = fn(*_args(w, dA, dB, dC, s))
    assert st == 0, binding.sgemm_status_string(st)
    for r in range(replays):
        Ar, Br, Cr = make_inputs(w.with_(seed=w.seed + 100 + r))
        dA.copy_(Ar)
        dB.copy_(Br)
        dC.copy_(Cr)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert binding.sgemm_poll_device_status(s.cuda_stream) == (0, 0)
        ref, mag = H.oracle_full(w, Ar, Br, Cr)
        H.assert_match(w, H.logical(dC.cpu().numpy(), w.M, w.N, w.LDC), ref, mag,
                       what=f"replay {r}")
    return binding.sgemm_last_config()


# few tiles and a long K: every tile split along K, partials behind flags
SPLIT = Workload("graphsplit", 256, 512, 9000, 1.25, -0.5, "int3", 91)
WHOLE = Workload("graphwhole", 1000, 1200, 300, 0.5, 3.0, "uniform", 92)


@pytest.mark.parametrize("w", [SPLIT, WHOLE, SPLIT.with_(dist="uniform")], ids=lambda w: w.name + w.dist)
def test_sgemm_graph_replays(w):
    cfg = _replay_and_check(binding.sgemm, w)
    if w is SPLIT:
        assert "split=" in cfg and "split=0" not in cfg


@pytest.mark.parametrize("form", binding.X3_FORMS)
@pytest.mark.parametrize("w", [Workload("x3graph", 300, 700, 3000, 1.25, -0.5, "int3", 93),
                               Workload("x3graphpairs", 128 * 2 * 76 * 2, 256, 64, 1.0, 1.0,
                                        "int3", 94)], ids=lambda w: w.name)
def test_3xtf32_graph_replays(w, form):
    prev = binding.sgemm_3xtf32_set_kernel_form(form)
    try:
        _replay_and_check(binding.sgemm_3xtf32, w, replays=2)
    finally:
        binding.sgemm_3xtf32_set_kernel_form(prev)


def test_batched_graph_replays():
    w = Workload("graphbatch", 96, 160, 4000, 1.0, 1.0, "int3", 95)
    fn = functools.partial(binding.sgemm_strided_batched, binding.SGEMM_OP_N, binding.SGEMM_OP_N)
    batch = 3
    gens = [make_inputs(w.with_(seed=w.seed + i)) for i in range(batch)]
    A = torch.cat([g[0] for g in gens]).cuda()
    B = torch.cat([g[1] for g in gens]).cuda()
    C = torch.cat([g[2] for g in gens]).cuda()
    sA, sB, sC = w.M * w.LDA, w.K * w.LDB, w.M * w.LDC
    s = torch.cuda.Stream()

    def call():
        return fn(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.LDA, sA, B.data_ptr(), w.LDB, sB, w.beta,
                  C.data_ptr(), w.LDC, sC, batch, s.cuda_stream)
    torch.cuda.synchronize()
    assert call() == 0
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert call() == 0
    for r in range(2):
        new = [make_inputs(w.with_(seed=w.seed + 50 + 10 * r + i)) for i in range(batch)]
        A.copy_(torch.cat([x[0] for x in new]))
        B.copy_(torch.cat([x[1] for x in new]))
        C.copy_(torch.cat([x[2] for x in new]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        out = C.cpu().numpy()
        for i, (Ai, Bi, Ci) in enumerate(new):
            ref, mag = H.oracle_full(w, Ai, Bi, Ci)
            H.assert_match(w, H.logical(out[i * sC:(i + 1) * sC], w.M, w.N, w.LDC), ref, mag,
                           what=f"replay {r} matrix {i}")


def test_capture_without_warm_up_is_refused():
    w = Workload("graphcold", 256, 512, 9000, 1.0, 0.0, "int3", 96)
    A, B, C = make_inputs(w)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    # device set-up happens on the first call of the process: do it on another
    # stream, so that only the capturing stream lacks its workspace
    assert binding.sgemm(*_args(w, dA, dB, dC, torch.cuda.current_stream())) == 0
    s = torch.cuda.Stream()  # a stream this process never used: no workspace yet
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = binding.sgemm(*_args(w, dA, dB, dC, s))
    assert st == binding.SGEMM_ERR_CAPTURE
    # the refusal left the process usable: a normal call on that stream works
    assert binding.sgemm(*_args(w, dA, dB, dC, s)) == 0
    s.synchronize()
    ref, mag = H.oracle_full(w, A, B, None)
    H.assert_match(w, H.logical(dC.cpu().numpy(), w.M, w.N, w.LDC), ref, mag)
