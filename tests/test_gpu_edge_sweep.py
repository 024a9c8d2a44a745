"""Every size from 1 to 67 on each dimension in turn (the others 67), against
the oracle, bit-exact on integer inputs: the automatic path (the small-problem
kernel at these sizes), the persistent kernel with the square-4096 tile
configuration forced (one ragged tile of 128 x 256 on every edge, a ragged
k-slice for every K), and the 3xTF32 path. Each case also rotates the pointer
offset (0-3 floats) and the padding of the leading dimensions, so 4-byte
alignment and every residue of lda, ldb, ldc modulo 4 occur; padding holds NaN
and C's guard bands must stay untouched."""
import pytest

from dense_fp32_gemm_gb300 import binding
from dense_fp32_gemm_gb300.workloads import Workload

import gpu_helpers as H

pytestmark = pytest.mark.gpu
EDGE = 67
CASES = [(d, EDGE, EDGE) for d in range(1, EDGE + 1)] + \
        [(EDGE, d, EDGE) for d in range(1, EDGE + 1)] + \
        [(EDGE, EDGE, d) for d in range(1, EDGE + 1)]
PATHS = ["auto", "persistent", "tf32x3"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("shape", CASES, ids=lambda s: "x".join(map(str, s)))
def test_edge_sizes(shape, path):
    M, N, K = shape
    i = CASES.index(shape)
    pad = i % 4
    w = Workload("edge", M, N, K, 1.25, -0.5, "int3", 60 + i % 7,
                 lda=K + pad, ldb=N + (pad + 1) % 4, ldc=N + (pad + 2) % 4)
    offsets = (i % 4, (i + 1) % 4, (i + 2) % 4)
    if path == "tf32x3":
        H.check_against_oracle(w, offsets=offsets, fn=binding.sgemm_3xtf32)
    else:
        config = None if path == "auto" else binding.sgemm_choose_config(4096, 4096, 4096)[0]
        H.check_against_oracle(w, offsets=offsets, config=config)
        if path == "auto":
            assert binding.sgemm_last_config().startswith("tiny_")
