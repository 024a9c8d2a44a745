"""Seeded synthetic inputs for the SGEMM workloads.

This module only draws random numbers and fixes shapes; it holds none of the
GEMM arithmetic, so both the CUDA path and the oracle can be fed from it.

Recipe (the pages measure at M = N = K = 4096 and give no data set; these are
the synthetic stand-ins, one seed per workload):
  * generator: ``torch.Generator('cpu').manual_seed(seed)``;
  * draw order: A, then B, then C, each as its full logical matrix;
  * uniform[-1, 1]: ``torch.rand(shape) * 2 - 1``;
  * N(0, 1):        ``torch.randn(shape)``;
  * integers {-3..3}: ``torch.randint(-3, 4, shape)`` converted to float32;
  * everything float32, generated on the host, then copied where it is needed.
A leading dimension larger than the row length leaves padding columns that are
filled with ``pad_value`` (NaN by default in tests, so any read of padding
shows up as a NaN in the result).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dist: str          # "uniform", "normal" or "int3"
    seed: int
    lda: int = 0       # 0 means the natural leading dimension
    ldb: int = 0
    ldc: int = 0

    @property
    def LDA(self) -> int:
        return self.lda or max(self.K, 1)

    @property
    def LDB(self) -> int:
        return self.ldb or max(self.N, 1)

    @property
    def LDC(self) -> int:
        return self.ldc or max(self.N, 1)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


SWEEP_SIZES = (256, 512, 1024, 2048, 4096, 8192, 16384)

# The five workloads: a small square case, the 4096 cube (the throughput
# headline), ragged edges with a leading dimension that is not a multiple of
# four, K-dominant and skinny shapes, and the square sweep.
WORKLOADS = {
    "square128": Workload("square128", 128, 128, 128, 1.0, 0.0, "uniform", 0),
    "square128_int": Workload("square128_int", 128, 128, 128, 1.0, 0.0, "int3", 0),
    "square4096": Workload("square4096", 4096, 4096, 4096, 0.5, 3.0, "uniform", 1),
    "edges8191x1000x777": Workload("edges8191x1000x777", 8191, 1000, 777, 1.25, -0.5, "normal", 2),
    "kdominant1024x1024x16384": Workload("kdominant1024x1024x16384", 1024, 1024, 16384, 1.0, 1.0,
                                         "uniform", 3),
    "skinny16384x64x4096": Workload("skinny16384x64x4096", 16384, 64, 4096, 1.0, 1.0, "uniform", 3),
}
for _n in SWEEP_SIZES:
    WORKLOADS[f"sweep{_n}"] = Workload(f"sweep{_n}", _n, _n, _n, 1.0, 0.0, "uniform", 4)
    WORKLOADS[f"sweep{_n}_int"] = Workload(f"sweep{_n}_int", _n, _n, _n, 1.0, 0.0, "int3", 4)


def integer_variant(w: Workload) -> Workload:
    """Same shape, alpha and beta with entries drawn from {-3..3}: every partial
    sum is an integer of magnitude at most 9*K, so it is exact in FP32 while
    9*K < 2^24."""
    return w.with_(name=w.name + "_int" if not w.name.endswith("_int") else w.name, dist="int3")


def _draw(gen: torch.Generator, rows: int, cols: int, dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand((rows, cols), generator=gen, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn((rows, cols), generator=gen, dtype=torch.float32)
    if dist == "int3":
        return torch.randint(-3, 4, (rows, cols), generator=gen).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def _embed(x: torch.Tensor, ld: int, pad_value: float) -> torch.Tensor:
    rows, cols = x.shape
    if ld == cols:
        return x.reshape(-1).contiguous()
    buf = torch.full((rows, ld), pad_value, dtype=torch.float32)
    buf[:, :cols] = x
    return buf.reshape(-1)


def make_inputs(w: Workload, pad_value: float = float("nan"), with_c: bool = True):
    """Host tensors (A, B, C) for workload ``w`` as flat float32 buffers of
    M*lda, K*ldb and M*ldc elements. C is drawn even when beta == 0 (the draw
    order stays fixed) unless ``with_c`` is False."""
    gen = torch.Generator("cpu").manual_seed(w.seed)
    A = _embed(_draw(gen, w.M, w.K, w.dist), w.LDA, pad_value)
    B = _embed(_draw(gen, w.K, w.N, w.dist), w.LDB, pad_value)
    C = _embed(_draw(gen, w.M, w.N, w.dist), w.LDC, pad_value) if with_c else None
    return A, B, C


def row_sample(M: int, count: int, seed: int):
    """Sorted distinct row indices used for sampled checks at large sizes."""
    gen = torch.Generator("cpu").manual_seed(1000 + seed)
    count = min(count, M)
    return torch.randperm(M, generator=gen)[:count].sort().values.tolist()


def element_sample(M: int, N: int, count: int, seed: int):
    """Random (row, col) pairs used for sampled checks at large sizes."""
    gen = torch.Generator("cpu").manual_seed(2000 + seed)
    r = torch.randint(0, M, (count,), generator=gen)
    c = torch.randint(0, N, (count,), generator=gen)
    return r.tolist(), c.tolist()


# ---- counter-based integer matrices for the largest sizes ----------------------
# A matrix of more than 2^31 elements is too large to draw on the host in one
# piece for every test run, and a sequential generator cannot produce a chosen
# row or column on its own. These matrices are instead a pure function of
# (seed, row, column): element (i, j) of a rows x cols matrix is
#     h = fmix32((idx mod 2^32) xor fmix32((idx div 2^32) xor seed)),  idx = i*cols + j
#     value = (h mod 7) - 3        (an integer in {-3..3})
# where fmix32 is the 32-bit finalizer of MurmurHash3 (Austin Appleby). The
# same torch integer arithmetic runs on the device (the whole matrix, in row
# blocks) and on the host (only the rows or columns a check needs).

_M32 = 0xFFFFFFFF


def fmix32(h: torch.Tensor) -> torch.Tensor:
    """MurmurHash3's 32-bit finalizer on int64 tensors holding values below
    2^32 (products wrap modulo 2^64; only their low 32 bits are kept)."""
    h = h ^ (h >> 16)
    h = (h * 0x85EBCA6B) & _M32
    h = h ^ (h >> 13)
    h = (h * 0xC2B2AE35) & _M32
    return h ^ (h >> 16)


def hashed_int3(seed: int, idx: torch.Tensor) -> torch.Tensor:
    """Values in {-3..3} (float32) of the elements with linear indices `idx`
    (int64, row-major) of a counter-based matrix with this seed."""
    hi = fmix32(((idx >> 32) ^ seed) & _M32)
    h = fmix32((idx & _M32) ^ hi)
    return ((h % 7) - 3).to(torch.float32)


def hashed_int3_rows(seed: int, cols: int, rows, device="cpu") -> torch.Tensor:
    """The listed rows (a list or a range) of a counter-based rows x cols
    matrix, as a len(rows) x cols float32 tensor on `device`."""
    r = torch.as_tensor(list(rows), dtype=torch.int64, device=device)
    j = torch.arange(cols, dtype=torch.int64, device=device)
    return hashed_int3(seed, r[:, None] * cols + j[None, :])


def hashed_int3_cols(seed: int, rows: int, cols: int, col_list, device="cpu") -> torch.Tensor:
    """The listed columns of a counter-based rows x cols matrix, as a
    rows x len(col_list) float32 tensor."""
    i = torch.arange(rows, dtype=torch.int64, device=device)
    c = torch.as_tensor(list(col_list), dtype=torch.int64, device=device)
    return hashed_int3(seed, i[:, None] * cols + c[None, :])


def hashed_int3_device(seed: int, rows: int, cols: int, device="cuda",
                       block_elems: int = 1 << 27) -> torch.Tensor:
    """The whole rows x cols counter-based matrix on `device` (dense,
    row-major), filled in blocks of rows."""
    out = torch.empty((rows, cols), dtype=torch.float32, device=device)
    step = max(1, block_elems // max(cols, 1))
    for r0 in range(0, rows, step):
        out[r0: r0 + step] = hashed_int3_rows(seed, cols, range(r0, min(rows, r0 + step)),
                                              device=device)
    return out
