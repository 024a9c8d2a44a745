"""The counter-based integer matrices used at the largest sizes: the torch
implementation against the published MurmurHash3 fmix32 finalizer written
with Python integers, and the row, column and whole-matrix views agree."""
import random

import torch

from dense_fp32_gemm_gb300.workloads import (fmix32, hashed_int3, hashed_int3_cols,
                                             hashed_int3_device, hashed_int3_rows)


def _fmix32(h):
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    return h ^ (h >> 16)


def test_fmix32_matches_python_integers():
    rng = random.Random(3)
    xs = [0, 1, 2, 0xFFFFFFFF, 0x80000000] + [rng.getrandbits(32) for _ in range(2000)]
    assert fmix32(torch.tensor(xs, dtype=torch.int64)).tolist() == [_fmix32(x) for x in xs]
    assert _fmix32(0) == 0  # the finalizer maps 0 to 0


def test_values_beyond_2_pow_31_and_2_pow_32():
    rng = random.Random(4)
    idx = [0, 2**31 - 1, 2**31, 2**32 - 1, 2**32, 2**33 + 5] + [rng.getrandbits(36) for _ in range(500)]
    seed = 12
    want = [(_fmix32((i & 0xFFFFFFFF) ^ _fmix32(((i >> 32) ^ seed) & 0xFFFFFFFF)) % 7) - 3
            for i in idx]
    assert hashed_int3(seed, torch.tensor(idx, dtype=torch.int64)).tolist() == want


def test_views_agree_and_values_cover_the_range():
    full = hashed_int3_device(5, 37, 53, device="cpu", block_elems=200)
    assert torch.equal(full[[0, 3, 36]], hashed_int3_rows(5, 53, [0, 3, 36]))
    assert torch.equal(full[:, [0, 52, 7]], hashed_int3_cols(5, 37, 53, [0, 52, 7]))
    counts = torch.bincount((full.flatten() + 3).long(), minlength=7)
    assert counts.numel() == 7 and int(counts.min()) > 0.7 * full.numel() / 7
