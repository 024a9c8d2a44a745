"""The tile-configuration legality checker, on the host.

Worked values from "Warp Tiling: A Third Level of Tiling": for the sweep
winner (BM, BN, BK, WM, WN, WNITER, TM, TN, threads) = (128, 64, 16, 64, 32,
2, 4, 4, 128) the page derives WMITER = (64*32)/(32*4*4*2) = 2 (section "The
Warp Tile Is Not Contiguous Either"), sub-tiles of WSUBM x WSUBN = 32 x 16
laid out as an 8 x 4 grid of lanes, and 2*4*2*4 = 64 accumulators per thread
("Mechanics" 2). Those values are stored in tests/golden/pages_analytic.json
with their citations.
"""
import json
import os

import pytest

from dense_fp32_gemm_gb300 import binding

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_analytic.json")))


def P(BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES=3, MINB=1, KU=4, ORDER=0):
    return [BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES, MINB, KU, ORDER]


def test_pages_winner_derived_values():
    g = GOLDEN["warp_tiling_winner"]
    rule, d = binding.sgemm_cfg_check(P(*g["params"]))
    assert rule == 0
    assert d["WMITER"] == g["WMITER"]
    assert d["WSUBM"] == g["WSUBM"] and d["WSUBN"] == g["WSUBN"]
    assert d["acc"] == g["accumulators"]
    lanes_m, lanes_n = d["WSUBM"] // 4, d["WSUBN"] // 4
    assert [lanes_m, lanes_n] == g["lane_grid"]


def test_default_config_derived_values():
    rule, d = binding.sgemm_cfg_check(P(128, 256, 16, 64, 64, 2, 4, 4, 256, 4, 1, 4, 0))
    assert rule == 0 and d["WMITER"] == 4 and d["acc"] == 128


# One tuple per rule, each breaking exactly the assumption that rule guards.
BAD = [
    (P(128, 64, 16, 64, 32, 2, 4, 4, 0), 1),          # no threads
    (P(128, 64, 16, 64, 32, 2, 4, 4, 100), 2),        # not whole warps
    (P(128, 64, 16, 48, 32, 2, 4, 4, 128), 3),        # warp tile does not divide BM
    (P(128, 64, 16, 64, 32, 2, 4, 4, 256), 4),        # warps != warp tiles
    (P(128, 64, 16, 64, 32, 3, 4, 4, 128), 5),        # WMITER not whole
    (P(128, 64, 16, 64, 32, 8, 4, 4, 128), 5),        # WMITER would be 1/2
    (P(128, 128, 16, 64, 24, 1, 4, 4, 256, 3, 1), 3),
    (P(64, 64, 16, 64, 64, 1, 4, 1, 32), 8),          # WSUBM = 2 is not a multiple of TM
    (P(64, 64, 16, 32, 32, 1, 4, 2, 128), 10),        # TN not a multiple of 4
    (P(128, 64, 4, 64, 32, 2, 4, 4, 128), 11),        # BK not a multiple of 8
    (P(32, 512, 16, 32, 32, 1, 4, 4, 512, 3, 1), 12), # BM not a multiple of NT/8
    (P(128, 512, 8, 64, 64, 2, 4, 4, 512, 3, 1), 13), # BN beyond one TMA box
    (P(128, 64, 16, 64, 32, 2, 4, 4, 128, 2, 1), 16), # two stages
    (P(128, 256, 64, 64, 64, 2, 4, 4, 256, 4, 1), 17),# shared memory per CTA
    (P(128, 256, 16, 64, 64, 2, 4, 4, 256, 6, 2), 18),# shared memory per SM
    (P(256, 128, 16, 128, 64, 2, 4, 4, 128, 3, 1), 19),# 256 accumulators
    (P(128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 5), 21), # register file at 5 CTAs/SM
    (P(128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 1, 3), 22),  # odd unroll chunk
    (P(128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 1, 32), 22), # chunk deeper than BK
]


@pytest.mark.parametrize("params,rule", BAD, ids=[str(r) for _, r in BAD])
def test_illegal_tuples_name_their_rule(params, rule):
    assert binding.sgemm_cfg_check(params)[0] == rule


def test_no_division_by_zero_on_degenerate_tuples():
    for bad in ([0] * 13, [1] * 13, [128, 64, 16, 0, 0, 0, 0, 0, 128, 3, 1, 4, 0],
                [-128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 1, 4, 0],
                [128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 1, 4, 4]):
        assert binding.sgemm_cfg_check(bad)[0] != 0
