"""Persistent-schedule invariants, on the host: every (tile, k-slice) unit is
computed exactly once; each tile has exactly one owner (the piece holding its
first k-slice); an owner's contributors are exactly the other pieces of its
tile, each the first split piece of the next CTAs in order and each a partial; no
CTA stores more than one partial; the tile numbering is a bijection onto the
tile grid; and the work per CTA is balanced."""
import itertools

import pytest

from dense_fp32_gemm_gb300 import binding

CASES = [
    (4096, 4096, 4096, 0, 152), (4096, 4096, 4096, 2, 304), (8191, 1000, 777, 0, 152),
    (1024, 1024, 16384, 0, 152), (16384, 64, 4096, 1, 304), (128, 128, 128, 0, 152),
    (256, 512, 9000, 3, 608), (1, 1, 1, 0, 152), (300, 520, 77, 2, 304), (2, 700, 2049, 1, 304),
    (16384, 16384, 16384, 0, 152), (100, 100, 100000, 0, 7), (5000, 5000, 64, 0, 152),
]


def enumerate_pieces(s):
    pieces = {}
    for b in range(s["grid"]):
        n, first = binding.sgemm_schedule_piece(s, b, 0)
        pieces[b] = [first] + [binding.sgemm_schedule_piece(s, b, i)[1] for i in range(1, n)]
    return pieces


@pytest.mark.parametrize("M,N,K,cid,cap", CASES)
def test_schedule_invariants(M, N, K, cid, cap):
    s = binding.sgemm_schedule_query(M, N, K, cid, cap)
    tiles = s["tiles_m"] * s["tiles_n"]
    assert 1 <= s["grid"] <= cap
    pieces = enumerate_pieces(s)
    covered = {}
    coords = {}
    for b, ps in pieces.items():
        assert ps, f"CTA {b} has no work"
        partials = [p for p in ps if p["is_partial"]]
        assert len(partials) <= 1
        split = [p for p in ps if p["tile"] >= s["dp_tiles"]]
        if partials:
            assert split[0]["is_partial"], "a partial must be the CTA's first split piece"
        for p in ps:
            assert 0 <= p["kb"] < p["ke"] <= s["kiters"]
            for k in range(p["kb"], p["ke"]):
                key = (p["tile"], k)
                assert key not in covered, f"unit {key} computed twice"
                covered[key] = b
            coords.setdefault(p["tile"], (p["tile_m"], p["tile_n"]))
            assert coords[p["tile"]] == (p["tile_m"], p["tile_n"])
    assert len(covered) == tiles * s["kiters"]
    assert sorted(coords.values()) == sorted(itertools.product(range(s["tiles_m"]), range(s["tiles_n"])))
    # owners and contributors
    for b, ps in pieces.items():
        for p in ps:
            if p["kb"] != 0:
                continue
            nc = p["contributors"]
            if p["ke"] == s["kiters"]:
                assert nc == 0
                continue
            assert nc >= 1
            k_next = p["ke"]
            for c in range(b + 1, b + nc + 1):
                q = [x for x in pieces[c] if x["tile"] >= s["dp_tiles"]][0]
                assert q["tile"] == p["tile"] and q["is_partial"] == 1 and q["kb"] == k_next
                k_next = q["ke"]
            assert k_next == s["kiters"], "contributors do not complete the tile"
    # balance: whole tiles differ by at most one per CTA, split units by one
    dp = [sum(1 for p in ps if p["tile"] < s["dp_tiles"]) for ps in pieces.values()]
    assert max(dp) - min(dp) <= 1
    sk = [sum(p["ke"] - p["kb"] for p in ps if p["tile"] >= s["dp_tiles"]) for ps in pieces.values()]
    assert max(sk) - min(sk) <= 1


def test_split_is_used_where_waves_are_ragged():
    s = binding.sgemm_schedule_query(4096, 4096, 4096, 0, 152)
    assert s["tiles_m"] * s["tiles_n"] == 512 and s["grid"] == 152
    assert s["dp_tiles"] == 304  # two whole waves; the last 208 tiles are split
    s = binding.sgemm_schedule_query(4096, 4096, 4096, 0, 128)
    assert s["dp_tiles"] == 512  # 512 tiles on 128 slots: whole waves, no split
