"""Persistent-schedule invariants, on the host: every (tile, k-slice) unit is
computed exactly once; each tile has exactly one owner (the piece holding its
first k-slice); an owner's contributors are exactly the other pieces of its
tile, each the first split piece of the next CTAs in order and each a partial; no
CTA stores more than one partial; the tile numbering is a bijection onto the
tile grid; and the work per CTA is balanced -- for every schedule policy."""
import itertools

import pytest

from dense_fp32_gemm_gb300 import binding

# (M, N, K, BM, BN, BK, capacity): the named workloads and edge cases on the
# tile shapes the configurations use
SHAPES = [
    (4096, 4096, 4096, 128, 256, 32, 152), (4096, 4096, 4096, 128, 128, 32, 304),
    (8191, 1000, 777, 128, 256, 32, 152), (1024, 1024, 16384, 128, 256, 32, 152),
    (16384, 64, 4096, 256, 64, 16, 304), (128, 128, 128, 128, 256, 32, 152),
    (256, 512, 9000, 128, 64, 16, 608), (1, 1, 1, 128, 256, 32, 152), (300, 520, 77, 128, 128, 16, 304),
    (2, 700, 2049, 64, 256, 24, 304), (16384, 16384, 16384, 128, 256, 32, 152),
    (100, 100, 100000, 128, 256, 16, 7), (5000, 5000, 64, 128, 256, 32, 152),
    (1024, 1024, 1024, 128, 256, 32, 152), (512, 512, 512, 128, 64, 32, 304),
]
H, HT, DP, SK, SPK = (binding.SCHED_HYBRID, binding.SCHED_HYBRID_TAIL, binding.SCHED_DATA_PARALLEL,
                      binding.SCHED_STREAM_K, binding.SCHED_SPLIT_K)
POLICIES = [(H, 8, 4, 1), (H, 1, 1, 1), (HT, 8, 4, 1), (HT, 4, 2, 1), (DP, 8, 4, 1), (DP, 16, 4, 1),
            (SK, 8, 4, 1), (SK, 8, 1, 1), (SPK, 8, 4, 2), (SPK, 4, 4, 3), (SPK, 8, 4, 8), (SPK, 8, 4, 1)]
CASES = [shape + (pol,) for shape in SHAPES for pol in POLICIES]


def enumerate_pieces(s):
    pieces = {}
    for b in range(s["grid"]):
        n, first = binding.sgemm_schedule_piece(s, b, 0)
        pieces[b] = [first] + [binding.sgemm_schedule_piece(s, b, i)[1] for i in range(1, n)]
    return pieces


@pytest.mark.parametrize("M,N,K,BM,BN,BK,cap,policy", CASES)
def test_schedule_invariants(M, N, K, BM, BN, BK, cap, policy):
    s = binding.sgemm_schedule_plan(M, N, K, BM, BN, BK, cap, policy)
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
    hybrid = (H, 8, 4, 1)
    s = binding.sgemm_schedule_plan(4096, 4096, 4096, 128, 128, 32, 152, hybrid)
    assert s["tiles_m"] * s["tiles_n"] == 1024 and s["grid"] == 152
    assert s["dp_tiles"] == 760  # five whole waves; the last 264 tiles (1.7 waves) are split
    s = binding.sgemm_schedule_plan(4096, 4096, 4096, 128, 256, 32, 152, hybrid)
    assert s["dp_tiles"] == 304  # two whole waves; the last 208 tiles are split
    s = binding.sgemm_schedule_plan(4096, 4096, 4096, 128, 256, 32, 128, hybrid)
    assert s["dp_tiles"] == 512  # 512 tiles on 128 slots: whole waves, no split


def test_each_policy_decomposes_as_documented():
    # 8191 x 1000 x 777 on 128 x 256 x 32 tiles: 64 x 4 = 256 tiles, 25 k-slices, 152 slots
    def plan(pol):
        return binding.sgemm_schedule_plan(8191, 1000, 777, 128, 256, 32, 152, pol)
    assert (plan((H, 8, 4, 1))["dp_tiles"], plan((H, 8, 4, 1))["grid"]) == (0, 152)
    t = plan((HT, 8, 4, 1))          # one whole wave, the 104 tiles of the last wave split
    assert (t["dp_tiles"], t["grid"]) == (152, 152)
    d = plan((DP, 8, 4, 1))
    assert (d["dp_tiles"], d["grid"], d["sk_q"], d["sk_r"]) == (256, 152, 0, 0)
    s = plan((SK, 8, 4, 1))          # every tile split, 6400 units over 152 CTAs
    assert (s["dp_tiles"], s["grid"], s["sk_q"], s["sk_r"]) == (0, 152, 42, 16)
    # 1024^3 on 128 x 256 x 32: 32 tiles of 32 k-slices
    k = binding.sgemm_schedule_plan(1024, 1024, 1024, 128, 256, 32, 152, (SPK, 8, 4, 4))
    assert (k["dp_tiles"], k["grid"], k["sk_q"], k["sk_r"]) == (0, 128, 8, 0)   # 4 k-ranges of 8
    k = binding.sgemm_schedule_plan(1024, 1024, 1024, 128, 256, 32, 152, (SPK, 8, 4, 8))
    assert k["grid"] == 152                                                   # capped at the slots
    g = binding.sgemm_schedule_plan(4096, 4096, 4096, 128, 256, 32, 152, (DP, 16, 4, 1))
    assert g["group_m"] == 16


def test_policy_argument_errors():
    for bad in [(5, 8, 4, 1), (-2, 8, 4, 1), (H, 0, 4, 1), (H, 8, 0, 1), (SPK, 8, 4, 0)]:
        with pytest.raises(binding.SgemmError):
            binding.sgemm_schedule_plan(64, 64, 64, 64, 64, 16, 152, bad)
        # a negative mode restores the tuned policy; any other bad field is refused
        want = 0 if bad[0] < 0 else binding.SGEMM_ERR_INVALID_VALUE
        assert binding.sgemm_force_schedule(bad) == want
    assert binding.sgemm_force_schedule(None) == 0


def test_forced_policy_reaches_the_schedule_query():
    cid, _ = binding.sgemm_choose_config(4096, 4096, 4096)
    st, auto = binding.sgemm_choose_policy(4096, 4096, 4096)
    assert st == 0 and 0 <= auto[0] < len(binding.SCHED_MODES)
    assert binding.sgemm_force_schedule((DP, 16, 4, 1)) == 0
    try:
        q = binding.sgemm_schedule_query(4096, 4096, 4096, cid, 152)
        assert q["dp_tiles"] == q["tiles_m"] * q["tiles_n"] and q["group_m"] == 16
    finally:
        assert binding.sgemm_force_schedule(None) == 0
    q = binding.sgemm_schedule_query(4096, 4096, 4096, cid, 152)
    prm = binding.sgemm_config_info(cid)[1]
    BM, BN, BK = prm["BM"], prm["BN"], prm["BK"]
    assert q == binding.sgemm_schedule_plan(4096, 4096, 4096, BM, BN, BK, 152, auto)
