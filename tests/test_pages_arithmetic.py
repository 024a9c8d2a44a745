"""The throughput and traffic accounting used by the benchmark, checked
against the numbers the pages print (tests/golden/pages_analytic.json)."""
import json
import os

import pytest

import bench

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_analytic.json")))


def test_flop_count_4096():
    assert bench.gemm_flops(4096, 4096, 4096) / 1e9 == pytest.approx(G["flops_4096"]["gflop"], abs=0.005)


@pytest.mark.parametrize("ms,gflops", G["timings_to_rate"]["cases"])
def test_rate_from_time(ms, gflops):
    assert bench.gflops(4096, 4096, 4096, ms / 1e3) == pytest.approx(gflops, rel=2e-4)


def test_gmem_accesses_per_result():
    g = G["gmem_accesses_per_result"]
    for BM, BN, want in g["cases"]:
        assert bench.gmem_accesses_per_result(g["K"], BM, BN) == pytest.approx(want)


def test_smem_loads_per_result():
    g = G["smem_loads_per_result"]
    TM, TN = g["thread_tile"]
    assert bench.smem_loads_per_result(g["K"], TM, TN) == pytest.approx(g["value"])


def test_smem_tiling_loads_per_cell():
    g = G["smem_tiling_loads_per_cell"]
    assert bench.gmem_accesses_per_result(g["K"], 1, 1) / 1 == pytest.approx(2 * g["K"])
    assert 2 * g["K"] == g["before"]
    assert bench.gmem_accesses_per_result(g["K"], g["tile"], g["tile"]) == pytest.approx(g["after"])
