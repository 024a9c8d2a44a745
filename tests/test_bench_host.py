"""bench.py's host-side accounting (no GPU): the FFMA peak and algorithmic
bytes, the committed ncu traffic lookup and the conditions under which it is
withheld, per-step statistics, the 3xTF32 roof choice, the clock samplers
(NVML through a fake library, nvidia-smi lines) and their timed-window
summaries, and the result check that backs the line's `verified`."""
import ctypes
import datetime as dt
import json
import os

import numpy as np
import pytest

import bench


def test_ffma_peak_and_algorithmic_bytes():
    assert bench.ffma_peak_tflops(152, 2070.0) == pytest.approx(80.548, abs=1e-3)
    # square 4096, beta != 0: A, B and C read once, C written once
    assert bench.min_bytes(4096, 4096, 4096, 3.0) == 4 * 4096 * 4096 * 4
    assert bench.min_bytes(4096, 4096, 4096, 0.0) == 4 * 4096 * 4096 * 3


def test_kernel_source_hash_is_stable():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert h == bench.kernel_source_hash()


def _committed(workload):
    table = json.load(open(bench.TRAFFIC_PATH))
    return table["ffma_sgemm"][workload]


@pytest.mark.parametrize("workload", ["square4096", "edges8191x1000x777", "kdominant1024x1024x16384",
                                      "skinny16384x64x4096"])
def test_profiled_traffic_follows_the_committed_figures(workload, monkeypatch):
    f = _committed(workload)
    # the figure is used while the kernel sources hash as they did at the capture
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: f["kernel_source_sha"])
    tile = f["tile_config"]
    assert bench.profiled_traffic(workload, tile + " a=rowT b=tma") == float(f["dram_bytes_per_launch"])
    # another tile configuration, or changed kernel sources: no figure
    assert bench.profiled_traffic(workload, "SomeOtherConfig_1x1") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic(workload, tile) is None


def test_profiled_traffic_unknown_workload_or_missing_file(tmp_path):
    assert bench.profiled_traffic("no_such_workload", "WideBk32F2Ku32") is None
    assert bench.profiled_traffic("square4096", "WideBk32F2Ku32", path=str(tmp_path / "none.json")) is None
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    assert bench.profiled_traffic("square4096", "WideBk32F2Ku32", path=str(bad)) is None


def test_committed_summaries_name_the_same_capture():
    # each workload's prose summary shows the identity its JSON entry holds
    table = json.load(open(bench.TRAFFIC_PATH))["ffma_sgemm"]
    for workload, e in table.items():
        text = open(os.path.join(bench.ROOT, e["summary"])).read()
        assert e["kernel_source_sha"] in text and e["tile_config"] in text, workload
        assert str(e["dram_bytes_per_launch"]) in text, workload


def test_step_stats():
    st = bench.step_stats([2.0, 2.1, 1.9, 2.4])
    assert st["n"] == 4 and st["min"] == 1.9 and st["max"] == 2.4
    assert st["median"] == pytest.approx(2.05) and st["mean"] == pytest.approx(2.1)
    assert st["spread_pct"] == pytest.approx(100 * 0.5 / 2.05, abs=0.01)
    assert bench.step_stats([3.0])["spread_pct"] == 0.0
    assert bench.step_stats([]) is None


class _FakeBinding:
    def __init__(self, single, pair):
        self.single, self.pair, self.calls = single, pair, []

    def sgemm_diag_tf32_mma_rate(self, iters):
        self.calls.append("single")
        return self.single

    def sgemm_diag_tf32_pair_mma_rate(self, iters):
        self.calls.append("pair")
        return self.pair


def test_tf32x3_roof_takes_the_probe_of_the_form_that_ran():
    b = _FakeBinding((0, 1200.0), (0, 1230.0))
    roof, basis, measured = bench.tf32x3_roof(b, {}, pair=True)
    assert (roof, measured, b.calls) == (410.0, 1230.0, ["pair"])
    assert "cta_group::2" in basis
    roof, basis, measured = bench.tf32x3_roof(b, {}, pair=False)
    assert (roof, measured, b.calls[-1]) == (400.0, 1200.0, "single")


def test_tf32x3_roof_falls_back_to_the_bf16_estimate():
    b = _FakeBinding((-6, 0.0), (-6, 0.0))
    roof, basis, measured = bench.tf32x3_roof(b, {"bf16_tflops": 2250.0}, pair=True)
    assert measured is None and roof == pytest.approx(2250.0 * 1.1 / 2.25 / 3)
    assert bench.tf32x3_roof(b, {}, pair=False)[0] is None


def _sampler_with(tmp_path, lines):
    s = object.__new__(bench.ClockSampler)
    s.proc = object()  # a sampler that ran
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def _line(t, mhz, reasons=("Not Active",) * 4):
    ts = t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, str(mhz), "2070", "900.00 W", "0x0"] + list(reasons))


def test_clock_summary_within_the_timed_window(tmp_path):
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line(t0 - dt.timedelta(seconds=5), 1000)]                 # before: ignored
    lines += [_line(t0 + dt.timedelta(milliseconds=100 * i), m) for i, m in enumerate([2070, 2055, 2070])]
    lines += [_line(t0 + dt.timedelta(seconds=5), 900,                   # after: ignored
                    ("Not Active", "Active", "Not Active", "Not Active"))]
    lines += ["garbage line"]
    s = _sampler_with(tmp_path, lines)
    out = s.summary(t0.timestamp() - 0.01, (t0 + dt.timedelta(seconds=1)).timestamp())
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": []}


def test_clock_summary_reports_throttle_reasons(tmp_path):
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line(t0, 1800, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + dt.timedelta(milliseconds=100), 1700, ("Active", "Not Active", "Not Active", "Active"))]
    s = _sampler_with(tmp_path, lines)
    out = s.summary(t0.timestamp() - 1, t0.timestamp() + 1)
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert out["sm_mhz"] == 1800.0 and out["samples"] == 2


def test_clock_summary_without_a_sampler():
    s = object.__new__(bench.ClockSampler)
    s.proc = None
    assert s.summary(0, 1)["reasons"] == ["nvidia-smi unavailable"]


# ---- NVML sampler, through a fake libnvidia-ml ---------------------------------------
class _FakeNvml:
    """Answers the NVML calls the sampler makes; clocks and reason bits come
    from the lists given, one per poll."""

    def __init__(self, clocks, reasons, max_mhz=2070):
        self.clocks, self.reasons, self.max_mhz, self.i = list(clocks), list(reasons), max_mhz, 0
        self.calls = []

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByPciBusId_v2(self, bus, h):
        self.calls.append(("bus", bus))
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, idx, h):
        self.calls.append(("index", idx.value))
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = self.max_mhz
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        assert kind == bench.NVML_CLOCK_SM
        out._obj.value = self.clocks[self.i % len(self.clocks)]
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = self.reasons[self.i % len(self.reasons)]
        self.i += 1
        return 0


def test_nvml_sampler_reads_clock_and_reasons():
    nv = _FakeNvml([2070, 1800], [0x0, 0x4 | 0x8])
    s = bench.NvmlClockSampler(pci_bus_id="00000000:1b:00.0", lib=nv)
    assert s.lib is nv and s.max_mhz == 2070.0 and nv.calls == [("bus", b"00000000:1b:00.0")]
    a, b = s.poll(), s.poll()
    assert a[1:] == (2070.0, 0) and b[1:] == (1800.0, 0xC)
    s.samples = [a, b]
    out = s.summary(a[0] - 1, b[0] + 1)
    assert out["samples"] == 2 and out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert out["sm_mhz"] == pytest.approx(1935.0) and out["sm_max_mhz"] == 2070.0
    assert out["source"] == "nvml"


def test_nvml_sampler_by_index_and_without_library():
    nv = _FakeNvml([2070], [0])
    bench.NvmlClockSampler(index=3, lib=nv)
    assert nv.calls == [("index", 3)]

    class _Broken:
        def nvmlInit_v2(self):
            return 1
    s = bench.NvmlClockSampler(lib=_Broken())
    assert s.lib is None
    out = s.summary(0, 1)
    assert out["sm_mhz"] is None and out["reasons"][0].startswith("NVML unavailable")


def test_nvml_sampler_thread_collects_samples():
    import time
    nv = _FakeNvml([2070], [0])
    s = bench.NvmlClockSampler(lib=nv, period_s=0.001).start()
    t0 = time.time()
    time.sleep(0.05)
    t1 = time.time()
    s.stop()
    out = s.summary(t0, t1)
    assert out["samples"] >= 5 and out["sm_mhz"] == 2070.0


def test_clock_summary_counts_only_the_window():
    samples = [(0.5, 1000.0, 0x8), (1.0, 2070.0, 0), (1.5, 2060.0, 0x4), (2.0, 2070.0, 0), (9.0, 900.0, 0x40)]
    out = bench.summarize_clock_samples(samples, 1.0, 2.0, 2070.0, "nvml")
    assert out["samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_mhz_min"] == 2060.0
    assert out["reasons"] == ["sw_power_cap"]
    none = bench.summarize_clock_samples(samples, 3.0, 4.0, 2070.0, "nvml")
    assert none["samples"] == 0 and none["sm_mhz"] is None


def test_nvml_bus_id_format():
    class P:
        pci_domain_id, pci_bus_id, pci_device_id = 0, 0x1B, 0
    assert bench.nvml_bus_id(P()) == "00000000:1b:00.0"
    assert bench.nvml_bus_id(object()) is None


# ---- the check behind `verified` -------------------------------------------------------
def test_check_against_reference_tolerance_and_exactness():
    ref = np.array([1.0, -2.0, 3.0])
    mag = np.array([10.0, 10.0, 10.0])
    ok, worst, bad = bench.check_against_reference(ref + [5e-5, -9e-5, 0], ref, mag, exact=False)
    assert ok and bad == 0 and worst == pytest.approx(0.9)
    ok, worst, bad = bench.check_against_reference(ref + [2e-4, 0, 0], ref, mag, exact=False)
    assert not ok and bad == 1
    # integer inputs: any difference fails, even inside the tolerance
    ok, _, bad = bench.check_against_reference(ref + [5e-5, 0, 0], ref, mag, exact=True)
    assert not ok and bad == 1
    ok, _, _ = bench.check_against_reference(np.array([1.0, np.nan, 3.0]), ref, mag, exact=False)
    assert not ok


def test_verify_sample_catches_a_wrong_element():
    import torch

    import oracle
    from dense_fp32_gemm_gb300.workloads import Workload, make_inputs
    w = Workload("vtest", 40, 24, 17, 1.25, -0.5, "int3", 5)
    A, B, C = make_inputs(w)
    ref, mag = oracle.sgemm_rows(w.M, w.N, w.K, w.alpha, A.numpy(), w.LDA, B.numpy(), w.LDB, w.beta,
                                 C.numpy(), w.LDC)
    good = np.zeros(w.M * w.LDC, dtype=np.float32)
    good.reshape(w.M, w.LDC)[:, :w.N] = ref.astype(np.float32)
    rows = (ref[:8], mag[:8])
    out = bench.verify_sample(w, A, B, C, {"ffma": good}, rows, n_elements=64)
    assert out["ffma"]["ok"] and out["ffma"]["rows_checked"] == 8 and out["ffma"]["bit_exact_required"]
    bad = good.copy()
    bad[(w.M - 1) * w.LDC + w.N - 1] += 1.0   # the last element is always sampled
    out = bench.verify_sample(w, A, B, C, {"ffma": bad}, rows, n_elements=64)
    assert not out["ffma"]["ok"] and out["ffma"]["mismatches"] >= 1
