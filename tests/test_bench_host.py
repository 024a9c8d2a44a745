"""bench.py's host-side accounting (no GPU): the FFMA peak and algorithmic
bytes, the committed ncu traffic lookup and the conditions under which it is
withheld, the 3xTF32 roof choice, and the clock summary's parsing of sampled
nvidia-smi lines (median clock, throttle reasons, the timed window)."""
import datetime as dt

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
    text = open(f"{bench.ROOT}/profiles/ffma_sgemm_{workload}.md").read()
    fields = dict(line.strip().split(": ", 1) for line in text.splitlines()
                  if line.strip().startswith(("kernel_source_sha:", "tile_config:",
                                              "dram_bytes_per_launch:")))
    return fields


@pytest.mark.parametrize("workload", ["square4096", "edges8191x1000x777", "kdominant1024x1024x16384",
                                      "skinny16384x64x4096"])
def test_profiled_traffic_follows_the_committed_summary(workload, monkeypatch):
    f = _committed(workload)
    # the figure is used while the kernel sources hash as they did at the capture
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: f["kernel_source_sha"])
    tile = f["tile_config"]
    assert bench.profiled_traffic(workload, tile + " a=rowT b=tma") == float(f["dram_bytes_per_launch"])
    # another tile configuration, or changed kernel sources: no figure
    assert bench.profiled_traffic(workload, "SomeOtherConfig_1x1") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic(workload, tile) is None


def test_profiled_traffic_unknown_workload():
    assert bench.profiled_traffic("no_such_workload", "WideBk32F2Ku32") is None


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
