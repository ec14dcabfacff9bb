"""CPU tests of bench.py's host logic: the clock sampler's parsing and timed
window, and the rule that a profiled DRAM-traffic figure is used only when it
was taken on the current kernel source."""
from __future__ import annotations

import os
import tempfile
import time

import bench


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _row(ts, sm, reasons=("Not Active",) * 4):
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(int(ts))) + f".{int((ts % 1) * 1000):03d}"
    return ", ".join(["0", str(sm), "2070", "900.0", "0x0", *reasons, stamp])


def _sampler_with(rows):
    s = bench.ClockSampler(0)
    s.window = None
    s.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.file.write("\n".join(rows) + "\n")
    s.file.flush()
    s.proc = _FakeProc()
    return s


def test_clock_sampler_keeps_the_timed_window():
    t0 = time.time() + 100.0  # a window in whole seconds away from the idle samples
    t0 = float(int(t0))
    rows = [_row(t0 - 2.0, 1200, ("Not Active", "Not Active", "Not Active", "Active")),  # idle, capped
            _row(t0 + 0.002, 2070), _row(t0 + 0.010, 2055),
            _row(t0 + 3.0, 990, ("Active", "Not Active", "Not Active", "Not Active"))]     # after the window
    s = _sampler_with(rows)
    s.mark(t0, t0 + 0.012)
    c = s.stop()
    assert c["samples_in_timed_region"] == 2 and c["samples"] == 2
    assert c["sm_mhz"] == (2070 + 2055) / 2 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == []  # reasons outside the window do not count


def test_clock_sampler_reports_reasons_inside_the_window():
    t0 = float(int(time.time()) + 200)
    rows = [_row(t0 + 0.005, 1800, ("Active", "Not Active", "Active", "Not Active"))]
    s = _sampler_with(rows)
    s.mark(t0, t0 + 0.010)
    c = s.stop()
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_samples_or_tool():
    s = bench.ClockSampler(0)
    assert s.stop() is None  # nvidia-smi never started
    s = _sampler_with(["garbage", ""])
    s.mark(0.0, 1.0)
    assert s.stop() is None


def test_profiled_traffic_needs_the_current_kernel_source(monkeypatch):
    with tempfile.TemporaryDirectory() as root:
        csrc = os.path.join(root, "transformer_scaled_dot_fwd_gb300", "csrc")
        os.makedirs(csrc)
        os.makedirs(os.path.join(root, "profiles"))
        for f, text in (("k.cu", "kernel v1"), ("ptx.cuh", "helpers"), ("kernels.h", "decls")):
            with open(os.path.join(csrc, f), "w") as fh:
                fh.write(text)
        monkeypatch.setattr(bench, "ROOT", root)
        digest = bench.kernel_source_digest("k.cu")
        with open(os.path.join(root, "profiles", "p.md"), "w") as fh:
            fh.write(f"kernel_source_digest: {digest}\ndram_bytes_per_launch: 123456\n")
        assert bench.profiled_traffic("p.md", "k.cu") == 123456.0
        with open(os.path.join(csrc, "k.cu"), "w") as fh:
            fh.write("kernel v2")  # the kernel changed after the capture
        assert bench.profiled_traffic("p.md", "k.cu") is None
        assert bench.profiled_traffic("missing.md", "k.cu") is None
