"""Host-side logic on the CPU: the binding refuses to run without its compiled
library (no fallback path exists), and the bench's DRAM-traffic figure is
reported only for the kernel sources it was measured on."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from speculative_decoding_moe_gb300 import dfv
    monkeypatch.setattr(dfv, "LIB_PATH", str(tmp_path / "libdfv.so"))
    monkeypatch.setattr(dfv, "_lib", None)
    with pytest.raises(ImportError, match="not built"):
        dfv._load()


def test_ncu_traffic_is_keyed_by_the_kernel_sources(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    name = "moe_fused_kernel"
    h = bench.kernel_hash(name)
    assert len(h) == 16 and int(h, 16) >= 0
    # the capture's bytes scale with the algorithmic bytes of the launch
    monkeypatch.setitem(bench.NCU_TRAFFIC, name, (h, 1000.0, 500.0))
    assert bench.ncu_traffic(name, 250.0) == 500.0
    # an edited kernel (another hash) reports no traffic rather than a stale one
    monkeypatch.setitem(bench.NCU_TRAFFIC, name, ("0" * 16, 1000.0, 500.0))
    assert bench.ncu_traffic(name, 250.0) is None
    assert bench.ncu_traffic("no_such_kernel", 250.0) is None


def test_peaks_come_from_the_measured_file():
    sys.path.insert(0, ROOT)
    import bench
    peaks, kind = bench.load_peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured"
        assert peaks["hbm_gbs"] > 1000
    else:
        assert kind == "fallback"


def test_cpu_baseline_reports_all_threads_one_thread_and_k1():
    sys.path.insert(0, ROOT)
    import bench
    line = bench.cpu_baseline_line(0.05)
    assert line["kind"] == "oracle" and line["unit"] == "GB/s"
    assert line["cores"] == bench.host_threads() and line["value"] > 0
    side = line["also"]
    assert side["k16_1thread"]["threads"] == 1 and side["k16_1thread"]["k"] == bench.KBLOCK
    assert side["k1_all_threads"]["k"] == 1 and side["k1_all_threads"]["threads"] == line["cores"]
    assert side["k1_1thread"]["threads"] == 1 and side["k1_1thread"]["k"] == 1
    assert all(side[n]["calls"] >= 1 and side[n]["value"] > 0 for n in ("k16_1thread", "k1_all_threads", "k1_1thread"))
    for n in ("stack_bf16", "stack_mxfp4"):
        st = side[n]
        assert st["layers_timed"] == 2 and st["tau"] == bench.KBLOCK + 1  # every planted draft token matches
        assert st["stack40_accept_ms_extrapolated"] == pytest.approx(20 * st["stack_ms"] + st["accept_ms"])


def test_spread_is_per_layer_percentiles():
    sys.path.insert(0, ROOT)
    import bench
    per_step_ms = [4.0, 5.0, 6.0, 5.5, 5.2, 4.8, 5.1, 5.0, 4.9, 7.0]  # 40-layer steps
    s = bench.spread_us(per_step_ms, 40)
    assert s["steps"] == 10
    assert s["median"] == pytest.approx(126.25)       # (5.0 + 5.1) / 2 ms over 40 layers, in µs
    assert s["p10"] == pytest.approx(120.0) and s["p90"] == pytest.approx(150.0)
    assert s["p10"] <= s["median"] <= s["p90"]
