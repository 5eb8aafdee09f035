"""Host-side pieces of bench.py on CPU: the clock sampler's summary over the timed window (median
SM clock, throttle reasons seen, an empty record), the measured-peak loaders and the source hash
that ties a recorded DRAM-traffic figure to the kernel sources it was measured on."""
import json

import bench


def _row(t, sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", pc="Not Active"):
    return (t, [str(sm), str(mx), hw, hwt, swt, pc])


def test_clock_summary_takes_the_timed_window():
    s = bench.ClockSampler(0)
    s.samples = [_row(0.0, 990, 2070, pc="Active"), _row(1.0, 2070, 2070), _row(2.0, 2055, 2070),
                 _row(3.0, 2070, 2070), _row(9.0, 1200, 2070, hwt="Active")]
    s.window = (0.5, 3.5)
    out = s.summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == [] and out["samples"] == 3
    s.window = None
    out = s.summary()
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"] and out["samples"] == 5


def test_clock_summary_without_samples():
    out = bench.ClockSampler(0).summary()
    assert out["sm_mhz"] is None and out["reasons"] == ["unsampled"] and out["samples"] == 0


def test_peaks_come_from_the_measured_file_when_present():
    gbs, kind = bench.load_peaks()
    tf, tkind = bench.load_tensor_peak()
    try:
        with open(bench.os.path.join(bench.ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
    except FileNotFoundError:
        assert (gbs, kind) == (6800.0, "fallback") and tkind == "fallback"
        return
    assert kind == "measured" and gbs == float(d["hbm_gbs"])
    if "bf16_tflops" in d:
        assert tf == float(d["bf16_tflops"]) and tkind.startswith("measured")


def test_source_hash_follows_the_bytes(tmp_path, monkeypatch):
    a, b = tmp_path / "a.cu", tmp_path / "b.cuh"
    a.write_text("kernel one")
    b.write_text("header")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.source_hash(["a.cu", "b.cuh"])
    assert h1 == bench.source_hash(["a.cu", "b.cuh"]) and len(h1) == 16
    a.write_text("kernel two")
    assert bench.source_hash(["a.cu", "b.cuh"]) != h1
    assert bench.source_hash(["b.cuh", "a.cu"]) != bench.source_hash(["a.cu", "b.cuh"])
