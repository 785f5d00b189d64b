"""Host-side helpers of the benchmark (CPU only)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_digest_ignores_comments_and_blank_space():
    a = "int f(int x) {\n    return x + 1;  // add one\n}\n"
    b = "/* header */\nint f(int x) {\n\n        return x + 1;\n}   // trailing\n"
    assert bench.code_digest([a]) == bench.code_digest([b])


def test_code_digest_follows_code_changes():
    a = "int f(int x) { return x + 1; }\n"
    b = "int f(int x) { return x + 2; }\n"
    assert bench.code_digest([a]) != bench.code_digest([b])
    # file boundaries and order matter
    assert bench.code_digest([a, b]) != bench.code_digest([b, a])


def test_captured_traffic_matches_committed_kernel():
    """The committed DRAM capture names the kernel code it was taken on; the bench reports its
    bytes only for that code (None otherwise)."""
    v = bench.captured_traffic("row_fwd")
    path = os.path.join(ROOT, "profiles", "dram_traffic_s2048_b4_h5120_ffn20480_p4.txt")
    recorded = [line.split()[1] for line in open(path) if line.startswith("kernel_code_sha256")]
    assert len(recorded) == 1
    if recorded[0] == bench.kernel_code_digest():
        assert isinstance(v, int) and v > 0
    else:
        assert v is None


def test_default_and_profiling_flags(monkeypatch):
    """Without flags the bench runs one GPU with a time-based warm-up; --next-rows-only is an
    opt-in profiling mode and never the default."""
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.warmup is None and a.impl == "tpmlp" and not a.next_rows_only
    monkeypatch.setattr(sys, "argv", ["bench.py", "--next-rows-only", "--steps", "8", "--warmup", "2"])
    a = bench.parse()
    assert a.next_rows_only and a.steps == 8 and a.warmup == 2


PEAKS = {"bf16_tflops": 1895.4, "bf16_tflops_sustained": 1707.2}


def test_peak_regime_short_region_is_burst():
    """A tenth of a second of load runs at the burst clock: the burst peak applies, whatever
    the sampled clock."""
    regime, peak, _ = bench.peak_regime({"sm_mhz": 1500.0, "sm_max_mhz": 2070.0}, 0.12, PEAKS)
    assert regime == "burst" and peak == 1895.4


def test_peak_regime_near_max_clock_is_burst():
    regime, peak, _ = bench.peak_regime({"sm_mhz": 2055.0, "sm_max_mhz": 2070.0}, 3.0, PEAKS)
    assert regime == "burst" and peak == 1895.4


def test_peak_regime_settled_long_region_is_sustained():
    regime, peak, why = bench.peak_regime({"sm_mhz": 1470.0, "sm_max_mhz": 2070.0}, 1.3, PEAKS)
    assert regime == "sustained" and peak == 1707.2
    assert "1470" in why and "2070" in why


def test_clock_summary_uses_samples_inside_the_window():
    """Samples stamped inside a marked window are summarised; a window with fewer than three
    samples falls back to every sample and says so."""
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.source, s.windows = "test", {"timed": [10.0, 10.1], "tiny": [20.0, 20.001]}
    s.rows = [(9.9, 1400.0, 2070.0, 1300.0, 0x4)] + \
        [(10.0 + 0.01 * i, 2000.0 + i, 2070.0, 900.0, 0x0) for i in range(1, 10)]
    c = s.summary("timed")
    assert c["window"] == "timed region" and c["samples"] == 9
    assert c["sm_mhz"] == 2005.0 and c["reasons"] == []
    t = s.summary("tiny")
    assert t["window"] == "whole run" and t["samples"] == 10 and t["reasons"] == ["sw_power_cap"]


def test_e2e_leg_times_as_many_steps_as_the_device_region(monkeypatch):
    """The end-to-end leg runs under the device-timed region's conditions: as many steps (at most
    60) unless --e2e-steps says otherwise, 0 skipping it."""
    for argv, want in ((["bench.py"], 60), (["bench.py", "--steps", "20", "--warmup", "5"], 20),
                       (["bench.py", "--steps", "20", "--e2e-steps", "7"], 7),
                       (["bench.py", "--e2e-steps", "0"], 0)):
        monkeypatch.setattr(sys, "argv", argv)
        assert bench.e2e_step_count(bench.parse()) == want


def test_e2e_leg_idles_as_long_as_the_set_up():
    """A short run's end-to-end leg starts after as long an idle as the buffer set-up gave the
    device-timed region, bounded on both sides."""
    assert bench.e2e_idle_seconds(3.2) == 3.2
    assert bench.e2e_idle_seconds(0.1) == bench.E2E_IDLE_SECONDS
    assert bench.e2e_idle_seconds(60.0) == bench.E2E_IDLE_MAX_SECONDS
