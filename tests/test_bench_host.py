"""Host checks of the bench's clock record: only samples inside the timed windows count, and
throttle reasons are read from the right columns."""
import datetime

import bench


def _line(t, clk, reasons=("Not Active",) * 4):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, "0", str(clk), "2070", "900.0", "0x0000000000000000", *reasons])


def test_clock_summary_keeps_only_timed_samples():
    s = bench.ClockSampler(0)
    t0 = 1_800_000_000.0
    s.lines = [_line(t0, 1000), _line(t0 + 1.0, 2070), _line(t0 + 1.02, 2060),
               _line(t0 + 1.04, 2070), _line(t0 + 3.0, 990)]
    r = s.summary([(t0 + 0.99, t0 + 1.05)])
    assert r["samples"] == 3 and r["samples_total"] == 5
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070 and r["reasons"] == []
    assert s.summary([])["samples"] == 5       # no windows recorded: every sample kept


def test_clock_summary_reads_reason_columns():
    s = bench.ClockSampler(0)
    t0 = 1_800_000_000.0
    s.lines = [_line(t0, 2000, ("Not Active", "Not Active", "Not Active", "Active")),
               _line(t0 + 5, 1500, ("Active", "Not Active", "Not Active", "Not Active"))]
    r = s.summary([(t0 - 0.01, t0 + 0.01)])
    assert r["reasons"] == ["sw_power_cap"]    # the hw_slowdown sample lies outside the window
    assert bench.ClockSampler(0).summary()["sm_mhz"] is None


def test_unique_kv_bytes_counts_each_page_once():
    # words: (block 5, 16 valid) twice, (block 7, 3 valid), (block 9, 16 valid); bit layout
    # block | offset << 32 | (n_valid - 1) << 58
    import numpy as np
    w = np.array([5 | (100 << 32) | (15 << 58), 5 | (900 << 32) | (15 << 58),
                  7 | (2 << 58), 9 | (15 << 58)], dtype=np.uint64)
    assert bench._unique_kv_bytes(w, 4096) == (16 + 3 + 16) * 4096
    assert bench._unique_kv_bytes(np.zeros(0, dtype=np.uint64), 4096) == 0


def test_traffic_commands_name_no_scratch_path():
    for name, run in bench.TRAFFIC_RUNS.items():
        assert "{csv}" in run["command"] and "gpurun" not in run["command"], name
        assert len(bench._kernel_hash(name)) == 16
