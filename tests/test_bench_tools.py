"""The benchmark's evidence tools on the CPU: the ncu-CSV-to-table conversion behind the
all-shape DRAM table, and the clock summary that flags throttled runs."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
          '"Metric Value"')


def _launch(i, mode, dur_ns, rd, wr, pct):
    name = "void rmsq::rmsq_row_kernel<0, 1, %d, 4, 1, 1>(rmsq::Params)" % mode
    rows = []
    for metric, unit, value in (("gpu__time_duration.sum", "ns", dur_ns),
                                ("dram__bytes_read.sum", "byte", rd),
                                ("dram__bytes_write.sum", "byte", wr),
                                ("dram__throughput.avg.pct_of_peak_sustained_elapsed", "%", pct)):
        rows.append('"%d","1","python","h","%s","1","7","(128, 1, 1)","(608, 1, 1)","0","10.3",'
                    '"Command line profiler metrics","%s","%s","%s"' % (i, name, metric, unit, value))
    return rows


def _csv(tmp_path, launches):
    lines = ["==PROF== Connected to process 1", HEADER]
    for i, l in enumerate(launches):
        lines += _launch(i, *l)
    p = tmp_path / "report.csv"
    p.write_text("\n".join(lines) + "\n")
    return str(p)


def test_ncu_table_takes_the_median_of_the_timed_launches(tmp_path, capsys):
    reps = 3
    seq = []
    # fp8_residual: allocation + 3 warm-ups (ignored), then 3 timed launches
    seq += [(0, 99_000, 1, 1, 1.0)] * 4
    seq += [(0, 40_000, 100_000_000, 50_000_000, 58.0), (0, 42_000, 110_000_000, 60_000_000, 60.0),
            (0, 41_000, 105_000_000, 55_000_000, 59.0)]
    # nvfp4: its global-scale pre-pass (mode 3) comes first and is dropped
    seq += [(3, 20_000, 1, 1, 1.0)]
    seq += [(1, 99_000, 1, 1, 1.0)] * 4
    seq += [(1, 88_000, 500_000_000, 70_000_000, 82.0)] * 3
    args = types.SimpleNamespace(ncu_table=_csv(tmp_path, seq), only="fp8_residual,nvfp4",
                                 report_reps=reps)
    bench.ncu_table(args)
    out = capsys.readouterr().out.splitlines()
    rows = [l for l in out if l.startswith("| fp8_residual") or l.startswith("| nvfp4")]
    assert len(rows) == 2
    f8 = [c.strip() for c in rows[0].split("|")[1:-1]]
    assert f8[2] == "41.0"                                   # median duration, us
    assert f8[3] == "%.1f" % ((105_000_000 + 55_000_000) / 1e6)
    assert f8[4] == "%.1f" % (W.config("fp8_residual").algorithmic_bytes() / 1e6)
    assert f8[5] == "59.0"
    nv = [c.strip() for c in rows[1].split("|")[1:-1]]
    assert nv[2] == "88.0" and nv[5] == "82.0"


def test_ncu_table_rejects_a_csv_from_another_run(tmp_path):
    seq = [(1, 40_000, 1, 1, 50.0)] * 7                     # NVFP4 launches where FP8 belongs
    args = types.SimpleNamespace(ncu_table=_csv(tmp_path, seq), only="fp8_residual",
                                 report_reps=3)
    with pytest.raises(SystemExit):
        bench.ncu_table(args)


def _clocks(lines):
    c = bench.ClockSampler(0)
    c.lines = lines
    return c.summary()


def test_clock_summary_reports_median_and_reasons():
    idle = "0, 2070, 2070, 700.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1800, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"
    hot = "0, 1500, 2070, 1400.0, 0x40, Not Active, Active, Not Active, Not Active"
    s = _clocks([idle, idle, capped])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    s = _clocks([idle, hot, hot])
    assert s["sm_mhz"] == 1500.0 and s["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_without_samples():
    assert _clocks([])["reasons"] == ["unsampled"]
    assert _clocks(["garbage"])["reasons"] == ["unsampled"]
