"""Host logic of bench.py that decides what its JSON line reports: the clock record of the timed
region (a throttled run is rejected on it) and the per-kernel DRAM traffic read from profiles/."""
import datetime
import os
import sys
import tempfile
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

FMT = "%Y/%m/%d %H:%M:%S.%f"


def at(clock: str) -> float:
    return datetime.datetime.strptime(f"2026/12/03 {clock}", FMT).timestamp()


def sampler(rows):
    """A ClockSampler whose nvidia-smi output is the given CSV rows."""
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    f.write("\n".join(rows) + "\n")
    f.flush()
    cs = bench.ClockSampler(0)
    cs.file, cs.proc = f, object()
    return cs


def row(clock, sm, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ", ".join("Active" if n in reasons else "Not Active" for n in names)
    return f"0, {sm}, 2070, 900.0, 0x0, {flags}, 2026/12/03 {clock}"


def test_clock_summary_keeps_only_the_timed_region():
    cs = sampler([row("10:00:00.000", 1200, ["hw_slowdown"]),     # before the region
                  row("10:00:01.000", 2070, ["sw_power_cap"]),
                  row("10:00:01.050", 2055),
                  row("10:00:01.100", 2040),
                  row("10:00:05.000", 900, ["hw_thermal_slowdown"])])  # after it
    cs.t_start, cs.t_end = at("10:00:00.500"), at("10:00:02.000")
    s = cs.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_of_a_region_shorter_than_the_sampling_period():
    cs = sampler([row("10:00:00.000", 1500), row("10:00:00.400", 2070, ["sw_thermal_slowdown"]),
                  row("10:00:00.450", 2000)])
    cs.t_start, cs.t_end = at("10:00:00.100"), at("10:00:00.120")
    s = cs.summary()  # no sample inside: the first one after the start stands for it
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0 and s["reasons"] == ["sw_thermal_slowdown"]


def test_clock_summary_without_nvidia_smi():
    cs = bench.ClockSampler(0)
    assert cs.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_record_of_the_long_context_workload():
    cfg = synth.config("4")
    shape = SimpleNamespace(**{k: cfg[k] for k in ("N", "M", "H", "Hkv", "D")}, k_type=synth.TYPE_Q8_0)
    assert (shape.N, shape.M, shape.H, shape.Hkv, shape.D) == (2048, 75520, 24, 4, 256)
    got = bench.read_traffic(shape)
    assert set(got) >= {"k_predecode", "k_rows_lse", "k_cols", "k_dq_gemm"}
    # per launch, at least the algorithmic bytes: K'/V' copies out; dS and dK/dV out; dS in
    assert got["k_predecode"] >= 309e6 and got["k_cols"] >= 8.39e9 and got["k_dq_gemm"] >= 7.42e9
    assert bench.read_traffic(SimpleNamespace(N=1, M=1, H=1, Hkv=1, D=64, k_type=synth.TYPE_F32)) == {}


def test_kernel_products_name_the_profiled_kernels():
    # the roofline's dominant kernel is looked up by these names in the library's profile record
    names = {"k_row_stats", "k_vsum", "k_finalize", "k_convert", "k_predecode", "k_rows_lse", "k_lse_merge",
             "k_rows_dq", "k_dq_reduce", "k_cols", "k_dq_gemm", "k_stats_in", "k_fwd", "k_fwd_merge",
             "k_cols_rowscale", "k_sink_grad", "k_dq_raw"}
    src = open(os.path.join(ROOT, "flash_attention_backward_gb300", "csrc", "fa_back.cu")).read()
    for n in names:
        assert f'"{n}"' in src, n
    assert set(bench.KERNEL_PRODUCTS) <= names
