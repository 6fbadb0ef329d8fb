"""Host-side logic of bench.py that needs no GPU: the kernel-source hash that keys the
committed ncu traffic table."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_drops_comments_not_code():
    src = ('int a = 1;  // trailing\n/* block\n comment */ const char* s = "x//y/*z*/";\n'
           "char q = '\"';\nint b = 2; /* inline */ int c = 3;\n")
    out = bench.code_only(src)
    assert "trailing" not in out and "block" not in out and "inline" not in out
    assert '"x//y/*z*/"' in out  # comment markers inside a string are code
    assert "char q = '\"';" in out
    assert out.startswith("int a = 1; ") and out.endswith("int c = 3;")


def test_comment_edits_keep_the_hash_code_edits_change_it():
    base = "int f(int x) {\n    return x + 1;  // add one\n}\n"
    assert bench.code_only(base) == bench.code_only(base.replace("add one", "increment"))
    assert bench.code_only(base) == bench.code_only("int f(int x) { return x + 1; }")
    assert bench.code_only(base) != bench.code_only(base.replace("x + 1", "x + 2"))


def test_traffic_table_is_keyed_by_a_current_hash_or_reads_null():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    h = bench.kernel_hash()
    assert len(h) == 16 and all(c in "0123456789abcdef" for c in h)
    for workload, row in table.items():
        got = bench.load_traffic(workload)
        if row["kernel_hash"] == h:
            assert got == row["traffic_bytes_per_launch"]
            # Only for the plan it was taken of.
            assert bench.load_traffic(workload, row["plan"]) == got
            assert bench.load_traffic(workload, row["plan"] + " other") is None
        else:
            assert got is None


def test_recorded_plans_are_the_planners_plans():
    # The traffic table's plans are what the planner gives these workloads on
    # a 152-SM GB300 (the plan string carries no device name; the grid does).
    import tile_primitive_tensor_gb300 as tp
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    for workload, row in table.items():
        w = bench.wl.BY_NAME[workload]
        if isinstance(w, bench.wl.MxWorkload):
            continue  # block-scaled plans are made inside tpgemm_gemm_mx
        st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
        assert st == tp.TPGEMM_OK
        assert text == row["plan"], (workload, text, row["plan"])


def _sample(t, sm, **reasons):
    d = {"t": t, "sm": sm, "sm_max": 2070.0, "power": 900.0, "hw_slowdown": False,
         "hw_thermal_slowdown": False, "sw_thermal_slowdown": False, "sw_power_cap": False}
    d.update(reasons)
    return d


def test_clock_summary_uses_only_samples_inside_the_timed_region():
    samples = [_sample(0.5, 900.0, sw_thermal_slowdown=True), _sample(1.01, 2070.0),
               _sample(1.02, 1900.0, sw_power_cap=True), _sample(1.03, 2000.0),
               _sample(2.5, 800.0, hw_slowdown=True)]
    s = bench.summarize_clocks(samples, 1.0, 1.05, "nvml every 1 ms")
    assert s["samples"] == 3 and s["sm_mhz"] == 2000.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_is_null_when_no_sample_fell_inside():
    # Samples before and after a short region are not substituted for it.
    samples = [_sample(0.5, 900.0), _sample(2.0, 2070.0)]
    s = bench.summarize_clocks(samples, 1.0, 1.012, "nvidia-smi every 50 ms")
    assert s["sm_mhz"] is None and s["samples"] == 0
    assert "12.0 ms timed region" in s["null_reason"]
    assert bench.summarize_clocks([], 1.0, 2.0, None)["null_reason"].startswith("no clock")


def test_host_cpu_reports_a_cpu_count():
    h = bench.host_cpu()
    assert h["logical_cpus"] == os.cpu_count()
    assert "cpu_model" in h
