"""bench.py host logic without a GPU: the clock-sample parser keeps the samples of the timed
region and reports every throttle reason seen there."""
import datetime
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _line(t, mhz, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, {thermal}, {power_cap}"


def test_clock_samples_restricted_to_timed_region():
    t0 = time.time()
    lines = [_line(t0 - 0.4, 1000), _line(t0 + 0.02, 2000), _line(t0 + 0.12, 1900, power_cap="Active"),
             _line(t0 + 0.6, 1500, thermal="Active"), "garbage"]
    c = bench.Clocks(0)
    c.lines, c.window = lines, (t0, t0 + 0.2)
    s = c.summary()
    assert s["samples"] == 2 and s["in_timed_region"]
    assert s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]          # the thermal sample lies outside the region


def test_clock_samples_fall_back_to_all_when_none_inside():
    t0 = time.time()
    c = bench.Clocks(0)
    c.lines, c.window = [_line(t0 - 1.0, 1200), _line(t0 + 2.0, 1800, thermal="Active")], (t0, t0 + 0.1)
    s = c.summary()
    assert s["samples"] == 2 and not s["in_timed_region"]
    assert s["reasons"] == ["sw_thermal_slowdown"]


def _profile(root, hashes, rows):
    os.makedirs(root / "profiles", exist_ok=True)
    text = "| kind | shape | launches | read MB | write MB | bytes per launch | algorithmic bytes per launch |\n"
    text += "|---|---|---:|---:|---:|---:|---:|\n"
    for kind, shape, nbytes in rows:
        text += f"| {kind} | {shape} | 2 | 1.0 | 1.0 | {nbytes} | 123 |\n"
    text += "\n| kernel type | sources sha256 |\n|---|---|\n"
    for kind, h in hashes.items():
        text += f"| {kind} sources | {h} |\n"
    (root / bench.TRAFFIC_PROFILE).write_text(text)


def test_measured_traffic_follows_each_kernels_sources(tmp_path, monkeypatch):
    """A kernel type's DRAM figure is the mean of its per-shape captures while that type's sources
    hash to the listed value, and is withdrawn once one of them changes; another type's edit
    leaves it."""
    import shutil
    root = tmp_path / "repo"
    for d in ("include", os.path.join("int8_mixed_precision_gb300", "csrc")):
        shutil.copytree(os.path.join(bench.ROOT, d), root / d)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.measured_traffic("gemm_int8") is None          # no profile yet
    hashes = {k: bench.kernel_sources_hash(k) for k in bench.KERNEL_SOURCES}
    _profile(root, hashes, [("gemm_int8", "qkv 17776x3072->9216", 100), ("gemm_int8", "out 17776x3072->3072", 300),
                            ("gemm_nvfp4", "qkv 17776x3072->9216", 50)])
    assert bench.measured_traffic("gemm_int8") == 200
    assert bench.measured_traffic("gemm_nvfp4") == 50
    assert bench.measured_traffic("quant_int8") is None          # a type without captures
    with open(root / "int8_mixed_precision_gb300" / "csrc" / "gemm_nvfp4.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.measured_traffic("gemm_nvfp4") is None
    assert bench.measured_traffic("gemm_int8") == 200
    with open(root / "int8_mixed_precision_gb300" / "csrc" / "common.cuh", "a") as f:
        f.write("\n// edited\n")
    assert all(bench.measured_traffic(k) is None for k in bench.KERNEL_SOURCES)
    assert bench.measured_traffic("no_such_kernel") is None


def test_algorithmic_bytes_follow_the_survey_accounting():
    """Quantisers are counted at the survey's algorithmic bytes per element (INT8: 2 in + 1 out +
    4 per row; NVFP4: 2 in + 0.5 + 1/16), not at the bytes of their containers."""
    assert bench.bytes_quant_int8(10, 64) == 10 * 64 * 3 + 40
    assert bench.bytes_quant_nvfp4(10, 64) == 10 * 64 * 2 + 10 * 32 + 10 * 4
    spec = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert spec["hidden"] == 3072 and spec["blocks"] == 42 and spec["tokens"] == 17776
    assert [s[1:] for s in bench.linears(spec)] == [(3072, 9216), (3072, 3072), (3072, 12288), (12288, 3072)]
