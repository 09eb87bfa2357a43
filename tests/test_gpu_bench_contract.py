"""bench.py's JSON line on the GPU: the keys and the consistency between
them that the measurement contract asks for (a short run of the default
workload)."""
import contextlib
import io
import json

import pytest

import bench

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_default_bench_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(["--steps", "8", "--warmup", "3"]) == 0
    d = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["unit"] == "resolves/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 8 and d["warmup"] == 3
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["dtype"] == "int32"
    assert d["config"]["workload"].startswith("tight_prefetch")   # the largest workload
    layers = 8
    # value = resolves of the timed steps over their device time
    resolves = d["config"]["resolves_per_step"] * d["steps"]
    assert abs(d["value"] - resolves / (d["ms_per_step"] * d["steps"] / 1e3)) <= 1e-6 * d["value"]
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] == "link" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) <= 1e-9 * r["frac"]
    assert 0 < r["frac"] < 1.5
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["unit"] == "resolves/s" and 0 < e["value"]
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == resolves // d["steps"] * 2048 * 4
    assert d["gpu_launches"] == d["steps"] * layers   # one launch per layer
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    # exact prefetch beside the value: every plan pair matched, nothing lost
    p = d["prefetch_on"]
    assert p["status"] == 0 and p["counters"]["plan_mismatches"] == 0
    assert p["counters"]["resolves"] == resolves
    assert p["counters"]["plan_hits"] * 1152 == p["counters"]["prefetched_bytes"]
    assert d["copy_only"]["status"] == 0 and d["copy_only"]["link_gbs"] > 0
    assert d["no_fetch"]["status"] == 0 and d["stages"]["status"] == 0
    assert d["no_fetch"]["roofline_hbm_metadata"]["bound"] == "hbm"
    assert "dsa_mla" in d["other_workloads"]
    # the step-time distribution beside the mean step that `value` is
    st = d["step_ms"]
    assert st["min"] <= st["median"] <= st["p90"] <= st["max"]
    assert st["min"] * (1 - 1e-9) <= d["ms_per_step"] <= st["max"] * (1 + 1e-9)
    assert st["resolves_per_s_at_median"] > 0
