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
    assert d["config"]["workload"].startswith("dsa_mla")
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
    assert d["gpu_launches"] == d["steps"] * 4       # four layers, one launch each
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
