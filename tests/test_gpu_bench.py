"""bench.py's JSON line on the GPU: the keys the contract names, the roofline and launch counts,
and the other workloads the default run appends, from one short default run."""
import contextlib
import io
import json

import pytest

import bench


@pytest.mark.gpu
def test_default_bench_line_and_other_workloads():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(["--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "3",
                           "--others-steps", "4"]) == 0
    d = json.loads(buf.getvalue().strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks",
              "e2e", "kernels"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # one step verifies B * N draft tokens
    assert d["value"] == pytest.approx(64 * 8 / (d["ms_per_step"] / 1e3), rel=1e-9)
    assert d["gpu_launches"] == 3 * 4          # verify, accept (rowmax + scan), rollback
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 2
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    others = d["other_workloads"]
    assert set(others) == {"qwen36_b16_n16_sample", "qwen36_b8_tree32", "qwen36_attn_b64_n8",
                           "qwen36_attn_b16_n16"}
    for name, o in others.items():
        assert o["value"] > 0 and o["ms_per_step"] > 0 and o["steps"] > 0, name
        assert o["roofline"]["frac"] > 0, name
        assert all(v["ms"] > 0 for v in o["kernels"].values()), name
