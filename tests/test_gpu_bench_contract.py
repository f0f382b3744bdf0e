"""bench.py's JSON line on a GPU: one line with every key of the contract
(metric, value, unit, n_gpus, steps, warmup, ms_per_step, higher_is_better,
scaling, vs_baseline, dtype, data, config.workload, roofline, cpu_baseline,
e2e, gpu_launches, clocks), run on a small workload."""
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_bench_prints_one_line_with_the_whole_contract(capsys):
    bench.main(["--workload", "opt125m_bf16_kahan", "--steps", "4", "--warmup", "3",
                "--no-ceiling"])
    lines = [l for l in capsys.readouterr().out.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["metric"] == bench.METRIC and d["unit"] == "params/s" and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "opt125m_bf16_kahan"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.2
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["traffic"] is None or r["traffic"] > 0
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # five timed repetitions of four one-launch steps
    assert d["repetitions"]["n"] == 5
    assert d["gpu_launches"] == 5 * 4
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
