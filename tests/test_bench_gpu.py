"""bench.py on the GPU, on a small cut of the OLMoE layer: the bench line
carries every key the measurement contract names, and the per-iteration
report gives one exact, consistent line per iteration."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


def test_bench_line_has_the_contract_keys():
    (d,) = _bench("--config", "2", "--variant", "experts4", "--steps", "3", "--warmup", "3",
                  "--no-cpu-baseline")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "cfg2_olmoe_moe_layer_experts4"
    assert d["config"]["raw_ahead"] is False
    assert d["value"] > 0 and d["gpu_launches"] == 3 * 3
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 2 * d["config"]["numel"]
    assert 0 < e["value"] <= 1.05 * e["link_bound"]
    assert len(e["passes"]) == len(e["link_passes"]) >= 3
    assert e["value"] == max(e["passes"]) and e["link_bound"] == max(e["link_passes"])


def test_per_iteration_report():
    lines = _bench("--per-iteration", "--config", "2", "--variant", "experts4", "--reps", "2")
    assert [d["iteration"] for d in lines] == list(range(1, 10))
    for d in lines:
        assert d["report"] == "per_iteration" and d["reps"] == 2
        assert d["compress_ms"] > 0 and d["decompress_ms"] > 0
        # every block of 4096 values changes at step 1e-5: RAW payloads
        assert d["modes"] == {"raw": 16}
        assert d["changed_fraction"] == 1.0 and d["wire_bytes_per_value"] == 2.0
        assert 0.001 < d["exponent_change_rate"] < 0.01
        # the times are printed to 0.1 us: allow for that rounding
        gbs = 2.0 * d["numel"] / ((d["compress_ms"] + d["decompress_ms"]) / 1e3) / 1e9
        assert abs(gbs - d["bf16_gbs"]) <= 0.005 * gbs


def test_per_iteration_report_compressed_payloads():
    lines = _bench("--per-iteration", "--config", "2", "--variant", "experts4,clustered0.1",
                   "--reps", "2", "--sender", "hash")
    assert len(lines) == 9
    for d in lines:
        assert d["modes"] == {"compressed": 16}
        assert 0.05 < d["changed_fraction"] < 0.15
        assert abs(d["wire_bytes_per_value"] - (1.0 + d["changed_fraction"])) < 0.01


def test_per_iteration_report_rans_payloads():
    """The RANS sender's histograms are part of the restored state: every
    repetition codes with the same table and rebuilds exactly."""
    lines = _bench("--per-iteration", "--config", "2", "--variant", "experts4", "--reps", "2",
                   "--sender", "rans")
    assert len(lines) == 9
    for d in lines:
        assert d["modes"] == {"rans": 16} and d["raw_ahead"] is None
        assert 1.2 < d["wire_bytes_per_value"] < 1.5
