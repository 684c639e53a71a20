"""CPU checks of bench.py's output contract (no GPU): the reference arm times
the FP64 oracle and prints one JSON line with the contract's keys; the
workload bookkeeping (launch counts, configuration, FLOPs) is consistent."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_tiled_attention_19_gb300 import workloads as W  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "n129_d32_f16_causal", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("n129_d32_f16_causal")


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_every_workload_has_consistent_bookkeeping(name):
    w = W.WORKLOADS[name]
    cfg = bench.workload_config(w, 1)
    assert cfg["workload"].startswith(name) and cfg["head_dim"] == w.D
    assert w.flops() > 0 and w.io_bytes() > 0
    n = bench.launches_per_call(w)
    assert n == (3 if w.backward else 2 if w.splitkv else 1)
    if w.window_left >= 0 or w.window_right >= 0:
        assert cfg["window"] == {"left": w.window_left, "right": w.window_right}
    if w.num_global:
        assert cfg["global_tokens"] == w.num_global
    if not w.square:
        assert w.flops() == pytest.approx(w.flops_exact() * (2.5 if w.backward else 1.0))


def test_per_workload_list_names_real_workloads():
    assert set(bench.PER_CONFIG) <= set(W.WORKLOADS)
    assert "global64_window4096_n16384" in bench.PER_CONFIG
