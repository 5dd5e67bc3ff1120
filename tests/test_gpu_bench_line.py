"""bench.py's JSON line on the GPU: one line with the keys of the benchmark
contract, the roofline of the dominant phase, the oracle baseline, the end-to-end
figure with its copied bytes, the clocks and the release manifest, on the
smallest workload and on the T = 1 MLP (whose norms run inside the clip call)."""

from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
        "phases_ms", "manifest"}


@pytest.mark.parametrize("workload,kernels", [(1, {"k_norm_ghost_cc", "k_grad_gemm_small"}),
                                              (4, {"k_sum_layers_pair_tc"})])
def test_bench_line_keys_and_values(workload, kernels):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", str(workload), "--steps", "3", "--warmup", "3",
           "--cpu-budget-s", "1"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["value"] == pytest.approx(d["config"]["B"] / (d["ms_per_step"] / 1e3), rel=1e-6)
    r = d["roofline"]
    assert r["kernel"] in kernels and r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] == max(e["pipelined_value"], e["serial_value"])
    assert d["gpu_launches"] > 0 and d["clocks"] is not None
    assert sum(d["manifest"]["kernels_per_step"].values()) * 3 == pytest.approx(d["gpu_launches"])
