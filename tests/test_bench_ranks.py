"""The multi-rank side of bench.py, on the CPU: world size 2 over gloo.

Under torchrun every rank steps its own batch (weak scaling, no collective on
the data path); the timing is the slowest rank's, and rank 0 alone prints
the JSON line.  The reference arm (the oracle) runs on rank 0 only; the
other ranks exit 0 without work.
"""

from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_max(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + 5 r ms; every rank must see the slowest one
        got = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_max, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks(3.25, torch.device("cpu")) == 3.25


def test_job_throughput_is_weak_scaling():
    # 2 ranks x 16 records x 4 steps in 8 ms of the slowest rank
    assert bench.job_throughput(2, 16, 4, 8.0) == pytest.approx(2 * 16 * 4 / 8e-3)
    assert bench.job_throughput(1, 16, 4, 8.0) * 2 == pytest.approx(bench.job_throughput(2, 16, 4, 8.0))


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload", "1",
           "--steps", "1", "--warmup", "1", "--cpu-budget-s", "0.5"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_dominant_kernel_names_the_runtime_choice():
    """The kernel each bench line names for its dominant phase is the one the
    runtime launches for that workload's dtype and shapes, and a kernel that
    exists in the CUDA sources."""
    import glob
    import re

    from synthetic import by_index

    src = "".join(open(f).read() for f in glob.glob(os.path.join(ROOT, "differentially_private_gb300", "csrc", "*.cu")))
    defined = set(re.findall(r"__global__\s+void\s+(?:__\w+__\([^)]*\)\s+)*(\w+)\s*\(", src))
    expected = {
        1: {("norm", "alu"): "k_norm_ghost_cc", ("grad", "alu"): "k_grad_gemm_small"},
        2: {("norm", "hbm"): "k_mat_skinny_tc", ("grad", "hbm"): "k_grad_wsum"},
        3: {("norm", "tensor"): "k_ghost_gram_tc", ("grad", "tensor"): "k_clipped_sum_fold_pair_tc"},
        4: {("norm", "hbm"): "k_norm_t1_group", ("grad", "tensor"): "k_sum_layers_pair_tc"},
        5: {("norm", "tensor"): "k_ghost_gram_tc", ("grad", "tensor"): "k_clipped_sum_fold_pair_tc"},
    }
    for i, cases in expected.items():
        w = by_index(i)
        for (phase, bound), name in cases.items():
            got = bench.dominant_kernel(w, phase, bound)
            assert got == name, (i, phase, bound, got)
            assert got in defined, (got, sorted(defined))


def test_release_record_keys_and_chooser():
    """The release record each bench line carries: every key, the public step
    parameters of the workload and the chooser's decision per layer."""
    from synthetic import by_index
    w = by_index(5)
    gpu = {"gpu": "NVIDIA GB300", "compute_capability": "10.3", "sms": 152, "driver": "580", "cuda": "13.0",
           "torch": "2.x"}
    rec = bench.release_record(w, gpu, {"version": 100, "sha256_16": "0" * 16},
                               {"k_ghost_gram_tc": 1.0}, {"cores": 16, "cpu_model": "cpu"})
    assert tuple(rec) == bench.MANIFEST_KEYS
    assert all(rec[k] is not None for k in bench.MANIFEST_KEYS)
    assert (rec["B"], rec["C"], rec["sigma"], rec["seed"], rec["step"], rec["L"]) == (32, 1.0, 1.0, 0, 0, 32.0)
    paths = [c[4] for c in rec["chooser"]]
    assert paths == ["materialize"] * 12 + ["ghost"]
    assert rec["chooser"][-1][:4] == ["down_proj", 14336, 4096, 2048]
