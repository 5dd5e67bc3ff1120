"""The record-sharded step's exchange logic on the CPU: world size 2 over gloo.

``sharded_step`` splits the records of a batch over the ranks, reduce-
scatters the partial clipped sums, adds the noise of each rank's coordinate
shard keyed by the global coordinate and all-gathers the result.  Here the
per-rank compute is the float64 oracle (``OracleShardOps``, test code) and
the collectives run on gloo, so the exchange itself is checked exactly:
the sharded G must equal the oracle's single-process step on the whole batch
to float64 rounding, for unequal record counts per rank, a coordinate count
that does not divide into the shards, layers with biases (odd coordinate
counts) and a public normalizer; and a non-finite norm on one rank must stop
the step on every rank.
"""

from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import dpsgd, philox


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleShardOps:
    """Per-rank compute of the sharded step in float64 (oracle), CPU tensors."""

    dtype = torch.float64

    def __init__(self, layers):
        self.layers = [dpsgd.Layer(d_in, d_out, hb) for (d_in, d_out, hb) in layers]
        self.offs, self.P = dpsgd.coordinate_offsets(self.layers)
        self.bad = False

    def partial_sum(self, A_list, E_list, T_list, C, S_flat):
        A64 = [a.numpy().astype(np.float64) for a in A_list]
        E64 = [e.numpy().astype(np.float64) for e in E_list]
        n2 = np.zeros(A64[0].shape[0])
        for ly, A, E in zip(self.layers, A64, E64):
            n2 = n2 + dpsgd.layer_sqnorms(A, E, ly.has_bias)
        if not np.all(np.isfinite(n2)):
            self.bad = True
            return
        c = dpsgd.clip_factors(n2, C)
        for ly, off, A, E in zip(self.layers, self.offs, A64, E64):
            S, sb = dpsgd.clipped_sum(A, E, c, ly.has_bias)
            flat = S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
            S_flat[off:off + flat.size] = torch.from_numpy(flat)

    def nonfinite(self):
        return self.bad

    def noise(self, S_shard, G_shard, k0, n, sigma, C, L, seed, step):
        if n == 0:
            return
        z = philox.normals(seed, step, k0, n)
        G_shard[:n] = (S_shard[:n] + torch.from_numpy(sigma * C * z)) / L


LAYERS = [(13, 7, True), (9, 5, False), (6, 11, True)]   # P = 98 + 45 + 77 = 220 coordinates
T = 3
SPLIT = (3, 2)                                          # records per rank


def _batch(B, seed, nan_record=None):
    g = torch.Generator().manual_seed(seed)
    A = [torch.randn(B, T, d_in, generator=g, dtype=torch.float64) for (d_in, _, _) in LAYERS]
    # records 0, 2 and 3 small enough to stay unclipped at C >= 0.4, records 1 and 4 clipped
    scale = torch.tensor([0.005, 0.3, 0.004, 0.006, 0.3], dtype=torch.float64)[:B].view(-1, 1, 1)
    E = [torch.randn(B, T, d_out, generator=g, dtype=torch.float64) * scale for (_, d_out, _) in LAYERS]
    if nan_record is not None:
        E[1][nan_record, 0, 0] = float("nan")
    return A, E


def _rank(rank, world, port, out, kw):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from differentially_private_gb300.sharded import NonFiniteNormError, sharded_step
        A, E = _batch(sum(SPLIT), 7, kw.get("nan_record"))
        lo = sum(SPLIT[:rank])
        hi = lo + SPLIT[rank]
        ops = OracleShardOps(LAYERS)
        try:
            G = sharded_step(ops, [a[lo:hi] for a in A], [e[lo:hi] for e in E], [T] * len(LAYERS),
                             C=kw["C"], sigma=kw["sigma"], seed=5, step=9, L=kw.get("L"))
            out[rank] = G.numpy().copy()
        except NonFiniteNormError:
            out[rank] = "nonfinite"
    finally:
        dist.destroy_process_group()


def _run(**kw):
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(len(SPLIT), port, out, kw), nprocs=len(SPLIT), join=True)
        return dict(out)


@pytest.mark.parametrize("C,sigma,L", [(1.2, 0.7, None), (0.4, 0.0, None), (0.9, 1.3, 17.5)])
def test_sharded_step_equals_single_process_oracle(C, sigma, L):
    got = _run(C=C, sigma=sigma, L=L)
    A, E = _batch(sum(SPLIT), 7)
    ref = dpsgd.step([dpsgd.Layer(*ly) for ly in LAYERS], [a.numpy() for a in A], [e.numpy() for e in E],
                     [T] * len(LAYERS), C=C, sigma=sigma, seed=5, step_index=9, L=L)
    want = np.concatenate(ref.grads)
    assert want.size == 220
    for r in range(len(SPLIT)):
        assert got[r].shape == want.shape
        np.testing.assert_allclose(got[r], want, rtol=1e-12, atol=1e-14 * np.abs(want).max())
    # some records are clipped and some are not, so both branches of the clip ran
    assert np.any(ref.clip < 1) and np.any(ref.clip == 1)


def test_nonfinite_norm_on_one_rank_stops_every_rank():
    got = _run(C=1.0, sigma=1.0, nan_record=4)     # record 4 belongs to rank 1
    assert got == {0: "nonfinite", 1: "nonfinite"}


@pytest.mark.parametrize("P,world", [(0, 1), (1, 2), (220, 2), (221, 3), (1000, 8), (59834368, 8)])
def test_shard_bounds_cover_every_coordinate_once(P, world):
    from differentially_private_gb300.sharded import shard_bounds
    seen = np.zeros(P, dtype=np.int64)
    for r in range(world):
        k0, n, n_shard = shard_bounds(P, world, r)
        assert n_shard % 4 == 0 and k0 == r * n_shard and 0 <= n <= n_shard
        seen[k0:k0 + n] += 1
    assert np.all(seen == 1)
