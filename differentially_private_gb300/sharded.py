"""Record-sharded DP-SGD step over the ranks of a torch.distributed group.

The records of one batch are split over the ranks (each GPU holds whole
records).  Every record's norm and clip factor depend on that record alone
("Sensitivity Inflation from Cross-Record Precision Routing in Private
Quantized Fine-Tuning", section 4.1, Proposition 2), so each rank clips its
own records and forms its partial clipped sum S_r = sum over its records of
c_i g_i with no exchange.  The only exchange is the sum over ranks:

1. each rank: its records' norms, clip factors and S_r (dp_clipped_sum);
2. one small all-reduce of (records, non-finite flag): the global batch size
   is the default normalizer L, and a non-finite norm on any rank stops the
   step on every rank;
3. reduce-scatter of S: rank r receives the total S over its shard of
   coordinates [k0_r, k0_r + n_r);
4. each rank adds sigma C z_k to its shard, z keyed by the GLOBAL coordinate
   k, and divides by L (dp_noise_shard), so every coordinate gets exactly one
   draw, the same one a single GPU would draw ("Privacy-Preserving Machine
   Learning", phases 4-5: noise once on the clipped sum, then the division;
   "Differential Privacy: DP-SGD, Privacy Budgets, and LLMs", implementation
   failures: noise on every component, once);
5. all-gather of the shards: every rank holds G.

The per-rank compute is an object with ``P``, ``dtype``, ``partial_sum``,
``nonfinite`` and ``noise``; ``LibraryShardOps`` is the library's.  All the
arithmetic of the path runs in the library's kernels; this module only
allocates the exchange buffers and calls the collectives.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import _binding as b


def shard_bounds(P: int, world: int, rank: int) -> tuple[int, int, int]:
    """(k0, n, n_shard): rank's coordinate range [k0, k0 + n) and the padded
    shard length every rank uses (a multiple of 4, so that shards start on a
    noise block and 16-byte boundaries)."""
    if P < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("need P >= 0, world >= 1 and 0 <= rank < world")
    n_shard = ((P + world - 1) // world + 3) // 4 * 4
    k0 = rank * n_shard
    n = max(0, min(n_shard, P - k0))
    return k0, n, n_shard


class NonFiniteNormError(RuntimeError):
    """A per-example norm was not finite on some rank; no gradient was released."""


class LibraryShardOps:
    """The per-rank compute of the sharded step through the library's C ABI."""

    dtype = torch.float32

    def __init__(self, pg):
        """pg: a ``PrivateGradient`` holding this rank's context and layers."""
        self.pg = pg
        self.P = int(pg.P)
        self.device = pg.device
        # the layers' slices of a flat [P] buffer can be handed to the library
        # directly when every layer starts on a 16-byte boundary
        self.aligned = all(off % 4 == 0 for (_, _, _, off, _) in pg.layers)

    def partial_sum(self, A_list, E_list, T_list, C: float, S_flat: torch.Tensor) -> None:
        """S_flat[:P] = this rank's clipped sum, in global coordinate order."""
        pg = self.pg
        B = int(A_list[0].shape[0])
        b.dp_begin_step(pg.ctx, B)
        b.dp_norm_accumulate_batch(pg.ctx, list(range(len(pg.layers))), A_list, E_list, T_list)
        b.dp_clip_factors(pg.ctx, C)
        if self.aligned:
            views = [S_flat[off:off + n] for (_, _, _, off, n) in pg.layers]
            b.dp_clipped_sum(pg.ctx, views)
        else:
            parts = [torch.empty(n, dtype=torch.float32, device=self.device) for (_, _, _, _, n) in pg.layers]
            b.dp_clipped_sum(pg.ctx, parts)
            for (_, _, _, off, n), p in zip(pg.layers, parts):
                S_flat[off:off + n].copy_(p)

    def nonfinite(self) -> bool:
        """Synchronize and report whether this rank saw a non-finite norm."""
        st = b.dp_step_status(self.pg.ctx)
        if st == b.DP_ERR_NONFINITE:
            return True
        if st != b.DP_OK:
            raise b.DPError(st, "dp_step_status", b.dp_last_error(self.pg.ctx))
        return False

    def noise(self, S_shard, G_shard, k0: int, n: int, sigma: float, C: float, L: float, seed: int,
              step: int) -> None:
        """G_shard[:n] = (S_shard[:n] + sigma C z_{k0 + j}) / L."""
        b.dp_noise_shard(S_shard, G_shard, k0, n, sigma, C, L, seed, step, self.pg.stream)


def sharded_step(ops, A_list, E_list, T_list, C: float, sigma: float, seed: int, step: int,
                 L: float | None = None, group=None, device=None) -> torch.Tensor:
    """One record-sharded step; returns G [P] (global coordinate order) on every rank.

    A_list / E_list hold this rank's records only.  L defaults to the number
    of records over all ranks."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    device = device if device is not None else (A_list[0].device if A_list else torch.device("cpu"))
    P = ops.P
    k0, n, n_shard = shard_bounds(P, world, rank)
    S = torch.zeros(world * n_shard, dtype=ops.dtype, device=device)
    B_local = int(A_list[0].shape[0])
    ops.partial_sum(A_list, E_list, T_list, C, S[:P])
    meta = torch.tensor([float(B_local), 1.0 if ops.nonfinite() else 0.0], dtype=torch.float64, device=device)
    dist.all_reduce(meta, op=dist.ReduceOp.SUM, group=group)
    B_global, bad = float(meta[0].item()), float(meta[1].item())
    if bad > 0:
        raise NonFiniteNormError("a per-example gradient norm was not finite on some rank; nothing released")
    Lg = B_global if L is None else float(L)
    S_shard = torch.empty(n_shard, dtype=ops.dtype, device=device)
    dist.reduce_scatter_tensor(S_shard, S, op=dist.ReduceOp.SUM, group=group)
    G_shard = torch.zeros(n_shard, dtype=ops.dtype, device=device)
    ops.noise(S_shard, G_shard, k0, n, sigma, C, Lg, seed, step)
    G = torch.empty(world * n_shard, dtype=ops.dtype, device=device)
    dist.all_gather_into_tensor(G, G_shard, group=group)
    return G[:P]
