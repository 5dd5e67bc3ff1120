"""The library side of the record-sharded step, on one GPU, through the C ABI.

dp_clipped_sum gives one rank's clipped sum without noise or normalizer;
dp_noise_shard adds the noise of a range of global coordinates and divides
by L.  Two "ranks" are run one after the other on the same GPU (no kernel
waits on another), their partial sums added, and the noise applied shard by
shard: the result must match the single-GPU step on the whole batch within
the clipped-sum tolerance, the noise must be bit-identical to the stream a
single GPU draws, and within 1e-6 of the float64 oracle's normals.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_harness import G_RTOL, Z_ATOL, noise_of, oracle_step, rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


@pytest.mark.parametrize("k0,n", [(0, 4096), (3, 1001), (8, 1), (1 << 33, 4099), (5, 0)])
def test_noise_shard_is_the_single_gpu_noise_stream(k0, n):
    import differentially_private_gb300 as dp
    zeros = torch.zeros(max(n, 1) + 8, dtype=torch.float32, device="cuda")
    G = torch.full_like(zeros, -7.0)
    dp.dp_noise_shard(zeros, G, k0, n, 1.0, 1.0, 1.0, 11, 4)
    z = torch.empty(max(n, 1), dtype=torch.float32, device="cuda")
    dp.dp_philox_normals(11, 4, k0, n, None, z)
    torch.cuda.synchronize()
    if n:
        assert torch.equal(G[:n], z[:n]), "shard noise differs from the generator's stream"
        assert np.max(np.abs(to64(G[:n]) - noise_of(11, 4, k0, n))) <= Z_ATOL
    assert torch.all(G[n:] == -7.0), "wrote past the range"


def test_noise_shard_scale_and_normalizer_and_misaligned_views():
    import differentially_private_gb300 as dp
    g = torch.Generator(device="cuda").manual_seed(1)
    S = torch.randn(10003, generator=g, device="cuda")
    sigma, C, L, k0 = 0.8, 0.5, 7.0, 12344
    for off in (0, 1, 2, 3):                      # off = 0: vector path; 4-byte aligned views: scalar path
        G = torch.empty_like(S)
        dp.dp_noise_shard(S[off:], G[off:], k0 + off, S.numel() - off, sigma, C, L, 2, 3)
        torch.cuda.synchronize()
        z = noise_of(2, 3, k0 + off, S.numel() - off)
        want = (to64(S[off:]) + np.float32(sigma * C) * z) / L
        assert np.max(np.abs(to64(G[off:]) - want)) <= 1e-6 * (1 + np.abs(want).max())
    # in place
    G = S.clone()
    dp.dp_noise_shard(G, G, k0, G.numel(), sigma, C, L, 2, 3)
    ref = torch.empty_like(S)
    dp.dp_noise_shard(S, ref, k0, S.numel(), sigma, C, L, 2, 3)
    torch.cuda.synchronize()
    assert torch.equal(G, ref)


def test_noise_shard_argument_errors():
    import differentially_private_gb300 as dp
    x = torch.zeros(8, device="cuda")
    for args, status in [((x, x, 0, -1, 1.0, 1.0, 1.0, 0, 0), dp.DP_ERR_SHAPE),
                         ((x, x, 2 ** 64 - 2, 4, 1.0, 1.0, 1.0, 0, 0), dp.DP_ERR_SHAPE),
                         ((x, x, 0, 4, -1.0, 1.0, 1.0, 0, 0), dp.DP_ERR_INVALID_ARG),
                         ((x, x, 0, 4, 1.0, 0.0, 1.0, 0, 0), dp.DP_ERR_INVALID_ARG),
                         ((x, x, 0, 4, 1.0, 1.0, 0.0, 0, 0), dp.DP_ERR_INVALID_ARG),
                         ((x, x, 0, 4, 1.0, 1.0, float("inf"), 0, 0), dp.DP_ERR_INVALID_ARG),
                         ((None, x, 0, 4, 1.0, 1.0, 1.0, 0, 0), dp.DP_ERR_INVALID_ARG)]:
        with pytest.raises(dp.DPError) as ei:
            dp.dp_noise_shard(*args)
        assert ei.value.status == status, args


LAYERS = [(256, 512, False), (768, 16, False), (40, 24, True), (512, 256, False)]
T_LIST = [128, 128, 10, 1]


def _inputs(B, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = [torch.randn(B, T, di, generator=g, device="cuda").to(dt)
         for (di, _, _), T, dt in zip(LAYERS, T_LIST, _DT)]
    scale = torch.exp(torch.randn(B, generator=g, device="cuda")).view(-1, 1, 1)
    E = [(0.02 * torch.randn(B, T, do, generator=g, device="cuda") * scale).to(dt)
         for (_, do, _), T, dt in zip(LAYERS, T_LIST, _DT)]
    return A, E


_DT = [torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.bfloat16]


@pytest.mark.parametrize("sigma", [0.0, 0.9])
def test_two_ranks_in_sequence_match_the_single_gpu_step(sigma):
    import differentially_private_gb300 as dp
    from differentially_private_gb300.sharded import shard_bounds
    B, split, C, seed, step = 7, (4, 3), 1.0, 21, 5
    A, E = _inputs(B, 3)
    # the whole batch on one GPU
    pg = dp.PrivateGradient(LAYERS, dtype=torch.bfloat16)
    full = pg.step(A, E, T_LIST, C=C, sigma=sigma, seed=seed, step=step)
    G_full = torch.cat([g for g in full.grads])
    P = pg.P
    # each "rank" its own records: partial clipped sums, added
    S_tot = torch.zeros(P, dtype=torch.float32, device="cuda")
    lo = 0
    for nrec in split:
        S_parts = [torch.empty(n, dtype=torch.float32, device="cuda") for (_, _, _, _, n) in pg.layers]
        dp.dp_begin_step(pg.ctx, nrec)
        dp.dp_norm_accumulate_batch(pg.ctx, list(range(len(LAYERS))), [a[lo:lo + nrec] for a in A],
                                    [e[lo:lo + nrec] for e in E], T_LIST)
        dp.dp_clip_factors(pg.ctx, C)
        dp.dp_clipped_sum(pg.ctx, S_parts)
        assert dp.dp_step_status(pg.ctx) == dp.DP_OK
        S_tot += torch.cat(S_parts)
        lo += nrec
    # the noise of each coordinate shard of a world of 3, keyed by the global coordinate
    G_sh = torch.empty(P, dtype=torch.float32, device="cuda")
    for r in range(3):
        k0, n, _ = shard_bounds(P, 3, r)
        dp.dp_noise_shard(S_tot[k0:k0 + n], G_sh[k0:k0 + n], k0, n, sigma, C, float(B), seed, step)
    torch.cuda.synchronize()
    assert rel_fro(to64(G_sh), to64(G_full)) <= G_RTOL
    ref = oracle_step(LAYERS, A, E, T_LIST, C, sigma, seed, step)
    assert rel_fro(to64(G_sh), np.concatenate(ref.grads)) <= G_RTOL
    # the partial sums hold no noise: with sigma = 0 the clipped sum over B alone
    if sigma == 0.0:
        S_ref = np.concatenate([S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
                                for (S, sb) in ref.clipped])
        assert rel_fro(to64(S_tot), S_ref) <= G_RTOL
    pg.close()


def test_clipped_sum_follows_the_step_state_machine():
    import differentially_private_gb300 as dp
    pg = dp.PrivateGradient([(64, 64, False)], dtype=torch.bfloat16)
    S = [torch.empty(64 * 64, dtype=torch.float32, device="cuda")]
    with pytest.raises(dp.DPError) as ei:
        dp.dp_clipped_sum(pg.ctx, S)                     # no step open
    assert ei.value.status == dp.DP_ERR_STATE
    A = torch.randn(2, 8, 64, device="cuda").bfloat16()
    dp.dp_begin_step(pg.ctx, 2)
    dp.dp_norm_accumulate(pg.ctx, 0, A, A, 8)
    with pytest.raises(dp.DPError) as ei:
        dp.dp_clipped_sum(pg.ctx, S)                     # before the clip factors
    assert ei.value.status == dp.DP_ERR_STATE
    dp.dp_clip_factors(pg.ctx, 1.0)
    dp.dp_clipped_sum(pg.ctx, S)
    with pytest.raises(dp.DPError) as ei:
        dp.dp_clipped_noisy_grad(pg.ctx, 1.0, 0, 0, S)   # the step is closed
    assert ei.value.status == dp.DP_ERR_STATE
    assert dp.dp_step_status(pg.ctx) == dp.DP_OK
    pg.close()


def test_sharded_step_over_nccl_with_one_rank():
    """The sharded step's exchange through NCCL on the GPU with one rank: the
    all-reduce, reduce-scatter and all-gather run on the library's device
    buffers (more ranks need more GPUs).  G matches the single-GPU step, and
    G(sigma) - G(0) is the float64 noise at every coordinate."""
    import torch.distributed as dist
    import differentially_private_gb300 as dp
    from differentially_private_gb300.sharded import LibraryShardOps, sharded_step
    if not dist.is_available() or not dist.is_nccl_available():
        pytest.skip("torch.distributed has no NCCL")
    if dist.is_initialized():
        pytest.skip("a process group is already initialized")
    dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1)
    try:
        B, C, sigma, seed, step = 7, 1.0, 0.9, 21, 5
        A, E = _inputs(B, 3)
        pg = dp.PrivateGradient(LAYERS, dtype=torch.bfloat16)
        full = pg.step(A, E, T_LIST, C=C, sigma=sigma, seed=seed, step=step)
        G_full = torch.cat([g for g in full.grads])
        ops = LibraryShardOps(pg)
        G = sharded_step(ops, A, E, T_LIST, C, sigma, seed, step).clone()
        G0 = sharded_step(ops, A, E, T_LIST, C, 0.0, seed, step).clone()
        torch.cuda.synchronize()
        assert rel_fro(to64(G), to64(G_full)) <= G_RTOL
        want = sigma * C * noise_of(seed, step, 0, pg.P) / B
        assert np.allclose(to64(G) - to64(G0), want, rtol=1e-4, atol=2e-6 * sigma * C / B)
        pg.close()
    finally:
        dist.destroy_process_group()
