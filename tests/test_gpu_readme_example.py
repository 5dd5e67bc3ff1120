"""The README's usage example, run as written on small tensors: one step, the
prepared step in a loop, the record-sharded step (one NCCL rank) and the int8
forward; each checked against the plain step or its own definition."""

from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_readme_usage_runs_as_written():
    import torch.distributed as dist
    import differentially_private_gb300 as dp
    from differentially_private_gb300.int8 import Int8Linear
    from differentially_private_gb300.sharded import LibraryShardOps, sharded_step
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    g = torch.Generator(device="cuda").manual_seed(3)
    B, T = 4, 128
    A0 = torch.randn(B, T, 768, generator=g, device="cuda").bfloat16()
    E0 = (0.01 * torch.randn(B, T, 8, generator=g, device="cuda")).bfloat16()
    A1 = torch.randn(B, T, 8, generator=g, device="cuda").bfloat16()
    E1 = (0.01 * torch.randn(B, T, 768, generator=g, device="cuda")).bfloat16()

    pg = dp.PrivateGradient([(768, 8, False), (8, 768, False)], dtype=torch.bfloat16)
    out = pg.step([A0, A1], [E0, E1], [T, T], C=1.0, sigma=1.0, seed=0, step=0)
    assert [x.numel() for x in out.grads] == [8 * 768, 768 * 8]
    assert out.clip.shape == (B,) and out.sqnorm.shape == (B,)

    prep = pg.prepare([A0, A1], [E0, E1], [T, T])
    for k in range(3):
        prep.run(C=1.0, sigma=1.0, seed=0, step=k)
    torch.cuda.synchronize()
    again = pg.step([A0, A1], [E0, E1], [T, T], C=1.0, sigma=1.0, seed=0, step=2)
    for a, b in zip(prep.grads, again.grads):
        assert torch.equal(a, b)                  # the prepared step is the same step

    if dist.is_available() and dist.is_nccl_available() and not dist.is_initialized():
        dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1)
        try:
            G = sharded_step(LibraryShardOps(pg), [A0, A1], [E0, E1], [T, T], C=1.0, sigma=1.0, seed=0, step=2)
            torch.cuda.synchronize()
            full = torch.cat([x for x in again.grads])
            assert G.shape == full.shape
            assert float((G - full).norm() / full.norm()) <= 5e-3
        finally:
            dist.destroy_process_group()

    W = (0.05 * torch.randn(96, 64, generator=g, device="cuda")).half()
    X = torch.randn(2 * 16, 64, generator=g, device="cuda").half()
    lin = Int8Linear(W)
    Y = lin(X, rows_per_record=16)
    assert Y.shape == (32, 96) and Y.dtype == torch.float16
    # no outliers (|x| < 6 almost surely): close to the fp32 product within the int8 error
    ref = X.float() @ W.float().t()
    assert float((Y.float() - ref).abs().max()) <= 0.05 * float(ref.abs().max()) + 1e-3
    pg.close()
