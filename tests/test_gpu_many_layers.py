"""Layer counts above one launch's group limits, and the status word across
a sequence of steps (two words that steps alternate between)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import differentially_private_gb300 as dp
from gpu_harness import assert_step_parity

pytestmark = pytest.mark.gpu


def test_more_lora_factors_than_one_skinny_launch_holds():
    # 60 materialized rank-8 factors: two skinny launches (48 + 12) and one
    # grouped weighted sum per 64 layers
    layers, A, E, T = [], [], [], []
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    for i in range(30):
        for (d_in, d_out) in ((256, 8), (8, 256)):
            layers.append((d_in, d_out, False))
            A.append(torch.randn(3, 96, d_in, device="cuda", generator=g).bfloat16())
            E.append((torch.randn(3, 96, d_out, device="cuda", generator=g) * 0.03).bfloat16())
            T.append(96)
    assert all(dp.dp_choose_path(t, a, b) == dp.DP_PATH_MATERIALIZE for (a, b, _), t in zip(layers, T))
    assert_step_parity(layers, A, E, T, C=0.5, sigma=1.0, seed=3, step=1)


def test_more_t1_layers_than_one_group_launch_holds():
    # 70 bf16 T = 1 layers: two grouped norm launches (64 + 6)
    layers, A, E, T = [], [], [], []
    g = torch.Generator(device="cuda")
    g.manual_seed(12)
    for i in range(70):
        d_in, d_out = 64 + 8 * (i % 5), 72 + 8 * (i % 3)
        layers.append((d_in, d_out, i % 7 == 0))
        A.append(torch.randn(5, 1, d_in, device="cuda", generator=g).bfloat16())
        E.append((torch.randn(5, 1, d_out, device="cuda", generator=g) * 0.1).bfloat16())
        T.append(1)
    assert_step_parity(layers, A, E, T, C=0.8, sigma=0.7, seed=4, step=2)


def test_status_across_a_sequence_of_steps():
    A = torch.randn(3, 4, 32, device="cuda")
    E = torch.randn(3, 4, 16, device="cuda")
    pg = dp.PrivateGradient([(32, 16, True)], dtype=torch.float32)
    bad = E.clone()
    bad[0, 0, 0] = float("inf")
    results = []
    for inp in (E, bad, E, E, bad, bad, E):
        try:
            pg.step([A], [inp], [4], C=1.0, sigma=1.0, seed=0, step=0)
            results.append(dp.DP_OK)
        except dp.DPError as err:
            results.append(err.status)
    assert results == [dp.DP_OK, dp.DP_ERR_NONFINITE, dp.DP_OK, dp.DP_OK, dp.DP_ERR_NONFINITE,
                       dp.DP_ERR_NONFINITE, dp.DP_OK]
    # a step abandoned before its clip factors (begin twice), then a full one
    dp.dp_begin_step(pg.ctx, 3)
    dp.dp_norm_accumulate(pg.ctx, 0, A, bad, 4, None)
    out = pg.step([A], [E], [4], C=1.0, sigma=1.0, seed=0, step=0)
    assert bool(torch.isfinite(out.grads[0]).all())
    assert dp.dp_step_status(pg.ctx) == dp.DP_OK
    pg.close()


def test_device_wait_timeout_is_reported_and_skips_writes():
    # a bounded device-side wait that gives up (a barrier nothing completes)
    # takes the same path as a stuck copy or MMA in the tensor-core kernels
    A = torch.randn(3, 4, 32, device="cuda")
    E = torch.randn(3, 4, 16, device="cuda")
    pg = dp.PrivateGradient([(32, 16, True)], dtype=torch.float32)
    G = [torch.full((16 * 32 + 16,), 5.0, device="cuda")]
    dp.dp_begin_step(pg.ctx, 3)
    dp.dp_norm_accumulate(pg.ctx, 0, A, E, 4, None)
    dp.dp_check_wait_timeout(pg.ctx, 20)
    dp.dp_clip_factors(pg.ctx, 1.0, None, None)
    dp.dp_clipped_noisy_grad(pg.ctx, 1.0, 0, 0, G)
    assert dp.dp_step_status(pg.ctx) == dp.DP_ERR_CUDA
    assert "timed out" in dp.dp_last_error(pg.ctx)
    assert bool((G[0] == 5.0).all())
    # outside a step the hook is refused; the next step is clean
    with pytest.raises(dp.DPError) as err:
        dp.dp_check_wait_timeout(pg.ctx, 20)
    assert err.value.status == dp.DP_ERR_STATE
    out = pg.step([A], [E], [4], C=1.0, sigma=1.0, seed=0, step=0)
    assert bool(torch.isfinite(out.grads[0]).all())
    pg.close()


def test_many_ragged_skinny_blocks_match_oracle_repeat_and_are_batch_invariant():
    # 2880 128-column blocks (8 layers x 40 records x 9 blocks, D = 1088 and
    # T = 140 both ragged) over the CTAs' ranges, ranges ending inside records
    layers, A, E, T = [], [], [], []
    g = torch.Generator(device="cuda")
    g.manual_seed(13)
    for i in range(4):
        for (d_in, d_out) in ((1088, 16), (16, 1088)):
            layers.append((d_in, d_out, False))
            A.append(torch.randn(40, 140, d_in, device="cuda", generator=g).bfloat16())
            E.append((torch.randn(40, 140, d_out, device="cuda", generator=g) * 0.02).bfloat16())
            T.append(140)
    assert all(dp.dp_choose_path(t, a, b) == dp.DP_PATH_MATERIALIZE for (a, b, _), t in zip(layers, T))
    out, _, _ = assert_step_parity(layers, A, E, T, C=0.5, sigma=1.0, seed=5, step=3)
    pg = dp.PrivateGradient(layers, dtype=torch.bfloat16)
    runs = [pg.step(A, E, T, C=0.5, sigma=1.0, seed=5, step=3, layer_norms=True) for _ in range(3)]
    torch.cuda.synchronize()
    for r in runs:
        assert torch.equal(r.sqnorm, out.sqnorm)
        for a, b in zip(r.grads, out.grads):
            assert torch.equal(a, b)
    # a record's norms alone equal its norms inside the batch
    one = pg.step([a[7:8].clone() for a in A], [e[7:8].clone() for e in E], T, C=0.5, sigma=1.0, seed=5, step=3,
                  layer_norms=True)
    torch.cuda.synchronize()
    for l in range(len(layers)):
        assert torch.equal(one.layer_sqnorm[l][0], out.layer_sqnorm[l][7])
    pg.close()


def test_two_contexts_from_two_host_threads():
    # one context per host thread, each on its own stream, stepping at the
    # same time: every result is bitwise the one of a lone run
    import threading
    g = torch.Generator(device="cuda")
    g.manual_seed(21)
    cases = []
    for (d_in, d_out, T) in ((768, 8, 128), (512, 512, 64), (1024, 256, 3)):
        A = torch.randn(6, T, d_in, device="cuda", generator=g).bfloat16()
        E = (torch.randn(6, T, d_out, device="cuda", generator=g) * 0.05).bfloat16()
        cases.append(([(d_in, d_out, False)], [A], [E], [T]))
    lone = []
    for layers, A, E, T in cases:
        pg = dp.PrivateGradient(layers, dtype=torch.bfloat16)
        out = pg.step(A, E, T, C=0.6, sigma=0.8, seed=9, step=4)
        torch.cuda.synchronize()
        lone.append(out.grads[0].clone())
        pg.close()
    results = [[None] * len(cases) for _ in range(2)]
    errors = []

    def worker(k):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for i, (layers, A, E, T) in enumerate(cases):
                    pg = dp.PrivateGradient(layers, dtype=torch.bfloat16, stream=stream)
                    for _ in range(3):
                        out = pg.step(A, E, T, C=0.6, sigma=0.8, seed=9, step=4)
                    stream.synchronize()
                    results[k][i] = out.grads[0].clone()
                    pg.close()
        except Exception as exc:   # surfaced in the main thread
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for k in range(2):
        for i in range(len(cases)):
            assert torch.equal(results[k][i], lone[i]), (k, i)
