"""GPU path against the CPU oracle, element by element, through the C ABI.

Sizes are small enough for the oracle to finish in seconds but span several
tiles and ragged tails; the five workloads appear at reduced size with their
value distributions (full sizes are in test_gpu_fullsize.py).
"""


import numpy as np
import pytest
import torch

from gpu_harness import (G_RTOL, Z_ATOL, assert_step_parity, gpu_step, oracle_step, rel_fro, to64)
from oracle import dpsgd, philox
from synthetic import by_index, generate_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


def _wl_inputs(w, device="cuda"):
    A, E, T = [], [], []
    for i, ly in enumerate(w.layers):
        a, e = generate_layer(w, i, device)
        A.append(a)
        E.append(e)
        T.append(ly.T)
    layers = [(ly.d_in, ly.d_out, ly.has_bias) for ly in w.layers]
    return layers, A, E, T


# ------------------------------------------------------------------ noise
@pytest.mark.parametrize("seed,step,k0,n", [
    (0, 0, 0, 1 << 22),
    (0x0123456789ABCDEF, 7, 3, 100_003),
    (2 ** 64 - 1, 2 ** 40 + 5, 2 ** 41 + 1, 4099),
])
def test_philox_raw_bits_and_normals(seed, step, k0, n):
    import differentially_private_gb300 as dp
    nb = (k0 + n - 1) // 4 - k0 // 4 + 1
    raw = torch.empty(4 * nb, dtype=torch.int32, device="cuda")
    z = torch.empty(n, dtype=torch.float32, device="cuda")
    dp.dp_philox_normals(seed, step, k0, n, raw, z)
    torch.cuda.synchronize()
    got_raw = raw.cpu().numpy().view(np.uint32).reshape(-1, 4)
    want_raw = philox.raw_blocks(seed, step, k0 // 4, nb)
    assert np.array_equal(got_raw, want_raw)
    err = np.abs(to64(z) - philox.normals(seed, step, k0, n))
    assert err.max() <= Z_ATOL, err.max()


# ------------------------------------------------------------ workloads
def test_workload1_linear_f32_bias():
    w = by_index(1)
    layers, A, E, T = _wl_inputs(w)
    out, out0, ref = assert_step_parity(layers, A, E, T, w.C, w.sigma, w.noise_seed, w.step,
                                        dtype=torch.float32, dtag="f32")
    assert ref.paths == [dpsgd.GHOST]
    assert np.all(ref.clip < 1.0)        # every record is clipped at N(0,1)


def test_workload1b_unclipped_records():
    w = by_index(1).scaled(a_scale=1e-2, e_std=1e-2)
    layers, A, E, T = _wl_inputs(w)
    out, _, ref = assert_step_parity(layers, A, E, T, w.C, w.sigma, 0, 1, dtype=torch.float32, dtag="f32")
    assert np.any(ref.clip == 1.0) and np.any(ref.clip < 1.0)
    c = to64(out.clip)
    assert np.array_equal(c[ref.clip == 1.0], np.ones(int((ref.clip == 1.0).sum())))


def test_workload2_lora_opt125m_full_size():
    w = by_index(2)
    layers, A, E, T = _wl_inputs(w)
    _, _, ref = assert_step_parity(layers, A, E, T, w.C, w.sigma, w.noise_seed, w.step)
    assert ref.paths == [dpsgd.MATERIALIZE] * 48


def test_workload3_dense_reduced():
    from synthetic.workloads import LayerSpec
    w = by_index(3).scaled(B=5, layers=(LayerSpec("linear", 320, 448, 200),))
    layers, A, E, T = _wl_inputs(w)
    _, _, ref = assert_step_parity(layers, A, E, T, w.C, w.sigma, 3, 0)
    assert ref.paths == [dpsgd.GHOST]


def test_workload4_mlp_t1_reduced():
    w = by_index(4).scaled(B=257)
    layers, A, E, T = _wl_inputs(w)
    _, _, ref = assert_step_parity(layers, A, E, T, w.C, w.sigma, 0, 0)
    assert ref.paths == [dpsgd.GHOST, dpsgd.GHOST]


def test_workload5_llama_layer_reduced():
    from synthetic.workloads import LayerSpec
    T = 176          # 176^2 >= 16 * 1792: every LoRA factor materializes, as at full size
    layers = []
    for t in ("q", "k", "v", "o"):
        layers += [LayerSpec(f"{t}.A", 512, 16, T), LayerSpec(f"{t}.B", 16, 512, T)]
    for t in ("gate", "up"):
        layers += [LayerSpec(f"{t}.A", 512, 16, T), LayerSpec(f"{t}.B", 16, 1792, T)]
    layers.append(LayerSpec("down", 1792, 512, T))
    w = by_index(5).scaled(B=3, layers=tuple(layers))
    ly, A, E, Ts = _wl_inputs(w)
    _, _, ref = assert_step_parity(ly, A, E, Ts, w.C, w.sigma, 0, 0)
    assert ref.paths == [dpsgd.MATERIALIZE] * 12 + [dpsgd.GHOST]


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("B,T,d_in,d_out,bias,dt", [
    (1, 1, 1, 1, True, torch.float32),
    (1, 3, 5, 2, True, torch.float32),       # ghost, tiny ragged
    (2, 7, 3, 3, False, torch.float32),      # materialize (49 >= 9)
    (3, 33, 70, 13, True, torch.bfloat16),   # ghost, ragged tiles
    (2, 65, 8, 9, False, torch.bfloat16),    # materialize, ragged
    (4, 1, 13, 29, True, torch.bfloat16),    # T = 1, no vector loads
])
def test_edge_shapes(B, T, d_in, d_out, bias, dt):
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + T)
    A = torch.randn(B, T, d_in, generator=g, device="cuda").to(dt)
    E = torch.randn(B, T, d_out, generator=g, device="cuda").to(dt)
    assert_step_parity([(d_in, d_out, bias)], [A], [E], [T], 0.9, 0.7, 11, 2,
                       dtype=dt, dtag="f32" if dt == torch.float32 else "bf16")


def test_zero_record_unclipped_and_public_normalizer():
    g = torch.Generator(device="cuda").manual_seed(5)
    A = torch.randn(4, 8, 48, generator=g, device="cuda")
    E = torch.randn(4, 8, 24, generator=g, device="cuda")
    A[2] = 0.0
    out, _, ref = assert_step_parity([(48, 24, False)], [A], [E], [8], 1.0, 1.0, 0, 0, L=64.0,
                                     dtype=torch.float32, dtag="f32")
    assert to64(out.clip)[2] == 1.0 and to64(out.sqnorm)[2] == 0.0


def test_nonfinite_input_reports_and_skips_writes():
    import differentially_private_gb300 as dp
    A = torch.randn(3, 4, 32, device="cuda")
    E = torch.randn(3, 4, 16, device="cuda")
    E[1, 2, 5] = float("nan")
    pg = dp.PrivateGradient([(32, 16, True)], dtype=torch.float32)
    grads, clip, sq = pg.alloc_outputs(3)
    grads[0].fill_(123.0)
    with pytest.raises(dp.DPError) as ei:
        pg.step([A], [E], [4], C=1.0, sigma=1.0, seed=0, step=0, outputs=(grads, clip, sq))
    assert ei.value.status == dp.DP_ERR_NONFINITE
    assert bool((grads[0] == 123.0).all())
    # the context stays usable
    E[1, 2, 5] = 0.0
    out = pg.step([A], [E], [4], C=1.0, sigma=1.0, seed=0, step=0)
    assert bool(torch.isfinite(out.grads[0]).all())


def test_call_order_and_argument_errors():
    import differentially_private_gb300 as dp
    ctx = dp.dp_create(0, torch.cuda.current_stream())
    try:
        l0 = dp.dp_register_layer(ctx, 16, 8, False, dp.DP_F32)
        l1 = dp.dp_register_layer(ctx, 8, 4, True, dp.DP_F32)
        A0, E0 = torch.randn(2, 3, 16, device="cuda"), torch.randn(2, 3, 8, device="cuda")
        A1, E1 = torch.randn(2, 3, 8, device="cuda"), torch.randn(2, 3, 4, device="cuda")
        G = [torch.empty(8 * 16, device="cuda"), torch.empty(8 * 4 + 4, device="cuda")]
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate(ctx, l0, A0, E0, 3)           # no open step
        assert e.value.status == dp.DP_ERR_STATE
        dp.dp_begin_step(ctx, 2)
        with pytest.raises(dp.DPError) as e:
            dp.dp_register_layer(ctx, 4, 4, False, dp.DP_F32)  # registration inside a step
        assert e.value.status == dp.DP_ERR_STATE
        dp.dp_norm_accumulate(ctx, l0, A0, E0, 3)
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate(ctx, l0, A0, E0, 3)           # twice in one step
        assert e.value.status == dp.DP_ERR_STATE
        with pytest.raises(dp.DPError) as e:
            dp.dp_clip_factors(ctx, 1.0)                        # layer 1 missing
        assert e.value.status == dp.DP_ERR_STATE
        with pytest.raises(dp.DPError) as e:
            dp.dp_clipped_noisy_grad(ctx, 1.0, 0, 0, G)         # grad before clip
        assert e.value.status == dp.DP_ERR_STATE
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate(ctx, l1, A1.view(-1)[1:].data_ptr(), E1, 3)  # misaligned
        assert e.value.status == dp.DP_ERR_INVALID_ARG
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate(ctx, 7, A1, E1, 3)
        assert e.value.status == dp.DP_ERR_INVALID_ARG
        sq = torch.empty(4, device="cuda")
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate(ctx, l1, A1, E1, 3, sq.data_ptr() + 2)  # output off a 4-byte boundary
        assert e.value.status == dp.DP_ERR_INVALID_ARG
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate_batch(ctx, [l1], [A1], [E1], [3], [sq.data_ptr() + 2])
        assert e.value.status == dp.DP_ERR_INVALID_ARG
        with pytest.raises(dp.DPError) as e:
            dp.dp_norm_accumulate(ctx, l1, A1, E1, 0)
        assert e.value.status == dp.DP_ERR_SHAPE
        dp.dp_norm_accumulate(ctx, l1, A1, E1, 3)
        for badC in (0.0, -1.0, float("inf"), float("nan")):
            with pytest.raises(dp.DPError) as e:
                dp.dp_clip_factors(ctx, badC)
            assert e.value.status == dp.DP_ERR_INVALID_ARG
        with pytest.raises(dp.DPError) as e:
            dp.dp_set_normalizer(ctx, 0.0)
        assert e.value.status == dp.DP_ERR_INVALID_ARG
        out = torch.empty(8, device="cuda")
        for c_out, n2_out in ((out.data_ptr() + 2, None), (None, out.data_ptr() + 1)):
            with pytest.raises(dp.DPError) as e:
                dp.dp_clip_factors(ctx, 1.0, c_out, n2_out)             # outputs off a 4-byte boundary
            assert e.value.status == dp.DP_ERR_INVALID_ARG
        dp.dp_clip_factors(ctx, 1.0)
        for bad_sigma in (-0.1, float("nan")):
            with pytest.raises(dp.DPError) as e:
                dp.dp_clipped_noisy_grad(ctx, bad_sigma, 0, 0, G)
            assert e.value.status == dp.DP_ERR_INVALID_ARG
        dp.dp_clipped_noisy_grad(ctx, 1.0, 0, 0, G)
        assert dp.dp_step_status(ctx) == dp.DP_OK
        with pytest.raises(dp.DPError) as e:
            dp.dp_clipped_noisy_grad(ctx, 1.0, 0, 0, G)         # the step is closed
        assert e.value.status == dp.DP_ERR_STATE
    finally:
        dp.dp_destroy(ctx)


# ------------------------------------------------------------- properties
def _batch(seed, B=6, T=40, d_in=96, d_out=48, dt=torch.bfloat16):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(B, T, d_in, generator=g, device="cuda").to(dt),
            torch.randn(B, T, d_out, generator=g, device="cuda").to(dt) * 0.1)


@pytest.mark.parametrize("shape", [(40, 96, 48), (1, 96, 48), (200, 16, 8)])
def test_norms_are_batch_invariant_bitwise(shape):
    T, d_in, d_out = shape
    A, E = _batch(1, 6, T, d_in, d_out)
    full, _ = gpu_step([(d_in, d_out, True)], [A], [E], [T], 1.0, 1.0, 0, 0)
    ref = full.layer_sqnorm[0].cpu()
    for r in range(6):
        one, _ = gpu_step([(d_in, d_out, True)], [A[r:r + 1].contiguous()], [E[r:r + 1].contiguous()], [T],
                          1.0, 1.0, 0, 0)
        assert torch.equal(one.layer_sqnorm[0].cpu()[0], ref[r])
    perm = torch.tensor([3, 0, 5, 1, 4, 2], device="cuda")
    pm, _ = gpu_step([(d_in, d_out, True)], [A[perm].contiguous()], [E[perm].contiguous()], [T], 1.0, 1.0, 0, 0)
    assert torch.equal(pm.layer_sqnorm[0].cpu(), ref[perm.cpu()])


def test_repeat_is_bitwise_deterministic_and_noise_covers_every_coordinate():
    A, E = _batch(2)
    a, _ = gpu_step([(96, 48, True)], [A], [E], [40], 0.5, 1.2, 9, 3)
    b, _ = gpu_step([(96, 48, True)], [A], [E], [40], 0.5, 1.2, 9, 3)
    z, _ = gpu_step([(96, 48, True)], [A], [E], [40], 0.5, 0.0, 9, 3)
    assert torch.equal(a.grads[0], b.grads[0])
    assert bool(((a.grads[0] - z.grads[0]) != 0).all())
    c, _ = gpu_step([(96, 48, True)], [A], [E], [40], 0.5, 1.2, 9, 4)
    assert not torch.equal(a.grads[0], c.grads[0])


def test_step_resume_independent_of_history():
    """z depends only on (seed, step, k): step 5 alone equals step 5 after steps 0..4."""
    import differentially_private_gb300 as dp
    A, E = _batch(3)
    pg = dp.PrivateGradient([(96, 48, False)], dtype=torch.bfloat16)
    for s in range(5):
        pg.step([A], [E], [40], C=1.0, sigma=1.0, seed=77, step=s)
    seq = pg.step([A], [E], [40], C=1.0, sigma=1.0, seed=77, step=5).grads[0].clone()
    alone, _ = gpu_step([(96, 48, False)], [A], [E], [40], 1.0, 1.0, 77, 5)
    assert torch.equal(seq, alone.grads[0])


def test_add_remove_and_replace_sensitivity_on_gpu():
    """With sigma = 0 and L = 1: removing one record moves G by <= C, replacing one by <= 2C."""
    A, E = _batch(4, B=7)
    C = 0.25
    E[0] *= 50.0
    full, _ = gpu_step([(96, 48, True)], [A], [E], [40], C, 0.0, 0, 0, L=1.0)
    rem, _ = gpu_step([(96, 48, True)], [A[1:].contiguous()], [E[1:].contiguous()], [40], C, 0.0, 0, 0, L=1.0)
    d = torch.linalg.norm(full.grads[0].double() - rem.grads[0].double()).item()
    assert d <= C * (1 + 1e-5)
    E2 = E.clone()
    E2[0] = -E[0]
    rep, _ = gpu_step([(96, 48, True)], [A], [E2], [40], C, 0.0, 0, 0, L=1.0)
    d2 = torch.linalg.norm(full.grads[0].double() - rep.grads[0].double()).item()
    assert d2 <= 2 * C * (1 + 1e-5) and d2 > 1.9 * C


def test_batched_and_single_accumulate_agree():
    A1, E1 = _batch(5)
    A2, E2 = _batch(6, T=40, d_in=48, d_out=96)
    layers = [(96, 48, True), (48, 96, False)]
    x, _ = gpu_step(layers, [A1, A2], [E1, E2], [40, 40], 1.0, 1.0, 1, 1, batch=True)
    y, _ = gpu_step(layers, [A1, A2], [E1, E2], [40, 40], 1.0, 1.0, 1, 1, batch=False)
    for g1, g2 in zip(x.grads, y.grads):
        assert torch.equal(g1, g2)
    assert torch.equal(x.sqnorm, y.sqnorm)


@pytest.mark.parametrize("fixed", ["u1", "u2"])
def test_box_muller_exhaustive_within_1e6(fixed):
    """Every one of the 2^24 values of one uniform, with the other at the values
    where the error is largest (u1 smallest: r = sqrt(48 ln 2), the longest
    radius; u2 at the axes and the diagonals), against the float64 map."""
    import differentially_private_gb300 as dp
    grid = (np.arange(1 << 24, dtype=np.uint64) << np.uint64(8)).astype(np.uint32)
    if fixed == "u1":
        others = [0, 1 << 8, (1 << 23) << 8, 0xFFFFFFFF]          # u1 = 2^-24, 2 2^-24, 1/2 + 2^-24, 1
    else:
        others = [(q * (1 << 21)) << 8 for q in range(8)] + [0xFFFFFF00, 0x00000100]
    worst = 0.0
    for o in others:
        w = np.empty((1 << 24, 2), dtype=np.uint32)
        if fixed == "u1":
            w[:, 0], w[:, 1] = np.uint32(o), grid
        else:
            w[:, 0], w[:, 1] = grid, np.uint32(o)
        words = torch.from_numpy(w.view(np.int32)).cuda()
        z = torch.empty((1 << 24, 2), dtype=torch.float32, device="cuda")
        dp.dp_box_muller(words, 1 << 24, z)
        torch.cuda.synchronize()
        za, zb = philox.box_muller(w[:, 0], w[:, 1])
        got = z.cpu().numpy().astype(np.float64)
        worst = max(worst, float(np.abs(got[:, 0] - za).max()), float(np.abs(got[:, 1] - zb).max()))
    assert worst <= Z_ATOL, worst


@pytest.mark.parametrize("kind", ["prescaled", "records", "stored"])
def test_nonfinite_on_each_tensor_core_path(kind):
    """A NaN in one record on each bf16 gradient path (pre-scaled single
    record written by the clip kernel, per-record fold, stored per-example
    gradients): the step reports it, no G is written, and the next clean step
    of the same context matches the oracle."""
    import differentially_private_gb300 as dp
    B, T, d_in, d_out = {"prescaled": (33, 3, 256, 192), "records": (6, 64, 320, 256),
                         "stored": (7, 96, 768, 8)}[kind]
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    A = torch.randn(B, T, d_in, device="cuda", generator=g).bfloat16()
    E = (torch.randn(B, T, d_out, device="cuda", generator=g) * 0.05).bfloat16()
    layers = [(d_in, d_out, True if kind == "prescaled" else False)]
    pg = dp.PrivateGradient(layers, dtype=torch.bfloat16)
    grads, clip, sq = pg.alloc_outputs(B)
    grads[0].fill_(-3.0)
    bad = E.clone()
    bad[B // 2, T - 1, d_out - 1] = float("nan")
    with pytest.raises(dp.DPError) as ei:
        pg.step([A], [bad], [T], C=0.5, sigma=0.7, seed=1, step=2, outputs=(grads, clip, sq))
    assert ei.value.status == dp.DP_ERR_NONFINITE
    assert bool((grads[0] == -3.0).all())
    out = pg.step([A], [E], [T], C=0.5, sigma=0.7, seed=1, step=2)
    ref = oracle_step(layers, [A], [E], [T], 0.5, 0.7, 1, 2)
    assert rel_fro(to64(out.grads[0]), ref.grads[0]) <= G_RTOL
    pg.close()
