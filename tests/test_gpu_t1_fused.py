"""Steps whose every layer has T = 1 (a non-sequence MLP) run their norms,
clip factors and pre-scaled operand copies in one kernel when the layers
come in one batch call with no per-layer norm outputs.  That path must give
bitwise the norms, clip factors and G of the two-kernel path (per-layer norm
calls, then the clip kernel), and the oracle's within the tolerances
("Privacy-Preserving Machine Learning", section "Differentially private
stochastic gradient descent", phases 2-5; "Differential Privacy in
Fine-Tuning (DP-SGD)", "Per-Sample Gradient Clipping")."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_harness import G_RTOL, NORM_RTOL, oracle_step, rel_fro, to64

pytestmark = pytest.mark.gpu


def _inputs(layers, B, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = [torch.nn.functional.gelu(torch.randn(B, 1, d_in, generator=g, device="cuda")).to(torch.bfloat16)
         for (d_in, _, _) in layers]
    # a few records well below the clip bound, the rest above it
    s = torch.where(torch.arange(B, device="cuda") % 5 == 0, 1e-4, 0.05)
    E = [(torch.randn(B, 1, d_out, generator=g, device="cuda") * s.view(-1, 1, 1)).to(torch.bfloat16)
         for (_, d_out, _) in layers]
    return A, E


def _step(layers, A, E, C, sigma, batch):
    import differentially_private_gb300 as dp
    pg = dp.PrivateGradient(layers, dtype=torch.bfloat16)
    before = dp.dp_kernel_launch_counts()
    out = pg.step(A, E, [1] * len(layers), C=C, sigma=sigma, seed=3, step=5, layer_norms=False, batch=batch)
    torch.cuda.synchronize()
    after = dp.dp_kernel_launch_counts()
    launched = {k: after[k] - before[k] for k in after if after[k] != before[k]}
    pg.close()
    return out, launched


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


@pytest.mark.parametrize("layers,B", [
    ([(64, 256, False), (256, 64, False)], 300),               # the MLP shape, records not a multiple of 8
    ([(128, 32, True), (32, 128, True), (96, 96, False)], 37),  # biases, three layers
    ([(64, 32, False)] * 5, 65),                               # five layers: the fifth copy by the grad phase
    ([(256, 512, False), (512, 256, False)], 1),               # one record
    ([(48, 40, False), (40, 48, True)] * 6, 19),               # twelve layers: one block per record, rows re-read
    ([(2048, 4096, False), (4096, 2048, False)], 24),          # pre-scaled rows too long to keep in registers
])
def test_fused_matches_two_kernel_path_bitwise_and_oracle(layers, B):
    A, E = _inputs(layers, B, seed=len(layers) * 100 + B)
    C = 1.0
    fused, kf = _step(layers, A, E, C, 0.9, batch=True)
    split, ks = _step(layers, A, E, C, 0.9, batch=False)
    assert kf.get("k_norm_clip_t1") == 1 and "k_clip" not in kf and "k_norm_t1_group" not in kf, kf
    assert "k_norm_clip_t1" not in ks and ks.get("k_clip") == 1, ks
    assert torch.equal(fused.sqnorm, split.sqnorm)
    assert torch.equal(fused.clip, split.clip)
    for a, b in zip(fused.grads, split.grads):
        assert torch.equal(a, b)
    ref = oracle_step(layers, A, E, [1] * len(layers), C, 0.9, 3, 5)
    n2 = to64(fused.sqnorm)
    assert np.all(np.abs(n2 - ref.total_sqnorm) <= NORM_RTOL["bf16"] * ref.total_sqnorm)
    c = to64(fused.clip)
    assert np.allclose(c, ref.clip, rtol=NORM_RTOL["bf16"], atol=0)
    assert np.any(c < 1.0) and np.any(c == 1.0) if B > 1 else True
    for l, G in enumerate(fused.grads):
        assert rel_fro(to64(G), ref.grads[l]) <= G_RTOL, l
    # sigma = 0: the clipped sum alone
    z0, _ = _step(layers, A, E, C, 0.0, batch=True)
    for l, G in enumerate(z0.grads):
        S, sb = ref.clipped[l]
        flat = S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
        assert rel_fro(to64(G), flat / B) <= G_RTOL, l


def test_more_layers_than_lanes_take_the_two_kernel_path():
    layers = [(16, 16, False)] * 33
    A, E = _inputs(layers, 9, seed=33)
    out, k = _step(layers, A, E, 1.0, 0.5, batch=True)
    assert "k_norm_clip_t1" not in k and k.get("k_clip") == 1, k
    ref = oracle_step(layers, A, E, [1] * 33, 1.0, 0.5, 3, 5)
    assert np.allclose(to64(out.clip), ref.clip, rtol=NORM_RTOL["bf16"], atol=0)


def test_per_layer_norm_outputs_keep_the_two_kernel_path():
    import differentially_private_gb300 as dp
    layers = [(64, 128, False), (128, 64, False)]
    A, E = _inputs(layers, 16, seed=7)
    pg = dp.PrivateGradient(layers, dtype=torch.bfloat16)
    before = dp.dp_kernel_launch_counts()
    out = pg.step(A, E, [1, 1], C=1.0, sigma=0.0, seed=0, step=0, layer_norms=True, batch=True)
    torch.cuda.synchronize()
    after = dp.dp_kernel_launch_counts()
    assert after["k_norm_clip_t1"] == before["k_norm_clip_t1"]
    assert torch.equal(out.sqnorm, out.layer_sqnorm[0] + out.layer_sqnorm[1])
    pg.close()


def test_nonfinite_input_on_the_fused_path():
    import differentially_private_gb300 as dp
    layers = [(64, 128, False), (128, 64, False)]
    A, E = _inputs(layers, 16, seed=9)
    A[1][4, 0, 7] = float("inf")
    pg = dp.PrivateGradient(layers, dtype=torch.bfloat16)
    grads, clip, sq = pg.alloc_outputs(16)
    for g in grads:
        g.fill_(-5.0)
    with pytest.raises(dp.DPError) as ei:
        pg.step(A, E, [1, 1], C=1.0, sigma=1.0, seed=0, step=0, outputs=(grads, clip, sq), batch=True)
    assert ei.value.status == dp.DP_ERR_NONFINITE
    assert all(bool((g == -5.0).all()) for g in grads)
    A[1][4, 0, 7] = 0.0
    out = pg.step(A, E, [1, 1], C=1.0, sigma=1.0, seed=0, step=0, batch=True)
    assert all(bool(torch.isfinite(g).all()) for g in out.grads)
    pg.close()
