"""Ghost norms of layers with T above 256 rows (several 256-column blocks of
the T x T Grams, the last one ragged): norms, clip factors and G against the
oracle, with and without a bias, and bitwise batch invariance of the norms
("Privacy-Preserving Machine Learning", section "Differentially private
stochastic gradient descent", phase 2: ghost clipping; "Sensitivity Inflation
from Cross-Record Precision Routing in Private Quantized Fine-Tuning",
Proposition 2)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_harness import assert_step_parity, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


def _inputs(B, T, d_in, d_out, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(B, T, d_in, generator=g, device="cuda").to(torch.bfloat16)
    scale = torch.exp(torch.randn(B, generator=g, device="cuda")).view(-1, 1, 1)
    E = (1e-3 * torch.randn(B, T, d_out, generator=g, device="cuda") * scale).to(torch.bfloat16)
    return A, E


@pytest.mark.parametrize("B,T,d_in,d_out,bias", [
    (3, 257, 512, 448, False),    # two 256-row blocks, the second one row deep
    (3, 300, 384, 320, True),     # ragged, with a bias
    (2, 520, 640, 512, False),    # three 256-column blocks
    (2, 1024, 1024, 1536, True),  # four blocks
])
def test_long_gram_against_oracle(B, T, d_in, d_out, bias):
    import differentially_private_gb300 as dp
    assert T * T < d_in * d_out    # the ghost path
    A, E = _inputs(B, T, d_in, d_out, seed=T)
    before = dp.dp_kernel_launch_counts()
    assert_step_parity([(d_in, d_out, bias)], [A], [E], [T], 0.5, 0.8, 4, 1)
    after = dp.dp_kernel_launch_counts()
    assert after["k_ghost_gram_tc"] > before["k_ghost_gram_tc"]


@pytest.mark.parametrize("T", [300, 700])
def test_long_gram_norms_are_batch_invariant_bitwise(T):
    import differentially_private_gb300 as dp
    d_in, d_out = 512, 1024
    A, E = _inputs(5, T, d_in, d_out, seed=T + 1)
    pg = dp.PrivateGradient([(d_in, d_out, False)], dtype=torch.bfloat16)
    full = pg.step([A], [E], [T], C=1.0, sigma=0.0, seed=0, step=0, layer_norms=True)
    for r in (0, 3):
        one = pg.step([A[r:r + 1]], [E[r:r + 1]], [T], C=1.0, sigma=0.0, seed=0, step=0, layer_norms=True)
        assert to64(one.layer_sqnorm[0])[0] == to64(full.layer_sqnorm[0])[r]
    perm = torch.tensor([4, 2, 0, 3, 1], device="cuda")
    shuf = pg.step([A[perm]], [E[perm]], [T], C=1.0, sigma=0.0, seed=0, step=0, layer_norms=True)
    assert np.array_equal(to64(shuf.layer_sqnorm[0]), to64(full.layer_sqnorm[0])[perm.cpu().numpy()])
    pg.close()
