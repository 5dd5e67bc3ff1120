"""Seeded random steps through the C ABI against the oracle: several layers
per step, each drawn from one of the shapes the chooser sends to a different
kernel (ghost Gram on the tensor cores, T = 1 closed form, materialized LoRA
factor on the tensor cores, small or odd shapes on the CUDA cores), ragged
sizes, biases, fp32 and bf16, clipped and unclipped records.  Norms, clip
factors and G at sigma and at sigma = 0 within the parity tolerances
("Privacy-Preserving Machine Learning", section "Differentially private
stochastic gradient descent", phases 2-5; "Differential Privacy in
Fine-Tuning (DP-SGD)", "Per-Sample Gradient Clipping" and "Calibrated
Gaussian Noise Addition")."""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from gpu_harness import assert_step_parity

pytestmark = pytest.mark.gpu

KINDS = ("ghost_tc", "t1", "skinny", "small")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


def _layer(rng, kind, bf16):
    """(d_in, d_out, has_bias, T) of one layer of the given kind."""
    m8 = lambda lo, hi: 8 * int(rng.integers(lo // 8, hi // 8 + 1))  # noqa: E731
    if kind == "ghost_tc" and bf16:
        d_in, d_out = m8(64, 320), m8(64, 320)
        T = int(rng.integers(2, min(300, int(math.isqrt(d_in * d_out - 1))) + 1))
        return d_in, d_out, bool(rng.integers(0, 2)), T
    if kind == "t1":
        if bf16 and rng.integers(0, 2):
            return m8(8, 256), m8(8, 256), bool(rng.integers(0, 2)), 1
        return int(rng.integers(1, 70)), int(rng.integers(1, 70)), bool(rng.integers(0, 2)), 1
    if kind == "skinny" and bf16:
        r, D = int(rng.choice([8, 16])), m8(64, 512)
        T = int(rng.integers(math.isqrt(r * D) + 1, 161))
        return (D, r, False, T) if rng.integers(0, 2) else (r, D, False, T)
    return int(rng.integers(1, 48)), int(rng.integers(1, 48)), bool(rng.integers(0, 2)), int(rng.integers(1, 48))


@pytest.mark.parametrize("case", range(64))
def test_random_step_against_oracle(case):
    rng = np.random.default_rng(9000 + case)
    bf16 = case % 4 != 3
    dt = torch.bfloat16 if bf16 else torch.float32
    B = int(rng.integers(1, 13))
    n = int(rng.integers(1, 4))
    specs = [_layer(rng, KINDS[int(rng.integers(0, len(KINDS)))], bf16) for _ in range(n)]
    g = torch.Generator(device="cuda").manual_seed(case)
    # one draw per record, common to its layers: some records far below the clip bound
    rec_scale = torch.exp(2.0 * torch.randn(B, generator=g, device="cuda")) * 1e-2
    A, E = [], []
    for d_in, d_out, _, T in specs:
        A.append(torch.randn(B, T, d_in, generator=g, device="cuda").to(dt))
        E.append((torch.randn(B, T, d_out, generator=g, device="cuda") * rec_scale.view(-1, 1, 1)).to(dt))
    layers = [(d_in, d_out, bias) for d_in, d_out, bias, _ in specs]
    T_list = [T for *_, T in specs]
    assert_step_parity(layers, A, E, T_list, 1.0, 0.7, int(rng.integers(0, 2 ** 40)), int(rng.integers(0, 100)),
                       dtype=dt, dtag="bf16" if bf16 else "f32")
