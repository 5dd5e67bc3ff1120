"""User-level clipping through the library ("Privacy-Preserving Machine
Learning", section "Differentially private stochastic gradient descent",
the user-level construction): users of equal and of different record
counts against the oracle's user-level step, and the page's printed
Alice/Bao example."""

from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

from differentially_private_gb300 import PrivateGradient
from gpu_harness import G_RTOL, NORM_RTOL, rel_fro, to64
from oracle import dpsgd

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "alice_users.json")


def test_alice_and_bao_on_the_gpu():
    gx = json.load(open(GOLDEN))
    alice, bao = gx["users"]["Alice"], gx["users"]["Bao"]
    vals = torch.tensor(alice + bao, dtype=torch.float32, device="cuda").view(-1, 1, 1)
    A = torch.ones_like(vals)
    pg = PrivateGradient([(1, 1, False)], dtype=torch.float32)
    out = pg.step_users([A], [vals], [1], [len(alice), len(bao)], C=gx["clip_bound"], sigma=0.0, seed=0, step=0,
                        L=gx["normalizer"])
    torch.cuda.synchronize()
    with_alice = float(out.grads[0][0])
    user_clipped = (out.clip.double() * out.sqnorm.double().sqrt()).cpu().numpy()
    assert user_clipped == pytest.approx([gx["user_clipped"]["Alice"], gx["user_clipped"]["Bao"]], abs=5e-3)
    out2 = pg.step_users([A[2:].clone()], [vals[2:].clone()], [1], [1], C=gx["clip_bound"], sigma=0.0,
                         seed=0, step=0, L=gx["normalizer"])
    torch.cuda.synchronize()
    without = float(out2.grads[0][0])
    assert with_alice == pytest.approx(gx["with_alice"], abs=1e-6)
    assert without == pytest.approx(gx["without_alice"], abs=1e-6)
    assert with_alice - without == pytest.approx(gx["change"], abs=1e-6)
    pg.close()


# a ghost tensor-core layer and a LoRA factor (materialized once users are stacked)
LAYERS = [(256, 128, False), (768, 8, False)]
T_LIST = [32, 64]


@pytest.mark.parametrize("sizes", [[2, 2, 2], [3, 1, 2, 3], [1, 0, 4]])
@pytest.mark.parametrize("sigma", [0.0, 0.9])
def test_users_match_oracle(sizes, sigma):
    B = sum(sizes)
    g = torch.Generator(device="cuda")
    g.manual_seed(sum(sizes) * 10 + len(sizes))
    A = [torch.randn(B, T, d_in, device="cuda", generator=g).bfloat16() for (d_in, _, _), T in zip(LAYERS, T_LIST)]
    E = [(torch.randn(B, T, d_out, device="cuda", generator=g) * 0.02).bfloat16()
         for (_, d_out, _), T in zip(LAYERS, T_LIST)]
    C, seed, step = 0.3, 7, 1
    pg = PrivateGradient(LAYERS)
    out = pg.step_users(A, E, T_LIST, sizes, C=C, sigma=sigma, seed=seed, step=step)
    torch.cuda.synchronize()
    ref = dpsgd.user_step([dpsgd.Layer(*ly) for ly in LAYERS], [to64(a) for a in A], [to64(e) for e in E], T_LIST,
                          sizes, C, sigma, seed, step)
    n2 = to64(out.sqnorm)
    nz = ref.user_sqnorm > 0
    assert np.all(np.abs(n2[nz] - ref.user_sqnorm[nz]) <= NORM_RTOL["bf16"] * ref.user_sqnorm[nz])
    assert np.all(n2[~nz] == 0.0)
    assert np.allclose(to64(out.clip), ref.clip, rtol=NORM_RTOL["bf16"], atol=0)
    for l, G in enumerate(out.grads):
        assert rel_fro(to64(G), ref.grads[l]) <= G_RTOL, (l, rel_fro(to64(G), ref.grads[l]))
    pg.close()
