"""The sensitivity audit run on the library's kernels ("Sensitivity Inflation
from Cross-Record Precision Routing in Private Quantized Fine-Tuning",
section 5, Algorithm 2's native arm, and Proposition 1 with no cross-record
influence): add/remove distances stay within C and replacement within 2C,
agree with the float64 oracle, and per-record norms do not depend on the
batch."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from differentially_private_gb300.audit import SensitivityAudit, epsilon_for
from gpu_harness import oracle_step

pytestmark = pytest.mark.gpu

# a ghost tensor-core layer, a materialized LoRA factor and a T = 1 layer
LAYERS = [(256, 128, False), (768, 8, False), (256, 512, False)]
T_LIST = [64, 128, 1]


def _batch(B, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    A, E = [], []
    for (d_in, d_out, _), T in zip(LAYERS, T_LIST):
        A.append(torch.randn(B, T, d_in, device="cuda", generator=g).bfloat16())
        E.append((torch.randn(B, T, d_out, device="cuda", generator=g) * 0.02 * scale).bfloat16())
    return A, E


def _oracle_F(A, E, C):
    ref = oracle_step(LAYERS, A, E, T_LIST, C, 0.0, 0, 0, L=1.0)
    return np.concatenate([g.reshape(-1) for g in ref.grads])


@pytest.mark.parametrize("C", [1e3, 1.0, 0.05, 1e-3])
def test_add_remove_within_C_and_matches_oracle(C):
    D = _batch(6, seed=1)
    x = _batch(1, seed=2, scale=10.0)        # a record far above most radii
    audit = SensitivityAudit(LAYERS)
    kappa = audit.add_remove(D, x, T_LIST, C)
    f0 = _oracle_F(*D, C)
    f1 = _oracle_F([torch.cat([a, b]) for a, b in zip(D[0], x[0])],
                   [torch.cat([e, b]) for e, b in zip(D[1], x[1])], C)
    want = float(np.linalg.norm(f1 - f0) / C)
    assert kappa <= 1.0 + 1e-5, kappa
    assert kappa == pytest.approx(want, rel=5e-3), (kappa, want)
    if C <= 0.05:
        # the added record is clipped: it moves the sum by exactly C
        assert kappa == pytest.approx(1.0, abs=1e-4)
    audit.close()


@pytest.mark.parametrize("C", [1.0, 1e-3])
def test_replace_within_2C(C):
    D = _batch(6, seed=3)
    x = _batch(1, seed=4, scale=10.0)
    audit = SensitivityAudit(LAYERS)
    rho = audit.replace(D, 2, x, T_LIST, C)
    A2 = [a.clone() for a in D[0]]
    E2 = [e.clone() for e in D[1]]
    for a2, b in zip(A2, x[0]):
        a2[2] = b[0]
    for e2, b in zip(E2, x[1]):
        e2[2] = b[0]
    want = float(np.linalg.norm(_oracle_F(A2, E2, C) - _oracle_F(*D, C)) / (2 * C))
    assert rho <= 1.0 + 1e-5, rho
    assert rho == pytest.approx(want, rel=5e-3)
    audit.close()


def test_norms_batch_invariant_and_epsilon_of_the_measured_pair():
    D = _batch(5, seed=6)
    audit = SensitivityAudit(LAYERS)
    assert audit.norms_batch_invariant(D, T_LIST)
    # at sigma = 1 a record-isolated computation's measured pair costs at most
    # the advertised one-step epsilon of mu = 1 (4.38 at delta = 1e-5)
    kappa = audit.add_remove(D, _batch(1, seed=7, scale=10.0), T_LIST, 1e-3)
    assert epsilon_for(1e-5, kappa) <= epsilon_for(1e-5, 1.0) + 1e-3
    audit.close()
