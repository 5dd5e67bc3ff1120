"""The one-step privacy loss of a neighbouring pair ("Sensitivity Inflation
from Cross-Record Precision Routing in Private Quantized Fine-Tuning",
section 3.2, Eq. 5), pinned to the values the page prints and to a direct
numerical integration of the hockey-stick divergence."""

from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

from differentially_private_gb300.audit import delta_pair, epsilon_for

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "eq5_one_step_epsilon.json")


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"])
def test_printed_epsilons(case):
    eps = epsilon_for(case["delta"], case["mu"])
    assert abs(eps - case["epsilon"]) <= case["abs_tol"], (case, eps)


def _hockey_stick_by_quadrature(eps: float, mu: float) -> float:
    """sup over events of P[N(mu,1) in S] - e^eps P[N(0,1) in S], integrated
    directly: the integral of max(0, phi(x - mu) - e^eps phi(x))."""
    from scipy.integrate import quad
    phi = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)  # noqa: E731
    f = lambda x: max(0.0, phi(x - mu) - math.exp(eps) * phi(x))  # noqa: E731
    # the integrand is positive only above x0 = mu/2 + eps/mu
    x0 = mu / 2.0 + eps / mu
    val, _ = quad(f, x0, x0 + 40.0, limit=400, epsabs=1e-15, epsrel=1e-12)
    return val


@pytest.mark.parametrize("eps,mu", [(0.0, 1.0), (0.5, 1.0), (2.0, 1.065), (4.0, 2.0), (1.0, 0.3)])
def test_matches_direct_integration(eps, mu):
    assert delta_pair(eps, mu) == pytest.approx(_hockey_stick_by_quadrature(eps, mu), rel=1e-7, abs=1e-15)


def test_zero_distance_and_monotone():
    assert delta_pair(3.0, 0.0) == 0.0
    assert epsilon_for(1e-5, 0.0) == 0.0
    d = [delta_pair(e, 1.0) for e in np.linspace(0.0, 8.0, 41)]
    assert all(a >= b for a, b in zip(d, d[1:]))
    # a larger distance costs more privacy at the same delta
    assert epsilon_for(1e-5, 1.2) > epsilon_for(1e-5, 1.0) > epsilon_for(1e-5, 0.8)


def test_inverse():
    for mu in (0.5, 1.0, 3.0):
        for delta in (1e-3, 1e-6):
            assert delta_pair(epsilon_for(delta, mu), mu) == pytest.approx(delta, rel=1e-8)
