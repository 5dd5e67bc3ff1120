"""Pins of the oracle's user-level clipping ("Privacy-Preserving Machine
Learning", section "Differentially private stochastic gradient descent",
the user-level construction and its sum-then-user-clip example)."""

from __future__ import annotations

import json
import os

import numpy as np
import pytest

from oracle import dpsgd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "alice_users.json")


def _scalar_batch(values):
    """A d_in = d_out = 1, T = 1 layer whose per-example gradient is the value:
    A = 1, E = value."""
    v = np.asarray(values, dtype=np.float64).reshape(-1, 1, 1)
    return np.ones_like(v), v


def test_alice_and_bao_printed_values():
    gx = json.load(open(GOLDEN))
    C, L = gx["clip_bound"], gx["normalizer"]
    alice, bao = gx["users"]["Alice"], gx["users"]["Bao"]
    layers = [dpsgd.Layer(1, 1, False)]
    A, E = _scalar_batch(alice + bao)
    with_alice = dpsgd.user_step(layers, [A], [E], [1], [len(alice), len(bao)], C, 0.0, 0, 0, L=L)
    # each user's clipped vector: c_u times the user's summed gradient
    user_clipped = with_alice.clip * np.sqrt(with_alice.user_sqnorm)
    assert user_clipped[0] == pytest.approx(gx["user_clipped"]["Alice"], abs=5e-3)
    assert user_clipped[1] == pytest.approx(gx["user_clipped"]["Bao"], abs=5e-3)
    assert with_alice.grads[0][0] == pytest.approx(gx["with_alice"], abs=5e-4)
    A2, E2 = _scalar_batch(bao)
    without = dpsgd.user_step(layers, [A2], [E2], [1], [len(bao)], C, 0.0, 0, 0, L=L)
    assert without.grads[0][0] == pytest.approx(gx["without_alice"], abs=5e-4)
    change = with_alice.grads[0][0] - without.grads[0][0]
    assert change == pytest.approx(gx["change"], abs=5e-4)
    assert abs(change) <= C / L * (1 + 1e-12)


def test_singleton_users_are_the_record_level_step():
    rng = np.random.default_rng(3)
    layers = [dpsgd.Layer(5, 4, True), dpsgd.Layer(3, 6, False)]
    T = [3, 2]
    A = [rng.normal(size=(6, t, ly.d_in)) for ly, t in zip(layers, T)]
    E = [rng.normal(size=(6, t, ly.d_out)) for ly, t in zip(layers, T)]
    rec = dpsgd.step(layers, A, E, T, 0.7, 1.3, 5, 2, L=6.0)
    usr = dpsgd.user_step(layers, A, E, T, [1] * 6, 0.7, 1.3, 5, 2, L=6.0)
    np.testing.assert_allclose(usr.user_sqnorm, rec.total_sqnorm, rtol=1e-12)
    for a, b in zip(usr.grads, rec.grads):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_aligned_records_clip_to_C_as_one_user():
    # two records with the same gradient direction, each of norm 0.8 C:
    # record-level clipping leaves 1.6 C, user-level clipping C
    C = 1.0
    layers = [dpsgd.Layer(1, 1, False)]
    A, E = _scalar_batch([0.8, 0.8])
    rec = dpsgd.step(layers, [A], [E], [1], C, 0.0, 0, 0, L=1.0)
    usr = dpsgd.user_step(layers, [A], [E], [1], [2], C, 0.0, 0, 0, L=1.0)
    assert rec.grads[0][0] == pytest.approx(1.6)
    assert usr.grads[0][0] == pytest.approx(1.0)


def test_user_level_add_remove_sensitivity_at_most_C():
    rng = np.random.default_rng(9)
    layers = [dpsgd.Layer(4, 3, True)]
    C = 0.5
    sizes = [2, 1, 3]
    A = rng.normal(size=(6, 2, 4))
    E = rng.normal(size=(6, 2, 3)) * 3.0
    full = dpsgd.user_step(layers, [A], [E], [2], sizes, C, 0.0, 0, 0, L=1.0)
    # remove the last user (its 3 records)
    part = dpsgd.user_step(layers, [A[:3]], [E[:3]], [2], sizes[:2], C, 0.0, 0, 0, L=1.0)
    d = np.linalg.norm(full.grads[0] - part.grads[0])
    assert d <= C * (1 + 1e-12)
    assert d == pytest.approx(C)      # the removed user's vector is clipped to exactly C


def test_zero_record_user_and_errors():
    layers = [dpsgd.Layer(1, 1, False)]
    A, E = _scalar_batch([0.3, 0.4])
    r = dpsgd.user_step(layers, [A], [E], [1], [2, 0], 1.0, 0.0, 0, 0, L=1.0)
    assert r.user_sqnorm[1] == 0.0 and r.clip[1] == 1.0
    with pytest.raises(ValueError):
        dpsgd.user_step(layers, [A], [E], [1], [1], 1.0, 0.0, 0, 0)
    with pytest.raises(ValueError):
        dpsgd.user_step(layers, [A], [E], [1], [3, -1], 1.0, 0.0, 0, 0)
