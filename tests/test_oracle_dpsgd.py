"""Pins for the oracle's DP-SGD step (CPU only).

Each test ties the oracle to something other than itself: a worked example
printed on the pages, exact integer brute force, independent autograd, or a
sensitivity bound the pages state.
"""

import itertools
import json
import os

import numpy as np
import pytest
import torch

from oracle import dpsgd, philox
from synthetic import WORKLOADS, by_index


def _rows_as_layer(rows):
    """Vectors g_r as one linear layer with d_in = 1, T = 1, A = 1, E = g_r."""
    g = np.asarray(rows, dtype=np.float64)
    B, d = g.shape
    return np.ones((B, 1, 1)), g.reshape(B, 1, d)


def test_clip_example_printed(golden_dir):
    gx = json.load(open(os.path.join(golden_dir, "clip_example.json")))
    A, E = _rows_as_layer(gx["sample_gradients"])
    n2 = dpsgd.layer_sqnorms(A, E, False)
    c = dpsgd.clip_factors(n2, gx["clip_bound"])
    clipped = c[:, None] * np.asarray(gx["sample_gradients"])
    assert np.round(clipped, 4).tolist() == gx["printed_clipped_4dp"]
    S, _ = dpsgd.clipped_sum(A, E, c, False)
    assert [round(v, 2) for v in S[:, 0]] == gx["printed_sum_2dp"]
    # and through the whole step with sigma = 0, L = 1
    res = dpsgd.step([dpsgd.Layer(1, 2)], [A], [E], [1], C=1.0, sigma=0.0, seed=0, step_index=0, L=1.0)
    assert np.allclose(res.grads[0], [1.6, 1.9], rtol=0, atol=1e-15)
    assert res.clip.tolist() == [1.0, 0.2, 1.0]


def test_rounding_caution(golden_dir):
    gx = json.load(open(os.path.join(golden_dir, "rounding_caution.json")))
    A, E = _rows_as_layer([gx["gradient"]])
    c = dpsgd.clip_factors(dpsgd.layer_sqnorms(A, E, False), gx["clip_bound"])
    h = c[0] * np.asarray(gx["gradient"])
    assert np.round(h, 4).tolist() == gx["printed_rounded_clipped"]
    assert np.linalg.norm(np.round(h, 4)) > gx["clip_bound"]            # what the page warns of
    assert np.linalg.norm(h) <= gx["clip_bound"] * (1 + 1e-12)           # full precision stays inside


def test_alice_row_clipping(golden_dir):
    gx = json.load(open(os.path.join(golden_dir, "alice_rows.json")))
    for who in ("alice", "bao"):
        A, E = _rows_as_layer([[v] for v in gx[who]])
        c = dpsgd.clip_factors(dpsgd.layer_sqnorms(A, E, False), gx["clip_bound"])
        S, _ = dpsgd.clipped_sum(A, E, c, False)
        assert round(float(S[0, 0]), 2) == gx[f"{who}_row_clipped_sum"]


def test_appendix_a_witness_exact(golden_dir):
    """Seven bias contributions flip from -C_f to +C_f; the replaced record is +C_f in both."""
    gx = json.load(open(os.path.join(golden_dir, "witness_appendix_a.json")))
    Cf = float(np.float32(gx["clip_bound_decimal"]))
    assert Cf == gx["clip_bound_fp32"]
    n = gx["unchanged_records"]
    layer = dpsgd.Layer(1, 1, has_bias=True)

    def F(deriv_unchanged, deriv_replaced):
        g = np.array([deriv_unchanged] * n + [deriv_replaced])
        A = np.zeros((n + 1, 1, 1))           # only the bias is trainable
        E = g.reshape(-1, 1, 1)
        c = dpsgd.clip_factors(dpsgd.layer_sqnorms(A, E, True), Cf)
        S, sb = dpsgd.clipped_sum(A, E, c, True)
        assert S[0, 0] == 0.0
        return sb

    D = F(gx["bias_derivative_D"], 100.0)
    Dp = F(gx["bias_derivative_Dprime"], 50.0)
    delta = float(np.linalg.norm(D - Dp))
    assert delta == pytest.approx(gx["replacement_distance"], rel=1e-15, abs=0)
    assert delta / (2 * Cf) == pytest.approx(gx["distance_over_2C"], rel=1e-15)


def _brute_ghost(A, E, has_bias):
    """<A A^T, E E^T> (+ 1^T E E^T 1) with plain Python integer loops."""
    T = len(A)
    tot = 0
    for s in range(T):
        for t in range(T):
            ga = sum(int(A[s][k]) * int(A[t][k]) for k in range(len(A[0])))
            ge = sum(int(E[s][k]) * int(E[t][k]) for k in range(len(E[0])))
            tot += ga * ge + (ge if has_bias else 0)
    return tot


def test_ghost_identity_brute_force_exact():
    rng = np.random.default_rng(1)
    for T, d_in, d_out in itertools.product([1, 2, 3, 4], [1, 2, 5], [1, 3, 4]):
        for has_bias in (False, True):
            A = rng.integers(-2, 3, size=(1, T, d_in))
            E = rng.integers(-2, 3, size=(1, T, d_out))
            mat = dpsgd.layer_sqnorms(A, E, has_bias)[0]
            assert mat == float(_brute_ghost(A[0].tolist(), E[0].tolist(), has_bias))


def test_t1_closed_form():
    rng = np.random.default_rng(2)
    A = rng.standard_normal((5, 1, 7))
    E = rng.standard_normal((5, 1, 3))
    n2 = dpsgd.layer_sqnorms(A, E, True)
    ref = (A[:, 0] ** 2).sum(1) * (E[:, 0] ** 2).sum(1) + (E[:, 0] ** 2).sum(1)
    assert np.allclose(n2, ref, rtol=1e-13, atol=0)


def test_per_example_grad_matches_autograd():
    torch.manual_seed(0)
    B, T, d_in, d_out = 3, 5, 6, 4
    A = torch.randn(B, T, d_in, dtype=torch.float64)
    E = torch.randn(B, T, d_out, dtype=torch.float64)
    for i in range(B):
        lin = torch.nn.Linear(d_in, d_out, dtype=torch.float64)
        y = lin(A[i])
        (y * E[i]).sum().backward()          # dL/dy = E_i
        g, b = dpsgd.per_example_grad(A[i].numpy(), E[i].numpy(), True)
        assert g.shape == tuple(lin.weight.shape)
        assert np.allclose(g, lin.weight.grad.numpy(), rtol=1e-13, atol=1e-13)
        assert np.allclose(b, lin.bias.grad.numpy(), rtol=1e-13, atol=1e-13)


def test_chooser_boundaries_and_workload_decisions():
    assert dpsgd.choose_path(3, 2, 4) == dpsgd.MATERIALIZE    # 9 < 8 is false
    assert dpsgd.choose_path(3, 3, 3) == dpsgd.MATERIALIZE    # equality materializes
    assert dpsgd.choose_path(3, 5, 2) == dpsgd.GHOST          # 9 < 10
    for n in (1, 7, 100, 4096, 65535, 3 * 10 ** 6):
        assert dpsgd.choose_path(n, n, n) == dpsgd.MATERIALIZE
        assert dpsgd.choose_path(n, n * n + 1, 1) == dpsgd.GHOST
        assert dpsgd.choose_path(n, n * n - 1, 1) == dpsgd.MATERIALIZE
        assert dpsgd.choose_path(n, n * n, 1) == dpsgd.MATERIALIZE
        assert dpsgd.choose_path(n, 1, n * n + 1) == dpsgd.GHOST
    # products beyond 2^63 stay exact
    assert dpsgd.choose_path(2 ** 32, 2 ** 32, 2 ** 32 + 1) == dpsgd.GHOST
    assert dpsgd.choose_path(2 ** 32, 2 ** 32, 2 ** 32) == dpsgd.MATERIALIZE
    decisions = {w.index: [dpsgd.choose_path(l.T, l.d_in, l.d_out) for l in w.layers] for w in WORKLOADS}
    assert decisions[1] == [dpsgd.GHOST]
    assert decisions[2] == [dpsgd.MATERIALIZE] * 48
    assert decisions[3] == [dpsgd.GHOST]
    assert decisions[4] == [dpsgd.GHOST, dpsgd.GHOST]
    assert decisions[5] == [dpsgd.MATERIALIZE] * 12 + [dpsgd.GHOST]


def test_clip_invariants():
    rng = np.random.default_rng(3)
    C = 0.7
    g = rng.standard_normal((200, 11)) * rng.uniform(0, 10 * C, size=(200, 1)) / np.sqrt(11)
    g[0] = 0.0
    n2 = (g ** 2).sum(1)
    c = dpsgd.clip_factors(n2, C)
    h = c[:, None] * g
    assert np.all(np.linalg.norm(h, axis=1) <= C * (1 + 1e-12))
    small = np.sqrt(n2) <= C
    assert np.all(c[small] == 1.0) and np.array_equal(h[small], g[small])
    assert c[0] == 1.0 and np.all(h[0] == 0.0)
    assert np.allclose(np.linalg.norm(h[~small], axis=1), C, rtol=1e-13)


def test_invalid_arguments_rejected():
    with pytest.raises(ValueError):
        dpsgd.clip_factors(np.ones(2), 0.0)
    with pytest.raises(ValueError):
        dpsgd.clip_factors(np.ones(2), float("inf"))
    with pytest.raises(ValueError):
        dpsgd.clip_factors(np.array([1.0, np.nan]), 1.0)
    with pytest.raises(ValueError):
        dpsgd.clip_factors(np.array([1.0, np.inf]), 1.0)
    A, E = np.ones((2, 1, 1)), np.ones((2, 1, 1))
    with pytest.raises(ValueError):
        dpsgd.step([dpsgd.Layer(1, 1)], [A], [E], [1], C=1.0, sigma=-1.0, seed=0, step_index=0)
    with pytest.raises(ValueError):
        dpsgd.step([dpsgd.Layer(1, 1)], [A], [E], [1], C=1.0, sigma=1.0, seed=0, step_index=0, L=0.0)


def _two_layer_batch(rng, B):
    layers = [dpsgd.Layer(4, 3, True), dpsgd.Layer(3, 2, False)]
    A = [rng.standard_normal((B, 2, 4)), rng.standard_normal((B, 2, 3))]
    E = [rng.standard_normal((B, 2, 3)), rng.standard_normal((B, 2, 2))]
    return layers, A, E


def _flat_sum(layers, A, E, C):
    res = dpsgd.step(layers, A, E, [2, 2], C=C, sigma=0.0, seed=0, step_index=0, L=1.0)
    return np.concatenate(res.grads)


def test_sensitivity_add_remove_and_replace():
    """Proposition 1 with m = 0: add/remove moves the clipped sum by <= C, replacement by <= 2C."""
    rng = np.random.default_rng(4)
    C = 0.5
    worst_add, worst_rep = 0.0, 0.0
    for trial in range(40):
        layers, A, E = _two_layer_batch(rng, 6)
        if trial % 4 == 0:             # adversarial: one record with norm >> C
            A[0][-1] *= 30.0
        base = _flat_sum(layers, A, E, C)
        rem = _flat_sum(layers, [a[:-1] for a in A], [e[:-1] for e in E], C)
        worst_add = max(worst_add, np.linalg.norm(base - rem) / C)
        A2 = [a.copy() for a in A]
        E2 = [e.copy() for e in E]
        A2[0][-1] = -40.0 * A[0][-1]
        E2[1][-1] = rng.standard_normal(E2[1][-1].shape)
        rep = _flat_sum(layers, A2, E2, C)
        worst_rep = max(worst_rep, np.linalg.norm(base - rep) / C)
    assert worst_add <= 1.0 + 1e-12
    assert worst_rep <= 2.0 + 1e-12
    assert worst_add > 0.99            # the bound is attained by clipped records


def test_clip_of_mean_anti_pattern_exceeds_bound():
    """Clipping the aggregate instead of each record breaks the add/remove bound C."""
    C = 1.0
    u = np.array([1.0, 0.0])
    D = [10 * C * u, 10 * C * u]
    Dp = D + [-100 * C * u]

    def clip_mean(rows):
        m = np.mean(rows, axis=0)
        return m * min(1.0, C / np.linalg.norm(m))

    assert np.linalg.norm(clip_mean(D) - clip_mean(Dp)) == pytest.approx(2 * C)
    A, E = _rows_as_layer(D)
    Ap, Ep = _rows_as_layer(Dp)
    s = dpsgd.clipped_sum(A, E, dpsgd.clip_factors(dpsgd.layer_sqnorms(A, E, False), C), False)[0]
    sp = dpsgd.clipped_sum(Ap, Ep, dpsgd.clip_factors(dpsgd.layer_sqnorms(Ap, Ep, False), C), False)[0]
    assert np.linalg.norm(s - sp) <= C * (1 + 1e-12)


def test_sigma_zero_and_noise_once():
    rng = np.random.default_rng(5)
    layers, A, E = _two_layer_batch(rng, 5)
    r0 = dpsgd.step(layers, A, E, [2, 2], C=0.3, sigma=0.0, seed=9, step_index=4)
    r1 = dpsgd.step(layers, A, E, [2, 2], C=0.3, sigma=1.3, seed=9, step_index=4)
    offs, P = dpsgd.coordinate_offsets(layers)
    assert P == 3 * 4 + 3 + 2 * 3
    z = philox.normals(9, 4, 0, P)
    for ly, g0, g1, S_sb, off in zip(layers, r0.grads, r1.grads, r0.clipped, offs):
        S, sb = S_sb
        flat = S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
        assert np.array_equal(g0, flat / 5.0)                       # L defaults to B
        diff = g1 - g0
        assert np.allclose(diff, 1.3 * 0.3 * z[off:off + ly.ncoords] / 5.0, rtol=1e-12, atol=1e-15)
        assert np.all(diff != 0.0)                                   # every coordinate noised
    # the public normalizer override
    r2 = dpsgd.step(layers, A, E, [2, 2], C=0.3, sigma=0.0, seed=9, step_index=4, L=64.0)
    assert np.allclose(r2.grads[0] * 64.0, r0.grads[0] * 5.0, rtol=1e-14)


def test_clipped_sum_at_matches_full():
    rng = np.random.default_rng(6)
    A = rng.standard_normal((4, 3, 5))
    E = rng.standard_normal((4, 3, 6))
    c = rng.uniform(0.1, 1.0, 4)
    S, _ = dpsgd.clipped_sum(A, E, c, False)
    rows = np.array([0, 5, 2, 2])
    cols = np.array([4, 0, 1, 3])
    assert np.allclose(dpsgd.clipped_sum_at(A, E, c, rows, cols), S[rows, cols], rtol=1e-13)


def test_workload_shapes_and_counts():
    w2 = by_index(2)
    assert len(w2.layers) == 48 and w2.ncoords == 294_912
    w5 = by_index(5)
    assert len(w5.layers) == 13 and w5.ncoords == 59_834_368
    assert by_index(3).ncoords == 16_777_216
    assert by_index(4).ncoords == 8_388_608
    assert by_index(1).ncoords == 2080
