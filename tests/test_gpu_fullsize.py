"""Full-size workloads, in the launch configuration bench.py times, on sampled outputs.

At these sizes the oracle cannot produce the whole step, so each check uses
outputs it can compute one by one:
* per-example norms of sampled records (materialized per record in float64)
  and their clip factors, at the workload's C and sigma;
* the clipped sum with every clip factor equal to one (C above every norm,
  sigma = 0) at sampled coordinates: sum_i E_i[:, m]^T A_i[:, n] / L;
* the noise at sampled coordinates: G(sigma) - G(0) = sigma C z_k / L, both
  runs with the same C.
* for the ghost-path workloads 3 and 5, the clipped sum at the workload's
  own C (clip factors below one, sigma = 0) at sampled coordinates:
  sum_i c_i E_i[:, m]^T A_i[:, n] / L with c_i from the oracle's norms of
  all B records (each record's gradient materialized in float64), which
  exercises the per-record fold of the clipped-sum kernel in the launch
  shape the bench times.
Clip factors below one are also covered element by element at reduced sizes
(test_gpu_parity.py).  No oracle input comes from the GPU path: the GPU only
supplies the input bytes (drawn by synthetic/) and the outputs under test.
"""

import numpy as np
import pytest
import torch

from gpu_harness import NORM_RTOL, to64
from oracle import dpsgd, philox
from synthetic import by_index, generate_layer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLED_RECORDS = {3: [0, 17, 63], 4: [0, 1, 2047, 4095], 5: [0, 31]}
SAMPLED_COORDS = 192
C_ALL_ONE = 1e30      # above every norm: every clip factor is 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


def _run(w, A, E, C, sigma, seed, step):
    import differentially_private_gb300 as dp
    layers = [(ly.d_in, ly.d_out, ly.has_bias) for ly in w.layers]
    pg = dp.PrivateGradient(layers, dtype=w.torch_dtype)
    out = pg.step(A, E, [ly.T for ly in w.layers], C=C, sigma=sigma, seed=seed, step=step, layer_norms=True)
    torch.cuda.synchronize()
    offs = [off for (_, _, _, off, _) in pg.layers]
    pg.close()
    return out, offs


@pytest.mark.parametrize("widx", [3, 4, 5])
def test_fullsize_workload(widx):
    w = by_index(widx)
    A, E = [], []
    for i in range(len(w.layers)):
        a, e = generate_layer(w, i, "cuda")
        A.append(a)
        E.append(e)
    rng = np.random.default_rng(widx)
    recs = SAMPLED_RECORDS[widx]

    # 1. norms and clip factors of sampled records, at the workload's C and sigma
    out, offs = _run(w, A, E, w.C, w.sigma, w.noise_seed, w.step)
    n2_tot = np.zeros(len(recs))
    for l, ly in enumerate(w.layers):
        got = to64(out.layer_sqnorm[l])[recs]
        want = np.array([dpsgd.record_sqnorm(to64(A[l][r]), to64(E[l][r]), ly.has_bias) for r in recs])
        assert np.all(np.abs(got - want) <= NORM_RTOL["bf16"] * want), (l, got, want)
        n2_tot += want
    c_want = dpsgd.clip_factors(n2_tot, w.C)
    assert np.allclose(to64(out.clip)[recs], c_want, rtol=NORM_RTOL["bf16"], atol=0)
    del out

    # 2. the sum with every clip factor one, at sampled coordinates
    g0, offs = _run(w, A, E, C_ALL_ONE, 0.0, 7, 3)
    assert bool((g0.clip == 1.0).all())
    ones = np.ones(w.B)
    for l, ly in enumerate(w.layers):
        rows = rng.integers(0, ly.d_out, SAMPLED_COORDS)
        cols = rng.integers(0, ly.d_in, SAMPLED_COORDS)
        Esub = to64(E[l][:, :, torch.as_tensor(rows, device="cuda")])
        Asub = to64(A[l][:, :, torch.as_tensor(cols, device="cuda")])
        q = np.arange(SAMPLED_COORDS)
        want = dpsgd.clipped_sum_at(Asub, Esub, ones, q, q) / w.B
        got = to64(g0.grads[l])[rows * ly.d_in + cols]
        err = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err <= 5e-3, (l, err)

    # 3. the noise: same C in both runs, so the clipped parts are identical
    sigma, C = 0.9, 1e3
    gs, _ = _run(w, A, E, C, sigma, 7, 3)
    gz, _ = _run(w, A, E, C, 0.0, 7, 3)
    for l, ly in enumerate(w.layers):
        p = rng.integers(0, ly.d_out * ly.d_in, SAMPLED_COORDS)
        diff = to64(gs.grads[l])[p] - to64(gz.grads[l])[p]
        want = sigma * C * philox.normals_at(7, 3, offs[l] + p) / w.B
        assert np.allclose(diff, want, rtol=1e-4, atol=2e-6 * sigma * C / w.B), l


@pytest.mark.parametrize("widx", [3, 5])
def test_fullsize_clipped_sum_at_the_workload_clip_bound(widx):
    w = by_index(widx)
    A, E = [], []
    for i in range(len(w.layers)):
        a, e = generate_layer(w, i, "cuda")
        A.append(a)
        E.append(e)
    # the oracle's clip factors: every record's gradient materialized in float64
    n2 = np.zeros(w.B)
    for r in range(w.B):
        for l, ly in enumerate(w.layers):
            n2[r] += dpsgd.record_sqnorm(to64(A[l][r]), to64(E[l][r]), ly.has_bias)
    c = dpsgd.clip_factors(n2, w.C)
    assert np.any(c < 1.0)
    out, _ = _run(w, A, E, w.C, 0.0, 7, 3)
    assert np.allclose(to64(out.clip), c, rtol=NORM_RTOL["bf16"], atol=0)
    rng = np.random.default_rng(100 + widx)
    # the ghost-path layer (the dense one): its sum is the per-record fold
    for l, ly in enumerate(w.layers):
        if dpsgd.choose_path(ly.T, ly.d_in, ly.d_out) != dpsgd.GHOST:
            continue
        rows = rng.integers(0, ly.d_out, SAMPLED_COORDS)
        cols = rng.integers(0, ly.d_in, SAMPLED_COORDS)
        Esub = to64(E[l][:, :, torch.as_tensor(rows, device="cuda")])
        Asub = to64(A[l][:, :, torch.as_tensor(cols, device="cuda")])
        q = np.arange(SAMPLED_COORDS)
        want = dpsgd.clipped_sum_at(Asub, Esub, c, q, q) / w.B
        got = to64(out.grads[l])[rows * ly.d_in + cols]
        err = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err <= 5e-3, (l, err)
