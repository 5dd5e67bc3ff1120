"""Tensor-core clipped sum with the tiles of a partial last wave split
into record ranges over the grid.

When a layer's tile count leaves a partial last wave, each remaining tile's
records are cut into ranges run side by side on otherwise idle SMs; every
range writes a partial sum and the CTA that arrives last at the tile adds
them in range order.  These cases put every tile, or the last wave, into
that mode and check G tile by tile against the oracle at sigma = 0, that the
noise of every coordinate is added exactly once, and that repeats are
bitwise equal.  Layers of one pre-scaled record (T not a multiple of 64:
the clip kernel writes c_i X_i, and the sum runs on whole tiles) are checked
the same way, several layers and several row counts in one step.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_harness import G_RTOL, gpu_step, oracle_step, to64
from oracle import philox

pytestmark = pytest.mark.gpu

# errors are checked per 128 x 256 block (rows of d_out x columns of d_in); the
# per-record fold runs on 256 x 256 tiles of CTA pairs, each CTA folding 128 rows
TILE_M, TILE_N = 128, 256


def _inputs(B, T, d_in, d_out, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    A = torch.randn(B, T, d_in, device="cuda", generator=g).bfloat16()
    scale = torch.exp(torch.randn(B, 1, 1, device="cuda", generator=g))
    E = (torch.randn(B, T, d_out, device="cuda", generator=g) * 0.05 * scale).bfloat16()
    return A, E


def _tile_errors(got, want, d_out, d_in):
    """Relative Frobenius error of every output tile."""
    errs = []
    for m0 in range(0, d_out, TILE_M):
        for n0 in range(0, d_in, TILE_N):
            w = want[m0:m0 + TILE_M, n0:n0 + TILE_N]
            gt = got[m0:m0 + TILE_M, n0:n0 + TILE_N]
            den = np.linalg.norm(w)
            errs.append(float(np.linalg.norm(gt - w) / (den if den > 0 else 1.0)))
    return np.array(errs)


@pytest.mark.parametrize("B,T,d_in,d_out", [
    (40, 512, 512, 256),    # 2 pair tiles of 40 records, each cut into 38 ranges (76 pairs)
    (20, 512, 2560, 2048),  # 80 pair tiles: one full wave of 76, then 4 tiles cut into 19 ranges
    (6500, 3, 256, 512),    # one pre-scaled record of 19500 rows: whole tiles
    (40, 128, 328, 200),    # widths not multiples of 64 (2D tensor maps), ragged in both
                            # directions: 2 pair tiles, each cut into 10 ranges of 4 records
    (12, 64, 640, 384),     # 3D maps, partial pair tiles: the second CTA of the last row
                            # block lies wholly past d_out (zero-filled loads, no stores)
])
def test_split_tiles_match_oracle(B, T, d_in, d_out):
    A, E = _inputs(B, T, d_in, d_out, seed=B * 7 + T)
    layers = [(d_in, d_out, False)]
    C, sigma, seed, step = 0.7, 0.9, 11, 4
    out0, _ = gpu_step(layers, [A], [E], [T], C, 0.0, seed, step, layer_norms=False)
    ref = oracle_step(layers, [A], [E], [T], C, 0.0, seed, step)
    S, _ = ref.clipped[0]
    G0 = to64(out0.grads[0]).reshape(d_out, d_in)
    errs = _tile_errors(G0, S / B, d_out, d_in)
    assert np.all(errs <= G_RTOL), (errs.max(), int(errs.argmax()))

    # the noise of every coordinate enters exactly once: G(sigma) - G(0) = sigma C z / L
    outs, _ = gpu_step(layers, [A], [E], [T], C, sigma, seed, step, layer_norms=False)
    Gs = to64(outs.grads[0]).reshape(d_out, d_in)
    z = philox.normals(seed, step, 0, d_out * d_in).reshape(d_out, d_in)
    diff = Gs - G0
    tol = 1e-3 * sigma * C / B + 4e-7 * np.abs(G0) + 1e-5 * np.abs(S).max() / B
    bad = np.abs(diff - sigma * C * z / B) > tol
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:4])


def test_split_tiles_repeat_bitwise():
    """The fixed summation order makes repeated steps of one context (new
    counter tags every launch) bitwise identical."""
    from differentially_private_gb300 import PrivateGradient
    B, T, d_in, d_out = 40, 512, 512, 256
    A, E = _inputs(B, T, d_in, d_out, seed=5)
    pg = PrivateGradient([(d_in, d_out, False)], dtype=torch.bfloat16)
    runs = []
    for _ in range(3):
        out = pg.step([A], [E], [T], C=1.0, sigma=1.0, seed=3, step=2)
        torch.cuda.synchronize()
        runs.append(out.grads[0].clone())
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])


def test_prescaled_layers_match_oracle_noise_once_and_repeat():
    """Four pre-scaled layers (all written by the clip kernel) of two row
    counts, ragged shapes (2D tensor maps, partial tiles), at sigma = 0 tile
    by tile, the noise once per coordinate, and bitwise repeats."""
    from differentially_private_gb300 import PrivateGradient
    B = 300
    shapes = [(1024, 512, 3), (512, 1024, 3), (320, 200, 3), (640, 384, 5)]
    layers = [(d_in, d_out, False) for (d_in, d_out, _) in shapes]
    A, E, T = [], [], []
    for i, (d_in, d_out, t) in enumerate(shapes):
        a, e = _inputs(B, t, d_in, d_out, seed=40 + i)
        A.append(a)
        E.append(e)
        T.append(t)
    C, sigma, seed, step = 0.8, 1.1, 21, 6
    out0, _ = gpu_step(layers, A, E, T, C, 0.0, seed, step, layer_norms=False)
    outs, _ = gpu_step(layers, A, E, T, C, sigma, seed, step, layer_norms=False)
    ref = oracle_step(layers, A, E, T, C, 0.0, seed, step)
    off = 0
    for l, (d_in, d_out, _) in enumerate(shapes):
        S, _ = ref.clipped[l]
        G0 = to64(out0.grads[l]).reshape(d_out, d_in)
        errs = _tile_errors(G0, S / B, d_out, d_in)
        assert np.all(errs <= G_RTOL), (l, errs.max(), int(errs.argmax()))
        Gs = to64(outs.grads[l]).reshape(d_out, d_in)
        z = philox.normals(seed, step, off, d_out * d_in).reshape(d_out, d_in)
        tol = 1e-3 * sigma * C / B + 4e-7 * np.abs(G0) + 1e-5 * np.abs(S).max() / B
        bad = np.abs(Gs - G0 - sigma * C * z / B) > tol
        assert not bad.any(), (l, int(bad.sum()), np.argwhere(bad)[:4])
        off += d_out * d_in
    pg = PrivateGradient(layers, dtype=torch.bfloat16)
    runs = []
    for _ in range(3):
        out = pg.step(A, E, T, C=C, sigma=sigma, seed=seed, step=step)
        torch.cuda.synchronize()
        runs.append([g.clone() for g in out.grads])
    for r in runs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(runs[0], r))
    pg.close()


def test_two_split_layers_in_one_step():
    """Two per-record layers whose last waves are both split into record
    ranges (one with 3D, one with 2D tensor maps) in one step: the second
    launch reuses the context's arrival counters under a new tag, and each
    layer's G matches the oracle tile by tile with its own noise once."""
    B, T = 40, 64
    shapes = [(512, 256), (328, 200)]
    layers = [(d_in, d_out, False) for d_in, d_out in shapes]
    A, E = [], []
    for i, (d_in, d_out) in enumerate(shapes):
        a, e = _inputs(B, T, d_in, d_out, seed=70 + i)
        A.append(a)
        E.append(e)
    C, sigma, seed, step = 0.6, 1.3, 8, 3
    out0, _ = gpu_step(layers, A, E, [T, T], C, 0.0, seed, step, layer_norms=False)
    outs, _ = gpu_step(layers, A, E, [T, T], C, sigma, seed, step, layer_norms=False)
    ref = oracle_step(layers, A, E, [T, T], C, 0.0, seed, step)
    off = 0
    for l, (d_in, d_out) in enumerate(shapes):
        S, _ = ref.clipped[l]
        G0 = to64(out0.grads[l]).reshape(d_out, d_in)
        errs = _tile_errors(G0, S / B, d_out, d_in)
        assert np.all(errs <= G_RTOL), (l, errs.max(), int(errs.argmax()))
        Gs = to64(outs.grads[l]).reshape(d_out, d_in)
        z = philox.normals(seed, step, off, d_out * d_in).reshape(d_out, d_in)
        tol = 1e-3 * sigma * C / B + 4e-7 * np.abs(G0) + 1e-5 * np.abs(S).max() / B
        bad = np.abs(Gs - G0 - sigma * C * z / B) > tol
        assert not bad.any(), (l, int(bad.sum()), np.argwhere(bad)[:4])
        off += d_out * d_in


def test_four_layers_in_one_sum_launch_and_a_fifth_beside():
    """Five pre-scaled layers of one row count: the clip kernel scales the
    first four, which are summed in one launch of four layers (the most one
    launch carries); the fifth is scaled by its own kernel and summed alone.
    Each G matches the oracle tile by tile at sigma = 0 and carries its own
    noise once at sigma."""
    B, T = 200, 3
    shapes = [(256, 512), (512, 256), (320, 200), (136, 264), (384, 640)]
    layers = [(d_in, d_out, False) for d_in, d_out in shapes]
    A, E = [], []
    for i, (d_in, d_out) in enumerate(shapes):
        a, e = _inputs(B, T, d_in, d_out, seed=90 + i)
        A.append(a)
        E.append(e)
    C, sigma, seed, step = 0.9, 0.8, 13, 5
    out0, _ = gpu_step(layers, A, E, [T] * 5, C, 0.0, seed, step, layer_norms=False)
    outs, _ = gpu_step(layers, A, E, [T] * 5, C, sigma, seed, step, layer_norms=False)
    ref = oracle_step(layers, A, E, [T] * 5, C, 0.0, seed, step)
    off = 0
    for l, (d_in, d_out) in enumerate(shapes):
        S, _ = ref.clipped[l]
        G0 = to64(out0.grads[l]).reshape(d_out, d_in)
        errs = _tile_errors(G0, S / B, d_out, d_in)
        assert np.all(errs <= G_RTOL), (l, errs.max(), int(errs.argmax()))
        Gs = to64(outs.grads[l]).reshape(d_out, d_in)
        z = philox.normals(seed, step, off, d_out * d_in).reshape(d_out, d_in)
        tol = 1e-3 * sigma * C / B + 4e-7 * np.abs(G0) + 1e-5 * np.abs(S).max() / B
        bad = np.abs(Gs - G0 - sigma * C * z / B) > tol
        assert not bad.any(), (l, int(bad.sum()), np.argwhere(bad)[:4])
        off += d_out * d_in


def test_batch_of_one_record_applies_its_clip_factor():
    """B = 1 with T a multiple of 64: the sum runs as one record of T rows
    with the record's own clip factor c_0 applied in the epilogue (no
    pre-scaled copy); the record is clipped (its norm is far above C)."""
    B, T, d_in, d_out = 1, 128, 320, 256
    A, E = _inputs(B, T, d_in, d_out, seed=123)
    layers = [(d_in, d_out, False)]
    C, sigma, seed, step = 0.05, 0.5, 2, 9
    out0, _ = gpu_step(layers, [A], [E], [T], C, 0.0, seed, step, layer_norms=False)
    ref = oracle_step(layers, [A], [E], [T], C, 0.0, seed, step)
    assert float(ref.clip[0]) < 0.5
    S, _ = ref.clipped[0]
    G0 = to64(out0.grads[0]).reshape(d_out, d_in)
    errs = _tile_errors(G0, S / B, d_out, d_in)
    assert np.all(errs <= G_RTOL), (errs.max(), int(errs.argmax()))
    outs, _ = gpu_step(layers, [A], [E], [T], C, sigma, seed, step, layer_norms=False)
    Gs = to64(outs.grads[0]).reshape(d_out, d_in)
    z = philox.normals(seed, step, 0, d_out * d_in).reshape(d_out, d_in)
    tol = 1e-3 * sigma * C / B + 4e-7 * np.abs(G0) + 1e-5 * np.abs(S).max() / B
    bad = np.abs(Gs - G0 - sigma * C * z / B) > tol
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:4])
