"""Shared helpers of the GPU parity tests: run a step through the C ABI and
through the CPU oracle on the same input bytes, and compare."""

from __future__ import annotations

import numpy as np
import torch

from oracle import dpsgd, philox

NORM_RTOL = {"f32": 1e-3, "bf16": 5e-3}
G_RTOL = 5e-3
Z_ATOL = 1e-6


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def gpu_step(layers, A_list, E_list, T_list, C, sigma, seed, step, L=None, dtype=torch.bfloat16,
             batch=True, layer_norms=True):
    """layers: list of (d_in, d_out, has_bias); A/E on cuda.  Returns (out, pg)."""
    from differentially_private_gb300 import PrivateGradient
    pg = PrivateGradient(layers, dtype=dtype)
    out = pg.step(A_list, E_list, T_list, C=C, sigma=sigma, seed=seed, step=step, L=L,
                  layer_norms=layer_norms, batch=batch)
    torch.cuda.synchronize()
    return out, pg


def oracle_step(layers, A_list, E_list, T_list, C, sigma, seed, step, L=None):
    ol = [dpsgd.Layer(d_in, d_out, hb) for (d_in, d_out, hb) in layers]
    return dpsgd.step(ol, [to64(a) for a in A_list], [to64(e) for e in E_list], T_list,
                      C=C, sigma=sigma, seed=seed, step_index=step, L=L)


def assert_step_parity(layers, A_list, E_list, T_list, C, sigma, seed, step, L=None,
                       dtype=torch.bfloat16, dtag="bf16"):
    """Norms, clip factors and G against the oracle, at sigma and at sigma = 0."""
    out, pg = gpu_step(layers, A_list, E_list, T_list, C, sigma, seed, step, L, dtype)
    ref = oracle_step(layers, A_list, E_list, T_list, C, sigma, seed, step, L)
    rtol = NORM_RTOL[dtag]
    for l, lsq in enumerate(out.layer_sqnorm):
        got = to64(lsq)
        want = ref.layer_sqnorms[l]
        assert np.all(np.abs(got - want) <= rtol * np.abs(want) + 1e-30), (l, got, want)
    n2 = to64(out.sqnorm)
    assert np.all(np.abs(n2 - ref.total_sqnorm) <= rtol * ref.total_sqnorm + 1e-30)
    c = to64(out.clip)
    assert np.allclose(c, ref.clip, rtol=rtol, atol=0)
    # the computed clip never lets c * n exceed C
    assert np.all(c * np.sqrt(n2.astype(np.float32).astype(np.float64)) <= C * (1 + 2e-7))
    for l, G in enumerate(out.grads):
        e = rel_fro(to64(G), ref.grads[l])
        assert e <= G_RTOL, (l, e)
    # sigma = 0: the clipped sum alone (the noise would hide GEMM errors)
    out0, _ = gpu_step(layers, A_list, E_list, T_list, C, 0.0, seed, step, L, dtype, layer_norms=False)
    B = A_list[0].shape[0]
    Ld = float(B) if L is None else float(L)
    for l, G in enumerate(out0.grads):
        S, sb = ref.clipped[l]
        flat = S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
        e = rel_fro(to64(G), flat / Ld)
        assert e <= G_RTOL, ("sigma=0", l, e)
    return out, out0, ref


def noise_of(seed, step, k0, n):
    return philox.normals(seed, step, k0, n)
