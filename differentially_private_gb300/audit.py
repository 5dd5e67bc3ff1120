"""Sensitivity audit of the clipped sum, run on the library's own kernels.

The release of one DP-SGD step is M(D) = F(D) + Z with F(D) the sum of the
records' clipped gradients and Z ~ N(0, sigma^2 C^2 I).  Its privacy rests on
the sensitivity of F: one record added or removed moves F by at most C, one
record replaced by at most 2C, provided every record's clipped gradient
depends on that record alone ("Sensitivity Inflation from Cross-Record
Precision Routing in Private Quantized Fine-Tuning", section 3.1,
Proposition 1 with no cross-record influence; section 4.1, Proposition 2).

This module measures that contract for the GPU computation itself
(section 5, Algorithm 2's native arm; the audit's distances are taken in
float64 from the float32 sums, with losses summed: L = 1):

* ``SensitivityAudit.add_remove`` -- kappa = ||F(D + x) - F(D)|| / C,
* ``SensitivityAudit.replace``    -- ||F(D') - F(D)|| / (2C), record i -> x,
* ``SensitivityAudit.norms_batch_invariant`` -- each record's norm is
  bitwise the same in the batch and alone,

and turns a measured distance into the privacy loss of the one-step
Gaussian mechanism (section 3.2, Eq. 5): ``delta_pair`` and its inverse
``epsilon_for``.  A kappa above 1 (beyond rounding) would be a sensitivity
witness against the computation.
"""

from __future__ import annotations

import math

import torch

from .step import PrivateGradient


# ------------------------------------------------------------- Eq. 5
def delta_pair(eps: float, mu: float) -> float:
    """Hockey-stick divergence of N(0, 1) and N(mu, 1) at eps:
    Phi(mu/2 - eps/mu) - e^eps Phi(-mu/2 - eps/mu), and 0 for mu = 0.

    mu = Delta / (sigma C) for a neighbouring pair at distance Delta.  The
    second term is formed in log space so that large eps does not overflow.
    """
    from scipy.special import log_ndtr

    if mu < 0 or not math.isfinite(mu) or not math.isfinite(eps):
        raise ValueError("mu must be finite and >= 0, eps finite")
    if mu == 0.0:
        return 0.0
    a = mu / 2.0 - eps / mu
    b = -mu / 2.0 - eps / mu
    return float(math.exp(log_ndtr(a)) - math.exp(eps + log_ndtr(b)))


def epsilon_for(delta: float, mu: float) -> float:
    """The smallest eps >= 0 with delta_pair(eps, mu) <= delta (the one-step
    privacy loss at delta of a pair at mu; delta_pair decreases in eps)."""
    from scipy.optimize import brentq

    if not (0.0 < delta < 1.0):
        raise ValueError("delta must lie in (0, 1)")
    if delta_pair(0.0, mu) <= delta:
        return 0.0
    hi = 1.0
    while delta_pair(hi, mu) > delta:
        hi *= 2.0
        if hi > 1e6:
            raise ValueError("no eps below 1e6 reaches this delta")
    return float(brentq(lambda e: delta_pair(e, mu) - delta, 0.0, hi, xtol=1e-12, rtol=1e-12, maxiter=500))


# ------------------------------------------------- the audit on the GPU
def _cat_records(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    return torch.cat([a, b], dim=0).contiguous()


class SensitivityAudit:
    """Neighbouring-batch distances of the clipped sum computed by the
    library (sigma = 0, L = 1: F(D) itself, nothing added)."""

    def __init__(self, layers, dtype=torch.bfloat16, device: int = 0):
        """layers: iterable of (d_in, d_out, has_bias), as for PrivateGradient."""
        self.pg = PrivateGradient(layers, dtype=dtype, device=device)

    def close(self):
        self.pg.close()

    def clipped_sum(self, A_list, E_list, T_list, C: float) -> torch.Tensor:
        """F(D) of every layer, concatenated in registration order, as float64."""
        out = self.pg.step(A_list, E_list, T_list, C=C, sigma=0.0, seed=0, step=0, L=1.0)
        return torch.cat([g.to(torch.float64) for g in out.grads])

    def add_remove(self, D, x, T_list, C: float) -> float:
        """kappa = ||F(D + {x}) - F(D)||_2 / C.  D and x are (A_list, E_list);
        x holds one record (batch dimension 1), appended after D's records."""
        A, E = D
        xa, xe = x
        f0 = self.clipped_sum(A, E, T_list, C)
        f1 = self.clipped_sum([_cat_records(a, b) for a, b in zip(A, xa)],
                              [_cat_records(e, b) for e, b in zip(E, xe)], T_list, C)
        return float(torch.linalg.vector_norm(f1 - f0).item() / C)

    def replace(self, D, i: int, x, T_list, C: float) -> float:
        """||F(D') - F(D)||_2 / (2C), D' = D with record i replaced by x."""
        A, E = D
        xa, xe = x
        A2 = [a.clone() for a in A]
        E2 = [e.clone() for e in E]
        for a2, b in zip(A2, xa):
            a2[i] = b[0]
        for e2, b in zip(E2, xe):
            e2[i] = b[0]
        f0 = self.clipped_sum(A, E, T_list, C)
        f1 = self.clipped_sum(A2, E2, T_list, C)
        return float(torch.linalg.vector_norm(f1 - f0).item() / (2.0 * C))

    def norms_batch_invariant(self, D, T_list) -> bool:
        """Each record's total squared norm is bitwise the same computed in
        the batch and computed alone (the record-isolation contract)."""
        A, E = D
        batched = self.pg.step(A, E, T_list, C=1.0, sigma=0.0, seed=0, step=0).sqnorm.clone()
        for i in range(A[0].shape[0]):
            alone = self.pg.step([a[i:i + 1].contiguous() for a in A], [e[i:i + 1].contiguous() for e in E],
                                 T_list, C=1.0, sigma=0.0, seed=0, step=0).sqnorm
            if not torch.equal(alone, batched[i:i + 1]):
                return False
        return True
