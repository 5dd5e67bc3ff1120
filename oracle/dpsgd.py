"""One DP-SGD private-gradient step in float64 numpy (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What it computes, in the order the pages give the steps
("Privacy-Preserving Machine Learning", section "Differentially private
stochastic gradient descent", phases 2-5; "Differential Privacy: DP-SGD,
Privacy Budgets, and LLMs", "Step 1: Per-example gradient clipping" and
"Step 2: Gaussian noise addition"; "Sensitivity Inflation from Cross-Record
Precision Routing in Private Quantized Fine-Tuning", section 2, Eq. 2 and 3):

1. per-example gradient of every trainable linear layer, MATERIALIZED:
   for a layer y = x W^T (+ b) with W in R^{d_out x d_in} (the orientation of
   "Privacy-Preserving Machine Learning", section "The privacy-utility
   trade-off in modern LLMs"), record i's activations A_i [T, d_in] and output
   errors E_i = dL/dy [T, d_out] give g_i = E_i^T A_i (d_out x d_in) and, for a
   bias, b_i = sum_t E_i[t, :].  The oracle never uses the ghost identity.
2. one L2 norm per record over the concatenation of every layer's weight and
   bias gradient ("Differential Privacy: DP-SGD, Privacy Budgets, and LLMs",
   the from-scratch implementation: weights and bias clipped together);
3. clip factor c_i = min(1, C / ||g_i||), with a zero vector left unchanged
   (c_i = 1), C finite and > 0, non-finite data rejected ("Privacy-Preserving
   Machine Learning", phase 3 and its clip example; "Differential Privacy in
   Fine-Tuning (DP-SGD)", "Per-Sample Gradient Clipping": g / max(1, ||g||/C));
4. clipped sum S = sum_i c_i g_i, accumulated in ascending record order
   (Eq. 3 of the Sensitivity Inflation paper, F(D) = sum_r h_r);
5. Gaussian noise sigma*C*z added once to every coordinate of the sum, z from
   ``oracle.philox`` ("Differential Privacy: DP-SGD, Privacy Budgets, and LLMs",
   implementation failures: noise on every component, once on the aggregate);
6. divide by the public normalizer L; L = B unless the caller gives one
   ("Differential Privacy: DP-SGD, Privacy Budgets, and LLMs", Step 2 divides
   by the minibatch size B; "Privacy-Preserving Machine Learning", phase 5 uses
   a fixed public L).

Coordinate layout of the flattened gradient (reading; the pages are silent):
layers in registration order; within a layer the weight gradient
[d_out][d_in] row-major (the layout of W), then the bias [d_out].  Coordinate
k = layer offset + row * d_in + col, or layer offset + d_out*d_in + row for a
bias entry.

Ghost / materialize chooser: ghost iff T*T < d_in*d_out in exact integers,
else materialize (equality materializes).  The pages only say that ghost
clipping avoids materializing every per-example gradient ("Privacy-Preserving
Machine Learning", phase 2; "Differential Privacy: DP-SGD, Privacy Budgets,
and LLMs", computational cost); the rule is this library's contract.

Pins (tests/test_oracle_dpsgd.py): the clip example printed on
"Privacy-Preserving Machine Learning" ([0.4,0.3],[3,4],[0.6,0.8] -> sum
[1.60, 1.90]) and its Alice example (1.5); the exact FP64 witness of the
Sensitivity Inflation paper, Appendix A (Delta = 14 C_f); brute-force
<A A^T, E E^T> on small integer inputs (exact equality with the materialized
norm); per-example gradients against independent torch autograd; the
add/remove <= C and replacement <= 2C sensitivity bounds (Proposition 1 with
m = 0) and the clip(mean) anti-pattern exceeding them; sigma = 0 reducing G to
S / L.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import philox

GHOST = 0
MATERIALIZE = 1


def choose_path(T: int, d_in: int, d_out: int) -> int:
    """GHOST (0) iff T^2 < d_in * d_out, computed in Python integers."""
    T, d_in, d_out = int(T), int(d_in), int(d_out)
    return GHOST if T * T < d_in * d_out else MATERIALIZE


@dataclass(frozen=True)
class Layer:
    d_in: int
    d_out: int
    has_bias: bool = False

    @property
    def ncoords(self) -> int:
        return self.d_out * self.d_in + (self.d_out if self.has_bias else 0)


def coordinate_offsets(layers: list[Layer]) -> tuple[list[int], int]:
    """First noise coordinate of every layer, and the total count P."""
    offs, p = [], 0
    for ly in layers:
        offs.append(p)
        p += ly.ncoords
    return offs, p


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def per_example_grad(A_i, E_i, has_bias: bool):
    """g_i = E_i^T A_i  [d_out, d_in]  and  b_i = sum_t E_i[t]  (or None)."""
    A_i, E_i = _f64(A_i), _f64(E_i)
    g = E_i.T @ A_i
    b = E_i.sum(axis=0) if has_bias else None
    return g, b


def layer_sqnorms(A, E, has_bias: bool) -> np.ndarray:
    """||g_i||_F^2 (+ ||b_i||^2) for every record of one layer: float64 [B]."""
    A, E = _f64(A), _f64(E)
    out = np.empty(A.shape[0], dtype=np.float64)
    for i in range(A.shape[0]):
        g, b = per_example_grad(A[i], E[i], has_bias)
        out[i] = np.sum(g * g) + (np.sum(b * b) if b is not None else 0.0)
    return out


def record_sqnorm(A_i, E_i, has_bias: bool) -> float:
    g, b = per_example_grad(A_i, E_i, has_bias)
    return float(np.sum(g * g) + (np.sum(b * b) if b is not None else 0.0))


def check_clip_bound(C: float) -> float:
    if isinstance(C, bool) or not isinstance(C, (int, float)) or not math.isfinite(C) or C <= 0:
        raise ValueError("clip bound C must be finite and > 0")
    return float(C)


def clip_factors(total_sqnorm, C: float) -> np.ndarray:
    """c_i = 1 if ||g_i|| <= C (zero vector included), else C / ||g_i||."""
    C = check_clip_bound(C)
    n2 = _f64(total_sqnorm)
    if not np.all(np.isfinite(n2)):
        raise ValueError("non-finite per-example gradient norm")
    n = np.sqrt(n2)
    c = np.ones_like(n)
    big = n > C
    c[big] = C / n[big]
    return c


def clipped_sum(A, E, c, has_bias: bool):
    """S = sum_i c_i g_i (ascending i) and the bias part, float64."""
    A, E, c = _f64(A), _f64(E), _f64(c)
    B, _, d_in = A.shape
    d_out = E.shape[2]
    S = np.zeros((d_out, d_in), dtype=np.float64)
    sb = np.zeros(d_out, dtype=np.float64) if has_bias else None
    for i in range(B):
        g, b = per_example_grad(A[i], E[i], has_bias)
        S += c[i] * g
        if has_bias:
            sb += c[i] * b
    return S, sb


def clipped_sum_at(A, E, c, rows, cols) -> np.ndarray:
    """S[rows[q], cols[q]] for sampled coordinates, by the per-record definition."""
    A, E, c = _f64(A), _f64(E), _f64(c)
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = np.zeros(rows.size, dtype=np.float64)
    for i in range(A.shape[0]):
        gi = np.einsum("tq,tq->q", E[i][:, rows], A[i][:, cols])
        out += c[i] * gi
    return out


def check_noise_args(sigma: float, L: float) -> None:
    if not math.isfinite(sigma) or sigma < 0:
        raise ValueError("noise multiplier sigma must be finite and >= 0")
    if not math.isfinite(L) or L <= 0:
        raise ValueError("normalizer L must be finite and > 0")


@dataclass
class StepResult:
    paths: list[int]
    layer_sqnorms: np.ndarray          # [n_layers, B]
    total_sqnorm: np.ndarray           # [B]
    clip: np.ndarray                   # [B]
    clipped: list[tuple[np.ndarray, np.ndarray | None]] = field(default_factory=list)
    noise: np.ndarray | None = None    # z over all P coordinates
    grads: list[np.ndarray] = field(default_factory=list)  # flattened per layer


def step(layers: list[Layer], A_list, E_list, T_list, C: float, sigma: float,
         seed: int, step_index: int, L: float | None = None) -> StepResult:
    """The whole step, every intermediate kept (small cases only)."""
    C = check_clip_bound(C)
    B = _f64(A_list[0]).shape[0]
    L = float(B) if L is None else float(L)
    check_noise_args(float(sigma), L)
    paths = [choose_path(T, ly.d_in, ly.d_out) for ly, T in zip(layers, T_list)]
    n2l = np.stack([layer_sqnorms(A, E, ly.has_bias)
                    for ly, A, E in zip(layers, A_list, E_list)])
    n2 = np.zeros(B, dtype=np.float64)
    for row in n2l:                      # registration order
        n2 = n2 + row
    c = clip_factors(n2, C)
    offs, P = coordinate_offsets(layers)
    z = philox.normals(seed, step_index, 0, P)
    res = StepResult(paths=paths, layer_sqnorms=n2l, total_sqnorm=n2, clip=c, noise=z)
    for ly, A, E, off in zip(layers, A_list, E_list, offs):
        S, sb = clipped_sum(A, E, c, ly.has_bias)
        res.clipped.append((S, sb))
        flat = S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
        G = (flat + sigma * C * z[off:off + ly.ncoords]) / L
        res.grads.append(G)
    return res


# ------------------------------------------------------------- user level
@dataclass
class UserStepResult:
    user_sqnorm: np.ndarray      # [U] squared norm of each user's summed gradient
    clip: np.ndarray             # [U]
    noise: np.ndarray            # [P]
    clipped: list = field(default_factory=list)   # per layer (S, sb) before noise and L
    grads: list = field(default_factory=list)     # per layer G = (S + sigma C z) / L


def user_step(layers: list[Layer], A_list, E_list, T_list, group_sizes, C: float, sigma: float,
              seed: int, step_index: int, L: float | None = None) -> UserStepResult:
    """User-level clipping ("Privacy-Preserving Machine Learning", section
    "Differentially private stochastic gradient descent", the user-level
    construction and its sum-then-user-clip example): the records are grouped
    in order (user u owns the next group_sizes[u] records), each user's vector
    is the sum of its records' gradients over all layers, that vector is
    clipped to C, the clipped user vectors are summed, noise N(0, sigma^2 C^2)
    is added once per coordinate, and the sum is divided by the public
    normalizer L (default: the number of users).  Zero-record users are
    allowed (their vector is zero)."""
    C = check_clip_bound(C)
    sizes = [int(k) for k in group_sizes]
    if any(k < 0 for k in sizes):
        raise ValueError("group sizes must be >= 0")
    B = _f64(A_list[0]).shape[0]
    if sum(sizes) != B:
        raise ValueError("group sizes must add up to the number of records")
    U = len(sizes)
    L = float(U) if L is None else float(L)
    check_noise_args(float(sigma), L)
    starts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    per_layer = []                       # per layer: list over users of (g_u, b_u)
    n2 = np.zeros(U, dtype=np.float64)
    for ly, A, E in zip(layers, A_list, E_list):
        A, E = _f64(A), _f64(E)
        users = []
        for u in range(U):
            g = np.zeros((ly.d_out, ly.d_in), dtype=np.float64)
            b = np.zeros(ly.d_out, dtype=np.float64) if ly.has_bias else None
            for i in range(starts[u], starts[u + 1]):
                gi, bi = per_example_grad(A[i], E[i], ly.has_bias)
                g += gi
                if ly.has_bias:
                    b += bi
            users.append((g, b))
            n2[u] += np.sum(g * g) + (np.sum(b * b) if b is not None else 0.0)
        per_layer.append(users)
    c = clip_factors(n2, C)
    offs, P = coordinate_offsets(layers)
    z = philox.normals(seed, step_index, 0, P)
    res = UserStepResult(user_sqnorm=n2, clip=c, noise=z)
    for ly, users, off in zip(layers, per_layer, offs):
        S = np.zeros((ly.d_out, ly.d_in), dtype=np.float64)
        sb = np.zeros(ly.d_out, dtype=np.float64) if ly.has_bias else None
        for u, (g, b) in enumerate(users):
            S += c[u] * g
            if ly.has_bias:
                sb += c[u] * b
        res.clipped.append((S, sb))
        flat = S.reshape(-1) if sb is None else np.concatenate([S.reshape(-1), sb])
        res.grads.append((flat + sigma * C * z[off:off + ly.ncoords]) / L)
    return res
