"""Oracle of the record-owned LLM.int8 forward of a frozen layer (test
infrastructure: only tests/, the entry's smoke check and the benchmark's
CPU leg use this package).

"Sensitivity Inflation from Cross-Record Precision Routing in Private
Quantized Fine-Tuning", section 4.2 (Eq. 6 and Algorithm 1) and Appendix A:

  M_ij = [ |A_ij| >= tau ]                      per-entry outlier test
  O_r  = { j : M_ij for some row i of record r } each record's own set
  U    = union of the O_r                        (batched LLM.int8 uses U for every row)
  s_i  = max over j with not M_ij of |A_ij|      row-local scale
  Q_ij = round(127 A_ij / s_i) if j not in O, else 0
  R_ij = A_ij if j in O, else 0
  Y    = dequant(Q Wq^T; s, sW) + R What^T

with O = O_rho(i) (record-owned) or U (batched).  The pages fix the
semantics, not the arithmetic order; the readings taken here (and by the
GPU kernels) are: A, What and Y are IEEE half; s_i, sW and the dequantized
product are float32; the weight is quantized per output row,
sW_n = max_j |W_nj|, Wq = rint(127 W / sW_n), What = half(Wq sW_n / 127);
a code is rint((127 a) / s) in float32 (round half to even; 0 when s = 0);
the integer product is exact (int64 here); dequant = ((float(acc) * s_i) *
sW_n) / 16129 in float32; the correction adds float(a) * float(w) over the
set's columns in ascending order, each step one float32 rounding of the
exact sum (a fused multiply-add); Y = half(dequant + correction).  Appendix
A pins it: the entry 1.234 of a row with scale 5 codes to 31 and comes out
as 1.220703125 through the integer path, as 1.234375 through the correction.
"""

from __future__ import annotations

import numpy as np

F32, F16 = np.float32, np.float16


def quantize_weight(W: np.ndarray):
    """Per-output-row absmax int8 weights: (Wq int8 [N, K], sW float32 [N], What half [N, K])."""
    W = np.asarray(W, dtype=F16).astype(F32)
    sW = np.max(np.abs(W), axis=1).astype(F32)
    safe = np.where(sW > 0, sW, F32(1))
    Wq = np.rint((F32(127) * W) / safe[:, None]).astype(np.int64)
    Wq = np.where(sW[:, None] > 0, Wq, 0)
    What = ((Wq.astype(F32) * sW[:, None]) / F32(127)).astype(F16)
    return Wq.astype(np.int8), sW, What


def outlier_sets(A: np.ndarray, rows_per_record: int, tau: float):
    """(O [records, K] bool, U [K] bool, M [n, K] bool) for half activations A [n, K]."""
    a = np.abs(np.asarray(A, dtype=F16).astype(F32))
    M = a >= F32(tau)
    n, K = M.shape
    if n % rows_per_record:
        raise ValueError("rows must split into whole records")
    O = M.reshape(n // rows_per_record, rows_per_record, K).any(axis=1)
    return O, O.any(axis=0), M


def forward(A: np.ndarray, rows_per_record: int, Wq: np.ndarray, sW: np.ndarray, What: np.ndarray,
            tau: float, record_owned: bool = True) -> np.ndarray:
    """Y [n, N] half: the layer's output under record-owned (or batched) routing."""
    A16 = np.asarray(A, dtype=F16)
    a = A16.astype(F32)
    n, K = a.shape
    O, U, M = outlier_sets(A16, rows_per_record, tau)
    owner = np.arange(n) // rows_per_record
    cols = O[owner] if record_owned else np.broadcast_to(U, (n, K))
    s = np.max(np.where(M, F32(0), np.abs(a)), axis=1).astype(F32)
    safe = np.where(s > 0, s, F32(1))
    q = np.rint((F32(127) * a) / safe[:, None]).astype(np.int64)
    q = np.where(cols | (s[:, None] == 0), 0, q)
    acc = q @ np.asarray(Wq, dtype=np.int64).T                       # exact
    deq = ((acc.astype(F32) * s[:, None]) * np.asarray(sW, F32)[None, :]) / F32(16129)
    w = np.asarray(What, dtype=F16).astype(np.float64)
    corr = np.zeros((n, w.shape[0]), dtype=F32)
    for i in range(n):
        for j in np.nonzero(cols[i])[0]:                             # ascending columns
            corr[i] = (a[i, j].astype(np.float64) * w[:, j] + corr[i].astype(np.float64)).astype(F32)
    return (deq.astype(F32) + corr).astype(F16)
