"""Pins of the record-owned LLM.int8 forward oracle ("Sensitivity Inflation
from Cross-Record Precision Routing in Private Quantized Fine-Tuning",
section 4.2 Eq. 6 and Algorithm 1, Appendix A)."""

from __future__ import annotations

import json
import os

import numpy as np

from oracle import int8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_witness_codes.json")


def _witness(eighth):
    gx = json.load(open(GOLDEN))
    A = np.array([gx["unchanged_row"]] * 7 + [eighth], dtype=np.float16)
    Wq, sW, What = int8.quantize_weight(np.array(gx["weight"], dtype=np.float16))
    return gx, A, Wq, sW, What


def test_appendix_a_codes_and_outputs():
    gx = json.load(open(GOLDEN))
    for eighth, batched_out in ((gx["eighth_row_D"], gx["int8_path_output"]),
                                (gx["eighth_row_Dprime"], gx["outlier_path_output"])):
        _, A, Wq, sW, What = _witness(eighth)
        assert int(Wq[0, 0]) == 127 and float(sW[0]) == 1.0 and float(What[0, 0]) == 1.0
        a = np.float32(A[0, 0])
        assert int(np.rint(np.float32(127) * a / np.float32(5.0))) == gx["code"]
        yb = int8.forward(A, 1, Wq, sW, What, gx["tau"], record_owned=False)
        yo = int8.forward(A, 1, Wq, sW, What, gx["tau"], record_owned=True)
        # batched: the other record's outlier moves the unchanged rows to the FP16 path
        assert np.all(yb[:7, 0].astype(np.float64) == batched_out)
        # record-owned: the unchanged rows stay on their own (INT8) path
        assert np.all(yo[:7, 0].astype(np.float64) == gx["int8_path_output"])


def _data(seed, n_rec=5, rows=4, K=48, N=24):
    rng = np.random.default_rng(seed)
    A = rng.normal(size=(n_rec * rows, K)).astype(np.float16)
    # a few outliers, each in one record
    for r, j in ((1, 3), (3, 17), (3, 40)):
        A[r * rows + 1, j] = np.float16(8.0 + r)
    W = (rng.normal(size=(N, K)) * 0.1).astype(np.float16)
    return A, W, rows


def test_record_owned_rows_ignore_other_records():
    A, W, rows = _data(1)
    Wq, sW, What = int8.quantize_weight(W)
    y0 = int8.forward(A, rows, Wq, sW, What, 6.0, record_owned=True)
    A2 = A.copy()
    A2[0 * rows + 2, 30] = np.float16(-9.0)        # a new outlier column in record 0
    A2[4 * rows:, :] = np.float16(0.5)             # and record 4 replaced
    y1 = int8.forward(A2, rows, Wq, sW, What, 6.0, record_owned=True)
    assert np.array_equal(y0[rows:4 * rows].view(np.uint16), y1[rows:4 * rows].view(np.uint16))
    # the batched special case couples them: column 30 joins every row's set
    b0 = int8.forward(A, rows, Wq, sW, What, 6.0, record_owned=False)
    b1 = int8.forward(A2, rows, Wq, sW, What, 6.0, record_owned=False)
    assert not np.array_equal(b0[rows:4 * rows], b1[rows:4 * rows])


def test_no_outliers_modes_agree_and_approximate_the_product():
    A, W, rows = _data(2)
    A = np.clip(A.astype(np.float32), -4, 4).astype(np.float16)
    Wq, sW, What = int8.quantize_weight(W)
    yo = int8.forward(A, rows, Wq, sW, What, 6.0, record_owned=True)
    yb = int8.forward(A, rows, Wq, sW, What, 6.0, record_owned=False)
    assert np.array_equal(yo.view(np.uint16), yb.view(np.uint16))
    exact = A.astype(np.float64) @ W.astype(np.float64).T
    rel = np.linalg.norm(yo.astype(np.float64) - exact) / np.linalg.norm(exact)
    assert rel < 0.03          # int8 vector-wise quantization error


def test_outlier_columns_are_exact_half_products():
    # every column an outlier: the output is the fp16 correction product alone
    A = np.full((2, 3), 7.0, dtype=np.float16)
    A[1] = np.float16(-6.5)
    W = np.array([[0.5, 0.25, -1.0], [1.0, 2.0, 0.125]], dtype=np.float16)
    Wq, sW, What = int8.quantize_weight(W)
    y = int8.forward(A, 1, Wq, sW, What, 6.0, record_owned=True)
    want = (A.astype(np.float64) @ What.astype(np.float64).T).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))
