"""Record-owned LLM.int8 forward on the GPU against the oracle, bit for bit
("Sensitivity Inflation from Cross-Record Precision Routing in Private
Quantized Fine-Tuning", section 4.2, Eq. 6 and Algorithm 1; Appendix A)."""

from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

from differentially_private_gb300.int8 import Int8Linear
from oracle import int8 as oint8

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_witness_codes.json")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


def test_quantized_weight_matches_oracle():
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    W = (torch.randn(70, 130, device="cuda", generator=g) * 0.2).half()
    W[5] = 0.0
    lin = Int8Linear(W)
    Wq, sW, What = oint8.quantize_weight(W.cpu().numpy())
    assert np.array_equal(lin.Wq.cpu().numpy(), Wq)
    assert np.array_equal(lin.sW.cpu().numpy().view(np.uint32), sW.view(np.uint32))
    assert np.array_equal(_bits(lin.What), What.view(np.uint16))


@pytest.mark.parametrize("record_owned", [True, False])
@pytest.mark.parametrize("shape", [(5, 37, 200, 96), (3, 64, 64, 64), (4, 1, 777, 130)])
def test_forward_bit_exact(record_owned, shape):
    records, rows, K, N = shape
    g = torch.Generator(device="cuda")
    g.manual_seed(records * 100 + K)
    A = torch.randn(records * rows, K, device="cuda", generator=g)
    # outliers in a few columns of a few records, one row that is all outliers
    A[rows // 2, 3] = 9.5
    A[(records - 1) * rows, K - 1] = -7.25
    if records > 2:
        A[2 * rows + rows - 1, :] = 6.5
    A = A.half()
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.05).half()
    lin = Int8Linear(W)
    Y = lin(A, rows, tau=6.0, record_owned=record_owned)
    torch.cuda.synchronize()
    want = oint8.forward(A.cpu().numpy(), rows, lin.Wq.cpu().numpy(), lin.sW.cpu().numpy(),
                         lin.What.cpu().numpy(), 6.0, record_owned=record_owned)
    got = _bits(Y)
    assert np.array_equal(got, want.view(np.uint16)), int((got != want.view(np.uint16)).sum())


@pytest.mark.parametrize("record_owned", [True, False])
def test_activations_off_a_16_byte_boundary(record_owned):
    """A view that starts one element into its buffer (K a multiple of 8): the
    rows are read element by element and the output is the same bits as from
    an aligned copy, and the oracle's."""
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    records, rows, K, N = 3, 40, 256, 72
    buf = torch.randn(records * rows * K + 1, device="cuda", generator=g).half()
    buf[1 + rows * K + 9] = 7.5                       # an outlier in record 1
    A = buf[1:].view(records * rows, K)
    assert A.data_ptr() % 16 != 0
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.05).half()
    lin = Int8Linear(W)
    Y = lin(A, rows, tau=6.0, record_owned=record_owned)
    Y2 = lin(A.clone(), rows, tau=6.0, record_owned=record_owned)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2)
    want = oint8.forward(A.cpu().numpy(), rows, lin.Wq.cpu().numpy(), lin.sW.cpu().numpy(),
                         lin.What.cpu().numpy(), 6.0, record_owned=record_owned)
    assert np.array_equal(_bits(Y), want.view(np.uint16))


def test_appendix_a_witness_on_the_gpu():
    gx = json.load(open(GOLDEN))
    W = torch.tensor(gx["weight"], dtype=torch.float16, device="cuda")
    lin = Int8Linear(W)
    for eighth, batched in ((gx["eighth_row_D"], gx["int8_path_output"]),
                            (gx["eighth_row_Dprime"], gx["outlier_path_output"])):
        A = torch.tensor([gx["unchanged_row"]] * 7 + [eighth], dtype=torch.float16, device="cuda")
        yb = lin(A, 1, tau=gx["tau"], record_owned=False)
        yo = lin(A, 1, tau=gx["tau"], record_owned=True)
        torch.cuda.synchronize()
        assert torch.all(yb[:7, 0].double() == batched)
        assert torch.all(yo[:7, 0].double() == gx["int8_path_output"])


def test_record_owned_rows_do_not_depend_on_other_records():
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    rows, K, N = 16, 256, 128
    A = torch.randn(6 * rows, K, device="cuda", generator=g).half()
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.05).half()
    lin = Int8Linear(W)
    y0 = lin(A, rows, record_owned=True)
    A2 = A.clone()
    A2[3 * rows + 2, 77] = 12.0             # a new outlier column in record 3
    A2[5 * rows:] = torch.randn(rows, K, device="cuda", generator=g).half() * 3
    y1 = lin(A2, rows, record_owned=True)
    torch.cuda.synchronize()
    others = [r for r in range(6) if r not in (3, 5)]
    for r in others:
        assert torch.equal(y0[r * rows:(r + 1) * rows], y1[r * rows:(r + 1) * rows])
    b0 = lin(A, rows, record_owned=False)
    b1 = lin(A2, rows, record_owned=False)
    torch.cuda.synchronize()
    assert not torch.equal(b0[:rows], b1[:rows])      # batched routing couples the records


@pytest.mark.parametrize("K,signs", [(1024, "same"), (1024, "random"), (2048, "same"), (3072, "random"),
                                     (4096, "same"), (4104, "random")])
def test_integer_product_exact_at_the_largest_partial_sums(K, signs):
    """Codes of +-127 on both sides: up to K, the partial sums reach 16129 K.
    Up to K = 4096 the product runs on the bf16 tensor cores in chunks of 1024
    (each below 2^24, exact in fp32, added in int32); beyond, on the CUDA
    cores.  Either way it must match the oracle's exact integer product bit
    for bit, including the float rounding of sums beyond 2^24."""
    import differentially_private_gb300 as dp
    g = torch.Generator(device="cuda").manual_seed(K)
    rows, records, N = 40, 3, 200
    n = rows * records
    if signs == "same":
        A = torch.ones(n, K, device="cuda")
        W = torch.full((N, K), 0.25, device="cuda")
    else:
        A = torch.where(torch.rand(n, K, device="cuda", generator=g) < 0.5, -1.0, 1.0)
        W = torch.where(torch.rand(N, K, device="cuda", generator=g) < 0.5, -0.25, 0.25)
    A[5, 7] = 9.0                          # one outlier column in record 0
    A = A.half()
    W = W.half()
    lin = Int8Linear(W)
    before = dp.dp_kernel_launch_counts()
    Y = lin(A, rows, tau=6.0, record_owned=True)
    torch.cuda.synchronize()
    after = dp.dp_kernel_launch_counts()
    tc_path = after["k_int8_gemm_tc"] - before["k_int8_gemm_tc"]
    assert tc_path == (1 if K <= 4096 else 0)
    assert after["k_int8_gemm"] - before["k_int8_gemm"] == (0 if K <= 4096 else 1)
    want = oint8.forward(A.cpu().numpy(), rows, lin.Wq.cpu().numpy(), lin.sW.cpu().numpy(),
                         lin.What.cpu().numpy(), 6.0, record_owned=True)
    got = _bits(Y)
    assert np.array_equal(got, want.view(np.uint16)), int((got != want.view(np.uint16)).sum())
