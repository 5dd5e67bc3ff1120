"""Record-owned LLM.int8 forward of a frozen layer through the library
("Sensitivity Inflation from Cross-Record Precision Routing in Private
Quantized Fine-Tuning", section 4.2, Eq. 6 and Algorithm 1): the producer of
a private adapter's activations kept record-isolated.  Thin wrappers over
dp_int8_quantize_weight / dp_int8_forward (argument marshalling only)."""

from __future__ import annotations

import torch

from . import _binding as b


class Int8Linear:
    """A frozen linear layer y = x W^T held as per-row absmax int8 weights."""

    def __init__(self, W: torch.Tensor, stream=None):
        if W.dtype != torch.float16 or W.dim() != 2 or not W.is_cuda:
            raise ValueError("W must be a CUDA float16 [N, K] tensor")
        self.N, self.K = W.shape
        self.stream = stream if stream is not None else torch.cuda.current_stream(W.device)
        W = W.contiguous()
        self.Wq = torch.empty(self.N, self.K, dtype=torch.int8, device=W.device)
        self.sW = torch.empty(self.N, dtype=torch.float32, device=W.device)
        self.What = torch.empty(self.N, self.K, dtype=torch.float16, device=W.device)
        b.dp_int8_quantize_weight(W, self.N, self.K, self.Wq, self.sW, self.What, self.stream)

    def __call__(self, A: torch.Tensor, rows_per_record: int, tau: float = 6.0,
                 record_owned: bool = True) -> torch.Tensor:
        """A: CUDA float16 [n, K] (rows of a record contiguous) -> float16 [n, N]."""
        if A.dtype != torch.float16 or A.dim() != 2 or A.shape[1] != self.K:
            raise ValueError("A must be float16 [n, K]")
        A = A.contiguous()
        n = A.shape[0]
        ws = b.dp_int8_workspace_bytes(n, self.K, self.N, rows_per_record)
        if ws < 0:
            raise ValueError("rows must split into whole records")
        work = torch.empty(max(ws, 16), dtype=torch.uint8, device=A.device)
        Y = torch.empty(n, self.N, dtype=torch.float16, device=A.device)
        b.dp_int8_forward(A, n, self.K, rows_per_record, self.Wq, self.sW, self.What, self.N, tau, record_owned, Y,
                          work, self.stream)
        return Y
