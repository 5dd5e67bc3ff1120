"""Per-example inputs A and output gradients E captured from a model's own
forward and backward, handed to the library for the private gradient.

A LoRA adapter adds B(A(x)) to a frozen projection.  Each adapter is two
trainable linear maps, registered as two layers: LoRA-A (d -> r), whose
activations are x and whose output gradients are dL/dh at h = x A^T, and
LoRA-B (r -> d_out), whose activations are h and whose output gradients are
dL/d(delta) at delta = h B^T.  With the loss a sum of per-record losses,
E's rows of record i are the gradients of record i's own loss, so
g_i = E_i^T A_i is record i's per-example gradient
("Privacy-Preserving Machine Learning", section "Differentially private
stochastic gradient descent", phase 2; "Sensitivity Inflation from
Cross-Record Precision Routing in Private Quantized Fine-Tuning", section
6.2: rank-8 LoRA on the query and value projections of OPT-125M).

``LoRAAdapter`` records (A, E) during a normal forward and backward;
``PrivateLoRA`` runs the library's step over all adapters and writes the
clipped, noised, normalized gradient into the adapters' ``.grad``.
"""

from __future__ import annotations

import torch
import torch.nn.functional as F

from .step import PrivateGradient


class LoRAAdapter(torch.nn.Module):
    """delta = (x A^T) B^T, with A [r, d_in] and B [d_out, r] trainable."""

    def __init__(self, d_in: int, d_out: int, r: int, dtype=torch.bfloat16, device="cuda", generator=None,
                 b_scale: float = 0.0):
        super().__init__()
        a = torch.randn(r, d_in, device=device, generator=generator) / d_in ** 0.5
        b = torch.randn(d_out, r, device=device, generator=generator) * b_scale
        self.A = torch.nn.Parameter(a.to(dtype))
        self.B = torch.nn.Parameter(b.to(dtype))
        self.capture = False
        self._acts = {}
        self._grads = {}

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        h = F.linear(x, self.A)
        delta = F.linear(h, self.B)
        if self.capture and torch.is_grad_enabled():
            self._acts["A"] = x.detach()
            self._acts["B"] = h.detach()
            h.register_hook(lambda g: self._grads.__setitem__("A", g.detach()))
            delta.register_hook(lambda g: self._grads.__setitem__("B", g.detach()))
        return delta

    def layers(self):
        """The two registered layers: (d_in, d_out, has_bias) of LoRA-A, LoRA-B."""
        r, d_in = self.A.shape
        d_out = self.B.shape[0]
        return [(d_in, r, False), (r, d_out, False)]

    def captured(self):
        """(A, E) of LoRA-A and of LoRA-B from the last forward and backward, as [B, T, d]."""
        if set(self._acts) != {"A", "B"} or set(self._grads) != {"A", "B"}:
            raise RuntimeError("no captured forward/backward: enable capture and run backward first")
        out = []
        for k in ("A", "B"):
            a, e = self._acts[k], self._grads[k]
            if a.dim() == 2:
                a, e = a.unsqueeze(1), e.unsqueeze(1)
            out.append((a.contiguous(), e.contiguous()))
        return out


class PrivateLoRA:
    """One DP-SGD gradient over a set of LoRA adapters through the library."""

    def __init__(self, adapters, dtype=torch.bfloat16, device: int = 0):
        self.adapters = list(adapters)
        layers = []
        for ad in self.adapters:
            layers += ad.layers()
        self.pg = PrivateGradient(layers, dtype=dtype, device=device)

    def set_capture(self, on: bool = True):
        for ad in self.adapters:
            ad.capture = on
            ad._acts.clear()
            ad._grads.clear()

    def step(self, C: float, sigma: float, seed: int, step: int, L: float | None = None, write_grads: bool = True):
        """Clip every record's gradient over all adapters to C, sum, add
        N(0, sigma^2 C^2) noise once and divide by L (default: the batch
        size); optionally write the result into the adapters' .grad.
        Returns the library's StepOutput."""
        A_list, E_list, T_list = [], [], []
        for ad in self.adapters:
            for a, e in ad.captured():
                A_list.append(a)
                E_list.append(e)
                T_list.append(a.shape[1])
        out = self.pg.step(A_list, E_list, T_list, C=C, sigma=sigma, seed=seed, step=step, L=L)
        if write_grads:
            i = 0
            for ad in self.adapters:
                for p in (ad.A, ad.B):
                    p.grad = out.grads[i].view(p.shape).to(p.dtype)
                    i += 1
        return out

    def close(self):
        self.pg.close()
