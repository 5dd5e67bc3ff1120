"""Activations and output gradients captured from a real forward and backward
of an OPT-shaped decoder with rank-8 LoRA on q and v, handed to the library.

Pin: each record's gradient of its own loss, taken by torch autograd on the
same batched graph (one backward per record), gives the per-example norms
and the clipped sum the library must reproduce from the captured A and E.
At T = 64 the chooser takes the ghost norm for the rank-8 factors (T^2 <
768 x 8), at T = 128 it materializes them (the tensor-core skinny kernel
and the weighted sum of stored gradients)."""

from __future__ import annotations

import pytest
import torch

from differentially_private_gb300.capture import PrivateLoRA
from differentially_private_gb300.opt_lora import OPTLoRA, random_tokens
from gpu_harness import G_RTOL, NORM_RTOL

pytestmark = pytest.mark.gpu


def _per_record_grads(model, tokens):
    params = [p for ad in model.adapters() for p in (ad.A, ad.B)]
    losses = model.record_losses(tokens)
    out = []
    for i in range(tokens.shape[0]):
        gs = torch.autograd.grad(losses[i], params, retain_graph=i + 1 < tokens.shape[0])
        out.append(torch.cat([g.reshape(-1).double() for g in gs]))
    return torch.stack(out)            # [B, P]


@pytest.mark.parametrize("T,C", [(64, 1e6), (64, 0.05), (128, 1e6), (128, 0.05)])
def test_captured_lora_step_matches_autograd(T, C):
    B, vocab = 4, 2048
    model = OPTLoRA(n_layers=2, vocab=vocab, seed=3)
    tokens = random_tokens(B, T, vocab, seed=4)
    g = _per_record_grads(model, tokens)
    n2 = (g * g).sum(dim=1)
    c = torch.clamp(C / n2.sqrt(), max=1.0)
    want = (c[:, None] * g).sum(dim=0)

    private = PrivateLoRA(model.adapters())
    private.set_capture(True)
    model.record_losses(tokens).sum().backward()
    out = private.step(C=C, sigma=0.0, seed=0, step=0, L=1.0)
    torch.cuda.synchronize()
    got_n2 = out.sqnorm.double()
    assert torch.allclose(got_n2, n2, rtol=NORM_RTOL["bf16"], atol=0), (got_n2, n2)
    got = torch.cat([x.double() for x in out.grads])
    rel = (torch.linalg.vector_norm(got - want) / torch.linalg.vector_norm(want)).item()
    assert rel <= G_RTOL, rel
    # the adapters' .grad now hold the clipped sum, parameter by parameter
    i = 0
    for ad in model.adapters():
        for p in (ad.A, ad.B):
            assert p.grad is not None and p.grad.shape == p.shape
            assert torch.equal(p.grad, out.grads[i].view(p.shape).to(p.dtype))
            i += 1
    private.close()


def test_opt125m_shape_registers_48_tensors():
    model = OPTLoRA(n_layers=12, vocab=512, seed=0)
    private = PrivateLoRA(model.adapters())
    assert len(private.pg.layers) == 48
    assert private.pg.P == 294_912    # 12 blocks x {q, v} x (768 x 8 + 8 x 768)
    private.close()
