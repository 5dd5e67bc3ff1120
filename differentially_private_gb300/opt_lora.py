"""An OPT-125M-shaped decoder with random frozen weights and rank-r LoRA
adapters on the query and value projections: a producer of the per-record
activations A and output gradients E of a real forward and backward.

Shapes follow the setting of "Sensitivity Inflation from Cross-Record
Precision Routing in Private Quantized Fine-Tuning", section 6.2 (OPT-125M:
12 blocks, d_model 768, 12 heads, FFN 3072; rank-8 LoRA on q and v, 48
trainable tensors; masked next-token loss of each window with a fixed
public divisor).  No pretrained weights or dataset are involved: weights
are seeded random draws and the tokens are seeded random ids.  The loss of
a batch is the sum of the records' losses, so record i's rows of every E
are the gradient of record i's own loss.
"""

from __future__ import annotations

import torch
import torch.nn.functional as F

from .capture import LoRAAdapter


class _Block(torch.nn.Module):
    def __init__(self, d, heads, ffn, r, dtype, g):
        super().__init__()
        self.heads = heads

        def w(o, i):
            return torch.nn.Parameter((torch.randn(o, i, device="cuda", generator=g) * 0.02).to(dtype),
                                      requires_grad=False)

        def bvec(n):
            return torch.nn.Parameter(torch.zeros(n, device="cuda", dtype=dtype), requires_grad=False)

        self.ln1_w = torch.nn.Parameter(torch.ones(d, device="cuda", dtype=dtype), requires_grad=False)
        self.ln1_b = bvec(d)
        self.q_w, self.k_w, self.v_w, self.o_w = w(d, d), w(d, d), w(d, d), w(d, d)
        self.q_b, self.k_b, self.v_b, self.o_b = bvec(d), bvec(d), bvec(d), bvec(d)
        self.ln2_w = torch.nn.Parameter(torch.ones(d, device="cuda", dtype=dtype), requires_grad=False)
        self.ln2_b = bvec(d)
        self.fc1_w, self.fc1_b = w(ffn, d), bvec(ffn)
        self.fc2_w, self.fc2_b = w(d, ffn), bvec(d)
        self.lora_q = LoRAAdapter(d, d, r, dtype=dtype, generator=g, b_scale=0.02)
        self.lora_v = LoRAAdapter(d, d, r, dtype=dtype, generator=g, b_scale=0.02)

    def forward(self, x):
        B, T, d = x.shape
        h = F.layer_norm(x, (d,), self.ln1_w, self.ln1_b)
        q = F.linear(h, self.q_w, self.q_b) + self.lora_q(h)
        k = F.linear(h, self.k_w, self.k_b)
        v = F.linear(h, self.v_w, self.v_b) + self.lora_v(h)
        sh = lambda t: t.view(B, T, self.heads, d // self.heads).transpose(1, 2)  # noqa: E731
        a = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
        x = x + F.linear(a.transpose(1, 2).reshape(B, T, d), self.o_w, self.o_b)
        h = F.layer_norm(x, (d,), self.ln2_w, self.ln2_b)
        return x + F.linear(F.relu(F.linear(h, self.fc1_w, self.fc1_b)), self.fc2_w, self.fc2_b)


class OPTLoRA(torch.nn.Module):
    """Decoder of n_layers blocks; ``adapters()`` lists the 2 * n_layers LoRA
    adapters (q then v of every block), i.e. 4 * n_layers registered layers."""

    def __init__(self, n_layers=12, d=768, heads=12, ffn=3072, vocab=50272, max_pos=2048, r=8,
                 dtype=torch.bfloat16, seed=0):
        super().__init__()
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        self.embed = torch.nn.Parameter((torch.randn(vocab, d, device="cuda", generator=g) * 0.02).to(dtype),
                                        requires_grad=False)
        self.pos = torch.nn.Parameter((torch.randn(max_pos, d, device="cuda", generator=g) * 0.02).to(dtype),
                                      requires_grad=False)
        self.blocks = torch.nn.ModuleList(_Block(d, heads, ffn, r, dtype, g) for _ in range(n_layers))
        self.lnf_w = torch.nn.Parameter(torch.ones(d, device="cuda", dtype=dtype), requires_grad=False)
        self.lnf_b = torch.nn.Parameter(torch.zeros(d, device="cuda", dtype=dtype), requires_grad=False)

    def adapters(self):
        out = []
        for b in self.blocks:
            out += [b.lora_q, b.lora_v]
        return out

    def record_losses(self, tokens: torch.Tensor, divisor: float | None = None) -> torch.Tensor:
        """Next-token cross entropy of every record, summed over its positions
        and divided by a fixed public divisor (default T - 1): float32 [B]."""
        B, T = tokens.shape
        x = self.embed[tokens] + self.pos[:T]
        for blk in self.blocks:
            x = blk(x)
        x = F.layer_norm(x, (x.shape[-1],), self.lnf_w, self.lnf_b)
        logits = F.linear(x[:, :-1], self.embed).float()
        ce = F.cross_entropy(logits.reshape(-1, logits.shape[-1]), tokens[:, 1:].reshape(-1), reduction="none")
        return ce.view(B, T - 1).sum(dim=1) / float(divisor if divisor is not None else T - 1)


def random_tokens(B: int, T: int, vocab: int, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(0, vocab, (B, T), device="cuda", generator=g)
