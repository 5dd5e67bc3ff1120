"""A small convenience wrapper over the C ABI: one object per model.

``PrivateGradient`` registers the trainable linear layers once and runs the
four calls of a step.  It only allocates the output tensors and forwards
pointers; all arithmetic is in the library's kernels.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _binding as b

_DT = {torch.float32: b.DP_F32, torch.bfloat16: b.DP_BF16}


@dataclass
class StepOutput:
    grads: list            # per layer, float32 [d_out*d_in (+ d_out)]
    clip: torch.Tensor     # float32 [B]
    sqnorm: torch.Tensor   # float32 [B], total over layers
    layer_sqnorm: list | None = None


class PrivateGradient:
    def __init__(self, layers, dtype=torch.bfloat16, device: int = 0, stream=None):
        """layers: iterable of (d_in, d_out, has_bias)."""
        self.device = torch.device("cuda", device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.ctx = b.dp_create(device, self.stream)
        self.layers = []
        self.dtype = dtype
        for (d_in, d_out, has_bias) in layers:
            lid = b.dp_register_layer(self.ctx, d_in, d_out, has_bias, _DT[dtype])
            off, n = b.dp_layer_info(self.ctx, lid)
            self.layers.append((d_in, d_out, bool(has_bias), off, n))
        self.P = b.dp_num_coords(self.ctx)

    def close(self):
        if self.ctx is not None:
            b.dp_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_outputs(self, B: int):
        grads = [torch.empty(n, dtype=torch.float32, device=self.device) for (_, _, _, _, n) in self.layers]
        clip = torch.empty(B, dtype=torch.float32, device=self.device)
        sq = torch.empty(B, dtype=torch.float32, device=self.device)
        return grads, clip, sq

    def step(self, A_list, E_list, T_list, C: float, sigma: float, seed: int, step: int,
             L: float | None = None, outputs=None, layer_norms: bool = False, batch: bool = True,
             check: bool = True) -> StepOutput:
        B = int(A_list[0].shape[0])
        grads, clip, sq = outputs if outputs is not None else self.alloc_outputs(B)
        lsq = [torch.empty(B, dtype=torch.float32, device=self.device) for _ in self.layers] if layer_norms else None
        b.dp_begin_step(self.ctx, B)
        if L is not None:
            b.dp_set_normalizer(self.ctx, L)
        ids = list(range(len(self.layers)))
        if batch:
            b.dp_norm_accumulate_batch(self.ctx, ids, A_list, E_list, T_list, lsq)
        else:
            for i in ids:
                b.dp_norm_accumulate(self.ctx, i, A_list[i], E_list[i], T_list[i], lsq[i] if lsq else None)
        b.dp_clip_factors(self.ctx, C, clip, sq)
        b.dp_clipped_noisy_grad(self.ctx, sigma, seed, step, grads)
        if check:
            st = b.dp_step_status(self.ctx)
            if st != b.DP_OK:
                raise b.DPError(st, "dp_step_status", b.dp_last_error(self.ctx))
        return StepOutput(grads=grads, clip=clip, sqnorm=sq, layer_sqnorm=lsq)
