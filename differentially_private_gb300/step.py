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

    def step_users(self, A_list, E_list, T_list, group_sizes, C: float, sigma: float, seed: int, step: int,
                   L: float | None = None, outputs=None) -> StepOutput:
        """User-level clipping: the records are grouped in order (user u owns
        the next group_sizes[u] records); each user's vector, the sum of its
        records' gradients, is clipped to C; noise is added once and the sum
        divided by L (default: the number of users).  A user is handed to the
        library as one record of its records stacked along T (users with
        fewer records than the largest one padded with zero records by
        dp_pack_groups).  The returned clip and sqnorm are per user."""
        sizes = [int(k) for k in group_sizes]
        B = int(A_list[0].shape[0])
        if any(k < 0 for k in sizes) or sum(sizes) != B:
            raise ValueError("group sizes must be >= 0 and add up to the number of records")
        U, kmax = len(sizes), max(sizes, default=0)
        if U == 0 or kmax == 0:
            raise ValueError("at least one user with a record is needed")
        if all(k == kmax for k in sizes):
            A_u = [a.reshape(U, kmax * a.shape[1], a.shape[2]) for a in A_list]
            E_u = [e.reshape(U, kmax * e.shape[1], e.shape[2]) for e in E_list]
        else:
            starts = torch.zeros(U + 1, dtype=torch.int64)
            starts[1:] = torch.cumsum(torch.tensor(sizes, dtype=torch.int64), 0)
            starts = starts.to(self.device)
            dt = _DT[self.dtype]

            def pack(x):
                out = torch.empty(U, kmax * x.shape[1], x.shape[2], dtype=x.dtype, device=self.device)
                b.dp_pack_groups(x, out, B, x.shape[1], x.shape[2], dt, starts, U, kmax, self.stream)
                return out
            A_u = [pack(a) for a in A_list]
            E_u = [pack(e) for e in E_list]
        T_u = [kmax * int(t) for t in T_list]
        return self.step(A_u, E_u, T_u, C=C, sigma=sigma, seed=seed, step=step, L=L, outputs=outputs)

    def prepare(self, A_list, E_list, T_list, outputs=None, L: float | None = None,
                layer_norms: bool = False) -> "PreparedStep":
        """Marshal the pointer arrays of a step once, for repeated steps on the same buffers."""
        B = int(A_list[0].shape[0])
        outputs = outputs if outputs is not None else self.alloc_outputs(B)
        return PreparedStep(self, A_list, E_list, T_list, outputs, L, layer_norms)

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


class PreparedStep:
    """The four C calls of a step with their pointer arguments marshalled once.

    Valid while the tensors given to ``PrivateGradient.prepare`` stay alive
    and keep their storage (refill them in place between steps).
    """

    def __init__(self, pg: PrivateGradient, A_list, E_list, T_list, outputs, L, layer_norms):
        import ctypes
        n = len(A_list)
        self.pg = pg
        self.lib = b.load_library()
        self.B = int(A_list[0].shape[0])
        self.L = L
        self.n = n
        self.tensors = (list(A_list), list(E_list), outputs)   # keep the storage alive
        self.grads, self.clip, self.sqnorm = outputs
        self.layer_sqnorm = ([torch.empty(self.B, dtype=torch.float32, device=pg.device) for _ in range(n)]
                             if layer_norms else None)
        self._ids = (ctypes.c_int * n)(*range(n))
        self._a = (ctypes.c_void_p * n)(*[int(x.data_ptr()) for x in A_list])
        self._e = (ctypes.c_void_p * n)(*[int(x.data_ptr()) for x in E_list])
        self._t = (ctypes.c_int64 * n)(*[int(t) for t in T_list])
        self._sq = (None if self.layer_sqnorm is None
                    else (ctypes.c_void_p * n)(*[int(x.data_ptr()) for x in self.layer_sqnorm]))
        self._g = (ctypes.c_void_p * n)(*[int(g.data_ptr()) for g in self.grads])
        self._clip = int(self.clip.data_ptr())
        self._sqn = int(self.sqnorm.data_ptr())

    def run(self, C: float, sigma: float, seed: int, step: int, events=None, after_phase=None) -> None:
        """Enqueue one step on the context's stream (asynchronous; no status check).

        events: optional four CUDA events recorded on the stream before the
        norms, after the norms, after the clip factors and after the gradient.
        after_phase: optional callable, called with "norm", "clip" and "grad"
        right after the calls of that phase were enqueued (instrumentation).
        """
        lib, ctx = self.lib, self.pg.ctx
        stream = self.pg.stream
        st = lib.dp_begin_step(ctx, self.B)
        if st == b.DP_OK and self.L is not None:
            st = lib.dp_set_normalizer(ctx, float(self.L))
        if events:
            events[0].record(stream)
        if st == b.DP_OK:
            st = lib.dp_norm_accumulate_batch(ctx, self.n, self._ids, self._a, self._e, self._t, self._sq)
        if events:
            events[1].record(stream)
        if after_phase and st == b.DP_OK:
            after_phase("norm")
        if st == b.DP_OK:
            st = lib.dp_clip_factors(ctx, C, self._clip, self._sqn)
        if events:
            events[2].record(stream)
        if after_phase and st == b.DP_OK:
            after_phase("clip")
        if st == b.DP_OK:
            st = lib.dp_clipped_noisy_grad(ctx, sigma, seed & (2 ** 64 - 1), step & (2 ** 64 - 1), self._g)
        if events:
            events[3].record(stream)
        if after_phase and st == b.DP_OK:
            after_phase("grad")
        if st != b.DP_OK:
            raise b.DPError(st, "PreparedStep.run", b.dp_last_error(ctx))
