"""ctypes binding of the C ABI in include/dp_clip.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  Device
arrays may be passed as torch tensors (their ``data_ptr()`` is used) or as
integer addresses; streams as ``torch.cuda.Stream`` or integer handles.
Nothing is computed in Python: every step of the path runs in the library's
CUDA kernels.  There is no fallback: if ``libdpclip.so`` is missing, or the
GPU is not sm_103, the calls raise.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdpclip.so")

DP_OK = 0
DP_ERR_INVALID_ARG = 1
DP_ERR_SHAPE = 2
DP_ERR_STATE = 3
DP_ERR_NONFINITE = 4
DP_ERR_CUDA = 5
DP_ERR_OOM = 6
DP_ERR_UNSUPPORTED = 7

DP_F32 = 0
DP_BF16 = 1

DP_PATH_GHOST = 0
DP_PATH_MATERIALIZE = 1

EXPORTS = (
    "dp_version", "dp_kernel_launches", "dp_status_string", "dp_create", "dp_destroy", "dp_register_layer",
    "dp_layer_info", "dp_num_coords", "dp_choose_path", "dp_begin_step", "dp_set_normalizer",
    "dp_norm_accumulate", "dp_norm_accumulate_batch", "dp_clip_factors", "dp_clipped_noisy_grad",
    "dp_step_status", "dp_last_error", "dp_philox_normals", "dp_layer_sqnorms_static", "dp_pack_groups",
    "dp_int8_quantize_weight", "dp_int8_workspace_bytes", "dp_int8_forward", "dp_check_wait_timeout", "dp_box_muller",
    "dp_kernel_launch_counts", "dp_clipped_sum", "dp_noise_shard", "dp_static_check_wait_timeout",
)


class DPError(RuntimeError):
    def __init__(self, status: int, func: str, message: str = ""):
        self.status = status
        super().__init__(f"{func} -> {status} ({_status_name(status)}){': ' + message if message else ''}")


_lib = None


def _status_name(s: int) -> str:
    names = {0: "DP_OK", 1: "DP_ERR_INVALID_ARG", 2: "DP_ERR_SHAPE", 3: "DP_ERR_STATE",
             4: "DP_ERR_NONFINITE", 5: "DP_ERR_CUDA", 6: "DP_ERR_OOM", 7: "DP_ERR_UNSUPPORTED"}
    return names.get(s, "?")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libdpclip.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with differentially_private_gb300.build.build()")
    lib = ctypes.CDLL(path)
    c = ctypes
    vp, i64, u64, i32 = c.c_void_p, c.c_int64, c.c_uint64, c.c_int
    sig = {
        "dp_version": (i32, []),
        "dp_kernel_launches": (i64, []),
        "dp_kernel_launch_counts": (i32, [c.POINTER(c.c_char_p), c.POINTER(i64), i32]),
        "dp_clipped_sum": (i32, [vp, c.POINTER(vp)]),
        "dp_noise_shard": (i32, [vp, vp, u64, i64, c.c_float, c.c_float, c.c_double, u64, u64, vp]),
        "dp_static_check_wait_timeout": (i32, [c.c_uint32, vp]),
        "dp_status_string": (c.c_char_p, [i32]),
        "dp_create": (i32, [c.POINTER(vp), i32, vp]),
        "dp_destroy": (i32, [vp]),
        "dp_register_layer": (i32, [vp, i64, i64, i32, i32, c.POINTER(i32)]),
        "dp_layer_info": (i32, [vp, i32, c.POINTER(i64), c.POINTER(i64)]),
        "dp_num_coords": (i64, [vp]),
        "dp_choose_path": (i32, [i64, i64, i64]),
        "dp_begin_step": (i32, [vp, i64]),
        "dp_set_normalizer": (i32, [vp, c.c_double]),
        "dp_norm_accumulate": (i32, [vp, i32, vp, vp, i64, vp]),
        "dp_norm_accumulate_batch": (i32, [vp, i32, c.POINTER(i32), c.POINTER(vp), c.POINTER(vp),
                                           c.POINTER(i64), c.POINTER(vp)]),
        "dp_clip_factors": (i32, [vp, c.c_float, vp, vp]),
        "dp_clipped_noisy_grad": (i32, [vp, c.c_float, u64, u64, c.POINTER(vp)]),
        "dp_step_status": (i32, [vp]),
        "dp_last_error": (c.c_char_p, [vp]),
        "dp_philox_normals": (i32, [u64, u64, u64, i64, vp, vp, vp]),
        "dp_check_wait_timeout": (i32, [vp, c.c_uint32]),
        "dp_box_muller": (i32, [vp, i64, vp, vp]),
        "dp_layer_sqnorms_static": (i32, [vp, vp, i64, i64, i64, i64, i32, i32, vp, vp]),
        "dp_pack_groups": (i32, [vp, vp, i64, i64, i64, i32, vp, i64, i64, vp]),
        "dp_int8_quantize_weight": (i32, [vp, i64, i64, vp, vp, vp, vp]),
        "dp_int8_workspace_bytes": (i64, [i64, i64, i64, i64]),
        "dp_int8_forward": (i32, [vp, i64, i64, i64, vp, vp, vp, i64, c.c_float, i32, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError(f"expected a tensor, an address or None, got {type(x)!r}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError("stream must be a torch.cuda.Stream, an integer handle or None")


def _check(status: int, func: str, ctx=None) -> None:
    if status != DP_OK:
        msg = ""
        if ctx is not None:
            raw = load_library().dp_last_error(ctx)
            msg = raw.decode() if raw else ""
        raise DPError(status, func, msg)


# ---------------------------------------------------------------- entry points
def dp_version() -> int:
    return load_library().dp_version()


def dp_kernel_launches() -> int:
    return load_library().dp_kernel_launches()


def dp_kernel_launch_counts() -> dict:
    """{kernel name: launches so far in this process} for every kernel of the library."""
    lib = load_library()
    k = lib.dp_kernel_launch_counts(None, None, 0)
    names = (ctypes.c_char_p * k)()
    counts = (ctypes.c_int64 * k)()
    lib.dp_kernel_launch_counts(names, counts, k)
    return {names[i].decode(): int(counts[i]) for i in range(k)}


def dp_status_string(status: int) -> str:
    return load_library().dp_status_string(status).decode()


def dp_create(device: int = 0, stream=None) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    _check(load_library().dp_create(ctypes.byref(ctx), int(device), _stream(stream)), "dp_create")
    return ctx


def dp_destroy(ctx) -> None:
    _check(load_library().dp_destroy(ctx), "dp_destroy")


def dp_register_layer(ctx, d_in: int, d_out: int, has_bias: bool, dtype: int) -> int:
    lid = ctypes.c_int()
    _check(load_library().dp_register_layer(ctx, int(d_in), int(d_out), int(bool(has_bias)), int(dtype),
                                            ctypes.byref(lid)), "dp_register_layer", ctx)
    return lid.value


def dp_layer_info(ctx, layer_id: int) -> tuple[int, int]:
    off, n = ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().dp_layer_info(ctx, int(layer_id), ctypes.byref(off), ctypes.byref(n)), "dp_layer_info")
    return off.value, n.value


def dp_num_coords(ctx) -> int:
    return load_library().dp_num_coords(ctx)


def dp_choose_path(T: int, d_in: int, d_out: int) -> int:
    return load_library().dp_choose_path(int(T), int(d_in), int(d_out))


def dp_begin_step(ctx, B: int) -> None:
    _check(load_library().dp_begin_step(ctx, int(B)), "dp_begin_step", ctx)


def dp_set_normalizer(ctx, L: float) -> None:
    _check(load_library().dp_set_normalizer(ctx, float(L)), "dp_set_normalizer", ctx)


def dp_norm_accumulate(ctx, layer_id: int, A, E, T: int, sqnorm_out=None) -> None:
    _check(load_library().dp_norm_accumulate(ctx, int(layer_id), _ptr(A), _ptr(E), int(T), _ptr(sqnorm_out)),
           "dp_norm_accumulate", ctx)


def dp_norm_accumulate_batch(ctx, layer_ids, A_list, E_list, T_list, sqnorm_out=None) -> None:
    n = len(layer_ids)
    ids = (ctypes.c_int * n)(*[int(i) for i in layer_ids])
    a = (ctypes.c_void_p * n)(*[_ptr(x) for x in A_list])
    e = (ctypes.c_void_p * n)(*[_ptr(x) for x in E_list])
    t = (ctypes.c_int64 * n)(*[int(x) for x in T_list])
    sq = None if sqnorm_out is None else (ctypes.c_void_p * n)(*[_ptr(x) for x in sqnorm_out])
    _check(load_library().dp_norm_accumulate_batch(ctx, n, ids, a, e, t, sq), "dp_norm_accumulate_batch", ctx)


def dp_clip_factors(ctx, C: float, c_out=None, total_sqnorm_out=None) -> None:
    _check(load_library().dp_clip_factors(ctx, float(C), _ptr(c_out), _ptr(total_sqnorm_out)),
           "dp_clip_factors", ctx)


def dp_clipped_noisy_grad(ctx, sigma: float, seed: int, step: int, G_list) -> None:
    n = len(G_list)
    g = (ctypes.c_void_p * n)(*[_ptr(x) for x in G_list])
    _check(load_library().dp_clipped_noisy_grad(ctx, float(sigma), int(seed) & (2 ** 64 - 1),
                                                int(step) & (2 ** 64 - 1), g), "dp_clipped_noisy_grad", ctx)


def dp_clipped_sum(ctx, S_list) -> None:
    """The clipped sum without noise or normalizer (one rank's partial sum); closes the step."""
    n = len(S_list)
    g = (ctypes.c_void_p * n)(*[_ptr(x) for x in S_list])
    _check(load_library().dp_clipped_sum(ctx, g), "dp_clipped_sum", ctx)


def dp_noise_shard(S, G, k0: int, n: int, sigma: float, C: float, L: float, seed: int, step: int,
                   stream=None) -> None:
    """G[j] = (S[j] + sigma C z_{k0+j}) / L over a contiguous range of global coordinates."""
    _check(load_library().dp_noise_shard(_ptr(S), _ptr(G), int(k0), int(n), float(sigma), float(C), float(L),
                                         int(seed) & (2 ** 64 - 1), int(step) & (2 ** 64 - 1), _stream(stream)),
           "dp_noise_shard")


def dp_step_status(ctx) -> int:
    """Synchronize and return the step's deferred status code (does not raise)."""
    return load_library().dp_step_status(ctx)


def dp_last_error(ctx) -> str:
    raw = load_library().dp_last_error(ctx)
    return raw.decode() if raw else ""


def dp_philox_normals(seed: int, step: int, k0: int, n: int, raw_out=None, z_out=None, stream=None) -> None:
    _check(load_library().dp_philox_normals(int(seed) & (2 ** 64 - 1), int(step) & (2 ** 64 - 1), int(k0), int(n),
                                            _ptr(raw_out), _ptr(z_out), _stream(stream)), "dp_philox_normals")


def dp_box_muller(words, npairs: int, z_out, stream=None) -> None:
    """The noise's Box-Muller map on given word pairs (test hook)."""
    _check(load_library().dp_box_muller(_ptr(words), int(npairs), _ptr(z_out), _stream(stream)), "dp_box_muller")


def dp_check_wait_timeout(ctx, limit_ms: int) -> None:
    """Enqueue the bounded wait that gives up (test hook of the timeout path)."""
    _check(load_library().dp_check_wait_timeout(ctx, int(limit_ms)), "dp_check_wait_timeout", ctx)


def dp_layer_sqnorms_static(A, E, B: int, T: int, d_in: int, d_out: int, has_bias: bool, dtype: int,
                            sqnorm_out, stream=None) -> None:
    """One layer's per-example squared norms through the entry point that allocates nothing."""
    _check(load_library().dp_layer_sqnorms_static(_ptr(A), _ptr(E), int(B), int(T), int(d_in), int(d_out),
                                                  int(bool(has_bias)), int(dtype), _ptr(sqnorm_out),
                                                  _stream(stream)), "dp_layer_sqnorms_static")


def dp_static_check_wait_timeout(limit_ms: int, stream=None) -> None:
    """Record a bounded wait that gave up for the next dp_layer_sqnorms_static call (test hook)."""
    _check(load_library().dp_static_check_wait_timeout(int(limit_ms), _stream(stream)),
           "dp_static_check_wait_timeout")


def dp_pack_groups(src, dst, B: int, T: int, d: int, dtype: int, group_starts, U: int, kmax: int,
                   stream=None) -> None:
    """Records grouped by user, laid out [U, kmax, T, d] with zero records where a user has fewer."""
    _check(load_library().dp_pack_groups(_ptr(src), _ptr(dst), int(B), int(T), int(d), int(dtype),
                                         _ptr(group_starts), int(U), int(kmax), _stream(stream)), "dp_pack_groups")


def dp_int8_quantize_weight(W, N: int, K: int, Wq, sW, What, stream=None) -> None:
    _check(load_library().dp_int8_quantize_weight(_ptr(W), int(N), int(K), _ptr(Wq), _ptr(sW), _ptr(What),
                                                  _stream(stream)), "dp_int8_quantize_weight")


def dp_int8_workspace_bytes(n: int, K: int, N: int, rows_per_record: int) -> int:
    return int(load_library().dp_int8_workspace_bytes(int(n), int(K), int(N), int(rows_per_record)))


def dp_int8_forward(A, n: int, K: int, rows_per_record: int, Wq, sW, What, N: int, tau: float, record_owned: bool,
                    Y, workspace, stream=None) -> None:
    _check(load_library().dp_int8_forward(_ptr(A), int(n), int(K), int(rows_per_record), _ptr(Wq), _ptr(sW),
                                          _ptr(What), int(N), float(tau), int(bool(record_owned)), _ptr(Y),
                                          _ptr(workspace), _stream(stream)), "dp_int8_forward")
