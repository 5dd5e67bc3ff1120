"""dp_layer_sqnorms_static: one layer's per-example norms with no allocation.

Callers that cannot call cudaMalloc (a process whose device memory is all
reserved by its own pool, a program whose memory belongs to another
framework's allocator, a latency-bound loop that cannot take the
synchronization cudaMalloc may cause) use this entry point: its scratch is
a fixed array inside the library.  These tests check, through the C ABI,
that it returns what dp_norm_accumulate returns for the same layer, on
calls made one after another that reuse the shared array, and that a
request larger than the array is refused before any work is launched.

This file is collected last, so a run that stops at the first failure has
run every other test already.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

NORM_RTOL = {torch.float32: 1e-3, torch.bfloat16: 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from differentially_private_gb300 import build
    build.build()


def _inputs(seed, B, T, d_in, d_out, dtype):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(B, T, d_in, generator=g, device="cuda").to(dtype)
    E = (0.1 * torch.randn(B, T, d_out, generator=g, device="cuda")).to(dtype)
    return A, E


def _with_context(A, E, T, d_in, d_out, has_bias, dtype):
    """The same norms through the context entry point dp_norm_accumulate."""
    import differentially_private_gb300 as dp
    B = A.shape[0]
    ctx = dp.dp_create(0, torch.cuda.current_stream())
    try:
        lid = dp.dp_register_layer(ctx, d_in, d_out, has_bias, dp.DP_F32 if dtype == torch.float32 else dp.DP_BF16)
        dp.dp_begin_step(ctx, B)
        out = torch.empty(B, dtype=torch.float32, device="cuda")
        dp.dp_norm_accumulate(ctx, lid, A, E, T, out)
        torch.cuda.synchronize()
        return out.cpu().numpy()
    finally:
        dp.dp_destroy(ctx)


def _static(A, E, T, d_in, d_out, has_bias, dtype):
    import differentially_private_gb300 as dp
    B = A.shape[0]
    out = torch.full((B,), -1.0, dtype=torch.float32, device="cuda")
    dp.dp_layer_sqnorms_static(A, E, B, T, d_in, d_out, has_bias,
                               dp.DP_F32 if dtype == torch.float32 else dp.DP_BF16, out,
                               torch.cuda.current_stream())
    torch.cuda.synchronize()
    return out.cpu().numpy()


CASES = [
    # (B, T, d_in, d_out, bias, dtype): tensor-core Gram, skinny materialize,
    # T = 1 closed form, CUDA-core Gram with a bias, CUDA-core materialize
    # with a bias (its per-example gradients are not kept here)
    (4, 128, 256, 128, False, torch.bfloat16),
    (3, 128, 768, 8, False, torch.bfloat16),
    (64, 1, 1024, 512, False, torch.bfloat16),
    (5, 24, 48, 40, True, torch.float32),
    (3, 64, 8, 8, True, torch.float32),
]


def test_cases_cover_every_norm_path():
    import differentially_private_gb300 as dp
    paths = [dp.dp_choose_path(T, d_in, d_out) for (_, T, d_in, d_out, _, _) in CASES]
    assert paths == [dp.DP_PATH_GHOST, dp.DP_PATH_MATERIALIZE, dp.DP_PATH_GHOST, dp.DP_PATH_GHOST,
                     dp.DP_PATH_MATERIALIZE]


def test_static_scratch_matches_context_entry_point_on_consecutive_calls():
    first = None
    for k, (B, T, d_in, d_out, bias, dt) in enumerate(CASES):
        A, E = _inputs(100 + k, B, T, d_in, d_out, dt)
        ref = _with_context(A, E, T, d_in, d_out, bias, dt)
        got1 = _static(A, E, T, d_in, d_out, bias, dt)
        got2 = _static(A, E, T, d_in, d_out, bias, dt)     # second call in a row, same shared array
        for got in (got1, got2):
            assert np.all(np.abs(got - ref) <= NORM_RTOL[dt] * np.abs(ref)), (k, got, ref)
        if first is None:
            first = (A, E, B, T, d_in, d_out, bias, dt, ref)
    # the array still holds the last case's partials; the first case is unaffected
    A, E, B, T, d_in, d_out, bias, dt, ref = first
    got = _static(A, E, T, d_in, d_out, bias, dt)
    assert np.all(np.abs(got - ref) <= NORM_RTOL[dt] * np.abs(ref))


def test_request_beyond_the_static_array_is_refused():
    import differentially_private_gb300 as dp
    # T = 1: one slot per record, so 2^20 + 1 records exceed the array
    B = (1 << 20) + 1
    A = torch.zeros(16, dtype=torch.bfloat16, device="cuda")   # never read: refused first
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(dp.DPError) as ei:
        dp.dp_layer_sqnorms_static(A, A, B, 1, 8, 8, False, dp.DP_BF16, out)
    assert ei.value.status == dp.DP_ERR_SHAPE
    with pytest.raises(dp.DPError) as ei:
        dp.dp_layer_sqnorms_static(None, A, 4, 1, 8, 8, False, dp.DP_BF16, out)
    assert ei.value.status == dp.DP_ERR_INVALID_ARG


def test_wait_that_gave_up_makes_the_norms_nan_and_the_next_call_is_clean():
    """A tensor-core wait that gives up leaves the partial sums unwritten: the
    call then reports NaN norms (the caller sees a non-finite norm) instead
    of summing stale partials.  The test hook records such a timeout exactly
    as a norm kernel's bounded wait would, without any fault."""
    import differentially_private_gb300 as dp
    B, T, d_in, d_out, bias, dt = CASES[0]
    A, E = _inputs(7, B, T, d_in, d_out, dt)
    ref = _with_context(A, E, T, d_in, d_out, bias, dt)
    dp.dp_static_check_wait_timeout(20, torch.cuda.current_stream())
    got = _static(A, E, T, d_in, d_out, bias, dt)
    assert np.all(np.isnan(got)), got
    got = _static(A, E, T, d_in, d_out, bias, dt)
    assert np.all(np.abs(got - ref) <= NORM_RTOL[dt] * np.abs(ref)), (got, ref)
    with pytest.raises(dp.DPError) as ei:
        dp.dp_static_check_wait_timeout(0)
    assert ei.value.status == dp.DP_ERR_INVALID_ARG
