"""GB300-native DP-SGD private-gradient hot path (clip + noise).

The work is done by ``libdpclip.so`` (hand-written CUDA for sm_103a) behind
the C ABI of ``include/dp_clip.h``; this package is its ctypes binding
(``_binding``, same names as the C entry points), a convenience wrapper
(``step.PrivateGradient``), the in-tree build (``build``), the sensitivity
audit of the computation (``audit``), and per-record activations and output
gradients captured from a model's own forward and backward (``capture``,
with an OPT-shaped LoRA producer in ``opt_lora``).
"""

from ._binding import (  # noqa: F401
    DP_BF16,
    DP_ERR_CUDA,
    DP_ERR_INVALID_ARG,
    DP_ERR_NONFINITE,
    DP_ERR_OOM,
    DP_ERR_SHAPE,
    DP_ERR_STATE,
    DP_ERR_UNSUPPORTED,
    DP_F32,
    DP_OK,
    DP_PATH_GHOST,
    DP_PATH_MATERIALIZE,
    DPError,
    EXPORTS,
    LIB_PATH,
    dp_begin_step,
    dp_box_muller,
    dp_check_wait_timeout,
    dp_choose_path,
    dp_clip_factors,
    dp_clipped_noisy_grad,
    dp_clipped_sum,
    dp_create,
    dp_destroy,
    dp_int8_forward,
    dp_int8_quantize_weight,
    dp_int8_workspace_bytes,
    dp_kernel_launch_counts,
    dp_kernel_launches,
    dp_last_error,
    dp_layer_info,
    dp_layer_sqnorms_static,
    dp_norm_accumulate,
    dp_noise_shard,
    dp_norm_accumulate_batch,
    dp_num_coords,
    dp_pack_groups,
    dp_philox_normals,
    dp_register_layer,
    dp_set_normalizer,
    dp_static_check_wait_timeout,
    dp_status_string,
    dp_step_status,
    dp_version,
    load_library,
)
from .step import PrivateGradient, StepOutput  # noqa: F401
