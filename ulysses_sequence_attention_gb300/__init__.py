"""GB300-native Ulysses sequence-parallel attention layer.

``_binding`` exposes the C-ABI calls of ``libulysses.so`` under their own names.
``layer.UlyssesLayer`` strings them together into the layer forward and backward
for P virtual ranks on one GPU. Importing this package fails loudly when the
CUDA library has not been built: there is no fallback path.
"""
from ._binding import (  # noqa: F401
    LIB_PATH, ULYSSES_BF16, ULYSSES_ERR_ALIGNMENT, ULYSSES_ERR_CUDA, ULYSSES_ERR_DIVISIBILITY,
    ULYSSES_ERR_INVALID_ARG, ULYSSES_ERR_TIMEOUT, ULYSSES_ERR_TOO_LARGE, ULYSSES_ERR_UNSUPPORTED, ULYSSES_FP32,
    ULYSSES_MAX_P, ULYSSES_OK, ULYSSES_NOALLOC_SCRATCH_BYTES, UlyssesError, UlyssesHandle, ulysses_attn_bwd,
    ulysses_attn_bwd_noalloc, ulysses_attn_fwd,
    ulysses_create, ulysses_destroy, ulysses_get_status, ulysses_head_to_seq, ulysses_launch_count, ulysses_seq_to_head,
    ulysses_strerror, ulysses_workspace_size, ulysses_set_ds_budget, ulysses_ds_bytes, ulysses_set_wait_limit, ulysses_inject_fault,
    ulysses_timing_enable, ulysses_timing_read, ULYSSES_KERNEL_COUNT, KERNEL_NAMES,
    ulysses_fused_supported, ulysses_layer_fwd, ulysses_layer_bwd,
    ulysses_host_begin, ulysses_host_step, ulysses_host_end, ulysses_create_varlen, ulysses_set_seq,
    ulysses_seq_to_head_qkv, ulysses_head_to_seq_qkv,
)
from .layer import HostSteps, UlyssesLayer, default_ds_budget  # noqa: F401
