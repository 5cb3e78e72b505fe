"""LowRAM compressed-cache decode attention for B300 (sm_103a).

The compute lives in ``liblowram.so`` (hand-written CUDA kernels behind the C ABI of
``include/lowram.h``); this package is its ctypes binding.  Build the library with
``python -m decode_attention_19_b300.build``.
"""
from .binding import (  # noqa: F401
    CHECK_LAYOUT, CHECK_NOT_PD, CHECK_POS_RANGE, FLAG_INT4_EXACT_SPLIT, CHECK_RES_INDEX, CHECK_TIMEOUT, LIB_PATH, LOWRAM_BF16, LOWRAM_F32, LOWRAM_INT4_G32, LOWRAM_INT8_VEC,
    LowramError, LowramShapeError, decode_shape, lib, lowram_clear_error, lowram_compress, lowram_compress_workspace_size,
    lowram_decode_attn, lowram_decode_attn_static, lowram_decode_attn_static_get_error, lowram_decode_shape, lowram_decode_uses_tensor_cores, lowram_compress_shape, lowram_decode_workspace_size,
    lowram_dense_decode_attn, lowram_dense_workspace_size, lowram_merge_attn, lowram_tail_append,
    lowram_tail_decode_attn, lowram_fit_basis, lowram_predictor_grad, lowram_fit_predictor,
    lowram_attention_mass, lowram_evict_plan, lowram_attention_mass_workspace_size, lowram_evict_plan_workspace_size, lowram_get_error, lowram_rope_table, lowram_version, lowram_set_wait_limit,
)
