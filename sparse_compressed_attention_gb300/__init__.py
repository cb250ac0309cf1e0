"""DeepSeek-V4-Flash compressed attention forward on one GB300 (sm_103a).

The compute lives in the CUDA library built from ``csrc/`` (C ABI in
``include/v4attn.h``); this package is its thin ctypes binding.
"""
from ._lib import (EXPORTS, V4Error, V4_BF16, V4_F32, V4_PATH_AUTO, V4_PATH_SIMT, V4_PATH_TC,  # noqa: F401
                   alloc_bwd_workspace, alloc_workspace, config_from_preset, lib, make_config, v4_attn_layer_fwd,
                   v4_compress, v4_config, v4_get_device_status, v4_grouped_o_proj,
                   v4_indexer_prep, v4_indexer_topk, v4_last_error, v4_launch_count, v4_profile_count, v4_profile_enable,
                   v4_profile_get, v4_profile_records,
                   v4_reset_device_status, v4_rope_inv_freq, v4_sparse_mqa_fwd, v4_sparse_mqa_fwd_noalloc,
                   v4_workspace_size, v4_bwd_workspace_size, v4_sparse_mqa_bwd, v4_quantize_e4m3,
                   v4_indexer_topk_e4m3, v4_q_proj, v4_indexer_kl_target, v4_selftest_wait_timeout,
                   v4_build_info)
