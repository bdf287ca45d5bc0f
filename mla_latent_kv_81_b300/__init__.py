"""B300-native Multi-head Latent Attention decode over a paged latent cache.

The compute lives in libmla.so (hand-written sm_103a CUDA behind a C ABI,
declared in include/mla.h); this package is its thin ctypes binding.
"""
from ._binding import (  # noqa: F401
    EXPORTED, LIB_PATH, MLA_BF16, MLA_F32, MlaError, default_scale, lib, make_cache, make_config, make_rope,
    mla_absorb_query, mla_absorb_workspace_bytes, mla_cache_bytes_per_token, mla_compress_append,
    mla_compress_append_noalloc,
    mla_compress_workspace_bytes, mla_config, mla_decode_attention, mla_decode_workspace_bytes,
    mla_get_device_status, mla_head_output_project, mla_head_output_workspace_bytes, mla_kernel_launches,
    mla_output_project, mla_output_workspace_bytes, mla_paged_cache, mla_prefill_attention,
    mla_prefill_workspace_bytes, mla_project_query, mla_project_workspace_bytes,
    mla_rope_table, mla_rope_table_create, mla_selftest_wait_timeout, mla_status_string, workspace)
