"""Fused attention forward for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library ``libattn.so`` (C ABI in
``include/attn.h``); ``attn`` is its thin ctypes binding and ``inputs`` the
seeded synthetic-input generator shared with the tests and the benchmark.
"""
from .attn import (  # noqa: F401
    ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_OK,
    MASK_ADDITIVE, MASK_CAUSAL, MASK_CAUSAL_ADDITIVE, MASK_NONE, AttnError, attention, attn_abi_version,
    attn_debug_inject_stall, attn_fwd, attn_fwd_f16, attn_fwd_splitkv, attn_fwd_splitkv_f16, attn_last_status,
    attn_set_wait_timeout_ns, attn_splitkv_num_splits, attn_splitkv_workspace_bytes, attn_status_string,
    attention_splitkv, attn_fwd_rope, attn_fwd_rope_f16, attn_rope_table, attn_rope_apply, attn_rope_apply_f16,
    attention_rope, rope_table, rope_apply, attn_fwd_host, attn_fwd_host_f16, attn_fwd_host_workspace_bytes,
    attention_host, attn_linear, attn_layernorm, attn_fwd_qkvpacked, attn_block_fwd, attn_block_workspace_bytes,
    linear, layernorm, attention_qkvpacked, attention_block)
