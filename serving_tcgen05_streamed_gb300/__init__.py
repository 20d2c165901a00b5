"""Streamed fused-QKV projection with rotated, group-scaled, packed INT4 K/V
and a dense attention that reads the packed K/V tile by tile, for one GB300
(sm_103a).  The computation is the CUDA library libkvq.so (C ABI in
include/kvq.h); this package is its binding plus seeded synthetic inputs.
"""
from ._lib import (  # noqa: F401
    EXPORTS, KVQ_ERR_ALIGN, KVQ_ERR_ARG, KVQ_ERR_CUDA, KVQ_ERR_TIMEOUT, KVQ_ERR_UNSUPPORTED, KVQ_OK, KvqError,
    PackedKV, codes_bytes, device_status, kv_rotate_quant_pack, kv_unpack, load, packed_kv_attention,
    packed_kv_attention_causal, packed_kv_attention_mixed, padded_rows, scales_bytes, selftest_wait_timeout, status_str,
    streamed_qkv_proj, streamed_qkv_proj_mixed, streamed_qkv_proj_ex, SECTION_Q, SECTION_KV, version,
    packed_kv_attention_partial, partial_state, PARTIAL_MERGE, PARTIAL_FINAL,
    packed_kv_attention_partial_static, STATIC_STATE_BYTES, KVQ_ERR_TOO_LARGE,
)
