"""GB300 (sm_103a) exact causal GQA attention: Python binding of libattn_gb300.so.

The binding only marshals arguments: it checks tensor dtypes, devices and
layouts, passes raw device pointers and the current CUDA stream to the C ABI
declared in include/attn_gb300.h, and raises on a non-zero status.  Every step
of the computation runs in the library's CUDA kernels; there is no fallback.
PyTorch provides device memory and streams.

Entry points (same names as the C ABI):
    rope_apply(x, positions, base)                      RoPE at absolute positions, in place
    rope_apply_qk(q, k, positions, base)                the same on queries and keys in one launch
    rope_table(positions, head_dim, base)               cos/sin table for on-the-fly rotation
    attn_prefill(..., q_rope_cs=table)                  attention with the query's RoPE fused in
    attn_kv_append_paged(k_new, v_new, positions, slots, k_cache, v_cache)
                                                        new K (rotated) / V into the paged cache
    attn_kv_append_paged_int8(..., k_scale, v_scale)    the same into an INT8 cache (quantising)
    attn_prefill(q, k, v, out, lse, cu_q, q_pos, ...)   tiled causal GQA attention
    attn_prefill_fp8(q, q_scale, k, k_scale, v_t, v_scale, ...)  the same on e4m3 codes (FP8 mode)
    quant_fp8_rows(x) / quant_fp8_heads(x, transposed)   e4m3 codes and scales for it
    rope_quant_fp8_rows / rope_quant_fp8_heads(x, positions)  RoPE fused into that quantisation
    attn_decode_paged(q, k_cache, v_cache, ...)         split-KV decode over a paged cache
    attn_decode_paged_int8(q, k_codes, v_codes, k_scale, v_scale, ...)   the same over an INT8 cache
    attn_lse_merge(part_out, part_lse, out, lse, ...)   log-sum-exp merge of partials

Sequence parallelism around the kernels (host code over torch.distributed):
    sp.ulysses_attention / sp.seq_to_heads / sp.heads_to_seq   the Ulysses all-to-all
    sp.ring_attention / sp.shard_rows                          ring context parallelism
"""
from ._binding import (ATTN_BF16, ATTN_FP32, AttnError, attn_decode_paged, attn_decode_paged_int8,
                       attn_device_status, attn_selftest_wait_timeout,
                       attn_kv_append_paged, attn_kv_append_paged_int8, attn_lse_merge, attn_prefill, attn_prefill_fp8,
                       decode_workspace, lib_path, library, prefill, quant_fp8_heads, quant_fp8_rows, rope_apply, rope_apply_qk, rope_quant_fp8_heads,
                       rope_quant_fp8_rows, rope_table)
from . import sp

__all__ = ["ATTN_BF16", "ATTN_FP32", "AttnError", "attn_decode_paged", "attn_decode_paged_int8", "attn_device_status",
           "attn_selftest_wait_timeout", "attn_kv_append_paged", "attn_kv_append_paged_int8", "attn_lse_merge", "attn_prefill", "attn_prefill_fp8", "decode_workspace", "lib_path", "library",
           "prefill", "quant_fp8_heads", "quant_fp8_rows", "rope_apply", "rope_apply_qk", "rope_quant_fp8_heads",
           "rope_quant_fp8_rows", "rope_table", "sp"]
