// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

struct RopeLaunch {
  void* x;
  int dtype;  // 0 bf16, 1 fp32
  int64_t tokens;
  int heads, head_dim;
  int64_t stride_token;
  const int32_t* positions;
  double base;
  void* x2 = nullptr;  // optional second tensor rotated at the same positions (keys with the queries)
  int heads2 = 0;
  int64_t stride2 = 0;
};
cudaError_t launch_rope(const RopeLaunch& a, cudaStream_t s);
cudaError_t launch_rope_table(float* cs_out, int64_t tokens, int head_dim, const int32_t* positions, double base,
                              cudaStream_t s);

struct AppendLaunch {
  const void* k_new;
  const void* v_new;
  const int32_t* positions;
  const int32_t* slots;
  int64_t tokens;
  int heads, head_dim;
  void* k_cache;
  void* v_cache;
  int64_t cache_rows;  // num_pages * page_size
  void* k_rot_out;
  double base;  // 0: copy keys unrotated
  unsigned* err;
  float* k_scale = nullptr;  // INT8 cache: per-row scales (k_cache / v_cache then hold int8 codes)
  float* v_scale = nullptr;
};
cudaError_t launch_kv_append(const AppendLaunch& a, cudaStream_t s);
cudaError_t launch_kv_append_int8(const AppendLaunch& a, cudaStream_t s);
cudaError_t launch_quant_fp8_rows(const void* x, int64_t rows, void* codes, float* scales, cudaStream_t s);
cudaError_t launch_quant_fp8_heads(const void* x, int64_t tokens, int heads, void* codes, float* scales,
                                   unsigned* amax_scratch, bool transposed, int64_t t_stride, cudaStream_t s);
// RoPE + e4m3 quantisation of a bf16 [tokens][heads][128] tensor: one scale per
// row when amax_scratch is null, else one per head (amax_scratch: [heads]).
constexpr int kMaxQuantHeads = 256;
cudaError_t launch_rope_quant_fp8(const void* x, int64_t tokens, int heads, const int32_t* positions, double base,
                                  void* codes, float* scales, unsigned* amax_scratch, cudaStream_t s);

struct MergeLaunch {
  const float* part_out;
  const float* part_lse;
  int n_parts;
  int64_t rows;
  int heads, head_dim;
  int64_t osp, osr, osh, lsp, lsr, lsh;
  void* out;
  int out_f32;
  float* lse_out;
};
cudaError_t launch_lse_merge(const MergeLaunch& a, cudaStream_t s);

struct PrefillLaunch {
  const void *q, *k, *v;
  void* out;
  int out_f32;
  float* lse;
  int in_f32;
  int batch;
  const int32_t *cu_q, *q_pos;
  int max_seqlen_q;
  const int32_t *cu_k, *k_pos;
  const int32_t *page_table, *k_lens;
  int max_pages, page_size;
  int64_t num_pages;
  int hq, hkv, d, h_lo, h_hi;
  float scale;
  int causal;
  unsigned* err;
  const float* q_rope_cs = nullptr;  // tcgen05 kernel only: [total_q][d/2][2] cos, sin; rotate Q on the fly
  // tcgen05 kernel only: q, k are e4m3 codes [T][H][128], v the transposed codes
  // [hkv][128][t_stride]; values are code * scale
  int fp8 = 0;
  const float *q_scale = nullptr, *k_scale = nullptr, *v_scale = nullptr;
};
// CUDA-core kernel: any supported dtype / head_dim / page size.
cudaError_t launch_prefill_simt(const PrefillLaunch& a, cudaStream_t s);
// tcgen05 tensor-core kernel: bf16, head_dim 128, page size 64 when paged.
// The tensor maps are built by the caller.
cudaError_t launch_prefill_tc(const PrefillLaunch& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t s);

struct DecodeLaunch {
  const void* q;
  const int32_t *page_table, *ctx_lens;
  int batch, max_pages;
  int64_t num_pages;
  int hq, hkv, num_splits;
  float scale;
  float *part_out, *part_lse;
  unsigned* err;
};
cudaError_t launch_decode_split(const DecodeLaunch& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t s);
cudaError_t launch_decode_split_int8(const DecodeLaunch& a, const float* k_scale, const float* v_scale,
                                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);

// Records `msg` as this thread's attn_last_error() text and returns `code`.
int set_last_error(int code, const char* msg);

}  // namespace attn
