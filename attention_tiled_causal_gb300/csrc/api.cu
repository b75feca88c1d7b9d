// C ABI of libattn_gb300.so: argument checks, TMA descriptors, kernel choice.
// The entry points and their contracts are documented in include/attn_gb300.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "../../include/attn_gb300.h"
#include "common.cuh"
#include "kernels.h"

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Device-side error word, one per device.  Kernels record a code with
// atomicCAS; attn_device_status() reads and clears it.
__device__ unsigned g_attn_dev_err;

constexpr int kMaxDev = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDev] = {};

int device_error_ptr(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev) return fail(ATTN_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_dev_err);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    g_err_ptr[dev] = (unsigned*)p;
  }
  *out = g_err_ptr[dev];
  return ATTN_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encode(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  static std::once_flag once;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (status == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = (EncodeTiledFn)p;
  });
  if (!cached) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorName(status));
  *fn = cached;
  return ATTN_OK;
}

// Tensor map of element type dt with a 128-byte swizzle (boxes whose innermost
// extent is 128 bytes: 64 bf16 or 128 one-byte elements).
int encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const cuuint64_t* dims,
                 const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  EncodeTiledFn fn = nullptr;
  int rc = get_encode(&fn);
  if (rc) return rc;
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return ATTN_OK;
}

int encode_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                const cuuint32_t* box) {
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box);
}

// [tokens][heads][128] bf16, box (64 dims, 1 head, 128 tokens).
int map_tokens(CUtensorMap* m, const void* base, int64_t tokens, int heads) {
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, 1, 128};
  return encode_bf16(m, base, 3, dims, strides, box);
}

// head-major paged cache [hkv][num_pages][64][128] bf16 as rows of 128, box (64 dims, 64 rows).
int map_pages(CUtensorMap* m, const void* base, int hkv, int64_t num_pages) {
  cuuint64_t dims[2] = {128, (cuuint64_t)hkv * (cuuint64_t)num_pages * 64};
  cuuint64_t strides[1] = {128 * 2};
  cuuint32_t box[2] = {64, 64};
  return encode_bf16(m, base, 2, dims, strides, box);
}

// e4m3 codes [tokens][heads][128] as rows of 128 bytes, box (128 bytes, 1 head, 128 tokens).
int map_tokens_i8(CUtensorMap* m, const void* base, int64_t tokens, int heads) {
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
  cuuint64_t strides[2] = {128, (cuuint64_t)heads * 128};
  cuuint32_t box[3] = {128, 1, 128};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 3, dims, strides, box);
}

// transposed e4m3 codes [heads][128][t_stride], box (128 keys, 128 dims, 1 head).
int map_vt_i8(CUtensorMap* m, const void* base, int64_t t_stride, int heads) {
  cuuint64_t dims[3] = {(cuuint64_t)t_stride, 128, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)t_stride, (cuuint64_t)t_stride * 128};
  cuuint32_t box[3] = {128, 128, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 3, dims, strides, box);
}

// head-major paged INT8 cache [hkv][num_pages][64][128] as rows of 128 bytes, box (128 bytes, 64 rows).
int map_pages_i8(CUtensorMap* m, const void* base, int hkv, int64_t num_pages) {
  cuuint64_t dims[2] = {128, (cuuint64_t)hkv * (cuuint64_t)num_pages * 64};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 64};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 2, dims, strides, box);
}

}  // namespace

namespace attn {
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

// One block whose thread 0 waits, through the helper `which` selects, on an
// mbarrier that nothing completes, so the wait runs out after its limit and
// its code is recorded: 0, mbar_wait (the prefill and decode pipelines'), code
// DEV_TIMEOUT_MMA; 1, mbar_wait_own (the staged appends'), DEV_TIMEOUT_APPEND.
__global__ void wait_timeout_selftest_kernel(unsigned* err, int which) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (which == 0)
    mbar_wait(&bar, 0, err, DEV_TIMEOUT_MMA);
  else if (!mbar_wait_own(&bar, 0))
    record_error(err, DEV_TIMEOUT_APPEND);
}
}  // namespace attn

extern "C" {

const char* attn_last_error(void) { return g_msg; }

int attn_selftest_wait_timeout(int which, void* stream) {
  if (which != 0 && which != 1) return fail(ATTN_ERR_ARG, "attn_selftest_wait_timeout: which must be 0 or 1");
  unsigned* err = nullptr;
  int rc = device_error_ptr(&err);
  if (rc) return rc;
  attn::wait_timeout_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, which);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_selftest_wait_timeout launch");
}

int attn_device_status(int clear) {
  unsigned* p = nullptr;
  int rc = device_error_ptr(&p);
  if (rc) return rc;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned v = 0;
  e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (clear) {
    e = cudaMemset(p, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  }
  if (v) {
    // the device codes of common.cuh: 0x10x wait timeouts, 0x20x bad inputs
    const char* what = v == 0x201   ? "page id outside the cache"
                       : v == 0x202 ? "cache slot outside the cache"
                       : v == 0x203 ? "INT8 decode value beyond the fp16 range"
                       : v == 0x204 ? "FP8 prefill key sequence not starting at a multiple of 16"
                       : v == 0x105 ? "cache append: a staged copy of new rows did not land in time"
                                    : "pipeline wait timed out";
    return fail(ATTN_ERR_DEVICE, "device error 0x%x (%s)", v, what);
  }
  return ATTN_OK;
}

int rope_apply(void* x, attn_dtype_t dtype, int64_t tokens, int heads, int head_dim, int64_t stride_token,
               const int32_t* positions, double base, void* stream) {
  if (tokens < 0 || heads < 0 || head_dim <= 0) return fail(ATTN_ERR_ARG, "rope_apply: negative size");
  if (tokens == 0 || heads == 0) return ATTN_OK;
  if (!x || !positions) return fail(ATTN_ERR_ARG, "rope_apply: null pointer");
  if (dtype != ATTN_BF16 && dtype != ATTN_FP32) return fail(ATTN_ERR_UNSUPPORTED, "rope_apply: dtype");
  const int V = dtype == ATTN_BF16 ? 8 : 4;
  if (head_dim % 2 || (head_dim / 2) % V || head_dim > 256)
    return fail(ATTN_ERR_SHAPE, "rope_apply: head_dim %d (need head_dim/2 a multiple of %d, <= 256)", head_dim, V);
  if (stride_token < (int64_t)heads * head_dim) return fail(ATTN_ERR_ARG, "rope_apply: stride_token too small");
  if (!aligned16(x) || stride_token % V) return fail(ATTN_ERR_ALIGN, "rope_apply: x / stride not 16-byte aligned");
  if (!(base > 0.0)) return fail(ATTN_ERR_ARG, "rope_apply: base must be positive");
  attn::RopeLaunch a{x, dtype == ATTN_BF16 ? 0 : 1, tokens, heads, head_dim, stride_token, positions, base};
  cudaError_t e = attn::launch_rope(a, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "rope_apply launch");
}

int rope_apply_qk(void* q, int q_heads, int64_t q_stride_token, void* k, int k_heads, int64_t k_stride_token,
                  attn_dtype_t dtype, int64_t tokens, int head_dim, const int32_t* positions, double base,
                  void* stream) {
  if (tokens < 0 || q_heads < 0 || k_heads < 0 || head_dim <= 0)
    return fail(ATTN_ERR_ARG, "rope_apply_qk: negative size");
  if (tokens == 0 || q_heads + k_heads == 0) return ATTN_OK;
  if ((q_heads && !q) || (k_heads && !k) || !positions) return fail(ATTN_ERR_ARG, "rope_apply_qk: null pointer");
  if (dtype != ATTN_BF16 && dtype != ATTN_FP32) return fail(ATTN_ERR_UNSUPPORTED, "rope_apply_qk: dtype");
  const int V = dtype == ATTN_BF16 ? 8 : 4;
  if (head_dim % 2 || (head_dim / 2) % V || head_dim > 256)
    return fail(ATTN_ERR_SHAPE, "rope_apply_qk: head_dim %d (need head_dim/2 a multiple of %d, <= 256)", head_dim, V);
  if ((q_heads && q_stride_token < (int64_t)q_heads * head_dim) ||
      (k_heads && k_stride_token < (int64_t)k_heads * head_dim))
    return fail(ATTN_ERR_ARG, "rope_apply_qk: stride_token too small");
  if ((q_heads && (!aligned16(q) || q_stride_token % V)) || (k_heads && (!aligned16(k) || k_stride_token % V)))
    return fail(ATTN_ERR_ALIGN, "rope_apply_qk: q / k / strides not 16-byte aligned");
  if (!(base > 0.0)) return fail(ATTN_ERR_ARG, "rope_apply_qk: base must be positive");
  attn::RopeLaunch a{q_heads ? q : k, dtype == ATTN_BF16 ? 0 : 1, tokens, q_heads ? q_heads : k_heads, head_dim,
                     q_heads ? q_stride_token : k_stride_token, positions, base};
  if (q_heads && k_heads) {
    a.x2 = k;
    a.heads2 = k_heads;
    a.stride2 = k_stride_token;
  }
  cudaError_t e = attn::launch_rope(a, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "rope_apply_qk launch");
}

int attn_kv_append_paged(const void* k_new, const void* v_new, const int32_t* positions, const int32_t* slots,
                         int64_t tokens, int num_kv_heads, int head_dim, void* k_cache, void* v_cache,
                         int64_t num_pages, int page_size, void* k_rot_out, double base, void* stream) {
  if (tokens < 0 || num_kv_heads < 0 || head_dim <= 0 || num_pages < 0 || page_size <= 0)
    return fail(ATTN_ERR_ARG, "attn_kv_append_paged: negative size");
  if (head_dim % 2 || (head_dim / 2) % 8 || head_dim > 256)
    return fail(ATTN_ERR_SHAPE, "attn_kv_append_paged: head_dim %d (need head_dim/2 a multiple of 8, <= 256)",
                head_dim);
  if (!(base >= 0.0)) return fail(ATTN_ERR_ARG, "attn_kv_append_paged: base must be >= 0 (0 = no rotation)");
  if (tokens == 0 || num_kv_heads == 0) return ATTN_OK;
  if (!k_new || !v_new || !slots || !k_cache || !v_cache || (base > 0.0 && !positions))
    return fail(ATTN_ERR_ARG, "attn_kv_append_paged: null pointer");
  if (num_pages == 0) return fail(ATTN_ERR_ARG, "attn_kv_append_paged: empty cache");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (k_rot_out && !aligned16(k_rot_out)))
    return fail(ATTN_ERR_ALIGN, "attn_kv_append_paged: tensors must be 16-byte aligned");
  unsigned* err = nullptr;
  int rc = device_error_ptr(&err);
  if (rc) return rc;
  attn::AppendLaunch a{k_new, v_new, positions, slots, tokens, num_kv_heads, head_dim, k_cache, v_cache,
                       num_pages * (int64_t)page_size, k_rot_out, base, err};
  cudaError_t e = attn::launch_kv_append(a, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_kv_append_paged launch");
}

int attn_kv_append_paged_int8(const void* k_new, const void* v_new, const int32_t* positions, const int32_t* slots,
                              int64_t tokens, int num_kv_heads, int head_dim, void* k_cache, void* v_cache,
                              float* k_scale, float* v_scale, int64_t num_pages, int page_size, void* k_rot_out,
                              double base, void* stream) {
  if (tokens < 0 || num_kv_heads < 0 || num_pages < 0 || page_size <= 0)
    return fail(ATTN_ERR_ARG, "attn_kv_append_paged_int8: negative size");
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "attn_kv_append_paged_int8: head_dim %d (need 128)", head_dim);
  if (!(base >= 0.0)) return fail(ATTN_ERR_ARG, "attn_kv_append_paged_int8: base must be >= 0 (0 = no rotation)");
  if (tokens == 0 || num_kv_heads == 0) return ATTN_OK;
  if (!k_new || !v_new || !slots || !k_cache || !v_cache || !k_scale || !v_scale || (base > 0.0 && !positions))
    return fail(ATTN_ERR_ARG, "attn_kv_append_paged_int8: null pointer");
  if (num_pages == 0) return fail(ATTN_ERR_ARG, "attn_kv_append_paged_int8: empty cache");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) ||
      !aligned16(v_scale) || (k_rot_out && !aligned16(k_rot_out)))
    return fail(ATTN_ERR_ALIGN, "attn_kv_append_paged_int8: tensors must be 16-byte aligned");
  unsigned* err = nullptr;
  int rc = device_error_ptr(&err);
  if (rc) return rc;
  attn::AppendLaunch a{k_new, v_new, positions, slots, tokens, num_kv_heads, head_dim, k_cache, v_cache,
                       num_pages * (int64_t)page_size, k_rot_out, base, err, k_scale, v_scale};
  cudaError_t e = attn::launch_kv_append_int8(a, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_kv_append_paged_int8 launch");
}

int quant_fp8_rows(const void* x, int64_t tokens, int heads, int head_dim, void* codes, float* scales,
                   void* stream) {
  if (tokens < 0 || heads < 0) return fail(ATTN_ERR_ARG, "quant_fp8_rows: negative size");
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "quant_fp8_rows: head_dim %d (need 128)", head_dim);
  if (tokens == 0 || heads == 0) return ATTN_OK;
  if (!x || !codes || !scales) return fail(ATTN_ERR_ARG, "quant_fp8_rows: null pointer");
  if (!aligned16(x) || !aligned16(codes)) return fail(ATTN_ERR_ALIGN, "quant_fp8_rows: x / codes not 16-byte aligned");
  cudaError_t e = attn::launch_quant_fp8_rows(x, tokens * heads, codes, scales, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "quant_fp8_rows launch");
}

static int rope_quant_check(const char* name, const void* x, int64_t tokens, int heads, int head_dim,
                            const int32_t* positions, double base, const void* codes, const float* scales) {
  if (tokens < 0 || heads < 0) return fail(ATTN_ERR_ARG, "%s: negative size", name);
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "%s: head_dim %d (need 128)", name, head_dim);
  if (!(base > 0.0)) return fail(ATTN_ERR_ARG, "%s: base must be positive", name);
  if (tokens == 0 || heads == 0) return ATTN_OK;
  if (!x || !positions || !codes || !scales) return fail(ATTN_ERR_ARG, "%s: null pointer", name);
  if (!aligned16(x) || !aligned16(codes)) return fail(ATTN_ERR_ALIGN, "%s: x / codes not 16-byte aligned", name);
  return ATTN_OK;
}

int rope_quant_fp8_rows(const void* x, int64_t tokens, int heads, int head_dim, const int32_t* positions,
                        double base, void* codes, float* scales, void* stream) {
  int rc = rope_quant_check("rope_quant_fp8_rows", x, tokens, heads, head_dim, positions, base, codes, scales);
  if (rc || tokens == 0 || heads == 0) return rc;
  cudaError_t e = attn::launch_rope_quant_fp8(x, tokens, heads, positions, base, codes, scales, nullptr,
                                              (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "rope_quant_fp8_rows launch");
}

int rope_quant_fp8_heads(const void* x, int64_t tokens, int heads, int head_dim, const int32_t* positions,
                         double base, void* codes, float* scales, unsigned* amax_scratch, void* stream) {
  int rc = rope_quant_check("rope_quant_fp8_heads", x, tokens, heads, head_dim, positions, base, codes, scales);
  if (rc || tokens == 0 || heads == 0) return rc;
  if (heads > attn::kMaxQuantHeads)
    return fail(ATTN_ERR_SHAPE, "rope_quant_fp8_heads: %d heads (at most %d)", heads, attn::kMaxQuantHeads);
  if (!amax_scratch) return fail(ATTN_ERR_ARG, "rope_quant_fp8_heads: null amax_scratch");
  cudaError_t e = attn::launch_rope_quant_fp8(x, tokens, heads, positions, base, codes, scales, amax_scratch,
                                              (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "rope_quant_fp8_heads launch");
}

int quant_fp8_heads(const void* x, int64_t tokens, int heads, int head_dim, void* codes, float* scales,
                    unsigned* amax_scratch, int transposed, int64_t t_stride, void* stream) {
  if (tokens < 0 || heads < 0) return fail(ATTN_ERR_ARG, "quant_fp8_heads: negative size");
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "quant_fp8_heads: head_dim %d (need 128)", head_dim);
  if (transposed && (t_stride < tokens || t_stride % 16))
    return fail(ATTN_ERR_ARG, "quant_fp8_heads: t_stride must be >= tokens and a multiple of 16");
  if (tokens == 0 || heads == 0) return ATTN_OK;
  if (!x || !codes || !scales || !amax_scratch) return fail(ATTN_ERR_ARG, "quant_fp8_heads: null pointer");
  if (!aligned16(x) || !aligned16(codes)) return fail(ATTN_ERR_ALIGN, "quant_fp8_heads: x / codes not 16-byte aligned");
  cudaError_t e = attn::launch_quant_fp8_heads(x, tokens, heads, codes, scales, amax_scratch, transposed != 0,
                                               t_stride, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "quant_fp8_heads launch");
}

int attn_prefill_fp8(const void* q, const float* q_scale, const void* k, const float* k_scale, const void* v_t,
                     const float* v_scale, int64_t v_t_stride, void* out, attn_dtype_t out_dtype, float* lse,
                     int batch, const int32_t* cu_q, const int32_t* q_pos, int64_t total_q, int max_seqlen_q,
                     const int32_t* cu_k, const int32_t* k_pos, int64_t total_k, int num_q_heads, int num_kv_heads,
                     int head_dim, int h_lo, int h_hi, float scale, int causal, void* stream) {
  if (batch < 0 || max_seqlen_q < 0 || total_q < 0 || total_k < 0)
    return fail(ATTN_ERR_ARG, "attn_prefill_fp8: negative size");
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return fail(ATTN_ERR_SHAPE, "attn_prefill_fp8: num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads,
                num_kv_heads);
  const int G = num_q_heads / num_kv_heads;
  if (h_lo < 0 || h_hi > num_q_heads || h_lo > h_hi || h_lo % G || h_hi % G)
    return fail(ATTN_ERR_SHAPE, "attn_prefill_fp8: head range [%d, %d) must be whole GQA groups of %d", h_lo, h_hi,
                G);
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "attn_prefill_fp8: head_dim %d (need 128)", head_dim);
  if (out_dtype != ATTN_BF16 && out_dtype != ATTN_FP32) return fail(ATTN_ERR_UNSUPPORTED, "attn_prefill_fp8: out_dtype");
  if (!(scale > 0.f)) return fail(ATTN_ERR_ARG, "attn_prefill_fp8: scale must be positive");
  if (v_t_stride < total_k || v_t_stride % 16)
    return fail(ATTN_ERR_ARG, "attn_prefill_fp8: v_t_stride must be >= total_k and a multiple of 16");
  if (batch == 0 || max_seqlen_q == 0 || h_lo == h_hi || total_q == 0) return ATTN_OK;
  if (!q || !q_scale || !k || !k_scale || !v_t || !v_scale || !out || !cu_q || !q_pos || !cu_k || !k_pos)
    return fail(ATTN_ERR_ARG, "attn_prefill_fp8: null pointer");
  if (total_q > 0x7fffffff || total_k > 0x7fffffff) return fail(ATTN_ERR_ARG, "attn_prefill_fp8: more than 2^31-1 tokens");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v_t) || !aligned16(out))
    return fail(ATTN_ERR_ALIGN, "attn_prefill_fp8: q/k/v_t/out must be 16-byte aligned");
  attn::PrefillLaunch a;
  a.q = q; a.k = k; a.v = v_t; a.out = out;
  a.out_f32 = out_dtype == ATTN_FP32;
  a.lse = lse;
  a.in_f32 = 0;
  a.batch = batch; a.cu_q = cu_q; a.q_pos = q_pos; a.max_seqlen_q = max_seqlen_q;
  a.cu_k = cu_k; a.k_pos = k_pos; a.page_table = nullptr; a.k_lens = nullptr;
  a.max_pages = 0; a.page_size = 0; a.num_pages = 0;
  a.hq = num_q_heads; a.hkv = num_kv_heads; a.d = head_dim; a.h_lo = h_lo; a.h_hi = h_hi;
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.fp8 = 1; a.q_scale = q_scale; a.k_scale = k_scale; a.v_scale = v_scale;
  int rc = device_error_ptr(&a.err);
  if (rc) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = map_tokens_i8(&tq, q, total_q, num_q_heads))) return rc;
  if ((rc = map_tokens_i8(&tk, k, total_k, num_kv_heads))) return rc;
  if ((rc = map_vt_i8(&tv, v_t, v_t_stride, num_kv_heads))) return rc;
  cudaError_t e = attn::launch_prefill_tc(a, tq, tk, tv, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_prefill_fp8 launch");
}

}  // extern "C"

namespace {

int prefill_impl(const void* q, const void* k, const void* v, void* out, attn_dtype_t out_dtype, float* lse,
                 attn_dtype_t dtype, int batch, const int32_t* cu_q, const int32_t* q_pos, int64_t total_q,
                 int max_seqlen_q, const int32_t* cu_k, const int32_t* k_pos, int64_t total_k,
                 const int32_t* page_table, const int32_t* k_lens, int max_pages, int page_size, int64_t num_pages,
                 int num_q_heads, int num_kv_heads, int head_dim, int h_lo, int h_hi, float scale, int causal,
                 const float* q_rope_cs, void* stream) {
  if (batch < 0 || max_seqlen_q < 0 || total_q < 0) return fail(ATTN_ERR_ARG, "attn_prefill: negative size");
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return fail(ATTN_ERR_SHAPE, "attn_prefill: num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads,
                num_kv_heads);
  const int G = num_q_heads / num_kv_heads;
  if (h_lo < 0 || h_hi > num_q_heads || h_lo > h_hi || h_lo % G || h_hi % G)
    return fail(ATTN_ERR_SHAPE, "attn_prefill: head range [%d, %d) must be whole GQA groups of %d", h_lo, h_hi, G);
  if (head_dim <= 0 || head_dim % 32 || head_dim > 256 || (head_dim & (head_dim - 1)))
    return fail(ATTN_ERR_SHAPE, "attn_prefill: head_dim %d (need 32, 64, 128 or 256)", head_dim);
  if (dtype != ATTN_BF16 && dtype != ATTN_FP32) return fail(ATTN_ERR_UNSUPPORTED, "attn_prefill: dtype");
  if (out_dtype != ATTN_BF16 && out_dtype != ATTN_FP32) return fail(ATTN_ERR_UNSUPPORTED, "attn_prefill: out_dtype");
  if (dtype == ATTN_FP32 && out_dtype != ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_prefill: fp32 inputs need an fp32 output");
  if (!(scale > 0.f)) return fail(ATTN_ERR_ARG, "attn_prefill: scale must be positive");
  if (batch == 0 || max_seqlen_q == 0 || h_lo == h_hi || total_q == 0) return ATTN_OK;
  if (!q || !k || !v || !out || !cu_q || !q_pos) return fail(ATTN_ERR_ARG, "attn_prefill: null pointer");
  if (total_q > 0x7fffffff) return fail(ATTN_ERR_ARG, "attn_prefill: total_q exceeds 2^31-1");
  const bool paged = page_table != nullptr;
  if (paged) {
    if (!k_lens || cu_k || k_pos) return fail(ATTN_ERR_ARG, "attn_prefill: paged source takes k_lens, not cu_k/k_pos");
    if (max_pages <= 0 || page_size <= 0 || num_pages <= 0)
      return fail(ATTN_ERR_ARG, "attn_prefill: paged source needs max_pages, page_size, num_pages > 0");
    if ((int64_t)num_kv_heads * num_pages * page_size > 0x7fffffffLL)
      return fail(ATTN_ERR_ARG, "attn_prefill: cache has more than 2^31-1 rows");
  } else {
    if (!cu_k || !k_pos) return fail(ATTN_ERR_ARG, "attn_prefill: contiguous source needs cu_k and k_pos");
    if (total_k < 0 || total_k > 0x7fffffff) return fail(ATTN_ERR_ARG, "attn_prefill: total_k out of range");
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(ATTN_ERR_ALIGN, "attn_prefill: q/k/v/out must be 16-byte aligned");

  attn::PrefillLaunch a;
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.out_f32 = out_dtype == ATTN_FP32;
  a.lse = lse;
  a.in_f32 = dtype == ATTN_FP32;
  a.batch = batch; a.cu_q = cu_q; a.q_pos = q_pos; a.max_seqlen_q = max_seqlen_q;
  a.cu_k = cu_k; a.k_pos = k_pos; a.page_table = page_table; a.k_lens = k_lens;
  a.max_pages = max_pages; a.page_size = page_size; a.num_pages = num_pages;
  a.hq = num_q_heads; a.hkv = num_kv_heads; a.d = head_dim; a.h_lo = h_lo; a.h_hi = h_hi;
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.q_rope_cs = q_rope_cs;
  int rc = device_error_ptr(&a.err);
  if (rc) return rc;

  const bool tc = dtype == ATTN_BF16 && head_dim == 128 && (!paged || page_size == 64);
  if (q_rope_cs && !tc)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_prefill_rope_q: fused RoPE needs bf16, head_dim 128 (tensor-core path)");
  cudaError_t e;
  if (tc) {
    CUtensorMap tq, tk, tv;
    if ((rc = map_tokens(&tq, q, total_q, num_q_heads))) return rc;
    if (paged) {
      if ((rc = map_pages(&tk, k, num_kv_heads, num_pages))) return rc;
      if ((rc = map_pages(&tv, v, num_kv_heads, num_pages))) return rc;
    } else {
      if ((rc = map_tokens(&tk, k, total_k, num_kv_heads))) return rc;
      if ((rc = map_tokens(&tv, v, total_k, num_kv_heads))) return rc;
    }
    e = attn::launch_prefill_tc(a, tq, tk, tv, (cudaStream_t)stream);
  } else {
    e = attn::launch_prefill_simt(a, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_prefill launch");
}

}  // namespace

extern "C" {

int attn_prefill(const void* q, const void* k, const void* v, void* out, attn_dtype_t out_dtype, float* lse,
                 attn_dtype_t dtype, int batch, const int32_t* cu_q, const int32_t* q_pos, int64_t total_q,
                 int max_seqlen_q, const int32_t* cu_k, const int32_t* k_pos, int64_t total_k,
                 const int32_t* page_table, const int32_t* k_lens, int max_pages, int page_size, int64_t num_pages,
                 int num_q_heads, int num_kv_heads, int head_dim, int h_lo, int h_hi, float scale, int causal,
                 void* stream) {
  return prefill_impl(q, k, v, out, out_dtype, lse, dtype, batch, cu_q, q_pos, total_q, max_seqlen_q, cu_k, k_pos,
                      total_k, page_table, k_lens, max_pages, page_size, num_pages, num_q_heads, num_kv_heads,
                      head_dim, h_lo, h_hi, scale, causal, nullptr, stream);
}

int attn_prefill_rope_q(const void* q, const void* k, const void* v, void* out, attn_dtype_t out_dtype, float* lse,
                        attn_dtype_t dtype, int batch, const int32_t* cu_q, const int32_t* q_pos, int64_t total_q,
                        int max_seqlen_q, const int32_t* cu_k, const int32_t* k_pos, int64_t total_k,
                        const int32_t* page_table, const int32_t* k_lens, int max_pages, int page_size,
                        int64_t num_pages, int num_q_heads, int num_kv_heads, int head_dim, int h_lo, int h_hi,
                        float scale, int causal, const float* q_rope_cs, void* stream) {
  if (!q_rope_cs) return fail(ATTN_ERR_ARG, "attn_prefill_rope_q: null RoPE table");
  if (!aligned16(q_rope_cs)) return fail(ATTN_ERR_ALIGN, "attn_prefill_rope_q: RoPE table must be 16-byte aligned");
  return prefill_impl(q, k, v, out, out_dtype, lse, dtype, batch, cu_q, q_pos, total_q, max_seqlen_q, cu_k, k_pos,
                      total_k, page_table, k_lens, max_pages, page_size, num_pages, num_q_heads, num_kv_heads,
                      head_dim, h_lo, h_hi, scale, causal, q_rope_cs, stream);
}

int rope_table(const int32_t* positions, int64_t tokens, int head_dim, double base, float* cs_out, void* stream) {
  if (tokens < 0 || head_dim <= 0) return fail(ATTN_ERR_ARG, "rope_table: negative size");
  if (head_dim % 2 || head_dim > 256) return fail(ATTN_ERR_SHAPE, "rope_table: head_dim %d (even, <= 256)", head_dim);
  if (!(base > 0.0)) return fail(ATTN_ERR_ARG, "rope_table: base must be positive");
  if (tokens == 0) return ATTN_OK;
  if (!positions || !cs_out) return fail(ATTN_ERR_ARG, "rope_table: null pointer");
  if (!aligned16(cs_out)) return fail(ATTN_ERR_ALIGN, "rope_table: cs_out must be 16-byte aligned");
  cudaError_t e = attn::launch_rope_table(cs_out, tokens, head_dim, positions, base, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "rope_table launch");
}

int attn_lse_merge(const float* part_out, const float* part_lse, int n_parts, int64_t rows, int heads, int head_dim,
                   int64_t o_stride_part, int64_t o_stride_row, int64_t o_stride_head, int64_t l_stride_part,
                   int64_t l_stride_row, int64_t l_stride_head, void* out, attn_dtype_t out_dtype, float* lse_out,
                   void* stream) {
  if (rows < 0 || heads < 0 || head_dim <= 0) return fail(ATTN_ERR_ARG, "attn_lse_merge: negative size");
  if (n_parts < 1 || n_parts > 1024) return fail(ATTN_ERR_ARG, "attn_lse_merge: n_parts %d not in [1, 1024]", n_parts);
  if (out_dtype != ATTN_BF16 && out_dtype != ATTN_FP32) return fail(ATTN_ERR_UNSUPPORTED, "attn_lse_merge: out_dtype");
  if (rows == 0 || heads == 0) return ATTN_OK;
  if (!part_out || !part_lse || !out) return fail(ATTN_ERR_ARG, "attn_lse_merge: null pointer");
  attn::MergeLaunch a{part_out, part_lse, n_parts, rows, heads, head_dim, o_stride_part, o_stride_row,
                      o_stride_head, l_stride_part, l_stride_row, l_stride_head, out, out_dtype == ATTN_FP32 ? 1 : 0,
                      lse_out};
  cudaError_t e = attn::launch_lse_merge(a, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_lse_merge launch");
}

int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* page_table,
                      const int32_t* ctx_lens, int batch, int max_pages, int page_size, int64_t num_pages,
                      int num_q_heads, int num_kv_heads, int head_dim, int num_splits, float scale, float* part_out,
                      float* part_lse, void* out, attn_dtype_t out_dtype, float* lse, void* stream) {
  if (batch < 0) return fail(ATTN_ERR_ARG, "attn_decode_paged: negative batch");
  if (num_kv_heads <= 0 || num_q_heads != 8 * num_kv_heads)
    return fail(ATTN_ERR_SHAPE, "attn_decode_paged: needs 8 query heads per KV head (got %d/%d)", num_q_heads,
                num_kv_heads);
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "attn_decode_paged: head_dim %d (need 128)", head_dim);
  if (page_size != 64) return fail(ATTN_ERR_SHAPE, "attn_decode_paged: page_size %d (need 64)", page_size);
  if (num_splits < 1 || num_splits > 256) return fail(ATTN_ERR_ARG, "attn_decode_paged: num_splits %d", num_splits);
  if (out && out_dtype != ATTN_BF16 && out_dtype != ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_paged: out_dtype");
  if (!(scale > 0.f)) return fail(ATTN_ERR_ARG, "attn_decode_paged: scale must be positive");
  if (batch == 0) return ATTN_OK;
  if (!q || !k_cache || !v_cache || !page_table || !ctx_lens || !part_out || !part_lse)
    return fail(ATTN_ERR_ARG, "attn_decode_paged: null pointer");
  if (max_pages <= 0 || num_pages <= 0) return fail(ATTN_ERR_ARG, "attn_decode_paged: max_pages/num_pages");
  if ((int64_t)num_kv_heads * num_pages * page_size > 0x7fffffffLL)
    return fail(ATTN_ERR_ARG, "attn_decode_paged: cache has more than 2^31-1 rows");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(part_out))
    return fail(ATTN_ERR_ALIGN, "attn_decode_paged: q / caches / part_out must be 16-byte aligned");
  unsigned* err = nullptr;
  int rc = device_error_ptr(&err);
  if (rc) return rc;
  CUtensorMap tk, tv;
  if ((rc = map_pages(&tk, k_cache, num_kv_heads, num_pages))) return rc;
  if ((rc = map_pages(&tv, v_cache, num_kv_heads, num_pages))) return rc;
  attn::DecodeLaunch a{q, page_table, ctx_lens, batch, max_pages, num_pages, num_q_heads, num_kv_heads, num_splits,
                       scale, part_out, part_lse, err};
  cudaError_t e = attn::launch_decode_split(a, tk, tv, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_paged launch");
  if (!out) return ATTN_OK;
  const int64_t S = num_splits, d = head_dim;
  attn::MergeLaunch m{part_out, part_lse, num_splits, batch, num_q_heads, head_dim, d, num_q_heads * S * d, S * d,
                      1, num_q_heads * S, S, out, out_dtype == ATTN_FP32 ? 1 : 0, lse};
  e = attn::launch_lse_merge(m, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_decode_paged merge launch");
}

int attn_decode_paged_int8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, const int32_t* page_table, const int32_t* ctx_lens, int batch,
                           int max_pages, int page_size, int64_t num_pages, int num_q_heads, int num_kv_heads,
                           int head_dim, int num_splits, float scale, float* part_out, float* part_lse, void* out,
                           attn_dtype_t out_dtype, float* lse, void* stream) {
  if (batch < 0) return fail(ATTN_ERR_ARG, "attn_decode_paged_int8: negative batch");
  if (num_kv_heads <= 0 || num_q_heads != 8 * num_kv_heads)
    return fail(ATTN_ERR_SHAPE, "attn_decode_paged_int8: needs 8 query heads per KV head (got %d/%d)", num_q_heads,
                num_kv_heads);
  if (head_dim != 128) return fail(ATTN_ERR_SHAPE, "attn_decode_paged_int8: head_dim %d (need 128)", head_dim);
  if (page_size != 64) return fail(ATTN_ERR_SHAPE, "attn_decode_paged_int8: page_size %d (need 64)", page_size);
  if (num_splits < 1 || num_splits > 256)
    return fail(ATTN_ERR_ARG, "attn_decode_paged_int8: num_splits %d", num_splits);
  if (out && out_dtype != ATTN_BF16 && out_dtype != ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_paged_int8: out_dtype");
  if (!(scale > 0.f)) return fail(ATTN_ERR_ARG, "attn_decode_paged_int8: scale must be positive");
  if (batch == 0) return ATTN_OK;
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !page_table || !ctx_lens || !part_out || !part_lse)
    return fail(ATTN_ERR_ARG, "attn_decode_paged_int8: null pointer");
  if (max_pages <= 0 || num_pages <= 0) return fail(ATTN_ERR_ARG, "attn_decode_paged_int8: max_pages/num_pages");
  if ((int64_t)num_kv_heads * num_pages * page_size > 0x7fffffffLL)
    return fail(ATTN_ERR_ARG, "attn_decode_paged_int8: cache has more than 2^31-1 rows");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) || !aligned16(v_scale) ||
      !aligned16(part_out))
    return fail(ATTN_ERR_ALIGN, "attn_decode_paged_int8: q / caches / scales / part_out must be 16-byte aligned");
  unsigned* err = nullptr;
  int rc = device_error_ptr(&err);
  if (rc) return rc;
  CUtensorMap tk, tv;
  if ((rc = map_pages_i8(&tk, k_cache, num_kv_heads, num_pages))) return rc;
  if ((rc = map_pages_i8(&tv, v_cache, num_kv_heads, num_pages))) return rc;
  attn::DecodeLaunch a{q, page_table, ctx_lens, batch, max_pages, num_pages, num_q_heads, num_kv_heads, num_splits,
                       scale, part_out, part_lse, err};
  cudaError_t e = attn::launch_decode_split_int8(a, k_scale, v_scale, tk, tv, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_paged_int8 launch");
  if (!out) return ATTN_OK;
  const int64_t S = num_splits, d = head_dim;
  attn::MergeLaunch m{part_out, part_lse, num_splits, batch, num_q_heads, head_dim, d, num_q_heads * S * d, S * d,
                      1, num_q_heads * S, S, out, out_dtype == ATTN_FP32 ? 1 : 0, lse};
  e = attn::launch_lse_merge(m, (cudaStream_t)stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_decode_paged_int8 merge launch");
}

}  // extern "C"
