// attn_decode_paged_noalloc: split-KV paged decode whose split partials live in
// a scratch array that the library holds statically, so the call itself
// allocates no device memory.
//
// Some callers cannot call cudaMalloc for a workspace: a serving engine that
// hands all free HBM to its KV-cache pool at start-up (a later cudaMalloc fails
// or carves into the pool), a plugin running inside a host framework whose
// caching allocator owns the device memory, or a latency-critical path where
// cudaMalloc/cudaFree would synchronise the device.  They pass inputs and
// outputs only; the partial O / LSE of every split go to g_decode_scratch.
//
// Limits and sharing:
//  - batch * num_q_heads * num_splits must not exceed kMaxPartRows (32768),
//    i.e. 32 requests x 64 query heads x 16 splits at head_dim 128; the array
//    takes 32768 * 129 floats (16.1 MiB) on every GPU that loads the library,
//    held until the process exits.  Larger calls are rejected.
//  - Every call on a device shares the one array, which keeps the previous
//    call's contents.  Nothing in it has to start at zero: the split kernel
//    writes every partial it covers (an empty split writes O = 0, LSE = -inf)
//    before the merge reads them.  Calls whose work overlaps on the GPU (two
//    streams, or two host threads) race on the array; serialise them.
//  - The first call on each device looks up the array's device address with
//    cudaGetSymbolAddress while that device is current and caches it; make that
//    first call before any stream capture.  The address belongs to the context
//    current at that first call (the device's primary context under the
//    runtime API); cudaDeviceReset() or another context on the same ordinal
//    would leave the cached address stale, so neither is supported afterwards.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn_gb300.h"
#include "kernels.h"

namespace {

constexpr long long kMaxPartRows = 32768;  // batch * num_q_heads * num_splits
constexpr long long kHeadDim = 128;        // the decode kernel's head_dim
constexpr long long kScratchFloats = kMaxPartRows * (kHeadDim + 1);

// Partial outputs [rows][128] followed by partial LSEs [rows].  In host code
// this name is only a stand-in for the device array; its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

std::mutex g_mu;
float* g_scratch[64] = {};

int scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn::set_last_error(ATTN_ERR_CUDA, "attn_decode_paged_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= 64) return attn::set_last_error(ATTN_ERR_CUDA, "attn_decode_paged_noalloc: device index >= 64");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return attn::set_last_error(ATTN_ERR_CUDA, "attn_decode_paged_noalloc: cudaGetSymbolAddress(scratch) failed");
    g_scratch[dev] = static_cast<float*>(p);
  }
  *out = g_scratch[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* page_table, const int32_t* ctx_lens, int batch,
                                         int max_pages, int page_size, int64_t num_pages, int num_q_heads,
                                         int num_kv_heads, int head_dim, int num_splits, float scale, void* out,
                                         attn_dtype_t out_dtype, float* lse, void* stream) {
  if (!out) return attn::set_last_error(ATTN_ERR_ARG, "attn_decode_paged_noalloc: out must not be NULL");
  if (batch < 0 || num_q_heads <= 0 || num_splits < 1)
    return attn::set_last_error(ATTN_ERR_ARG, "attn_decode_paged_noalloc: negative or empty size");
  if (head_dim != kHeadDim)
    return attn::set_last_error(ATTN_ERR_SHAPE, "attn_decode_paged_noalloc: head_dim must be 128");
  if ((long long)batch * num_q_heads * num_splits > kMaxPartRows)
    return attn::set_last_error(ATTN_ERR_ARG,
                                "attn_decode_paged_noalloc: batch * num_q_heads * num_splits exceeds the static "
                                "scratch (32768 partial rows, 16.1 MiB)");
  if (batch == 0) return ATTN_OK;
  float* s = nullptr;
  int rc = scratch_for_current_device(&s);
  if (rc) return rc;
  float* part_out = s;
  float* part_lse = s + kMaxPartRows * kHeadDim;
  return attn_decode_paged(q, k_cache, v_cache, page_table, ctx_lens, batch, max_pages, page_size, num_pages,
                           num_q_heads, num_kv_heads, head_dim, num_splits, scale, part_out, part_lse, out,
                           out_dtype, lse, stream);
}
