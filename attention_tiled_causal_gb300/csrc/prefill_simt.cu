// CUDA-core prefill: exact attention with the online softmax of the Flash
// Attention page, section 18.3, one warp per (query row, query head).
//
// This kernel serves the shapes the tensor-core kernel does not take (fp32
// inputs, head_dim other than 128, page sizes other than 64) and small
// problems.  Per block of 32 keys each lane scores one key against the query
// row held in shared memory; the warp then updates the running max m and
// denominator l, rescales its output slice by exp(m_old - m_new) and adds the
// 32 weighted value rows, one coalesced row read per key.  Normalisation by l
// is deferred to the end (section 18.4).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {

__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ld_f(const float* p) { return *p; }

template <typename T, typename OT, int D, bool PAGED>
__global__ void __launch_bounds__(128) prefill_simt_kernel(const PrefillLaunch a) {
  constexpr int E = D / 32;
  __shared__ float qs[4][D];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.z;
  const int h = a.h_lo + blockIdx.y;
  const int q_beg = a.cu_q[b];
  const int Sq = a.cu_q[b + 1] - q_beg;
  const int r = blockIdx.x * 4 + w;
  if (r >= Sq) return;
  const int g = h / (a.hq / a.hkv);
  int k_beg = 0, Sk;
  if (PAGED)
    Sk = a.k_lens[b];
  else {
    k_beg = a.cu_k[b];
    Sk = a.cu_k[b + 1] - k_beg;
  }
  const int qp = a.q_pos[q_beg + r];
  const T* q = (const T*)a.q + ((int64_t)(q_beg + r) * a.hq + h) * D;
  for (int i = lane; i < D; i += 32) qs[w][i] = ld_f(q + i);
  __syncwarp();

  const T* K = (const T*)a.k;
  const T* V = (const T*)a.v;
  auto row_ptr = [&](const T* base, int j, bool& ok) -> const T* {
    if (PAGED) {
      const int lp = j / a.page_size;
      const int pid = lp < a.max_pages ? a.page_table[(int64_t)b * a.max_pages + lp] : -1;
      if (pid < 0 || pid >= a.num_pages) {
        ok = false;
        return base;
      }
      return base + (((int64_t)g * a.num_pages + pid) * a.page_size + (j % a.page_size)) * D;
    }
    return base + ((int64_t)(k_beg + j) * a.hkv + g) * D;
  };

  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int kb = 0; kb < Sk; kb += 32) {
    if (a.causal) {  // positions are non-decreasing: nothing visible beyond this point
      const int first = PAGED ? kb : a.k_pos[k_beg + kb];
      if (first > qp) break;
    }
    const int j = kb + lane;
    bool vis = j < Sk;
    if (vis && a.causal) vis = (PAGED ? j : a.k_pos[k_beg + j]) <= qp;
    float s = -INFINITY;
    if (vis) {
      bool ok = true;
      const T* kr = row_ptr(K, j, ok);
      if (ok) {
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < D; ++i) acc = fmaf(qs[w][i], ld_f(kr + i), acc);
        s = acc * a.scale;
      } else {
        record_error(a.err, DEV_BAD_PAGE);
        vis = false;
      }
    }
    float mb = s;
#pragma unroll
    for (int off = 16; off; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    if (mb == -INFINITY) continue;
    const float m_new = fmaxf(m, mb);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float p = vis ? expf(s - m_new) : 0.f;
    float ps = p;
#pragma unroll
    for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= alpha;
    const int nvalid = min(32, Sk - kb);
    for (int jj = 0; jj < nvalid; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      if (pj == 0.f) continue;  // uniform across the warp
      bool ok = true;
      const T* vr = row_ptr(V, kb + jj, ok);
      if (!ok) continue;
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf(pj, ld_f(vr + lane + 32 * e), o[e]);
    }
    m = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  OT* out = (OT*)a.out + ((int64_t)(q_beg + r) * a.hq + h) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if constexpr (sizeof(OT) == 4)
      out[lane + 32 * e] = o[e] * inv;
    else
      out[lane + 32 * e] = __float2bfloat16_rn(o[e] * inv);
  }
  if (a.lse && lane == 0) a.lse[(int64_t)(q_beg + r) * a.hq + h] = l > 0.f ? m + logf(l) : -INFINITY;
}

template <typename T, typename OT, int D>
static cudaError_t launch_d(const PrefillLaunch& a, cudaStream_t s) {
  dim3 grid((a.max_seqlen_q + 3) / 4, a.h_hi - a.h_lo, a.batch);
  if (a.page_table)
    prefill_simt_kernel<T, OT, D, true><<<grid, 128, 0, s>>>(a);
  else
    prefill_simt_kernel<T, OT, D, false><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, typename OT>
static cudaError_t launch_t(const PrefillLaunch& a, cudaStream_t s) {
  switch (a.d) {
    case 32: return launch_d<T, OT, 32>(a, s);
    case 64: return launch_d<T, OT, 64>(a, s);
    case 128: return launch_d<T, OT, 128>(a, s);
    case 256: return launch_d<T, OT, 256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill_simt(const PrefillLaunch& a, cudaStream_t s) {
  if (a.max_seqlen_q == 0 || a.batch == 0 || a.h_hi == a.h_lo) return cudaSuccess;
  if (a.in_f32) return launch_t<float, float>(a, s);
  if (a.out_f32) return launch_t<__nv_bfloat16, float>(a, s);
  return launch_t<__nv_bfloat16, __nv_bfloat16>(a, s);
}

}  // namespace attn
