// RoPE at absolute positions, in place (Ulysses page, sections 3.2 and 5.3).
//
// Each block takes kTok consecutive tokens: it first computes their cos/sin
// tables (d/2 angles per token, once) into shared memory, then streams every
// head of those tokens.  A thread rotates one 16-byte vector of the first half
// of a head together with the matching vector of the second half; consecutive
// threads take consecutive vectors, so a warp covers whole 128-byte segments.
#include "common.cuh"
#include "kernels.h"

namespace attn {

struct InvFreq {
  double v[128];  // base^(-2i/d), i < d/2 <= 128
};

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
};

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ void from_f(float x, __nv_bfloat16& y) { y = __float2bfloat16_rn(x); }
__device__ __forceinline__ void from_f(float x, float& y) { y = x; }

constexpr int kTok = 4;  // tokens per block

template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(T* __restrict__ x, int64_t tokens, int heads, int d,
                                                   int64_t stride_tok, const int32_t* __restrict__ pos,
                                                   const InvFreq f) {
  constexpr int V = Vec<T>::N;
  __shared__ float cs_s[kTok][128], sn_s[kTok][128];
  const int half = d / 2;
  const int chunks = half / V;
  const int64_t t0 = (int64_t)blockIdx.x * kTok;
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
  for (int i = threadIdx.x; i < kTok * half; i += blockDim.x) {
    const int tt = i / half, ii = i % half;
    const int64_t t = t0 + tt;
    if (t < tokens) {
      const double a = (double)__ldg(pos + t) * f.v[ii];
      const double r = fma(-rint(a * kInvTwoPi), kTwoPi, a);
      sincosf((float)r, &sn_s[tt][ii], &cs_s[tt][ii]);
    }
  }
  __syncthreads();
  const int items = kTok * heads * chunks;
#pragma unroll 4
  for (int w = threadIdx.x; w < items; w += blockDim.x) {
    const int c = w % chunks;
    const int h = (w / chunks) % heads;
    const int tt = w / (chunks * heads);
    const int64_t t = t0 + tt;
    if (t >= tokens) continue;
    T* p1 = x + t * stride_tok + (int64_t)h * d + c * V;
    T* p2 = p1 + half;
    uint4 u1 = *reinterpret_cast<const uint4*>(p1);
    uint4 u2 = *reinterpret_cast<const uint4*>(p2);
    const T* a1 = reinterpret_cast<const T*>(&u1);
    const T* a2 = reinterpret_cast<const T*>(&u2);
    uint4 w1, w2;
    T* b1 = reinterpret_cast<T*>(&w1);
    T* b2 = reinterpret_cast<T*>(&w2);
#pragma unroll
    for (int e = 0; e < V; ++e) {
      const float cs = cs_s[tt][c * V + e], sn = sn_s[tt][c * V + e];
      const float x1 = to_f(a1[e]), x2 = to_f(a2[e]);
      from_f(x1 * cs - x2 * sn, b1[e]);
      from_f(x2 * cs + x1 * sn, b2[e]);
    }
    *reinterpret_cast<uint4*>(p1) = w1;
    *reinterpret_cast<uint4*>(p2) = w2;
  }
}

cudaError_t launch_rope(const RopeLaunch& a, cudaStream_t s) {
  InvFreq f;
  const int half = a.head_dim / 2;
  for (int i = 0; i < half; ++i) f.v[i] = pow(a.base, -2.0 * (double)i / (double)a.head_dim);
  if (a.tokens == 0) return cudaSuccess;
  const int64_t blocks = (a.tokens + kTok - 1) / kTok;
  if (a.dtype == 0)
    rope_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
        (__nv_bfloat16*)a.x, a.tokens, a.heads, a.head_dim, a.stride_token, a.positions, f);
  else
    rope_kernel<float><<<(unsigned)blocks, 256, 0, s>>>((float*)a.x, a.tokens, a.heads, a.head_dim,
                                                        a.stride_token, a.positions, f);
  return cudaGetLastError();
}

}  // namespace attn
