// RoPE at absolute positions, in place (Ulysses page, sections 3.2 and 5.3).
//
// One thread owns one token and one vector of V consecutive pair indices i
// (16 bytes of the first half of the head plus the matching 16 bytes of the
// second half) and walks every head of that token, so each angle is computed
// once per token and reused across heads.  A warp covers whole 128-byte
// segments of a few tokens per head: the access is a coalesced HBM stream.
//
// Angle accuracy: a = pos * base^(-2i/d) reaches ~1.3e5 rad at 128K positions,
// where an fp32 product alone would be off by ~1e-2 rad.  The product and its
// reduction to [-pi, pi] are done in fp64 (a few fp64 operations per token and
// pair, shared by all heads); the rotation itself is fp32.
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

template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(T* __restrict__ x, int64_t tokens, int heads, int d,
                                                   int64_t stride_tok, const int32_t* __restrict__ pos,
                                                   const InvFreq f) {
  constexpr int V = Vec<T>::N;
  const int half = d / 2;
  const int chunks = half / V;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t t = gid / chunks;
  const int c = (int)(gid % chunks);
  if (t >= tokens) return;
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
  const double p = (double)__ldg(pos + t);
  float cs[V], sn[V];
#pragma unroll
  for (int e = 0; e < V; ++e) {
    const double a = p * f.v[c * V + e];
    const double r = fma(-rint(a * kInvTwoPi), kTwoPi, a);
    sincosf((float)r, &sn[e], &cs[e]);
  }
  T* row = x + t * stride_tok + c * V;
  for (int h = 0; h < heads; ++h) {
    T* p1 = row + (int64_t)h * d;
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
      const float x1 = to_f(a1[e]), x2 = to_f(a2[e]);
      from_f(x1 * cs[e] - x2 * sn[e], b1[e]);
      from_f(x2 * cs[e] + x1 * sn[e], b2[e]);
    }
    *reinterpret_cast<uint4*>(p1) = w1;
    *reinterpret_cast<uint4*>(p2) = w2;
  }
}

cudaError_t launch_rope(const RopeLaunch& a, cudaStream_t s) {
  InvFreq f;
  const int half = a.head_dim / 2;
  for (int i = 0; i < half; ++i) f.v[i] = pow(a.base, -2.0 * (double)i / (double)a.head_dim);
  const int V = a.dtype == 0 ? 8 : 4;
  const int64_t threads = a.tokens * (half / V);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  if (a.dtype == 0)
    rope_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
        (__nv_bfloat16*)a.x, a.tokens, a.heads, a.head_dim, a.stride_token, a.positions, f);
  else
    rope_kernel<float><<<(unsigned)blocks, 256, 0, s>>>((float*)a.x, a.tokens, a.heads, a.head_dim,
                                                        a.stride_token, a.positions, f);
  return cudaGetLastError();
}

}  // namespace attn
