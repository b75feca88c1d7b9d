// FP8 (e4m3) quantisation of Q, K and V for the FP8 prefill (Flash Attention
// page, section 18.5: an FP8 mode with block quantisation).  A group of values
// shares one fp32 scale = max|x| / 448 (the largest e4m3 value), and each value
// is stored as e4m3(x / scale), rounded to nearest even with x / scale in fp32
// (correctly rounded; div_rn_recip computes it in three instructions); an
// all-zero group gets scale 0 and codes 0.
//
//   rows:  a group is one (token, head) row of head_dim values (the queries);
//   heads: a group is one head over all tokens (keys, values); the codes keep
//          the [tokens][heads][d] layout, or are written transposed as
//          [heads][d][t_stride] (values: the P V contraction reads V^T rows
//          with the keys contiguous).
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace q8 {

// Codes of 8 values x / s: the three-instruction division for normal scales,
// the full one below kFastDivMinScale; 0 for a zero scale.
__device__ __forceinline__ uint2 e4m3x8(const float (&v)[4], const float (&u)[4], float s) {
  uint2 out = make_uint2(0u, 0u);
  if (s >= kFastDivMinScale) {
    const float r = __frcp_rn(s);
    out.x = e4m3x4_div<true>(v[0], v[1], v[2], v[3], s, r);
    out.y = e4m3x4_div<true>(u[0], u[1], u[2], u[3], s, r);
  } else if (s != 0.0f) {
    out.x = e4m3x4_div<false>(v[0], v[1], v[2], v[3], s, 0.f);
    out.y = e4m3x4_div<false>(u[0], u[1], u[2], u[3], s, 0.f);
  }
  return out;
}

__device__ __forceinline__ void unpack_bf16x4(uint2 w, float (&x)[4]) {
  x[0] = __uint_as_float(w.x << 16);
  x[1] = __uint_as_float(w.x & 0xffff0000u);
  x[2] = __uint_as_float(w.y << 16);
  x[3] = __uint_as_float(w.y & 0xffff0000u);
}

// One warp per (token, head) row of 128 values, 4 per lane.
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                         uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float v[4];
  unpack_bf16x4(__ldg(reinterpret_cast<const uint2*>(x + r * 128) + lane), v);
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax / 448.0f;
  uint32_t packed = 0;
  if (s >= kFastDivMinScale)
    packed = e4m3x4_div<true>(v[0], v[1], v[2], v[3], s, __frcp_rn(s));
  else if (s != 0.0f)
    packed = e4m3x4_div<false>(v[0], v[1], v[2], v[3], s, 0.f);
  reinterpret_cast<uint32_t*>(codes + r * 128)[lane] = packed;
  if (lane == 0) scales[r] = s;
}

// Per-head max |x|: block column y = the head; each block reduces its share of
// the head's tokens (8 values per thread per step) and folds the result, as the
// bits of a non-negative float (which order like the integers), into
// amax_bits[head] with one atomic.
__global__ void __launch_bounds__(256) head_amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens, int heads,
                                                        unsigned* __restrict__ amax_bits) {
  __shared__ float wmax[8];
  const int h = blockIdx.y;
  float m = 0.f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < tokens * 16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i >> 4;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + (t * heads + h) * 128) + (i & 15));
    float v[4];
    unpack_bf16x4(make_uint2(w.x, w.y), v);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    unpack_bf16x4(make_uint2(w.z, w.w), v);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mm = fmaxf(mm, wmax[w]);
    atomicMax(amax_bits + h, __float_as_uint(mm));
  }
}

// Codes with the head's scale max|x| / 448: 8 values per thread, row layout.
__global__ void __launch_bounds__(256) quant_heads_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens,
                                                          int heads, const unsigned* __restrict__ amax_bits,
                                                          uint8_t* __restrict__ codes) {
  const int64_t chunks = tokens * heads * 16;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rw = c >> 4;  // (token, head) row; 32-bit division while it fits
    const int h = rw < 0x7fffffff ? (int)((uint32_t)rw % (uint32_t)heads) : (int)(rw % heads);
    const float s = __uint_as_float(__ldg(amax_bits + h)) / 448.0f;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(x) + c);
    float v[4], u[4];
    unpack_bf16x4(make_uint2(w.x, w.y), v);
    unpack_bf16x4(make_uint2(w.z, w.w), u);
    reinterpret_cast<uint2*>(codes)[c] = e4m3x8(v, u, s);
  }
}

// Transposed codes [heads][128][t_stride]: a block takes 32 tokens x one head,
// reads the 32 rows coalesced, and writes 128 rows of 32 contiguous bytes.  The
// grid spans t_stride, so columns [tokens, t_stride) are written as zero codes
// (the prefill's last K/V tile reads them, with weight 0).
__global__ void __launch_bounds__(256) quant_heads_t_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens,
                                                            int heads, const unsigned* __restrict__ amax_bits,
                                                            uint8_t* __restrict__ codes_t, int64_t t_stride,
                                                            float* __restrict__ scales) {
  __shared__ uint8_t tile[128][33];  // [dim][token], padded
  const int64_t t0 = (int64_t)blockIdx.x * 32;
  const int h = blockIdx.y;
  const float s = __uint_as_float(__ldg(amax_bits + h)) / 448.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) scales[h] = s;
  // read: 32 tokens x 128 dims, 16 threads per token row (8 values each)
  for (int i = threadIdx.x; i < 32 * 16; i += blockDim.x) {
    const int tt = i >> 4, c = i & 15;
    const int64_t t = t0 + tt;
    uint2 out = make_uint2(0u, 0u);
    if (t < tokens && s != 0.0f) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + (t * heads + h) * 128) + c);
      float v[4], u[4];
      unpack_bf16x4(make_uint2(w.x, w.y), v);
      unpack_bf16x4(make_uint2(w.z, w.w), u);
      out = e4m3x8(v, u, s);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) tile[c * 8 + e][tt] = (uint8_t)((e < 4 ? out.x : out.y) >> (8 * (e & 3)));
  }
  __syncthreads();
  // write: 128 dim rows x 32 tokens (bytes), 4 bytes per thread
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int dd = i >> 3, q = i & 7;
    const int64_t t = t0 + q * 4;
    if (t >= t_stride) continue;  // t_stride is a multiple of 16: the word fits whole
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) w |= (uint32_t)tile[dd][q * 4 + e] << (8 * e);
    *reinterpret_cast<uint32_t*>(codes_t + ((int64_t)h * 128 + dd) * t_stride + t) = w;
  }
}

__global__ void head_scales_kernel(const unsigned* __restrict__ amax_bits, int heads, float* __restrict__ scales) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < heads) scales[h] = __uint_as_float(amax_bits[h]) / 448.0f;
}

}  // namespace q8

cudaError_t launch_quant_fp8_rows(const void* x, int64_t rows, void* codes, float* scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows * 32 + 255) / 256;
  q8::quant_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>((const __nv_bfloat16*)x, rows, (uint8_t*)codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_fp8_heads(const void* x, int64_t tokens, int heads, void* codes, float* scales,
                                   unsigned* amax_scratch, bool transposed, int64_t t_stride, cudaStream_t s) {
  if (tokens == 0 || heads == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(amax_scratch, 0, sizeof(unsigned) * heads, s);
  if (e != cudaSuccess) return e;
  const int64_t chunks = tokens * heads * 16;
  const unsigned blocks = (unsigned)min((chunks + 255) / 256, (int64_t)4096);
  dim3 agrid((unsigned)min((tokens * 16 + 255) / 256, (int64_t)512), (unsigned)heads);
  q8::head_amax_kernel<<<agrid, 256, 0, s>>>((const __nv_bfloat16*)x, tokens, heads, amax_scratch);
  if (transposed) {
    dim3 grid((unsigned)((t_stride + 31) / 32), (unsigned)heads);
    q8::quant_heads_t_kernel<<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, tokens, heads, amax_scratch,
                                                  (uint8_t*)codes, t_stride, scales);
  } else {
    q8::quant_heads_kernel<<<blocks, 256, 0, s>>>((const __nv_bfloat16*)x, tokens, heads, amax_scratch,
                                                  (uint8_t*)codes);
    q8::head_scales_kernel<<<(heads + 127) / 128, 128, 0, s>>>(amax_scratch, heads, scales);
  }
  return cudaGetLastError();
}

}  // namespace attn
