// Log-sum-exp merge of partial attention results over disjoint key sets:
//   LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
// (Flash Attention page, section 18.3: the exp(m_old - m_new) rescale that
// combines running softmax states).  Parts with LSE_s = -inf weigh 0.
//
// One warp per (row, head).  The part LSEs are read once per lane-strided
// slice and reduced with shuffles; the weighted sum streams the part outputs
// with lanes spread over head_dim, so every part row is one coalesced read.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {

template <bool OUT_F32>
__global__ void __launch_bounds__(256) lse_merge_kernel(MergeLaunch a) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= a.rows * a.heads) return;
  const int64_t r = w / a.heads;
  const int h = (int)(w % a.heads);
  const float* L = a.part_lse + r * a.lsr + h * a.lsh;
  float mx = -INFINITY;
  for (int p = lane; p < a.n_parts; p += 32) mx = fmaxf(mx, __ldg(L + p * a.lsp));
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int64_t out_off = (r * a.heads + h) * (int64_t)a.head_dim;
  if (mx == -INFINITY) {
    for (int i = lane; i < a.head_dim; i += 32) {
      if (OUT_F32)
        ((float*)a.out)[out_off + i] = 0.f;
      else
        ((__nv_bfloat16*)a.out)[out_off + i] = __float2bfloat16_rn(0.f);
    }
    if (a.lse_out && lane == 0) a.lse_out[r * a.heads + h] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int p = lane; p < a.n_parts; p += 32) {
    const float l = __ldg(L + p * a.lsp);
    sum += (l == -INFINITY) ? 0.f : expf(l - mx);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = mx + logf(sum);
  const float* O = a.part_out + r * a.osr + h * a.osh;
  for (int i = lane; i < a.head_dim; i += 32) {
    float acc = 0.f;
    for (int p = 0; p < a.n_parts; ++p) {
      const float l = __ldg(L + p * a.lsp);
      if (l == -INFINITY) continue;
      acc += expf(l - lse) * __ldg(O + p * a.osp + i);
    }
    if (OUT_F32)
      ((float*)a.out)[out_off + i] = acc;
    else
      ((__nv_bfloat16*)a.out)[out_off + i] = __float2bfloat16_rn(acc);
  }
  if (a.lse_out && lane == 0) a.lse_out[r * a.heads + h] = lse;
}

// The same merge with each lane owning 4 consecutive elements of head_dim
// (16-byte loads of the part outputs), the part weights exp(LSE_s - LSE)
// computed once per part, and two parts in flight per iteration.  Used when
// head_dim is a multiple of 4 and every part row starts on a 16-byte boundary.
template <bool OUT_F32>
__global__ void __launch_bounds__(256) lse_merge_vec_kernel(MergeLaunch a) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= a.rows * a.heads) return;
  const int64_t r = w / a.heads;
  const int h = (int)(w % a.heads);
  const float* L = a.part_lse + r * a.lsr + h * a.lsh;
  float mx = -INFINITY;
  for (int p = lane; p < a.n_parts; p += 32) mx = fmaxf(mx, __ldg(L + p * a.lsp));
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int64_t out_off = (r * a.heads + h) * (int64_t)a.head_dim;
  float lse = -INFINITY;
  if (mx != -INFINITY) {
    float sum = 0.f;
    for (int p = lane; p < a.n_parts; p += 32) {
      const float l = __ldg(L + p * a.lsp);
      sum += (l == -INFINITY) ? 0.f : expf(l - mx);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    lse = mx + logf(sum);
  }
  const float* O = a.part_out + r * a.osr + h * a.osh;
  for (int i = lane * 4; i < a.head_dim; i += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse != -INFINITY) {
      int p = 0;
      for (; p + 1 < a.n_parts; p += 2) {
        const float l0 = __ldg(L + p * a.lsp), l1 = __ldg(L + (p + 1) * a.lsp);
        float4 o0 = make_float4(0.f, 0.f, 0.f, 0.f), o1 = o0;
        if (l0 != -INFINITY) o0 = __ldg(reinterpret_cast<const float4*>(O + p * a.osp + i));
        if (l1 != -INFINITY) o1 = __ldg(reinterpret_cast<const float4*>(O + (p + 1) * a.osp + i));
        const float w0 = (l0 == -INFINITY) ? 0.f : expf(l0 - lse);
        const float w1 = (l1 == -INFINITY) ? 0.f : expf(l1 - lse);
        acc.x += w0 * o0.x;
        acc.y += w0 * o0.y;
        acc.z += w0 * o0.z;
        acc.w += w0 * o0.w;
        acc.x += w1 * o1.x;
        acc.y += w1 * o1.y;
        acc.z += w1 * o1.z;
        acc.w += w1 * o1.w;
      }
      if (p < a.n_parts) {
        const float l0 = __ldg(L + p * a.lsp);
        if (l0 != -INFINITY) {
          const float4 o0 = __ldg(reinterpret_cast<const float4*>(O + p * a.osp + i));
          const float w0 = expf(l0 - lse);
          acc.x += w0 * o0.x;
          acc.y += w0 * o0.y;
          acc.z += w0 * o0.z;
          acc.w += w0 * o0.w;
        }
      }
    }
    if (OUT_F32) {
      *reinterpret_cast<float4*>((float*)a.out + out_off + i) = acc;
    } else {
      uint2 v;
      v.x = pack_bf16x2(acc.x, acc.y);
      v.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>((__nv_bfloat16*)a.out + out_off + i) = v;
    }
  }
  if (a.lse_out && lane == 0) a.lse_out[r * a.heads + h] = lse;
}

cudaError_t launch_lse_merge(const MergeLaunch& a, cudaStream_t s) {
  const int64_t warps = a.rows * a.heads;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  const bool vec = a.head_dim % 4 == 0 && ((uintptr_t)a.part_out & 15) == 0 && a.osp % 4 == 0 && a.osr % 4 == 0 &&
                   a.osh % 4 == 0 && ((uintptr_t)a.out & (a.out_f32 ? 15 : 7)) == 0;
  if (vec) {
    if (a.out_f32)
      lse_merge_vec_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
      lse_merge_vec_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(a);
  } else if (a.out_f32) {
    lse_merge_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(a);
  } else {
    lse_merge_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace attn
