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

// (row, head) of item w = row * heads + head, in 32-bit arithmetic when w fits
// (a 64-bit division is a long instruction sequence).
__device__ __forceinline__ void split_item(int64_t w, int heads, int64_t& row, int& h) {
  if (w < 0x7fffffff) {
    const uint32_t r32 = (uint32_t)w / (uint32_t)heads;
    row = r32;
    h = (int)((uint32_t)w - r32 * (uint32_t)heads);
  } else {
    row = w / heads;
    h = (int)(w % heads);
  }
}

template <bool OUT_F32>
__global__ void __launch_bounds__(256) lse_merge_kernel(MergeLaunch a) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= a.rows * a.heads) return;
  int64_t r;
  int h;
  split_item(w, a.heads, r, h);
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
// (16-byte loads of the part outputs) and the part weights exp(LSE_s - LSE)
// computed per part.  The first kPre parts' outputs are requested before the
// part LSEs are reduced, so a warp waits for one memory latency, not two.
// Used when head_dim is a multiple of 4 and every part row starts on a 16-byte
// boundary.  A part whose LSE is -inf contributes nothing, whatever its output
// row holds.
constexpr int kPre = 4;

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& o) {
  acc.x = fmaf(w, o.x, acc.x);
  acc.y = fmaf(w, o.y, acc.y);
  acc.z = fmaf(w, o.z, acc.z);
  acc.w = fmaf(w, o.w, acc.w);
}

template <bool OUT_F32>
__global__ void __launch_bounds__(256) lse_merge_vec_kernel(MergeLaunch a) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= a.rows * a.heads) return;
  int64_t r;
  int h;
  split_item(w, a.heads, r, h);
  const float* L = a.part_lse + r * a.lsr + h * a.lsh;
  const float* O = a.part_out + r * a.osr + h * a.osh;
  const int i0 = lane * 4;
  float4 pre[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k)
    if (k < a.n_parts && i0 < a.head_dim) pre[k] = __ldg(reinterpret_cast<const float4*>(O + k * a.osp + i0));
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
  for (int i = i0; i < a.head_dim; i += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse != -INFINITY) {
#pragma unroll
      for (int k = 0; k < kPre; ++k) {
        if (k < a.n_parts) {
          const float l = __ldg(L + k * a.lsp);
          const float4 o = (i == i0) ? pre[k] : __ldg(reinterpret_cast<const float4*>(O + k * a.osp + i));
          if (l != -INFINITY) fma4(acc, expf(l - lse), o);
        }
      }
      for (int p = kPre; p < a.n_parts; ++p) {
        const float l = __ldg(L + p * a.lsp);
        if (l != -INFINITY) fma4(acc, expf(l - lse), __ldg(reinterpret_cast<const float4*>(O + p * a.osp + i)));
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

// head_dim 128 and at most 32 parts: a warp takes R consecutive (row, head)
// items, lane l holding dims 4l..4l+3 and the LSE of part l.  The part weights
// exp(LSE_s - LSE) are computed by the lane that holds part s and broadcast by
// shuffle; the part outputs are read G parts at a time for all R items, every
// load of a group issued before any is used, so a warp has R * G 16-byte loads
// in flight.  The sum runs over the parts in order, as in the kernels above.
template <bool OUT_F32, int R, int G>
__global__ void __launch_bounds__(256) lse_merge_d128_kernel(MergeLaunch a) {
  const int64_t items = a.rows * a.heads;
  const int64_t w0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * R;
  const int lane = threadIdx.x & 31;
  if (w0 >= items) return;  // the whole warp
  const int i = lane * 4;
  const float* O[R];
  float wgt[R], lse[R];
  bool valid[R];
  float4 o[R][G];
  const bool one_group = a.n_parts <= G;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t w = w0 + r;
    valid[r] = w < items;
    // items < 2^31 (checked at launch): 32-bit division, not the 64-bit sequence
    const uint32_t w32 = valid[r] ? (uint32_t)w : 0u;
    const uint32_t row = w32 / (uint32_t)a.heads;
    const int h = (int)(w32 - row * (uint32_t)a.heads);
    O[r] = a.part_out + (int64_t)row * a.osr + h * a.osh + i;
    // with all parts in one group, their rows are requested first: they need
    // only addresses, so their latency overlaps the LSE loads and the weights
    if (one_group)
#pragma unroll
      for (int k = 0; k < G; ++k)
        if (valid[r] && k < a.n_parts) o[r][k] = __ldg(reinterpret_cast<const float4*>(O[r] + k * a.osp));
    wgt[r] = (valid[r] && lane < a.n_parts) ? __ldg(a.part_lse + (int64_t)row * a.lsr + h * a.lsh + lane * a.lsp)
                                              : -INFINITY;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float mx = wgt[r];
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = (wgt[r] == -INFINITY) ? 0.f : expf(wgt[r] - mx);
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    lse[r] = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    wgt[r] = (wgt[r] == -INFINITY || lse[r] == -INFINITY) ? 0.f : expf(wgt[r] - lse[r]);
  }
  float4 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p0 = 0; p0 < a.n_parts; p0 += G) {
    if (!one_group)
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < G; ++k)
          if (valid[r] && p0 + k < a.n_parts) o[r][k] = __ldg(reinterpret_cast<const float4*>(O[r] + (p0 + k) * a.osp));
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wgt[r], (p0 + k) & 31);
        if (valid[r] && p0 + k < a.n_parts && wk != 0.f) fma4(acc[r], wk, o[r][k]);
      }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!valid[r]) continue;
    const int64_t out_off = (w0 + r) * 128 + i;  // (row * heads + h) * 128
    if (OUT_F32) {
      *reinterpret_cast<float4*>((float*)a.out + out_off) = acc[r];
    } else {
      uint2 v;
      v.x = pack_bf16x2(acc[r].x, acc[r].y);
      v.y = pack_bf16x2(acc[r].z, acc[r].w);
      *reinterpret_cast<uint2*>((__nv_bfloat16*)a.out + out_off) = v;
    }
    if (a.lse_out && lane == 0) a.lse_out[w0 + r] = lse[r];
  }
}

// head_dim 128, at most 2 parts: a warp merges 16 (row, head) items.  First
// lane 2i + k holds part k's LSE of item i; one exchange with the partner lane
// gives the item's max, sum, LSE and the lane's weight -- the same arithmetic
// as lse_merge_d128_kernel, done once per 32 lanes instead of once per item.
// Then the items go two at a time: both parts' 16-byte slices requested
// first, the weights taken from their lanes by shuffle.
template <bool OUT_F32>
__global__ void __launch_bounds__(256) lse_merge_d128_x16_kernel(MergeLaunch a) {
  constexpr int W = 16;
  const int64_t items = a.rows * a.heads;
  const int64_t w0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * W;
  const int lane = threadIdx.x & 31;
  if (w0 >= items) return;  // the whole warp
  // items < 2^31 (checked at launch): 32-bit row / head arithmetic
  const uint32_t first = (uint32_t)w0;
  const uint32_t row0 = first / (uint32_t)a.heads;
  const int h0 = (int)(first - row0 * (uint32_t)a.heads);
  float wgt, lse;
  {
    const int i = lane >> 1, k = lane & 1;
    const int64_t w = w0 + i;
    float l = -INFINITY;
    if (w < items && k < a.n_parts) {
      const uint32_t row = (uint32_t)w / (uint32_t)a.heads;
      const int h = (int)((uint32_t)w - row * (uint32_t)a.heads);
      l = __ldg(a.part_lse + (int64_t)row * a.lsr + h * a.lsh + k * a.lsp);
    }
    const float lp = __shfl_xor_sync(0xffffffffu, l, 1);
    const float mx = fmaxf(l, lp);
    const float sum = (l == -INFINITY ? 0.f : expf(l - mx)) + (lp == -INFINITY ? 0.f : expf(lp - mx));
    lse = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    wgt = (l == -INFINITY || lse == -INFINITY) ? 0.f : expf(l - lse);
    if (a.lse_out && k == 0 && w < items) a.lse_out[w] = lse;
  }
  const int c = lane * 4;
  uint32_t row = row0;
  int h = h0;
  for (int i = 0; i < W; i += 2) {
    const float* O[2];
    bool valid[2];
    float4 o[2][2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      valid[r] = w0 + i + r < items;
      O[r] = a.part_out + (int64_t)row * a.osr + h * a.osh + c;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (valid[r] && k < a.n_parts) o[r][k] = __ldg(reinterpret_cast<const float4*>(O[r] + k * a.osp));
      if (++h == a.heads) {
        h = 0;
        ++row;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wgt, 2 * (i + r) + k);
        if (valid[r] && k < a.n_parts && wk != 0.f) fma4(acc, wk, o[r][k]);
      }
      if (!valid[r]) continue;
      const int64_t out_off = (w0 + i + r) * 128 + c;  // (row * heads + h) * 128
      if (OUT_F32) {
        *reinterpret_cast<float4*>((float*)a.out + out_off) = acc;
      } else {
        uint2 v;
        v.x = pack_bf16x2(acc.x, acc.y);
        v.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>((__nv_bfloat16*)a.out + out_off) = v;
      }
    }
  }
}

template <bool OUT_F32>
static void launch_d128(const MergeLaunch& a, int64_t items, cudaStream_t s) {
  if (a.n_parts <= 2) {
    const int64_t warps = (items + 15) / 16;
    lse_merge_d128_x16_kernel<OUT_F32><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(a);
  } else if (a.n_parts <= 4) {
    const int64_t warps = (items + 1) / 2;
    lse_merge_d128_kernel<OUT_F32, 2, 4><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(a);
  } else {
    lse_merge_d128_kernel<OUT_F32, 1, 8><<<(unsigned)((items * 32 + 255) / 256), 256, 0, s>>>(a);
  }
}

cudaError_t launch_lse_merge(const MergeLaunch& a, cudaStream_t s) {
  const int64_t warps = a.rows * a.heads;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  const bool vec = a.head_dim % 4 == 0 && ((uintptr_t)a.part_out & 15) == 0 && a.osp % 4 == 0 && a.osr % 4 == 0 &&
                   a.osh % 4 == 0 && ((uintptr_t)a.out & (a.out_f32 ? 15 : 7)) == 0;
  if (vec && a.head_dim == 128 && a.n_parts <= 32 && warps < 0x7fffffff) {
    if (a.out_f32)
      launch_d128<true>(a, warps, s);
    else
      launch_d128<false>(a, warps, s);
  } else if (vec) {
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
