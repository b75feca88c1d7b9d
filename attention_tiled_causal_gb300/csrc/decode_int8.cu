// Split-KV decode over a head-major paged INT8 KV cache.
//
// The cache holds symmetric int8 codes and one fp32 scale per (KV head, cached
// token): value = code * scale.  An INT8 cache halves the bytes a decode step
// streams (Flash Attention page, section 18.12); the Ulysses page, section 5.4,
// describes such grouped codes with their scales.  Per head and page: 64 x 128
// code bytes of K (one 8 KB block), the same for V, and 64 scales each.
//
// Structure as the bf16 split kernel: one CTA per (split s, KV head g, request
// b); a producer thread streams pages through a 6-stage ring (TMA for the code
// blocks, 128-byte swizzled; a bulk copy for the two 256-byte scale rows); four
// consumer warps take 16 tokens of each page, two pages per iteration, and keep
// online-softmax states that are merged at the end.  The group contraction runs on mma.sync m16n8k16 with
// fp16 operands, because an int8 code becomes an fp16 value exactly with two
// integer instructions and one packed subtract (0x6400 | (code + 128) is the
// fp16 number 1024 + code + 128), and fp16 holds the bf16 query and the
// softmax weights without loss over their ranges.  The scales stay outside the
// MMAs: S[h][t] = k_scale[t] * (q_h . kcode_t), and the weight P[h][t] is
// multiplied by v_scale[t] before O += P Vcode.  A query or scaled weight
// beyond the fp16 range is recorded as a device error.
//
//   scores: A = q (k order permuted so a thread's 4 dims of a k-step are
//           consecutive; the same permutation is used for K), B = K codes via
//           ldmatrix on the code rows viewed as 16-bit pairs: a thread receives
//           4 consecutive dims of one token.
//   values: A = P * v_scale (k = the warp's 16 tokens), B = V codes via
//           ldmatrix.trans on the same 16-bit view: a thread receives two
//           dims of two tokens; a byte permute splits them into an even-dim
//           and an odd-dim operand, so output column n of an MMA is dim
//           16 c + 2 n (even) or 16 c + 2 n + 1 (odd).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace dec8 {

constexpr int D = 128, PAGE = 64, G = 8;
constexpr int NST = 6;                                    // pipeline stages
constexpr int PAGE_BYTES = PAGE * D;                      // 8 KB of codes (one head's K or V page)
constexpr int SCALE_BYTES = PAGE * 4;                     // 256 B of scales
constexpr int OFF_V = PAGE_BYTES, OFF_KS = 2 * PAGE_BYTES, OFF_VS = OFF_KS + SCALE_BYTES;
constexpr int STAGE_TX = 2 * PAGE_BYTES + 2 * SCALE_BYTES;
constexpr int STAGE_BYTES = 17408;                        // STAGE_TX rounded up to 1 KB (swizzle alignment)
constexpr int OFF_BAR = NST * STAGE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 2 * NST * 8 + 1024;
constexpr int NCONS = 4;                                  // consumer warps
constexpr int NTHREADS = (NCONS + 1) * 32;
constexpr float kHalfMax = 65504.f;
static_assert(STAGE_BYTES >= STAGE_TX && STAGE_BYTES % 1024 == 0, "stage layout");
static_assert(NCONS * G * D * 4 + 2 * NCONS * G * 4 <= OFF_BAR, "merge scratch fits in the ring");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two int8 codes, selected from a code word already XOR-ed with 0x80808080
// (each byte = code + 128) by a byte-permute selector, as an fp16 pair:
// 0x64uu is the fp16 number 1024 + uu, and 1024 + code + 128 - 1152 = code.
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t biased, uint32_t sel) {
  const uint32_t h = __byte_perm(biased, 0x64646464u, sel);
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));  // 0x6480 = 1152.0
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte offset of (token row, 16-byte chunk 0..7) in a staged 8 KB code page:
// 64 rows of 128 bytes, 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t code_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(NTHREADS, 2)
    decode_split_int8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const DecodeLaunch a, const float* __restrict__ k_scale,
                             const float* __restrict__ v_scale) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + OFF_BAR);
  uint64_t* empty = full + NST;

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int S = a.num_splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ctx = a.ctx_lens[b];
  const int n_pages = (ctx + PAGE - 1) / PAGE;
  const int pps = (n_pages + S - 1) / S;
  const int p_beg = min(s * pps, n_pages);
  const int npg = min(p_beg + pps, n_pages) - p_beg;
  const int64_t part_row = ((int64_t)b * a.hq + g * G) * S + s;  // (b, h = g*G, s)

  if (npg <= 0) {  // empty split: O = 0, LSE = -inf
    for (int i = threadIdx.x; i < G * D; i += NTHREADS)
      a.part_out[(part_row + (int64_t)(i / D) * S) * D + (i % D)] = 0.f;
    if (threadIdx.x < G) a.part_lse[part_row + (int64_t)threadIdx.x * S] = -INFINITY;
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCONS);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NCONS) {
    // ---------------- producer: one thread streams this split's pages
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int32_t* table = a.page_table + (int64_t)b * a.max_pages;
      int issued = 0;
      for (int i = 0; i < npg; ++i) {
        const int st = i % NST;
        if (i >= NST && !mbar_wait(&empty[st], ((i / NST) - 1) & 1, a.err, DEV_TIMEOUT_DECODE)) break;
        int pid = table[p_beg + i];
        if (pid < 0 || pid >= a.num_pages) {
          record_error(a.err, DEV_BAD_PAGE);
          pid = 0;
        }
        const int64_t row0 = ((int64_t)g * a.num_pages + pid) * PAGE;
        uint8_t* dst = smem + st * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[st], STAGE_TX);
        tma_load_2d(dst, &tm_k, &full[st], 0, (int)row0);
        tma_load_2d(dst + OFF_V, &tm_v, &full[st], 0, (int)row0);
        bulk_load(dst + OFF_KS, k_scale + row0, SCALE_BYTES, &full[st]);
        bulk_load(dst + OFF_VS, v_scale + row0, SCALE_BYTES, &full[st]);
        issued = i + 1;
      }
      // leave no copy in flight: wait (bounded) for the last stages issued
      for (int i = max(0, issued - NST); i < issued; ++i)
        mbar_wait(&full[i % NST], (i / NST) & 1, nullptr, 0);
    }
    return;
  }

  // ---------------- consumers
  const int grp = lane >> 2, tig = lane & 3;  // mma fragment coordinates
  const float sl2 = a.scale * 1.4426950408889634f;
  // A fragments of q (fp16): row grp = head g*G + grp; in k-step ks the thread's
  // slots 2tig, 2tig+1 hold dims 16ks + 4tig + {0, 1} and slots 2tig+8, 2tig+9
  // hold dims 16ks + 4tig + {2, 3}.
  uint32_t qa[8][2];
  {
    const uint2* qrow = (const uint2*)((const __nv_bfloat16*)a.q + ((int64_t)b * a.hq + g * G + grp) * D);
    bool in_range = true;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint2 w = __ldg(qrow + ks * 4 + tig);  // 4 bf16: dims 16ks + 4tig .. +3
      const float x0 = __uint_as_float(w.x << 16), x1 = __uint_as_float(w.x & 0xffff0000u);
      const float x2 = __uint_as_float(w.y << 16), x3 = __uint_as_float(w.y & 0xffff0000u);
      in_range &= fabsf(x0) <= kHalfMax && fabsf(x1) <= kHalfMax && fabsf(x2) <= kHalfMax && fabsf(x3) <= kHalfMax;
      qa[ks][0] = pack_half2(x0, x1);
      qa[ks][1] = pack_half2(x2, x3);
    }
    if (!in_range) record_error(a.err, DEV_FP16_RANGE);
  }
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int kb = warp * 16;  // this warp's 16 tokens of each page
  const uint32_t sbase = smem_u32(smem);
  const int mat = lane >> 3, rr = lane & 7;
  const int key = kb + (mat & 1) * 8 + rr;  // ldmatrix row this lane addresses
  bool ok = true;

  // Two pages per iteration: 32 tokens of this warp, whose score chains are
  // independent, under one online-softmax update.  An odd last page runs alone.
  for (int i = 0; i < npg; i += 2) {
    const bool two = i + 1 < npg;
    const int st0 = i % NST, st1 = (i + 1) % NST;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[st0], (i / NST) & 1, a.err, DEV_TIMEOUT_DECODE) &&
                                     (!two || mbar_wait(&full[st1], ((i + 1) / NST) & 1, a.err, DEV_TIMEOUT_DECODE)));
    if (!ok) break;
    // S = q Kcode^T: n-tiles (page 0, tokens 0-7), (page 0, 8-15), (page 1, 0-7), (page 1, 8-15)
    float sc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int pg = 0; pg < 2; ++pg) {
      if (pg == 1 && !two) break;
      const uint32_t kst = sbase + (pg ? st1 : st0) * STAGE_BYTES;
#pragma unroll
      for (int ks = 0; ks < 8; ks += 2) {
        uint32_t r0, r1, r2, r3;  // (n-tile 0, ks), (n-tile 1, ks), (n-tile 0, ks+1), (n-tile 1, ks+1)
        ldsm_x4(kst + code_off(key, ks + (mat >> 1)), r0, r1, r2, r3);
        r0 ^= 0x80808080u;
        r1 ^= 0x80808080u;
        r2 ^= 0x80808080u;
        r3 ^= 0x80808080u;
        mma_f16(sc[2 * pg], qa[ks][0], 0u, qa[ks][1], 0u, codes_to_half2(r0, 0x5140), codes_to_half2(r0, 0x7362));
        mma_f16(sc[2 * pg + 1], qa[ks][0], 0u, qa[ks][1], 0u, codes_to_half2(r1, 0x5140),
                codes_to_half2(r1, 0x7362));
        mma_f16(sc[2 * pg], qa[ks + 1][0], 0u, qa[ks + 1][1], 0u, codes_to_half2(r2, 0x5140),
                codes_to_half2(r2, 0x7362));
        mma_f16(sc[2 * pg + 1], qa[ks + 1][0], 0u, qa[ks + 1][1], 0u, codes_to_half2(r3, 0x5140),
                codes_to_half2(r3, 0x7362));
      }
    }
    // K scales, mask of tokens past the context (and of a missing second page),
    // online softmax for head row grp
    float mx = -INFINITY;
#pragma unroll
    for (int pg = 0; pg < 2; ++pg) {
      const float* kss = (const float*)(smem + (pg ? st1 : st0) * STAGE_BYTES + OFF_KS);
      const int tok0 = (p_beg + i + pg) * PAGE + kb + 2 * tig;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        float2 ksc = make_float2(0.f, 0.f);
        if (pg == 0 || two) ksc = *reinterpret_cast<const float2*>(kss + kb + n * 8 + 2 * tig);
        sc[2 * pg + n][0] *= ksc.x;
        sc[2 * pg + n][1] *= ksc.y;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if ((pg == 1 && !two) || tok0 + n * 8 + e >= ctx) sc[2 * pg + n][e] = -INFINITY;
          mx = fmaxf(mx, sc[2 * pg + n][e]);
        }
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2((m - m_new) * sl2);
    const float mb = (m_new == -INFINITY) ? 0.f : m_new * sl2;
    float p[4][2];
    l *= alpha;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[n][e] = fast_exp2(fmaf(sc[n][e], sl2, -mb));
        l += p[n][e];
      }
    m = m_new;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= alpha;
      o[n][1] *= alpha;
    }
    // O += (P v_scale) Vcode, page by page: A = weighted P (rows = heads, k = the page's 16 tokens)
#pragma unroll
    for (int pg = 0; pg < 2; ++pg) {
      if (pg == 1 && !two) break;
      const uint32_t vst = sbase + (pg ? st1 : st0) * STAGE_BYTES + OFF_V;
      const float* vss = (const float*)(smem + (pg ? st1 : st0) * STAGE_BYTES + OFF_VS);
      uint32_t pa0, pa2;
      {
        const float2 v0 = *reinterpret_cast<const float2*>(vss + kb + 2 * tig);
        const float2 v1 = *reinterpret_cast<const float2*>(vss + kb + 8 + 2 * tig);
        const float w00 = p[2 * pg][0] * v0.x, w01 = p[2 * pg][1] * v0.y;
        const float w10 = p[2 * pg + 1][0] * v1.x, w11 = p[2 * pg + 1][1] * v1.y;
        if (!(fabsf(w00) <= kHalfMax && fabsf(w01) <= kHalfMax && fabsf(w10) <= kHalfMax &&
              fabsf(w11) <= kHalfMax))
          record_error(a.err, DEV_FP16_RANGE);
        pa0 = pack_half2(w00, w01);
        pa2 = pack_half2(w10, w11);
      }
#pragma unroll
      for (int c = 0; c < 8; c += 2) {
        uint32_t r0, r1, r2, r3;  // (tokens 0-7, chunk c), (tokens 8-15, c), (0-7, c+1), (8-15, c+1)
        ldsm_x4_t(vst + code_off(key, c + (mat >> 1)), r0, r1, r2, r3);
        r0 ^= 0x80808080u;
        r1 ^= 0x80808080u;
        r2 ^= 0x80808080u;
        r3 ^= 0x80808080u;
        // even dims 16c + 2n use bytes 0 and 2 of each register, odd dims bytes 1 and 3
        mma_f16(o[2 * c], pa0, 0u, pa2, 0u, codes_to_half2(r0, 0x5240), codes_to_half2(r1, 0x5240));
        mma_f16(o[2 * c + 1], pa0, 0u, pa2, 0u, codes_to_half2(r0, 0x5341), codes_to_half2(r1, 0x5341));
        mma_f16(o[2 * c + 2], pa0, 0u, pa2, 0u, codes_to_half2(r2, 0x5240), codes_to_half2(r3, 0x5240));
        mma_f16(o[2 * c + 3], pa0, 0u, pa2, 0u, codes_to_half2(r2, 0x5341), codes_to_half2(r3, 0x5341));
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[st0]);
      if (two) mbar_arrive(&empty[st1]);
    }
  }

  // ---------------- merge the four warps' states through shared memory
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  asm volatile("bar.sync 1, %0;" ::"r"(NCONS * 32) : "memory");  // every page consumed: ring is free
  float* red = (float*)smem;                                       // [NCONS][G][D]
  float* ms = red + NCONS * G * D;                                 // [NCONS][G]
  float* ls = ms + NCONS * G;                                      // [NCONS][G]
  if (tig == 0) {
    ms[warp * G + grp] = ok ? m : -INFINITY;
    ls[warp * G + grp] = ok ? l : 0.f;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCONS * 32) : "memory");
  float M = -INFINITY;
#pragma unroll
  for (int w2 = 0; w2 < NCONS; ++w2) M = fmaxf(M, ms[w2 * G + grp]);
  const float wself = (M == -INFINITY || m == -INFINITY || !ok) ? 0.f : fast_exp2((m - M) * sl2);
  // accumulator o[2c + par] column n is dim 16c + 2n + par; this thread holds n = 2tig, 2tig+1
#pragma unroll
  for (int idx = 0; idx < 16; ++idx) {
    const int dim = (idx >> 1) * 16 + 4 * tig + (idx & 1);
    red[(warp * G + grp) * D + dim] = o[idx][0] * wself;
    red[(warp * G + grp) * D + dim + 2] = o[idx][1] * wself;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCONS * 32) : "memory");
  for (int idx = threadIdx.x; idx < G * D; idx += NCONS * 32) {
    const int h = idx / D, dd = idx % D;
    float Mh = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < NCONS; ++w2) Mh = fmaxf(Mh, ms[w2 * G + h]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < NCONS; ++w2) {
      const float mw = ms[w2 * G + h];
      if (mw != -INFINITY) L += ls[w2 * G + h] * fast_exp2((mw - Mh) * sl2);
      acc += red[(w2 * G + h) * D + dd];
    }
    const int64_t prow = part_row + (int64_t)h * S;
    a.part_out[prow * D + dd] = L > 0.f ? acc / L : 0.f;
    if (dd == 0) a.part_lse[prow] = L > 0.f ? Mh * a.scale + logf(L) : -INFINITY;
  }
}

}  // namespace dec8

cudaError_t launch_decode_split_int8(const DecodeLaunch& a, const float* k_scale, const float* v_scale,
                                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dec8::decode_split_int8_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, dec8::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (a.batch == 0) return cudaSuccess;
  dim3 grid(a.num_splits, a.hkv, a.batch);
  dec8::decode_split_int8_kernel<<<grid, dec8::NTHREADS, dec8::SMEM_BYTES, s>>>(tk, tv, a, k_scale, v_scale);
  return cudaGetLastError();
}

}  // namespace attn
