// Split-KV decode over a head-major paged KV cache.
//
// One CTA per (split s, KV head g, request b).  The split owns a run of whole
// 64-token pages; each page of one head is one contiguous 16 KB block of K and
// one of V (the head-sharded cache of the Ulysses page, section 2.3).  A
// producer thread streams the pages through a 3-stage shared-memory ring with
// TMA (128-byte swizzled boxes, completion on mbarriers), and four consumer
// warps each take 16 of the 64 tokens of every page.
//
// All 8 query heads of the GQA group read the same page, so the page is read
// from HBM once per group.  The group's work is a small dense contraction
// (8 heads x 128 dims x 64 tokens, twice per page: 8 flops per cached byte),
// too much for fp32 CUDA-core FMAs to hide behind the HBM stream, so each warp
// runs it on the tensor cores with mma.sync m16n8k16 (bf16 in, fp32 out):
// the 8 heads fill rows 0-7 of the 16-row A operand (rows 8-15 are zero).
//   scores:  S[h][t] = q_h . k_t   A = q (registers), B = K rows (ldmatrix)
//   values:  O[h][:] += P[h][t] V_t   A = P (the score accumulators re-packed
//            to bf16 in registers), B = V rows (ldmatrix.trans)
// Each warp keeps its own online-softmax state (m, l, O) across pages
// (Flash Attention page, section 18.3); the four warps are merged through
// shared memory at the end, and the split writes its partial O and LSE.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace dec {

constexpr int D = 128, PAGE = 64, G = 8;
constexpr int NST = 3;                    // pipeline stages
constexpr int PAGE_BYTES = PAGE * D * 2;  // 16 KB (one head's K or V page)
constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
constexpr int OFF_BAR = NST * STAGE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 2 * NST * 8 + 1024;
constexpr int NCONS = 4;                  // consumer warps
constexpr int NTHREADS = (NCONS + 1) * 32;

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
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of (token row, 16-byte chunk 0..15) inside one staged page: the
// two 64-element halves of head_dim are two TMA boxes of 64 rows x 128 bytes,
// each stored with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t page_off(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * (PAGE_BYTES / 2) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(NTHREADS, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeLaunch a) {
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
      for (int i = 0; i < npg; ++i) {
        const int st = i % NST;
        if (i >= NST && !mbar_wait(&empty[st], ((i / NST) - 1) & 1, a.err, DEV_TIMEOUT_DECODE)) break;
        int pid = table[p_beg + i];
        if (pid < 0 || pid >= a.num_pages) {
          record_error(a.err, DEV_BAD_PAGE);
          pid = 0;
        }
        const int row0 = (int)(((int64_t)g * a.num_pages + pid) * PAGE);
        uint8_t* dst = smem + st * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
        tma_load_2d(dst, &tm_k, &full[st], 0, row0);
        tma_load_2d(dst + PAGE_BYTES / 2, &tm_k, &full[st], 64, row0);
        tma_load_2d(dst + PAGE_BYTES, &tm_v, &full[st], 0, row0);
        tma_load_2d(dst + PAGE_BYTES + PAGE_BYTES / 2, &tm_v, &full[st], 64, row0);
      }
    }
    return;
  }

  // ---------------- consumers
  const int grp = lane >> 2, tig = lane & 3;  // mma fragment coordinates
  const float sl2 = a.scale * 1.4426950408889634f;
  // A fragments of q: row grp = head g*G + grp, 16 dims per k-step.
  uint32_t qa[8][2];
  {
    const uint32_t* qrow =
        (const uint32_t*)((const __nv_bfloat16*)a.q + ((int64_t)b * a.hq + g * G + grp) * D);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = __ldg(qrow + ks * 8 + tig);
      qa[ks][1] = __ldg(qrow + ks * 8 + 4 + tig);
    }
  }
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int kb = warp * 16;  // this warp's 16 tokens of each page
  const uint32_t sbase = smem_u32(smem);
  const int mat = lane >> 3, rr = lane & 7;
  bool ok = true;

  for (int i = 0; i < npg; ++i) {
    const int st = i % NST;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / NST) & 1, a.err, DEV_TIMEOUT_DECODE));
    if (!ok) break;
    const uint32_t kst = sbase + st * STAGE_BYTES;
    const uint32_t vst = kst + PAGE_BYTES;
    // S = q K^T for tokens kb..kb+15 (two n-tiles of 8 tokens)
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int key = kb + (mat >> 1) * 8 + rr;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + page_off(key, 2 * ks + (mat & 1)), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
        mma_bf16(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
      }
    }
    // mask tokens past the context, online softmax for head row grp
    const int tok0 = (p_beg + i) * PAGE + kb + 2 * tig;
    float mx = -INFINITY;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (tok0 + n * 8 + e >= ctx) sc[n][e] = -INFINITY;
        mx = fmaxf(mx, sc[n][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2((m - m_new) * sl2);
    const float mb = (m_new == -INFINITY) ? 0.f : m_new * sl2;
    float p[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[n][e] = fast_exp2(fmaf(sc[n][e], sl2, -mb));
        l = (n == 0 && e == 0) ? l * alpha + p[n][e] : l + p[n][e];
      }
    m = m_new;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= alpha;
      o[n][1] *= alpha;
    }
    // O += P V: A = P (rows = heads, k = the warp's 16 tokens)
    const uint32_t pa0 = pack_bf16x2(p[0][0], p[0][1]);
    const uint32_t pa2 = pack_bf16x2(p[1][0], p[1][1]);
    {
      const int key = kb + (mat & 1) * 8 + rr;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vst + page_off(key, c + (mat >> 1)), b0, b1, b2, b3);
        mma_bf16(o[c], pa0, 0u, pa2, 0u, b0, b1);
        mma_bf16(o[c + 1], pa0, 0u, pa2, 0u, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
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
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    red[(warp * G + grp) * D + n * 8 + 2 * tig] = o[n][0] * wself;
    red[(warp * G + grp) * D + n * 8 + 2 * tig + 1] = o[n][1] * wself;
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

}  // namespace dec

cudaError_t launch_decode_split(const DecodeLaunch& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dec::decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         dec::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (a.batch == 0) return cudaSuccess;
  dim3 grid(a.num_splits, a.hkv, a.batch);
  dec::decode_split_kernel<<<grid, dec::NTHREADS, dec::SMEM_BYTES, s>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace attn
