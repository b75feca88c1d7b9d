// Causal GQA prefill on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// The method is the tiled attention of the Flash Attention page: scores of one
// query tile against one K/V tile (section 18.3, step 1), the running max m and
// denominator l updated per tile with the old output rescaled by
// exp(m_old - m_new) (steps 2-6), the query tile as the outer loop and the
// division by l deferred to the end (section 18.4), and TMA loads overlapped
// with compute by warp specialisation (section 18.5).  What is GB300-specific:
//
//  * One CTA owns TWO 128-row query tiles (A and B) of one query head and
//    streams the K/V tiles of that head's KV group once for both.
//  * Warp 8 (one thread) is the TMA producer: Q tiles once, then K_j and V_j
//    tiles (128 tokens x 128 dims, two 128-byte-swizzled boxes each) into a
//    3-slot shared-memory ring, each slot guarded by full/empty mbarriers.
//    The Q tiles and K_0 are requested before the CTA knows how many key
//    tiles it needs; warp 11 works that out meanwhile.
//  * Warps 9 and 10 issue tcgen05.mma, each as a converged warp with one
//    elected lane: warp 9 the scores S_t = Q_t K_j^T into TMEM (M = 128,
//    N = 128, K = 16 per instruction, bf16 in, fp32 accumulate), warp 10 the
//    updates O_t += P_t V_j into a second TMEM accumulator.  tcgen05.commit
//    arrives on mbarriers when the tensor core is done.
//  * Warps 0-3 (tile A) and 4-7 (tile B) are the softmax warpgroups: thread r
//    of a warpgroup owns query row r (TMEM lane r), loads its 128 scores with
//    tcgen05.ld, applies the absolute-position causal mask (Ulysses page,
//    section 5.3), updates m and l, writes P = exp(S - m) as bf16 into shared
//    memory in the swizzled K-major layout the MMA reads, and rescales its O
//    row in TMEM when m grows.  While one warpgroup works on its softmax the
//    tensor core runs the other tile's MMAs.
//  * The rescale is thresholded: m only moves (and O is only rescaled) when
//    some row of the warp would grow by more than 2^8 in exp2 units; P then
//    stays <= 256, and the final O / l is exact whatever reference max was
//    used, because numerator and denominator share it.
//  * TMEM: 512 columns = S_A | S_B | O_A | O_B, 128 fp32 columns each.
//
// Every mbarrier wait is bounded; on expiry the kernel records an error code,
// unwinds, frees its TMEM and returns (no trap).
#include <math.h>
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace tc {

constexpr int BM = 128, BN = 128, D = 128;
constexpr int HALF = 16384;  // one 128-byte-swizzled TMA box: 128 rows x 128 bytes

// Tile geometry of the two element types.  bf16: a 128 x 128 tile is two
// boxes of 64 elements (32 KB); an MMA k-step is 16 elements.  e4m3: one box of
// 128 elements (16 KB); a k-step is 32 elements.  Both step through a
// 128-byte swizzle row 32 bytes at a time.
//
// PBUF is the number of P buffers per query tile.  With two, the softmax could
// write P_t(j) while O_t += P_t(j-1) V_{j-1} still reads the other; the e4m3
// tiles leave room for that (bf16 does not: 224 KB of 227 are in use), but it
// measured slower (1755 against 1881 TFLOP/s on the 8K workload), so both
// kernels keep one.  The barriers are indexed per buffer either way.
template <bool FP8>
struct Cfg {
  static constexpr int TILE = FP8 ? 16384 : 32768;
  static constexpr int NBOX = FP8 ? 1 : 2;
  static constexpr int KSTEPS = FP8 ? 4 : 8;
  static constexpr int NSLOT = 3;
  static constexpr int PBUF = 1;
  // barriers: q_full[2], k_full[NSLOT], v_full[NSLOT], kv_empty[NSLOT],
  // s_full[2], s_free[2], p_full[2][PBUF], o_done[2][PBUF], q_rot[2]
  static constexpr int NBAR = 2 + 3 * NSLOT + 2 + 2 + 4 * PBUF + 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + 2 * TILE;
  static constexpr int OFF_P = OFF_KV + NSLOT * TILE;
  static constexpr int OFF_BAR = OFF_P + 2 * PBUF * TILE;
  static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 32 + 1024;
};
// 12 warps = 3 warpgroups.  The register file is split across the SM's four
// sub-partitions, so 3 warps per sub-partition launch with at most 168
// registers each; every role fits in that without spilling.
constexpr int NTHREADS = 384;
constexpr int WARP_TMA = 8, WARP_MMA_S = 9, WARP_MMA_PV = 10, WARP_IDLE = 11;
constexpr int REGS_LAUNCH = 168;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false, false);  // Q, K both K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, false, true);    // P K-major, V MN-major
// e4m3 x e4m3 -> fp32 (kind::f8f6f4: A and B format 0), both operands K-major:
// P V reads V^T rows (values stored transposed), since 8-bit MMA operands are K-major.
constexpr uint32_t IDESC_FP8 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
constexpr float kRescaleLog2 = 8.f;
// The e4m3 kernel's lazy reference (see the softmax loop) keeps a tile whose
// weight sum is at most this: every weight is then <= 256, inside e4m3's 448.
constexpr float kLazySumFp8 = 256.f;
// Register split of the e4m3 kernel: the producer / issuer warpgroup drops to
// REGS_SIDE so the two softmax warpgroups can hold a tile's scores through the
// lazy pass (2 x REGS_SOFTMAX + REGS_SIDE <= 3 x REGS_LAUNCH per thread).
constexpr uint32_t REGS_SOFTMAX = 200, REGS_SIDE = 88;
static_assert(2 * REGS_SOFTMAX + REGS_SIDE <= 3 * 168, "register split exceeds the launch total");

// Every mbarrier below is waited on by one role only, and that role waits for
// every phase in turn, so no barrier ever runs two phases ahead of its waiter
// (a parity wait cannot tell phase k from phase k+2).  That is why a ring slot
// has one "full" barrier for K tiles and one for V tiles: the slot alternates
// between K and V, whose consumers are different warps, and one shared
// barrier could run ahead of the warp that skipped the other kind's fills.
// For the same reason p_full and o_done have one barrier per P buffer.
struct Smem {
  uint64_t* q_full;    // [2]  TMA -> MMA: Q tile landed
  uint64_t* k_full;    // [NSLOT]  TMA -> score MMA: a K tile landed in the slot
  uint64_t* v_full;    // [NSLOT]  TMA -> value MMA: a V tile landed in the slot
  uint64_t* kv_empty;  // [NSLOT]  MMA -> TMA: ring slot consumed
  uint64_t* s_full;    // [2]  MMA -> softmax: S_t ready in TMEM
  uint64_t* s_free;    // [2]  softmax -> MMA: S_t read out of TMEM (128 arrivals)
  uint64_t* p_full;    // [2][PBUF]  softmax -> MMA: P_t written, O_t rescaled (128 arrivals)
  uint64_t* o_done;    // [2][PBUF]  MMA -> softmax: O_t += P_t V_j finished (buffer j % PBUF)
  uint64_t* q_rot;     // [2]  softmax -> MMA: Q_t rotated in place (128 arrivals; only when RoPE is fused)
  uint32_t* tmem_slot;
  int* nkv;            // [2]  K/V tiles each query tile needs
  int* nfull;          // [2]  leading K/V tiles every row of the query tile sees in full
};

struct Params {
  const int32_t *cu_q, *q_pos, *cu_k, *k_pos, *page_table, *k_lens;
  void* out;
  float* lse;
  unsigned* err;
  int64_t num_pages;
  int max_pages, hq, hkv, h_lo, causal, out_f32;
  float scale;
  int wave;  // CTAs resident at once (one per SM): the CTA `wave` launches later likely follows this one
  const float4* q_cs;  // NULL, or [total_q][32] float4: (cos, sin) of the 64 RoPE angles of each query row
  // e4m3 inputs: the value of a code is code * scale
  const float* q_scale;  // [total_q][hq]: one scale per query row
  const float* k_scale;  // [hkv]
  const float* v_scale;  // [hkv]
};

// Number of keys with position <= qp among k_pos[0..n), positions
// non-decreasing (first = k_pos[0]), if a guess that is exact for consecutive
// positions checks out (one thread, one round of loads); -1 otherwise.
__device__ int count_le_guess(const int32_t* k_pos, int n, int first, int qp) {
  if (n <= 0) return 0;
  if (first > qp) return 0;
  const int64_t g = (int64_t)qp - first + 1;  // the count if positions are consecutive
  if (g >= n) return __ldg(k_pos + n - 1) <= qp ? n : -1;
  return (__ldg(k_pos + g - 1) <= qp && __ldg(k_pos + g) > qp) ? (int)g : -1;
}

// The same count by one whole warp (every lane gets the result): a 32-way
// search; each round the lanes probe 32 evenly spaced keys of the open
// interval and a ballot keeps the segment where the positions pass qp
// (8192 keys: three rounds).
__device__ int count_le_warp(const int32_t* k_pos, int n, int qp, int lane) {
  if (n <= 0 || __ldg(k_pos) > qp) return 0;
  int lo = 1, hi = n;  // the count lies in [lo, hi]: k_pos[lo-1] <= qp, k_pos[hi] > qp or hi = n
  while (lo < hi) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < hi && __ldg(k_pos + idx) <= qp;
    const int c = __popc(__ballot_sync(0xffffffffu, le));  // lanes 0..c-1 passed (positions are sorted)
    if (c > 0) {
      const int nlo = lo + (c - 1) * step + 1;
      hi = min(hi, lo + c * step);
      lo = nlo;
    } else {
      hi = min(hi, lo);
    }
  }
  return lo;
}

// Row max of 128 scores over eight independent chains of 3-input maxima.
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
  for (int c = 24; c < 120; c += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + i], s[c + 8 + i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], s[120 + i]);
  return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
}

// One row of e4m3 softmax weights P = exp2(S * c*log2e - mb), sixteen keys per
// 16-byte chunk of the swizzled K-major P tile (prow = this row's 128-byte
// line); returns their sum, taken on four fp32 pairs (pair k holds
// accumulators 2k and 2k+1).
__device__ __forceinline__ float weights_e4m3(const float (&s)[128], float sl2, float mb, uint8_t* prow, int row) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2), nmbx2 = f2_pack(-mb, -mb);
  uint64_t accp[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) accp[k] = f2_pack(0.f, 0.f);
#pragma unroll
  for (int c16 = 0; c16 < 8; ++c16) {
    float e[16];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(s[c16 * 16 + i], s[c16 * 16 + i + 1]), sl2x2, nmbx2), x0, x1);
      e[i] = fast_exp2(x0);
      e[i + 1] = fast_exp2(x1);
      accp[(i >> 1) & 3] = f2_add(accp[(i >> 1) & 3], f2_pack(e[i], e[i + 1]));
    }
    uint4 v;
    v.x = (uint32_t)pack_e4m3x2(e[0], e[1]) | ((uint32_t)pack_e4m3x2(e[2], e[3]) << 16);
    v.y = (uint32_t)pack_e4m3x2(e[4], e[5]) | ((uint32_t)pack_e4m3x2(e[6], e[7]) << 16);
    v.z = (uint32_t)pack_e4m3x2(e[8], e[9]) | ((uint32_t)pack_e4m3x2(e[10], e[11]) << 16);
    v.w = (uint32_t)pack_e4m3x2(e[12], e[13]) | ((uint32_t)pack_e4m3x2(e[14], e[15]) << 16);
    *reinterpret_cast<uint4*>(prow + ((c16 ^ (row & 7)) << 4)) = v;
  }
  float acc[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) f2_unpack(accp[k], acc[2 * k], acc[2 * k + 1]);
  return ((acc[0] + acc[2]) + (acc[4] + acc[6])) + ((acc[1] + acc[3]) + (acc[5] + acc[7]));
}

// Warpgroup-wide change of the per-thread register budget (PTX setmaxnreg);
// each call sits at the top of its warpgroup's role branch.
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// K/V ring order.  K runs one tile ahead of V: K0, K1, V0, K2, V1, ...,
// K_{n-1}, V_{n-2}, V_{n-1}, matching the MMA order S(j) then PV(j-1), so
// slots are consumed and released first in, first out.
__device__ __forceinline__ int ring_pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int ring_pos_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

// S_t = Q_t K_j^T over head_dim, both operands K-major: bf16 eight k-steps of
// 16 (two boxes), e4m3 four k-steps of 32 (one box).
template <bool FP8>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint64_t a0, uint64_t b0) {
#pragma unroll
  for (int kk = 0; kk < Cfg<FP8>::KSTEPS; ++kk) {
    const uint64_t o = (uint64_t)(((kk >> 2) * HALF + (kk & 3) * 32) >> 4);
    if constexpr (FP8)
      tc_mma_fp8_warp(d_tmem, a0 + o, b0 + o, IDESC_FP8, kk > 0 ? 1u : 0u);
    else
      tc_mma_bf16_warp(d_tmem, a0 + o, b0 + o, IDESC_QK, kk > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V_j.  bf16: eight k-steps of 16 tokens; P K-major, V MN-major
// (16 tokens = two 8-row swizzle atoms = 2048 bytes).  e4m3: four k-steps of
// 32 tokens; P and V^T both K-major.
template <bool FP8>
__device__ __forceinline__ void mma_values(uint32_t d_tmem, uint64_t a0, uint64_t b0, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < Cfg<FP8>::KSTEPS; ++kk) {
    const uint64_t o = (uint64_t)(((kk >> 2) * HALF + (kk & 3) * 32) >> 4);
    if constexpr (FP8)
      tc_mma_fp8_warp(d_tmem, a0 + o, b0 + o, IDESC_FP8, (accumulate || kk > 0) ? 1u : 0u);
    else
      tc_mma_bf16_warp(d_tmem, a0 + o, b0 + (uint64_t)(kk * (2048 >> 4)), IDESC_PV,
                       (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <bool PAGED, bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  using C = Cfg<FP8>;
  constexpr int TILE = C::TILE, OFF_Q = C::OFF_Q, OFF_KV = C::OFF_KV, OFF_P = C::OFF_P, OFF_BAR = C::OFF_BAR;
  constexpr int NSLOT = C::NSLOT, PBUF = C::PBUF, NBAR = C::NBAR;

  // Work item: query head h, pair of 128-row query tiles (longest first), sequence b.
  const int h = p.h_lo + blockIdx.x;
  const int pair = gridDim.y - 1 - blockIdx.y;
  const int b = blockIdx.z;
  const int q_beg = p.cu_q[b];
  const int Sq = p.cu_q[b + 1] - q_beg;
  const int q0 = pair * 2 * BM;
  if (q0 >= Sq) return;  // the whole CTA leaves together
  const int g = h / (p.hq / p.hkv);
  int k_beg = 0, Sk;
  if (PAGED) {
    Sk = p.k_lens[b];
  } else {
    k_beg = p.cu_k[b];
    Sk = p.cu_k[b + 1] - k_beg;
  }
  // e4m3 V^T tiles are addressed by key index in the innermost (byte)
  // dimension, which a TMA copy needs at a multiple of 16: the whole CTA leaves,
  // before any barrier or TMEM is set up, if the sequence does not start there.
  if (FP8 && (k_beg & 15)) {
    if (threadIdx.x == 0) record_error(p.err, DEV_FP8_ALIGN);
    return;
  }

  Smem sm;
  uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
  sm.q_full = bars;
  sm.k_full = sm.q_full + 2;
  sm.v_full = sm.k_full + NSLOT;
  sm.kv_empty = sm.v_full + NSLOT;
  sm.s_full = sm.kv_empty + NSLOT;
  sm.s_free = sm.s_full + 2;
  sm.p_full = sm.s_free + 2;
  sm.o_done = sm.p_full + 2 * PBUF;
  sm.q_rot = sm.o_done + 2 * PBUF;
  sm.tmem_slot = (uint32_t*)(bars + NBAR);
  sm.nkv = (int*)(sm.tmem_slot + 4);
  sm.nfull = sm.nkv + 2;

  if (warp == WARP_IDLE) {
    // Per query tile: K/V tiles needed (keys up to the tile's last position) and
    // leading tiles visible in full to every row (keys up to its first position);
    // only tiles in between need the per-element mask.  Lane c < 4 handles count
    // c (tile c / 2; its last row if c is even, its first row if odd), so the
    // four counts' loads are in flight together.  It touches no barrier, so it
    // runs before the barriers are even set up.
    const int c = lane & 3, t = c >> 1;
    const int r0 = q0 + t * BM;
    const bool rows = r0 < Sq;
    int qp = 0, cnt = 0;
    if (rows && p.causal) {
      qp = __ldg(p.q_pos + q_beg + ((c & 1) ? r0 : min(r0 + BM, Sq) - 1));
      const int first = (!PAGED && Sk > 0) ? __ldg(p.k_pos + k_beg) : 0;  // in flight with qp
      cnt = PAGED ? max(0, min(Sk, qp + 1)) : count_le_guess(p.k_pos + k_beg, Sk, first, qp);
    } else if (rows) {
      cnt = Sk;
    }
    for (int cc = 0; cc < 4; ++cc) {  // the rare counts whose guess failed, by the whole warp
      const int got = __shfl_sync(0xffffffffu, cnt, cc);
      if (got < 0) {
        const int v = count_le_warp(p.k_pos + k_beg, Sk, __shfl_sync(0xffffffffu, qp, cc), lane);
        if (c == cc) cnt = v;
      }
    }
    const int cnt_first = __shfl_sync(0xffffffffu, cnt, lane | 1);  // the same tile's first-row count
    if (lane == 0 || lane == 2) {
      sm.nkv[t] = (cnt + BN - 1) / BN;
      sm.nfull[t] = cnt_first / BN;
    }
  }
  if (warp == WARP_MMA_S) tmem_alloc(sm.tmem_slot, TMEM_COLS);
  // K or V tile j into ring slot `slot` (TMA, completion on k_full[slot] or v_full[slot]).
  const int32_t* table = PAGED ? p.page_table + (int64_t)b * p.max_pages : nullptr;
  auto load_kv = [&](int slot, bool is_v, int j) {
    const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
    uint8_t* dst = smem + OFF_KV + slot * TILE;
    uint64_t* full = is_v ? &sm.v_full[slot] : &sm.k_full[slot];
    mbar_arrive_expect_tx(full, TILE);
    if (FP8 && is_v) {  // V^T codes [hkv][128][keys]: one box of 128 keys x 128 dims
      tma_load_3d(dst, tm, full, k_beg + j * BN, 0, g);
    } else if (!PAGED) {
      for (int hf = 0; hf < C::NBOX; ++hf)
        tma_load_3d(dst + hf * HALF, tm, full, hf * 64, g, k_beg + j * BN);
    } else {
      for (int pp = 0; pp < 2; ++pp) {  // two 64-token pages per tile
        const int lp = j * 2 + pp;
        int pid = lp < p.max_pages ? table[lp] : -1;
        if (pid < 0 || pid >= p.num_pages) {
          if (lp * 64 < Sk) record_error(p.err, DEV_BAD_PAGE);
          pid = 0;  // tokens past Sk are masked; keep the byte count whole
        }
        const int row0 = (int)(((int64_t)g * p.num_pages + pid) * 64);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(dst + hf * HALF + pp * (HALF / 2), tm, full, hf * 64, row0);
      }
    }
  };
  // The producer sets the barriers up itself and requests the Q tiles and K_0
  // at once: none of them depends on the K/V extent, which warp 11 may still
  // be working out.  K_0 is load 0 of the ring whenever any key is visible; if
  // none is, the producer still waits for it before exiting.  The __syncthreads
  // below publishes the initialised barriers to every other role.
  const bool k0_early = Sk > 0;
  if (warp == WARP_TMA && lane == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.q_full[t], 1);
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.s_free[t], 128);
      for (int b = 0; b < PBUF; ++b) {
        mbar_init(&sm.p_full[t * PBUF + b], 128);
        mbar_init(&sm.o_done[t * PBUF + b], 1);
      }
      mbar_init(&sm.q_rot[t], 128);
    }
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int t = 0; t < 2; ++t) {
      if (q0 + t * BM >= Sq) continue;
      mbar_arrive_expect_tx(&sm.q_full[t], TILE);
      for (int hf = 0; hf < C::NBOX; ++hf)
        tma_load_3d(smem + OFF_Q + t * TILE + hf * HALF, &tm_q, &sm.q_full[t], hf * 64, h, q_beg + q0 + t * BM);
    }
    if (k0_early) load_kv(0, false, 0);
    // Q comes from HBM and its latency opens every CTA.  Blocks start in
    // launch order as SMs free up, so the block `wave` places later in that
    // order will likely start on some SM when a block of this wave ends: bring
    // its Q tiles into L2 now.
    const int64_t L = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    const int64_t Ln = L + p.wave;
    if (p.wave > 0 && Ln < (int64_t)gridDim.x * gridDim.y * gridDim.z) {
      const int xn = (int)(Ln % gridDim.x), yn = (int)((Ln / gridDim.x) % gridDim.y);
      const int bn = (int)(Ln / ((int64_t)gridDim.x * gridDim.y));
      const int qbn = __ldg(p.cu_q + bn), sqn = __ldg(p.cu_q + bn + 1) - qbn;
      const int q0n = (gridDim.y - 1 - yn) * 2 * BM;
      for (int t = 0; t < 2; ++t)
        if (q0n + t * BM < sqn)
          for (int hf = 0; hf < C::NBOX; ++hf) tma_prefetch_l2_3d(&tm_q, hf * 64, p.h_lo + xn, qbn + q0n + t * BM);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  const int nkv_a = sm.nkv[0], nkv_b = sm.nkv[1];
  const int nkv = max(nkv_a, nkv_b);

  if (warp >= 8) {
   if constexpr (FP8) regs_dec<REGS_SIDE>();
   if (warp == WARP_TMA) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Per slot (bit s): the parity of the K and of the V fills issued so far,
      // whether the last fill was a V tile, and whether the slot was used --
      // what the final drain needs to wait for each slot's last load.
      uint32_t kpar = 0, vpar = 0, lastv = 0, used = 0;
      auto note = [&](int i, bool is_v) {
        const uint32_t bit = 1u << (i % NSLOT);
        if (is_v) {
          vpar ^= bit;
          lastv |= bit;
        } else {
          kpar ^= bit;
          lastv &= ~bit;
        }
        used |= bit;
      };
      int issued = 0;
      if (k0_early) {
        note(0, false);
        issued = 1;
      }
      for (int i = issued; i < 2 * nkv; ++i) {
        // load i of the ring order (see ring_pos_k / ring_pos_v)
        bool is_v;
        int j;
        if (i == 0) {
          is_v = false, j = 0;
        } else if (i == 2 * nkv - 1) {
          is_v = true, j = nkv - 1;
        } else {
          is_v = !(i & 1), j = is_v ? (i >> 1) - 1 : (i + 1) >> 1;
        }
        const int slot = i % NSLOT;
        if (i >= NSLOT && !mbar_wait(&sm.kv_empty[slot], ((i / NSLOT) - 1) & 1, p.err, DEV_TIMEOUT_TMA)) break;
        load_kv(slot, is_v, j);
        note(i, is_v);
        issued = i + 1;
      }
      // Leave no copy in flight: wait (bounded) for the last load of each slot
      // (the phase of its kind's barrier that it completes has the parity of
      // that kind's fill count minus one) and for the Q tiles (loaded even
      // when a tile turns out to need no keys).
#pragma unroll
      for (int sl = 0; sl < NSLOT; ++sl) {
        if (!((used >> sl) & 1u)) continue;
        const bool v = (lastv >> sl) & 1u;
        mbar_wait(v ? &sm.v_full[sl] : &sm.k_full[sl], (((v ? vpar : kpar) >> sl) & 1u) ^ 1u, nullptr, 0);
      }
      for (int t = 0; t < 2; ++t)
        if (q0 + t * BM < Sq) mbar_wait(&sm.q_full[t], 0, nullptr, 0);
    }
  } else if (warp == WARP_MMA_S || warp == WARP_MMA_PV) {
    // ------------------------------------------------------------ MMA issuers
    // Two converged warps on different sub-partitions feed the tensor core:
    // warp 9 issues the scores S_t(j) = Q_t K_j^T, warp 10 the updates
    // O_t += P_t(j) V_j.  tcgen05.mma issue blocks once a few MMAs are queued,
    // so whatever an issuer does between its groups (barrier waits, fences,
    // commits) would leave the tensor core idle; with two issuers the other
    // one's MMAs fill that time.  Each accumulator still has a single issuer,
    // so its MMAs run in program order and results do not depend on how the
    // two streams interleave.  The K/V ring holds K0, K1, V0, K2, V1, ..., so
    // each softmax has from the end of S_t(j) until PV_t(j) -- which follows
    // S_t(j+1) -- to produce P_t(j).  P lives in shared memory, so S_t(j+1) may
    // overwrite S_t in TMEM while P_t(j) still waits for its PV.
    if (nkv > 0) {
      // Warp-uniform bounded waits, so every elect.sync below sees all 32 lanes.
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.err, DEV_TIMEOUT_MMA));
      };
      // Descriptors of every tile base; a k-step adds a constant byte offset
      // (>> 4) to the 14-bit start-address field, which never carries out of it
      // because shared-memory addresses stay below 256 KB.
      constexpr uint64_t kTile16 = TILE >> 4;
      if (warp == WARP_MMA_S) {
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t)
          if (sm.nkv[t] > 0) ok = wait(p.q_cs ? &sm.q_rot[t] : &sm.q_full[t], 0);
        tc_fence_after();
        const uint64_t dQ = sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
        const uint64_t dK = sdesc_sw128(smem_u32(smem + OFF_KV), 16, 1024);
        uint32_t kph = 0;  // bit s: parity of the next K fill of slot s
        for (int j = 0; j < nkv && ok; ++j) {
          const int iK = ring_pos_k(j), slotK = iK % NSLOT;
          if (!(ok = wait(&sm.k_full[slotK], (kph >> slotK) & 1u))) break;
          kph ^= 1u << slotK;
          tc_fence_after();
          // S_t(j) overwrites S_t(j-1) in TMEM only after the softmax has
          // signalled (s_free) that S_t(j-1) is in its registers.
          for (int t = 0; t < 2; ++t) {
            if (j >= (t ? nkv_b : nkv_a)) continue;
            if (j > 0) {
              if (!(ok = wait(&sm.s_free[t], (j - 1) & 1))) break;
              tc_fence_after();
            }
            mma_scores<FP8>(tmem + t * BN, dQ + t * kTile16, dK + slotK * kTile16);
            tc_commit_warp(&sm.s_full[t]);
          }
          if (!ok) break;
          tc_commit_warp(&sm.kv_empty[slotK]);  // K_j consumed
        }
      } else {
        const uint64_t dP = sdesc_sw128(smem_u32(smem + OFF_P), 16, 1024);
        const uint64_t dV = sdesc_sw128(smem_u32(smem + OFF_KV), FP8 ? 16 : HALF, 1024);
        bool ok = true;
        uint32_t vph = 0;  // bit s: parity of the next V fill of slot s
        for (int j = 0; j < nkv && ok; ++j) {
          const int iV = ring_pos_v(j, nkv), slotV = iV % NSLOT;
          if (!(ok = wait(&sm.v_full[slotV], (vph >> slotV) & 1u))) break;
          vph ^= 1u << slotV;
          tc_fence_after();
          for (int t = 0; t < 2; ++t) {
            if (j >= (t ? nkv_b : nkv_a)) continue;
            if (!(ok = wait(&sm.p_full[t * PBUF + j % PBUF], (j / PBUF) & 1))) break;
            tc_fence_after();
            mma_values<FP8>(tmem + 2 * BN + t * D, dP + (t * PBUF + j % PBUF) * kTile16, dV + slotV * kTile16,
                            j > 0);
            tc_commit_warp(&sm.o_done[t * PBUF + j % PBUF]);
          }
          if (!ok) break;
          tc_commit_warp(&sm.kv_empty[slotV]);  // V_j consumed
        }
      }
    }
   }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    if constexpr (FP8) regs_inc<REGS_SOFTMAX>();
    const int t = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const int rq = q0 + t * BM + row;  // row index inside the sequence
    const bool rv = rq < Sq;
    const int qp = rv ? p.q_pos[q_beg + rq] : 0;
    const int nkv_t = sm.nkv[t];
    const int nfull_t = sm.nfull[t];
    // score = c_row * (MMA output): the softmax scale, times the query row's and
    // the key head's e4m3 scales when the inputs are codes.  A zero scale (an
    // all-zero group, whose codes are all zero) makes every score 0; c_row is
    // kept at least FLT_MIN so that masked scores (-inf) still give weight 0.
    const float c_row = FP8 ? fmaxf(p.scale * (rv ? __ldg(p.q_scale + (int64_t)(q_beg + rq) * p.hq + h) : 0.f) *
                                        __ldg(p.k_scale + g),
                                    FLT_MIN)
                            : p.scale;
    const float sl2 = c_row * 1.4426950408889634f;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * BN;
    const uint32_t tO = tmem + lane_base + 2 * BN + t * D;
    uint8_t* const prow0 = smem + OFF_P + t * PBUF * TILE + (row >> 3) * 1024 + (row & 7) * 128;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;

    if (!FP8 && p.q_cs && nkv_t > 0) {
      // RoPE of the query, fused: the warp rotates its 32 rows of Q_t in shared
      // memory with the same cos/sin and the same rounding as rope_apply, so the
      // scores are those of rope_apply followed by this kernel, bit for bit.
      // Lane l takes pairs 2l and 2l+1 (dims 2l, 2l+1 with partners 64+2l,
      // 65+2l) of every row, so each table load reads one row's 512 bytes
      // contiguously across the warp; the loads are issued before Q lands.
      const int r_first = wq * 32;
      const int nrows = max(0, min(32, Sq - (q0 + t * BM + r_first)));
      const float4* src = p.q_cs + (int64_t)(q_beg + q0 + t * BM + r_first) * 32 + lane;
      float4 tab[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nrows) tab[i] = __ldg(src + i * 32);
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full[t], 0, p.err, DEV_TIMEOUT_SOFTMAX));
      if (ok) {
        const int chunk = lane >> 2, within = (lane & 3) * 4;  // dims 2l, 2l+1: chunk l/4, bytes 4(l%4)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i >= nrows) break;
          const int rr = r_first + i;
          uint8_t* qrow = smem + OFF_Q + t * TILE + (rr >> 3) * 1024 + (rr & 7) * 128 + ((chunk ^ (rr & 7)) << 4) +
                          within;
          uint32_t* p1 = reinterpret_cast<uint32_t*>(qrow);
          uint32_t* p2 = reinterpret_cast<uint32_t*>(qrow + HALF);
          const uint32_t u1 = *p1, u2 = *p2;
          float y0, y1, z0, z1;
          rope_rotate(__uint_as_float(u1 << 16), __uint_as_float(u2 << 16), tab[i].x, tab[i].y, y0, z0);
          rope_rotate(__uint_as_float(u1 & 0xffff0000u), __uint_as_float(u2 & 0xffff0000u), tab[i].z, tab[i].w, y1,
                      z1);
          *p1 = pack_bf16x2(y0, y1);
          *p2 = pack_bf16x2(z0, z1);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.q_rot[t]);
    }

    for (int j = 0; j < nkv_t && ok; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], j & 1, p.err, DEV_TIMEOUT_SOFTMAX));
      if (!ok) break;
      tc_fence_after();
      uint8_t* const prow = prow0 + (j % PBUF) * TILE;
      // Scores: one row of S_t (128 fp32) per thread, in one TMEM load.
      float s[128];
      float mx[8];
      {
        uint32_t sr[128];
        tmem_ld128(tS, sr);
        tmem_wait_ld();
        tmem_regs_ready128(sr);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      }
      tc_fence_before();
      mbar_arrive(&sm.s_free[t]);  // S_t may now be overwritten by S_t(j+1)
      if (!FP8 && j < nfull_t) {  // no mask on this tile: reduce the first half right away
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
        for (int c = 24; c < 64; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + i], s[c + 8 + i]);
      }

      // Causal mask by absolute position, and keys past the sequence: only the
      // tiles from nfull_t on (the diagonal band and a ragged last tile).  Rows
      // past the sequence compute values that are never stored.
      if (j >= nfull_t) {
        const int key0 = j * BN;
        if (PAGED) {  // cached token j sits at position j: one bound per row
          const int lim = (p.causal ? min(qp, Sk - 1) : Sk - 1) - key0;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) s[c] = -INFINITY;
        } else {  // positions are sorted: the visible keys of the tile are a prefix
          const int n = min(BN, Sk - key0);
          int lim = n - 1;
          if (p.causal) {
            const int32_t* kp = p.k_pos + k_beg + key0;
            int lo = 0, hi = n;  // count of keys with position <= qp
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (__ldg(kp + mid) <= qp)
                lo = mid + 1;
              else
                hi = mid;
            }
            lim = lo - 1;
          }
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
      }

      float alpha = 1.f;
      bool any_grow = false;
      // The e4m3 kernel checks its reference lazily: once every row of the
      // warp has one (its first tile with a visible key), the weights are
      // computed against the reference as it stands, with no row-max pass; the
      // tile's weight sum bounds every weight, and only a sum above
      // kLazySumFp8 sends the warp back for the row max, a new reference, an O
      // rescale and a second pass.  Until then -- and always in the bf16
      // kernel -- the row max comes first and moves the reference when it
      // grows by more than 2^8 in exp2 units.  Either way every weight stays
      // <= 2^8, and the final O / l is exact for whatever reference was used.
      const bool need_ref = !FP8 || __any_sync(0xffffffffu, m_ref == -INFINITY);
      if (need_ref) {
        float mt;
        if constexpr (FP8) {
          mt = row_max128(s);
        } else {
          if (j >= nfull_t) {  // masked tile: the first half was not reduced yet
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
            for (int c = 24; c < 64; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + i], s[c + 8 + i]);
          }
#pragma unroll
          for (int c = 64; c < 128; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + i], s[c + 8 + i]);
          mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        }
        const float m_new = fmaxf(m_ref, mt);
        const bool grow = (m_new - m_ref) * sl2 > kRescaleLog2;  // false when both are -inf
        any_grow = __any_sync(0xffffffffu, grow);
        if (any_grow && m_new > m_ref) {
          alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2((m_ref - m_new) * sl2);
          l *= alpha;
          m_ref = m_new;
        }
      }

      // P_t's buffer j % PBUF is free once O_t += P_t V finished for tile
      // j - PBUF (its barrier o_done[t][j % PBUF] completes once per use).
      if (j >= PBUF) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_done[t * PBUF + j % PBUF], (j / PBUF - 1) & 1, p.err,
                                               DEV_TIMEOUT_SOFTMAX));
        if (!ok) break;
        tc_fence_after();
      }
      float tsum;
      if constexpr (!FP8) {
        // P = exp2(S * scale*log2e - m*scale*log2e), bf16, into the swizzled
        // K-major tile.  The affine step runs on fp32 pairs; the row sum on
        // eight scalar accumulators (key i goes to accumulator i mod 8), which
        // measured faster than paired adds and gives the same sums.
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref * sl2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nmbx2 = f2_pack(-mb, -mb);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
          float e[8];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[c8 * 8 + i], s[c8 * 8 + i + 1]), sl2x2, nmbx2), x0, x1);
            e[i] = fast_exp2(x0);
            e[i + 1] = fast_exp2(x1);
            acc[i] += e[i];
            acc[i + 1] += e[i + 1];
          }
          uint4 v;
          v.x = pack_bf16x2(e[0], e[1]);
          v.y = pack_bf16x2(e[2], e[3]);
          v.z = pack_bf16x2(e[4], e[5]);
          v.w = pack_bf16x2(e[6], e[7]);
          *reinterpret_cast<uint4*>(prow + (c8 >> 3) * HALF + (((c8 & 7) ^ (row & 7)) << 4)) = v;
        }
        tsum = ((acc[0] + acc[2]) + (acc[4] + acc[6])) + ((acc[1] + acc[3]) + (acc[5] + acc[7]));
      } else {
        for (int pass = 0;; ++pass) {
          tsum = weights_e4m3(s, sl2, (m_ref == -INFINITY) ? 0.f : m_ref * sl2, prow, row);
          if (need_ref || pass > 0) break;
          const bool over = !(tsum <= kLazySumFp8);  // also true for inf and NaN
          if (!__any_sync(0xffffffffu, over)) break;
          const float m_new = fmaxf(m_ref, row_max128(s));
          const bool grew = m_new > m_ref;
          if (grew) {
            alpha = fast_exp2((m_ref - m_new) * sl2);
            l *= alpha;
            m_ref = m_new;
          }
          any_grow = __any_sync(0xffffffffu, grew);
        }
      }
      l += tsum;
      if (any_grow && j > 0) {
        // O_t *= alpha in TMEM, once the last O_t += P_t V finished (with one
        // P buffer the wait above already covered it).  tcgen05.st reads its
        // source registers asynchronously, so all four chunks keep their own
        // registers until the single wait::st.
        if (PBUF > 1) {
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_done[t * PBUF + (j - 1) % PBUF], ((j - 1) / PBUF) & 1, p.err,
                                                 DEV_TIMEOUT_SOFTMAX));
          if (!ok) break;
          tc_fence_after();
        }
        uint32_t o[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tO + c * 32, o[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_regs_ready(o[c]);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[c][i] = __float_as_uint(__uint_as_float(o[c][i]) * alpha);
          tmem_st32(tO + c * 32, o[c]);
        }
        tmem_wait_st();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_regs_ready(o[c]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.p_full[t * PBUF + j % PBUF]);
    }

    // epilogue: O / l to global memory, LSE = scale * m + ln l
    if (ok && nkv_t > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_done[t * PBUF + (nkv_t - 1) % PBUF], ((nkv_t - 1) / PBUF) & 1,
                                             p.err, DEV_TIMEOUT_SOFTMAX));
      tc_fence_after();
    }
    const bool have_o = ok && nkv_t > 0;
    const float inv = l > 0.f ? (FP8 ? __ldg(p.v_scale + g) : 1.f) / l : 0.f;
    const int64_t orow = ((int64_t)(q_beg + rq) * p.hq + h) * D;
    // The bf16 kernel's output goes through shared memory the tile no longer
    // reads, then out whole rows per warp store instruction; stored straight
    // from each thread's row, a warp instruction would touch 32 rows (that
    // cost 4% of the kernel with bf16 output).
    //  - bf16 output: the two 16 KB boxes of Q_t hold dims 0-63 and 64-127 of
    //    each row as 128-byte rows, 16-byte chunks XOR-swizzled by row; a warp
    //    instruction stores two 256-byte rows.
    //  - fp32 output (partials for a merge): Q_t (32 KB) holds dims 0-63 and
    //    P_t (32 KB, free once the last P V finished) dims 64-127, as 256-byte
    //    rows swizzled by row; a warp instruction stores one 512-byte row.
    // (In the e4m3 kernel the tiles are half the size, and staging bf16 output
    // measured slower.)
    constexpr bool kStage = !FP8;
    const bool stage = kStage;
    uint8_t* const stg0 = smem + OFF_Q + t * TILE;
    uint8_t* const stg1 = p.out_f32 ? smem + OFF_P + t * PBUF * TILE : stg0 + HALF;
    // a tile that saw no key had no score MMA wait for its Q: let that copy land first
    if (stage && nkv_t == 0 && q0 + t * BM < Sq)
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full[t], 0, p.err, DEV_TIMEOUT_SOFTMAX)) && ok;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
        tmem_regs_ready(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (p.out_f32) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                       __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
          const int k = c * 8 + i;  // 16-byte chunk of the 512-byte row, 0..31
          if (stage)
            *reinterpret_cast<float4*>((k < 16 ? stg0 : stg1) + row * 256 + (((k & 15) ^ (row & 15)) << 4)) = v;
          else if (rv)
            reinterpret_cast<float4*>((float*)p.out + orow)[k] = v;
        }
      } else if (stage || rv) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
          const int k = c * 4 + i;  // 16-byte chunk of the row, 0..15
          if (stage)
            *reinterpret_cast<uint4*>((k < 8 ? stg0 : stg1) + row * 128 + (((k & 7) ^ (row & 7)) << 4)) = v;
          else
            reinterpret_cast<uint4*>((__nv_bfloat16*)p.out + orow)[k] = v;
        }
      }
    }
    if (stage) {
      __syncwarp();
      if (p.out_f32) {
        // the warp's 32 staged rows go out one 512-byte row per store instruction
#pragma unroll 4
        for (int r = wq * 32; r < wq * 32 + 32; ++r) {
          const float4 v = *reinterpret_cast<const float4*>((lane < 16 ? stg0 : stg1) + r * 256 +
                                                            (((lane & 15) ^ (r & 15)) << 4));
          const int rq_r = q0 + t * BM + r;
          if (rq_r < Sq) reinterpret_cast<float4*>((float*)p.out + ((int64_t)(q_beg + rq_r) * p.hq + h) * D)[lane] = v;
        }
      } else {
        // the warp's 32 staged rows go out two 256-byte rows per store instruction
        const int chunk = lane & 15;
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
          const int r = wq * 32 + 2 * it + (lane >> 4);
          const uint4 v =
              *reinterpret_cast<const uint4*>((chunk < 8 ? stg0 : stg1) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
          const int rq_r = q0 + t * BM + r;
          if (rq_r < Sq)
            reinterpret_cast<uint4*>((__nv_bfloat16*)p.out + ((int64_t)(q_beg + rq_r) * p.hq + h) * D)[chunk] = v;
        }
      }
    }
    if (rv && p.lse) p.lse[(int64_t)(q_beg + rq) * p.hq + h] = l > 0.f ? m_ref * c_row + logf(l) : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA_S) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace tc

namespace {

template <bool PAGED, bool FP8>
cudaError_t launch_variant(const tc::Params& p, dim3 grid, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t s) {
  // per device: raise the dynamic shared-memory limit once, and check the
  // compiled register count (384 threads fit on an SM only at <= 168 registers),
  // so a toolchain change shows up as an error, not a failed launch
  static int ready[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc::prefill_tc_kernel<PAGED, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Cfg<FP8>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, tc::prefill_tc_kernel<PAGED, FP8>);
    if (e != cudaSuccess) return e;
    // the e4m3 kernel's register split hands out exactly the launch total, so
    // it must be launched with 168 registers per thread
    if (FP8 ? fa.numRegs != tc::REGS_LAUNCH : fa.numRegs > tc::REGS_LAUNCH) return cudaErrorInvalidConfiguration;
    ready[dev] = 1;
  }
  tc::prefill_tc_kernel<PAGED, FP8><<<grid, tc::NTHREADS, tc::Cfg<FP8>::SMEM_BYTES, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillLaunch& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const bool paged = a.page_table != nullptr;
  if (a.fp8 && paged) return cudaErrorInvalidValue;
  if (a.max_seqlen_q == 0 || a.batch == 0 || a.h_hi == a.h_lo) return cudaSuccess;
  tc::Params p;
  p.cu_q = a.cu_q;
  p.q_pos = a.q_pos;
  p.cu_k = a.cu_k;
  p.k_pos = a.k_pos;
  p.page_table = a.page_table;
  p.k_lens = a.k_lens;
  p.out = a.out;
  p.lse = a.lse;
  p.err = a.err;
  p.num_pages = a.num_pages;
  p.max_pages = a.max_pages;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.h_lo = a.h_lo;
  p.causal = a.causal;
  p.out_f32 = a.out_f32;
  p.scale = a.scale;
  p.q_cs = reinterpret_cast<const float4*>(a.q_rope_cs);
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  {
    static int sms[64] = {};
    if (dev < 64 && sms[dev] == 0) {
      int n = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
      sms[dev] = n;
    }
    p.wave = dev < 64 ? sms[dev] : 0;
  }
  const int pairs = (a.max_seqlen_q + 2 * tc::BM - 1) / (2 * tc::BM);
  dim3 grid(a.h_hi - a.h_lo, pairs, a.batch);
  if (a.fp8) return launch_variant<false, true>(p, grid, tq, tk, tv, s);
  if (paged) return launch_variant<true, false>(p, grid, tq, tk, tv, s);
  return launch_variant<false, false>(p, grid, tq, tk, tv, s);
}

}  // namespace attn
