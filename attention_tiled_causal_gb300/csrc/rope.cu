// RoPE at absolute positions, in place (Ulysses page, sections 3.2 and 5.3).
//
// Each block takes NT consecutive tokens: it first computes their cos/sin
// tables (d/2 angles per token, once) into shared memory, then streams every
// head of those tokens.  A thread rotates one 16-byte vector of the first half
// of a head together with the matching vector of the second half; consecutive
// threads take consecutive vectors, so a warp covers whole 128-byte segments.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attn {

// The rotation frequencies as fractions of a turn per position step:
// theta_i = base^(-2i/d) / (2 pi), held as theta_i * 2^64 in a 64-bit integer
// (i < d/2 <= 128).  The angle of position p is then p * theta_i turns, and its
// fractional part -- all a rotation needs -- is the low 64 bits of the integer
// product p * turns[i], exactly.
struct InvFreq {
  uint64_t turns[128];
};

// theta_i in units of 2^-64 turns, from the fp64 frequency (53 significant
// bits; the product with a 32-bit position keeps the phase to about 2^-22
// relative, as an fp64 angle would).  base <= 0 gives 0: no rotation.
static InvFreq make_inv_freq(double base, int head_dim) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  InvFreq f;
  for (int i = 0; i < 128; ++i) f.turns[i] = 0;
  if (base > 0.0)
    for (int i = 0; i < head_dim / 2 && i < 128; ++i)
      f.turns[i] = (uint64_t)ldexp(pow(base, -2.0 * (double)i / (double)head_dim) / kTwoPi, 64);
  return f;
}

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

// The items w = w0, w0 + step, w0 + 2 step, ... of a block, where item w is
// chunk w % inner of row w / inner, and row r is head r % heads of token
// r / heads: the coordinates advance by constants, so the loop body does no
// integer division (three per item were most of these kernels' instructions).
struct GridWalk {
  int c, h, tt;
  int dc, dh, dt, inner, heads;
  __device__ __forceinline__ GridWalk(int w0, int step, int inner_, int heads_) : inner(inner_), heads(heads_) {
    c = w0 % inner;
    const int r = w0 / inner;
    h = r % heads;
    tt = r / heads;
    dc = step % inner;
    const int dr = step / inner;
    dh = dr % heads;
    dt = dr / heads;
  }
  __device__ __forceinline__ void next() {
    c += dc;
    const int carry = c >= inner;
    if (carry) c -= inner;
    h += dh + carry;  // < 2 heads
    tt += dt;
    if (h >= heads) {
      h -= heads;
      ++tt;
    }
  }
};

// sin and cos of p * base^(-2i/d) (turns = InvFreq::turns[i]).  The angle is
// reduced modulo one turn exactly, in integers; its top 32 bits, as a signed
// fraction of a turn in [-1/2, 1/2), go to sincospif.  No fp64 arithmetic,
// which runs at a small fraction of the fp32 rate on this GPU.  Every kernel
// that rotates takes its angles from here, so their results agree bit for bit.
__device__ __forceinline__ void pair_sincos(int32_t p, uint64_t turns, float& sn, float& cs) {
  const uint64_t phase = (uint64_t)(int64_t)p * turns;  // mod 2^64: the fraction of a turn
  const int32_t hi = (int32_t)(phase >> 32);            // turns * 2^32 in [-2^31, 2^31)
  sincospif((float)hi * 0x1p-31f, &sn, &cs);            // angle = 2 pi * turns
}

// The block's NT tokens' tables (cos and sin for i < d/2) in shared memory.
template <int NT = kTok, int W = 128>
__device__ __forceinline__ void angle_tables(float (*cs_s)[W], float (*sn_s)[W], int64_t t0, int64_t tokens,
                                             int half, const int32_t* __restrict__ pos, const InvFreq& f) {
  for (int i = threadIdx.x; i < NT * half; i += blockDim.x) {
    const int tt = i / half, ii = i % half;
    const int64_t t = t0 + tt;
    if (t < tokens) pair_sincos(__ldg(pos + t), f.turns[ii], sn_s[tt][ii], cs_s[tt][ii]);
  }
  __syncthreads();
}

// Rotates the heads of x and, when heads2 > 0, those of x2 at the same token
// positions (queries and keys in one launch): a token's rows are its heads of
// x, then its heads of x2, all sharing the block's angle tables.
template <typename T, int NT>
__global__ void __launch_bounds__(256) rope_kernel(T* __restrict__ x, int64_t tokens, int heads, int d,
                                                   int64_t stride_tok, T* __restrict__ x2, int heads2,
                                                   int64_t stride2, const int32_t* __restrict__ pos,
                                                   const InvFreq f) {
  constexpr int V = Vec<T>::N;
  __shared__ float cs_s[NT][128], sn_s[NT][128];
  const int half = d / 2;
  const int chunks = half / V;
  const int hall = heads + heads2;
  const int64_t t0 = (int64_t)blockIdx.x * NT;
  angle_tables<NT, 128>(cs_s, sn_s, t0, tokens, half, pos, f);
  const int items = NT * hall * chunks;
  GridWalk gw(threadIdx.x, blockDim.x, chunks, hall);
#pragma unroll 4
  for (int w = threadIdx.x; w < items; w += blockDim.x, gw.next()) {
    const int c = gw.c, h = gw.h, tt = gw.tt;
    const int64_t t = t0 + tt;
    if (t >= tokens) continue;
    T* p1 = (h < heads ? x + t * stride_tok + (int64_t)h * d : x2 + t * stride2 + (int64_t)(h - heads) * d) + c * V;
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
      float y1, y2;
      rope_rotate(x1, x2, cs, sn, y1, y2);
      from_f(y1, b1[e]);
      from_f(y2, b2[e]);
    }
    *reinterpret_cast<uint4*>(p1) = w1;
    *reinterpret_cast<uint4*>(p2) = w2;
  }
}

// New tokens' K and V into the head-major paged cache (SGLang page, sections
// 2.1-2.2), K rotated as rope_kernel rotates it.  Each block takes NT tokens:
// angle tables first, then per thread one 16-byte vector of the first half of
// a head's key and value rows with its partner vector of the second half (the
// key pair rotated), written to the cache rows and optionally the rotated keys
// to k_rot_out.  Slots are checked per token: -1 skips, out of range is
// recorded and skipped.  kv_append_staged_kernel below does the same per item
// with the rows staged in shared memory; this kernel serves the shapes whose
// staged groups would not fit.
template <int NT>
__global__ void __launch_bounds__(256, 4) kv_append_kernel(AppendLaunch a, const InvFreq f) {
  constexpr int V = 8;  // bf16 per 16-byte vector
  __shared__ float cs_s[NT][128], sn_s[NT][128];
  __shared__ int64_t slot_s[NT];
  const int d = a.head_dim, half = d / 2;
  const int64_t t0 = (int64_t)blockIdx.x * NT;
  const __nv_bfloat16* kn = (const __nv_bfloat16*)a.k_new;
  const __nv_bfloat16* vn = (const __nv_bfloat16*)a.v_new;
  __nv_bfloat16* kc = (__nv_bfloat16*)a.k_cache;
  __nv_bfloat16* vc = (__nv_bfloat16*)a.v_cache;
  __nv_bfloat16* ko = (__nv_bfloat16*)a.k_rot_out;
  // One item is one (token, head, chunk pair): chunk c of the first half of the
  // key and value rows with its partner chunk of the second half.  Items go in
  // batches of kB whose loads (four 16-byte vectors each) are all issued before
  // the first store: the compiler may not move loads above stores to memory it
  // cannot tell apart.  The first batch is requested before the slots and the
  // angle tables, which its loads do not need.
  const int chunks = half / V;
  const int items = NT * a.heads * chunks;
  constexpr int kB = 2;
  GridWalk gw(threadIdx.x, blockDim.x, chunks, a.heads);
  uint4 k1[kB], k2[kB], v1[kB], v2[kB];
  int64_t src[kB];
  int tts[kB], cc[kB], hh[kB];
  auto load_batch = [&](int w0) {
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      tts[u] = gw.tt;
      cc[u] = gw.c;
      hh[u] = gw.h;
      src[u] = -1;
      if (w0 + u * (int)blockDim.x < items && t0 + gw.tt < a.tokens) {
        src[u] = ((t0 + gw.tt) * a.heads + gw.h) * d + gw.c * V;
        k1[u] = __ldg(reinterpret_cast<const uint4*>(kn + src[u]));
        k2[u] = __ldg(reinterpret_cast<const uint4*>(kn + src[u] + half));
        v1[u] = __ldg(reinterpret_cast<const uint4*>(vn + src[u]));
        v2[u] = __ldg(reinterpret_cast<const uint4*>(vn + src[u] + half));
      }
      gw.next();
    }
  };
  load_batch(threadIdx.x);
  if (threadIdx.x < NT) {
    const int64_t t = t0 + threadIdx.x;
    int64_t sl = -1;
    if (t < a.tokens) {
      sl = __ldg(a.slots + t);
      if (sl < -1 || sl >= a.cache_rows) {
        record_error(a.err, DEV_BAD_SLOT);
        sl = -1;
      }
    }
    slot_s[threadIdx.x] = sl;
  }
  const bool rotate = a.base > 0.0;
  if (rotate) angle_tables<NT, 128>(cs_s, sn_s, t0, a.tokens, half, a.positions, f);
  __syncthreads();
  for (int w0 = threadIdx.x; w0 < items; w0 += kB * blockDim.x) {
    if (w0 != (int)threadIdx.x) load_batch(w0);
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      if (src[u] < 0) continue;
      const int64_t sl = slot_s[tts[u]];
      if (sl < 0) continue;
      const int64_t dst = ((int64_t)hh[u] * a.cache_rows + sl) * d + cc[u] * V;
      if (rotate) {
        const __nv_bfloat16* a1 = reinterpret_cast<const __nv_bfloat16*>(&k1[u]);
        const __nv_bfloat16* a2 = reinterpret_cast<const __nv_bfloat16*>(&k2[u]);
        uint4 w1, w2;
        __nv_bfloat16* b1 = reinterpret_cast<__nv_bfloat16*>(&w1);
        __nv_bfloat16* b2 = reinterpret_cast<__nv_bfloat16*>(&w2);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float cs = cs_s[tts[u]][cc[u] * V + e], sn = sn_s[tts[u]][cc[u] * V + e];
          float y1, y2;
          rope_rotate(to_f(a1[e]), to_f(a2[e]), cs, sn, y1, y2);
          from_f(y1, b1[e]);
          from_f(y2, b2[e]);
        }
        k1[u] = w1;
        k2[u] = w2;
      }
      *reinterpret_cast<uint4*>(kc + dst) = k1[u];
      *reinterpret_cast<uint4*>(kc + dst + half) = k2[u];
      *reinterpret_cast<uint4*>(vc + dst) = v1[u];
      *reinterpret_cast<uint4*>(vc + dst + half) = v2[u];
      if (ko) {
        *reinterpret_cast<uint4*>(ko + src[u]) = k1[u];
        *reinterpret_cast<uint4*>(ko + src[u] + half) = k2[u];
      }
    }
  }
}

// kv_append_kernel, for the shapes whose staged groups would not fit in 64 KB
// of shared memory.
static cudaError_t launch_kv_append_unstaged(const AppendLaunch& a, const InvFreq& f, cudaStream_t s) {
  // enough rows per block that the angle tables and the block's start-up are
  // amortised: 16 tokens for up to 16 heads, else 4
  if (a.heads <= 16) {
    const int64_t blocks = (a.tokens + 15) / 16;
    kv_append_kernel<16><<<(unsigned)blocks, 256, 0, s>>>(a, f);
  } else {
    const int64_t blocks = (a.tokens + kTok - 1) / kTok;
    kv_append_kernel<kTok><<<(unsigned)blocks, 256, 0, s>>>(a, f);
  }
  return cudaGetLastError();
}

// A thread's share of one (token, head) row of 128 values in the chunk-pair
// layout: chunk c (dims 8c..8c+7) of the first half and its RoPE partner chunk
// (dims 64+8c..64+8c+7) of the second half, as fp32.  Eight consecutive lanes
// hold a row.
struct RowChunk {
  float a[8], b[8];
};

__device__ __forceinline__ void load_chunk(const __nv_bfloat16* __restrict__ rowp, int c, bool ok, RowChunk& r) {
  uint4 u1 = make_uint4(0u, 0u, 0u, 0u), u2 = u1;
  if (ok) {
    u1 = __ldg(reinterpret_cast<const uint4*>(rowp + 8 * c));
    u2 = __ldg(reinterpret_cast<const uint4*>(rowp + 64 + 8 * c));
  }
  const uint32_t w1[4] = {u1.x, u1.y, u1.z, u1.w}, w2[4] = {u2.x, u2.y, u2.z, u2.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    r.a[e] = __uint_as_float((e & 1) ? (w1[e >> 1] & 0xffff0000u) : (w1[e >> 1] << 16));
    r.b[e] = __uint_as_float((e & 1) ? (w2[e >> 1] & 0xffff0000u) : (w2[e >> 1] << 16));
  }
}

// The raw 16-byte vectors of a chunk pair (chunk c of the first half of a
// 128-value row and its partner chunk of the second half), before widening.
struct RawPair {
  uint4 lo, hi;
};

// Loads the key and value chunk pairs of the walker's current item (token
// t0 + gw.tt, head gw.h, pair gw.c); tokens past the end read as zeros.
__device__ __forceinline__ void load_raw(const __nv_bfloat16* __restrict__ kn, const __nv_bfloat16* __restrict__ vn,
                                         int64_t t0, const GridWalk& gw, int heads, int64_t tokens, RawPair& k,
                                         RawPair& v) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  k.lo = k.hi = v.lo = v.hi = z;
  if (t0 + gw.tt < tokens) {
    const int64_t src = ((t0 + gw.tt) * heads + gw.h) * 128 + 8 * gw.c;
    k.lo = __ldg(reinterpret_cast<const uint4*>(kn + src));
    k.hi = __ldg(reinterpret_cast<const uint4*>(kn + src + 64));
    v.lo = __ldg(reinterpret_cast<const uint4*>(vn + src));
    v.hi = __ldg(reinterpret_cast<const uint4*>(vn + src + 64));
  }
}

__device__ __forceinline__ void unpack_chunk(const RawPair& p, RowChunk& r) {
  const uint32_t w1[4] = {p.lo.x, p.lo.y, p.lo.z, p.lo.w}, w2[4] = {p.hi.x, p.hi.y, p.hi.z, p.hi.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    r.a[e] = __uint_as_float((e & 1) ? (w1[e >> 1] & 0xffff0000u) : (w1[e >> 1] << 16));
    r.b[e] = __uint_as_float((e & 1) ? (w2[e >> 1] & 0xffff0000u) : (w2[e >> 1] << 16));
  }
}

// Rotates the chunk pair exactly as rope_kernel rotates it and rounds to bf16,
// the value rope_apply stores.  cs, sn: the token's 64 cos / sin values.
__device__ __forceinline__ void rotate_chunk(RowChunk& r, const float* cs_row, const float* sn_row, int c) {
  // the chunk's 8 cos and 8 sin values as four 16-byte shared loads
  const float4 ca = reinterpret_cast<const float4*>(cs_row)[2 * c], cb = reinterpret_cast<const float4*>(cs_row)[2 * c + 1];
  const float4 sa = reinterpret_cast<const float4*>(sn_row)[2 * c], sb = reinterpret_cast<const float4*>(sn_row)[2 * c + 1];
  const float cs[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
  const float sn[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float y1[2], y2[2];
    rope_rotate(r.a[e], r.b[e], cs[e], sn[e], y1[0], y2[0]);
    rope_rotate(r.a[e + 1], r.b[e + 1], cs[e + 1], sn[e + 1], y1[1], y2[1]);
    // round each pair to bf16 with one packed conversion, then widen back
    const uint32_t pa = pack_bf16x2(y1[0], y1[1]), pb = pack_bf16x2(y2[0], y2[1]);
    r.a[e] = __uint_as_float(pa << 16), r.a[e + 1] = __uint_as_float(pa & 0xffff0000u);
    r.b[e] = __uint_as_float(pb << 16), r.b[e + 1] = __uint_as_float(pb & 0xffff0000u);
  }
}

// rotate_chunk on packed pairs of lanes e, e + 1: y1 = x1 cos + RN(x2 * -sin)
// and y2 = x2 cos + RN(x1 sin), each one two-lane FMA after a two-lane
// product.  x2 * -sin is -(x2 * sin) exactly, so the bits are rope_rotate's.
// nsn_row: the token's sines with the sign flipped.
__device__ __forceinline__ void rotate_chunk_packed(RowChunk& r, const float* cs_row, const float* sn_row,
                                                    const float* nsn_row, int c) {
  const float4* c4 = reinterpret_cast<const float4*>(cs_row) + 2 * c;
  const float4* s4 = reinterpret_cast<const float4*>(sn_row) + 2 * c;
  const float4* n4 = reinterpret_cast<const float4*>(nsn_row) + 2 * c;
  const float4 ca = c4[0], cb = c4[1], sa = s4[0], sb = s4[1], na = n4[0], nb = n4[1];
  const uint64_t cs[4] = {f2_pack(ca.x, ca.y), f2_pack(ca.z, ca.w), f2_pack(cb.x, cb.y), f2_pack(cb.z, cb.w)};
  const uint64_t sn[4] = {f2_pack(sa.x, sa.y), f2_pack(sa.z, sa.w), f2_pack(sb.x, sb.y), f2_pack(sb.z, sb.w)};
  const uint64_t ns[4] = {f2_pack(na.x, na.y), f2_pack(na.z, na.w), f2_pack(nb.x, nb.y), f2_pack(nb.z, nb.w)};
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const uint64_t x1 = f2_pack(r.a[e], r.a[e + 1]), x2 = f2_pack(r.b[e], r.b[e + 1]);
    float y10, y11, y20, y21;
    f2_unpack(f2_fma(x1, cs[e >> 1], f2_mul(x2, ns[e >> 1])), y10, y11);
    f2_unpack(f2_fma(x2, cs[e >> 1], f2_mul(x1, sn[e >> 1])), y20, y21);
    const uint32_t pa = pack_bf16x2(y10, y11), pb = pack_bf16x2(y20, y21);
    r.a[e] = __uint_as_float(pa << 16), r.a[e + 1] = __uint_as_float(pa & 0xffff0000u);
    r.b[e] = __uint_as_float(pb << 16), r.b[e + 1] = __uint_as_float(pb & 0xffff0000u);
  }
}

// max |x| over the row (the eight lanes holding it).  Its shuffles take all 32
// lanes of the warp, so every caller runs it warp-uniformly.
__device__ __forceinline__ float chunk_amax(const RowChunk& r) {
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmax3(m, fabsf(r.a[e]), fabsf(r.b[e]));
#pragma unroll
  for (int o = 4; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// Symmetric int8 codes of the chunk pair: code = x / sc rounded to the nearest
// integer (ties to even) and clamped to [-127, 127], the quotient correctly
// rounded in fp32 (div_rn_recip for normal scales); 0 for a zero scale.  The
// quotient is rounded by adding 1.5 * 2^23: an fp32 add then rounds it to an
// integer, ties to even, whose two's complement is the low byte of the sum's
// bits, and three byte permutes pack four such bytes -- no conversion
// instruction and no shifts or masks per code.
//
// With sc = RN(amax / 127) >= (amax / 127)(1 - 2^-24) and |x| <= amax, the
// correctly rounded quotient is at most 127 (1 + 2^-24) rounded, 127 + 2^-17 <
// 127.5, so its nearest integer never leaves [-127, 127] and the fast path
// needs no clamp.  The full division (scales below 2^-90, where sc may be
// subnormal and carry a large relative error) clamps.
__device__ __forceinline__ uint32_t code_bits(float q) { return (uint32_t)__float_as_int(__fadd_rn(q, 12582912.0f)); }

// RN(m / 127), the row scale: div_rn_recip with RN(1/127) for maxima whose
// quotient is a normal number far from overflow (Markstein's conditions hold
// there), the division otherwise (zero, tiny, infinite or NaN maxima).
__device__ __forceinline__ float scale127(float m) {
  constexpr float kRcp127 = 0x1.020408p-7f;  // RN(1/127)
  return (m >= 0x1p-80f && m <= 0x1p120f) ? div_rn_recip(m, 127.0f, kRcp127) : m / 127.0f;
}

__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Fast path, two lanes per instruction: q = x rc, then div_rn_recip's one
// correction q + (x - q sc) rc with the remainder formed as fma(q, -sc, x) (the
// same exact value), then the rounding add.  nsc2 = (-sc, -sc), rc2 = (rc, rc).
__device__ __forceinline__ uint32_t int8x4_fast(const float* x, uint64_t nsc2, uint64_t rc2) {
  const uint64_t m2 = f2_pack(12582912.0f, 12582912.0f);
  uint32_t b[4];
#pragma unroll
  for (int e = 0; e < 4; e += 2) {
    const uint64_t xx = f2_pack(x[e], x[e + 1]);
    const uint64_t q = f2_mul(xx, rc2);
    float lo, hi;
    f2_unpack(f2_add(f2_fma(f2_fma(q, nsc2, xx), rc2, q), m2), lo, hi);
    b[e] = __float_as_uint(lo), b[e + 1] = __float_as_uint(hi);
  }
  return pack_low_bytes(b[0], b[1], b[2], b[3]);
}

// The full division, clamped, for scales below the fast path's range.
__device__ __forceinline__ uint32_t int8x4_full(const float* x, float sc) {
  uint32_t b[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) b[e] = code_bits(fminf(fmaxf(x[e] / sc, -127.0f), 127.0f));
  return pack_low_bytes(b[0], b[1], b[2], b[3]);
}

__device__ __forceinline__ void chunk_store_int8(const RowChunk& r, float sc, int8_t* row_codes, int c) {
  uint2 a = make_uint2(0u, 0u), b = a;
  if (sc >= kFastDivMinScale) {
    const float rc = __frcp_rn(sc);
    const uint64_t rc2 = f2_pack(rc, rc), nsc2 = f2_pack(-sc, -sc);
    a = make_uint2(int8x4_fast(r.a, nsc2, rc2), int8x4_fast(r.a + 4, nsc2, rc2));
    b = make_uint2(int8x4_fast(r.b, nsc2, rc2), int8x4_fast(r.b + 4, nsc2, rc2));
  } else if (sc != 0.0f) {
    a = make_uint2(int8x4_full(r.a, sc), int8x4_full(r.a + 4, sc));
    b = make_uint2(int8x4_full(r.b, sc), int8x4_full(r.b + 4, sc));
  }
  *reinterpret_cast<uint2*>(row_codes + 8 * c) = a;
  *reinterpret_cast<uint2*>(row_codes + 64 + 8 * c) = b;
}

// kv_append_kernel for an INT8 cache, in the chunk-pair layout.  One thread
// takes one (token, head, chunk pair) for both the key row and the value row:
// it issues the four 16-byte loads first, then rotates the key chunks (rounded
// to bf16 -- the value a bf16 cache would hold), takes each row's max |x| over
// the eight lanes that hold it, and writes both rows' codes, each row with one
// fp32 scale = max|x| / 127.  A block holds kAppendTok tokens, so each of its
// loops covers 32 * heads items: every warp takes whole rows and runs the loop
// as often as the others, as chunk_amax's shuffles require.  The launcher takes
// this kernel only where the staged one below does not apply (more than 64
// heads); both write the same bits.
constexpr int kAppendTok = 4;
__global__ void __launch_bounds__(256, 4) kv_append_int8_kernel(AppendLaunch a, const InvFreq f) {
  __shared__ __align__(16) float cs_s[kAppendTok][64], sn_s[kAppendTok][64];
  __shared__ int64_t slot_s[kAppendTok];
  const int64_t t0 = (int64_t)blockIdx.x * kAppendTok;
  const __nv_bfloat16* kn = (const __nv_bfloat16*)a.k_new;
  const __nv_bfloat16* vn = (const __nv_bfloat16*)a.v_new;
  __nv_bfloat16* ko = (__nv_bfloat16*)a.k_rot_out;
  const int items = kAppendTok * a.heads * 8;
  GridWalk gw(threadIdx.x, blockDim.x, 8, a.heads);
  // The first item's key and value chunks are requested before anything else:
  // they depend on neither the slots nor the angle tables.
  RawPair kraw, vraw;
  if (threadIdx.x < items) load_raw(kn, vn, t0, gw, a.heads, a.tokens, kraw, vraw);
  if (threadIdx.x < kAppendTok) {
    const int64_t t = t0 + threadIdx.x;
    int64_t sl = -1;
    if (t < a.tokens) {
      sl = __ldg(a.slots + t);
      if (sl < -1 || sl >= a.cache_rows) {
        record_error(a.err, DEV_BAD_SLOT);
        sl = -1;
      }
    }
    slot_s[threadIdx.x] = sl;
  }
  const bool rotate = a.base > 0.0;
  if (rotate) angle_tables<kAppendTok, 64>(cs_s, sn_s, t0, a.tokens, 64, a.positions, f);
  __syncthreads();
  for (int it = threadIdx.x; it < items; it += blockDim.x, gw.next()) {
    const int c = gw.c, tt = gw.tt, h = gw.h;
    if (it != (int)threadIdx.x) load_raw(kn, vn, t0, gw, a.heads, a.tokens, kraw, vraw);
    const int64_t sl = slot_s[tt];
    const bool ok = sl >= 0;  // tokens past the end carry slot -1
    const int64_t src = ((t0 + tt) * a.heads + h) * 128;
    RowChunk rk, rv;
    unpack_chunk(kraw, rk);
    unpack_chunk(vraw, rv);
    if (rotate) rotate_chunk(rk, cs_s[tt], sn_s[tt], c);
    if (ko && ok) {
      uint4 o1, o2;
      o1.x = pack_bf16x2(rk.a[0], rk.a[1]), o1.y = pack_bf16x2(rk.a[2], rk.a[3]);
      o1.z = pack_bf16x2(rk.a[4], rk.a[5]), o1.w = pack_bf16x2(rk.a[6], rk.a[7]);
      o2.x = pack_bf16x2(rk.b[0], rk.b[1]), o2.y = pack_bf16x2(rk.b[2], rk.b[3]);
      o2.z = pack_bf16x2(rk.b[4], rk.b[5]), o2.w = pack_bf16x2(rk.b[6], rk.b[7]);
      *reinterpret_cast<uint4*>(ko + src + 8 * c) = o1;
      *reinterpret_cast<uint4*>(ko + src + 64 + 8 * c) = o2;
    }
    const float sk = scale127(chunk_amax(rk));
    const float sv = scale127(chunk_amax(rv));
    if (ok) {
      const int64_t row = (int64_t)h * a.cache_rows + sl;
      chunk_store_int8(rk, sk, (int8_t*)a.k_cache + row * 128, c);
      chunk_store_int8(rv, sv, (int8_t*)a.v_cache + row * 128, c);
      if (c == 0) {
        a.k_scale[row] = sk;
        a.v_scale[row] = sv;
      }
    }
  }
}

// Contiguous global bytes into shared memory (cp.async.bulk), counted on bar.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// kv_append_int8_kernel with the new rows staged through shared memory.  A
// persistent block walks groups of G whole tokens, whose G * heads key rows
// (and value rows) are contiguous in k_new (v_new).  Its thread 0 copies each
// group into one of two buffers (two cp.async.bulk, counted on that buffer's
// mbarrier) as soon as the buffer is free, so while the block rotates and
// quantises one group the next one is already in flight.  Per item it writes
// the same bits as kv_append_int8_kernel; the key rotation runs on packed lane
// pairs (rotate_chunk_packed).
//
// Shared memory: four buffers of G * heads * 256 bytes (K and V of buffers 0
// and 1), then cos, sin and -sin tables [G][64] and the group's slots [G].
// The item loop runs over whole warps (chunk_amax's shuffles take all 32
// lanes); the lanes past G * heads * 8 items form whole 8-lane rows, take
// zeros and store nothing.  A copy that does not land within the wait limit
// records DEV_TIMEOUT_APPEND; the block then lets the copies it has in flight
// land (bounded) and returns.
__global__ void __launch_bounds__(256, 4) kv_append_int8_staged_kernel(AppendLaunch a, const InvFreq f, int G,
                                                                       int64_t groups) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t full[2];
  const int heads = a.heads;
  const uint32_t gbytes = (uint32_t)G * heads * 256;  // one group of K (or V)
  float (*cs_s)[64] = reinterpret_cast<float (*)[64]>(dsm + 4 * gbytes);
  float (*sn_s)[64] = cs_s + G;
  float (*nsn_s)[64] = sn_s + G;
  int64_t* slot_s = reinterpret_cast<int64_t*>(nsn_s + G);
  const char* kn = (const char*)a.k_new;
  const char* vn = (const char*)a.v_new;
  __nv_bfloat16* ko = (__nv_bfloat16*)a.k_rot_out;
  auto issue = [&](int64_t g, int b) {
    const int64_t t0 = g * G;
    const uint32_t bytes = (uint32_t)(min((int64_t)G, a.tokens - t0) * heads * 256);
    mbar_arrive_expect_tx(&full[b], 2 * bytes);
    bulk_copy_g2s(dsm + (2 * b) * gbytes, kn + t0 * heads * 256, bytes, &full[b]);
    bulk_copy_g2s(dsm + (2 * b + 1) * gbytes, vn + t0 * heads * 256, bytes, &full[b]);
  };
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    issue(blockIdx.x, 0);
    if (blockIdx.x + gridDim.x < groups) issue(blockIdx.x + gridDim.x, 1);
  }
  const int items = G * heads * 8;
  const int items_w = (items + 31) & ~31;
  const GridWalk gw0(threadIdx.x, blockDim.x, 8, heads);
  const bool rotate = a.base > 0.0;
  int i = 0;
  bool failed = false;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x, ++i) {
    const int b = i & 1;
    const int64_t t0 = g * G;
    if (threadIdx.x < G) {
      const int64_t t = t0 + threadIdx.x;
      int64_t sl = -1;
      if (t < a.tokens) {
        sl = __ldg(a.slots + t);
        if (sl < -1 || sl >= a.cache_rows) {
          record_error(a.err, DEV_BAD_SLOT);
          sl = -1;
        }
      }
      slot_s[threadIdx.x] = sl;
    }
    if (rotate)
      for (int j = threadIdx.x; j < G * 64; j += blockDim.x) {
        const int tt = j >> 6, ii = j & 63;
        if (t0 + tt < a.tokens) {
          float sn, cs;
          pair_sincos(__ldg(a.positions + t0 + tt), f.turns[ii], sn, cs);
          sn_s[tt][ii] = sn;
          nsn_s[tt][ii] = -sn;
          cs_s[tt][ii] = cs;
        }
      }
    // one barrier publishes the tables and slots and agrees on the wait
    if (!__syncthreads_and(mbar_wait_own(&full[b], (i >> 1) & 1))) {
      failed = true;
      break;
    }
    const uint8_t* kb = dsm + (2 * b) * gbytes;
    const uint8_t* vb = kb + gbytes;
    GridWalk gw = gw0;
    for (int it = threadIdx.x; it < items_w; it += blockDim.x, gw.next()) {
      const bool live = it < items;
      const int c = gw.c, tt = gw.tt, h = gw.h;
      const int64_t sl = live ? slot_s[tt] : -1;
      const bool ok = sl >= 0;  // tokens past the end carry slot -1
      RawPair kraw, vraw;
      kraw.lo = kraw.hi = vraw.lo = vraw.hi = make_uint4(0u, 0u, 0u, 0u);
      if (live) {
        const uint32_t off = (uint32_t)((tt * heads + h) * 256 + 16 * c);
        kraw.lo = *reinterpret_cast<const uint4*>(kb + off);
        kraw.hi = *reinterpret_cast<const uint4*>(kb + off + 128);
        vraw.lo = *reinterpret_cast<const uint4*>(vb + off);
        vraw.hi = *reinterpret_cast<const uint4*>(vb + off + 128);
      }
      RowChunk rk, rv;
      unpack_chunk(kraw, rk);
      unpack_chunk(vraw, rv);
      if (rotate && live) rotate_chunk_packed(rk, cs_s[tt], sn_s[tt], nsn_s[tt], c);
      if (ko && ok) {
        const int64_t src = ((t0 + tt) * heads + h) * 128;
        uint4 o1, o2;
        o1.x = pack_bf16x2(rk.a[0], rk.a[1]), o1.y = pack_bf16x2(rk.a[2], rk.a[3]);
        o1.z = pack_bf16x2(rk.a[4], rk.a[5]), o1.w = pack_bf16x2(rk.a[6], rk.a[7]);
        o2.x = pack_bf16x2(rk.b[0], rk.b[1]), o2.y = pack_bf16x2(rk.b[2], rk.b[3]);
        o2.z = pack_bf16x2(rk.b[4], rk.b[5]), o2.w = pack_bf16x2(rk.b[6], rk.b[7]);
        *reinterpret_cast<uint4*>(ko + src + 8 * c) = o1;
        *reinterpret_cast<uint4*>(ko + src + 64 + 8 * c) = o2;
      }
      const float sk = scale127(chunk_amax(rk));
      const float sv = scale127(chunk_amax(rv));
      if (ok) {
        const int64_t row = (int64_t)h * a.cache_rows + sl;
        chunk_store_int8(rk, sk, (int8_t*)a.k_cache + row * 128, c);
        chunk_store_int8(rv, sv, (int8_t*)a.v_cache + row * 128, c);
        if (c == 0) {
          a.k_scale[row] = sk;
          a.v_scale[row] = sv;
        }
      }
    }
    __syncthreads();  // buffer b, the tables and the slots are free again
    if (threadIdx.x == 0 && g + 2 * gridDim.x < groups) issue(g + 2 * gridDim.x, b);
  }
  if (failed && threadIdx.x == 0) {
    record_error(a.err, DEV_TIMEOUT_APPEND);
    for (int k = i; k < i + 2; ++k)
      if (blockIdx.x + (int64_t)k * gridDim.x < groups) mbar_wait_own(&full[k & 1], (k >> 1) & 1);
  }
}

// kv_append_kernel with the new rows staged through shared memory, as
// kv_append_int8_staged_kernel stages them: a persistent block walks groups of
// G whole tokens (contiguous in k_new and v_new), thread 0 keeping the next
// group's bytes in flight on one of two mbarriers while the block rotates the
// current group's keys and writes its rows to the cache.  Per item (a key and a
// value chunk pair) the arithmetic is kv_append_kernel's.  Shared memory: four
// buffers of G * heads * d * 2 bytes, then cos and sin tables [G][d/2] and the
// slots [G].
__global__ void __launch_bounds__(256, 4) kv_append_staged_kernel(AppendLaunch a, const InvFreq f, int G,
                                                                  int64_t groups) {
  constexpr int V = 8;  // bf16 per 16-byte vector
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint64_t full[2];
  const int heads = a.heads, d = a.head_dim, half = d / 2, chunks = half / V;
  const uint32_t rbytes = (uint32_t)d * 2;
  const uint32_t gbytes = (uint32_t)G * heads * rbytes;  // one group of K (or V)
  float* cs_s = reinterpret_cast<float*>(dsm + 4 * gbytes);  // [G][half]
  float* sn_s = cs_s + G * half;
  int64_t* slot_s = reinterpret_cast<int64_t*>(sn_s + G * half);
  const char* kn = (const char*)a.k_new;
  const char* vn = (const char*)a.v_new;
  __nv_bfloat16* kc = (__nv_bfloat16*)a.k_cache;
  __nv_bfloat16* vc = (__nv_bfloat16*)a.v_cache;
  __nv_bfloat16* ko = (__nv_bfloat16*)a.k_rot_out;
  auto issue = [&](int64_t g, int b) {
    const int64_t t0 = g * G;
    const uint32_t bytes = (uint32_t)(min((int64_t)G, a.tokens - t0) * heads * rbytes);
    mbar_arrive_expect_tx(&full[b], 2 * bytes);
    bulk_copy_g2s(dsm + (2 * b) * gbytes, kn + t0 * heads * rbytes, bytes, &full[b]);
    bulk_copy_g2s(dsm + (2 * b + 1) * gbytes, vn + t0 * heads * rbytes, bytes, &full[b]);
  };
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    issue(blockIdx.x, 0);
    if (blockIdx.x + gridDim.x < groups) issue(blockIdx.x + gridDim.x, 1);
  }
  const int items = G * heads * chunks;
  const GridWalk gw0(threadIdx.x, blockDim.x, chunks, heads);
  const bool rotate = a.base > 0.0;
  int i = 0;
  bool failed = false;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x, ++i) {
    const int b = i & 1;
    const int64_t t0 = g * G;
    if (threadIdx.x < G) {
      const int64_t t = t0 + threadIdx.x;
      int64_t sl = -1;
      if (t < a.tokens) {
        sl = __ldg(a.slots + t);
        if (sl < -1 || sl >= a.cache_rows) {
          record_error(a.err, DEV_BAD_SLOT);
          sl = -1;
        }
      }
      slot_s[threadIdx.x] = sl;
    }
    if (rotate)
      for (int j = threadIdx.x; j < G * half; j += blockDim.x) {
        const int tt = j / half, ii = j - tt * half;
        if (t0 + tt < a.tokens) pair_sincos(__ldg(a.positions + t0 + tt), f.turns[ii], sn_s[j], cs_s[j]);
      }
    if (!__syncthreads_and(mbar_wait_own(&full[b], (i >> 1) & 1))) {
      failed = true;
      break;
    }
    const uint8_t* kb = dsm + (2 * b) * gbytes;
    const uint8_t* vb = kb + gbytes;
    GridWalk gw = gw0;
    for (int it = threadIdx.x; it < items; it += blockDim.x, gw.next()) {
      const int c = gw.c, tt = gw.tt, h = gw.h;
      const int64_t sl = slot_s[tt];
      if (sl < 0) continue;  // tokens past the end and skipped slots
      const uint32_t off = (uint32_t)(tt * heads + h) * rbytes + 16u * c;
      uint4 k1 = *reinterpret_cast<const uint4*>(kb + off);
      uint4 k2 = *reinterpret_cast<const uint4*>(kb + off + half * 2);
      const uint4 v1 = *reinterpret_cast<const uint4*>(vb + off);
      const uint4 v2 = *reinterpret_cast<const uint4*>(vb + off + half * 2);
      if (rotate) {
        const __nv_bfloat16* a1 = reinterpret_cast<const __nv_bfloat16*>(&k1);
        const __nv_bfloat16* a2 = reinterpret_cast<const __nv_bfloat16*>(&k2);
        uint4 w1, w2;
        __nv_bfloat16* b1 = reinterpret_cast<__nv_bfloat16*>(&w1);
        __nv_bfloat16* b2 = reinterpret_cast<__nv_bfloat16*>(&w2);
        const float* cs = cs_s + tt * half + c * V;
        const float* sn = sn_s + tt * half + c * V;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          float y1, y2;
          rope_rotate(to_f(a1[e]), to_f(a2[e]), cs[e], sn[e], y1, y2);
          from_f(y1, b1[e]);
          from_f(y2, b2[e]);
        }
        k1 = w1;
        k2 = w2;
      }
      const int64_t dst = ((int64_t)h * a.cache_rows + sl) * d + c * V;
      *reinterpret_cast<uint4*>(kc + dst) = k1;
      *reinterpret_cast<uint4*>(kc + dst + half) = k2;
      *reinterpret_cast<uint4*>(vc + dst) = v1;
      *reinterpret_cast<uint4*>(vc + dst + half) = v2;
      if (ko) {
        const int64_t src = ((t0 + tt) * heads + h) * d + c * V;
        *reinterpret_cast<uint4*>(ko + src) = k1;
        *reinterpret_cast<uint4*>(ko + src + half) = k2;
      }
    }
    __syncthreads();  // buffer b, the tables and the slots are free again
    if (threadIdx.x == 0 && g + 2 * gridDim.x < groups) issue(g + 2 * gridDim.x, b);
  }
  if (failed && threadIdx.x == 0) {
    record_error(a.err, DEV_TIMEOUT_APPEND);
    for (int k = i; k < i + 2; ++k)
      if (blockIdx.x + (int64_t)k * gridDim.x < groups) mbar_wait_own(&full[k & 1], (k >> 1) & 1);
  }
}

// SMs of device dev, cached per device; 0 if they cannot be read.
static int device_sms(int dev) {
  static int sms[64] = {};
  if (dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) sms[dev] = n;
  }
  return sms[dev];
}

// Grid of a persistent staged kernel of 256 threads: its resident blocks for
// `smem` bytes of dynamic shared memory, at most `groups`; 0 if it does not
// fit.  The first call on a device raises the kernel's dynamic shared-memory
// limit to `max_smem` (attr_set: one flag per device, kept by the caller for
// its kernel).
static cudaError_t staged_grid(const void* kernel, bool (&attr_set)[64], size_t smem, size_t max_smem,
                               int64_t groups, int64_t& grid) {
  grid = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sms = device_sms(dev);
  if (sms == 0) return cudaSuccess;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem);
  if (e != cudaSuccess) return e;
  grid = std::min<int64_t>(groups, (int64_t)sms * per_sm);
  return cudaSuccess;
}

// Shared memory of kv_append_staged_kernel for G tokens per group.
static size_t staged_bf16_smem_bytes(int heads, int d, int G) {
  return (size_t)4 * G * heads * d * 2 + (size_t)2 * G * (d / 2) * sizeof(float) + (size_t)G * sizeof(int64_t);
}
constexpr size_t kStagedMaxSmem = 64 * 1024;

cudaError_t launch_kv_append(const AppendLaunch& a, cudaStream_t s) {
  const InvFreq f = make_inv_freq(a.base, a.head_dim);
  if (a.tokens == 0) return cudaSuccess;
  // G tokens per group: about one item (a key and a value chunk pair) per thread
  const int per_token = a.heads * (a.head_dim / 16);
  const int G = std::max(1, 256 / per_token);
  const size_t smem = staged_bf16_smem_bytes(a.heads, a.head_dim, G);
  if (smem <= kStagedMaxSmem) {
    static bool attr_set[64] = {};
    const int64_t groups = (a.tokens + G - 1) / G;
    int64_t grid = 0;
    const cudaError_t e =
        staged_grid((const void*)kv_append_staged_kernel, attr_set, smem, kStagedMaxSmem, groups, grid);
    if (e != cudaSuccess) return e;
    if (grid > 0) {
      kv_append_staged_kernel<<<(unsigned)grid, 256, smem, s>>>(a, f, G, groups);
      return cudaGetLastError();
    }
  }
  return launch_kv_append_unstaged(a, f, s);
}

// Heads the staged kernel takes: its four group buffers then stay within 64 KB.
constexpr int kStagedMaxHeads = 64;

static size_t staged_smem_bytes(int heads, int G) {
  return (size_t)4 * G * heads * 256 + (size_t)3 * G * 64 * sizeof(float) + (size_t)G * sizeof(int64_t);
}

cudaError_t launch_kv_append_int8(const AppendLaunch& a, cudaStream_t s) {
  const InvFreq f = make_inv_freq(a.base, 128);
  if (a.tokens == 0) return cudaSuccess;
  if (a.heads <= kStagedMaxHeads) {
    // G tokens per group: 32 rows (one item per thread) where the heads divide
    // into 32, else whole tokens below that; one token from 32 heads up.  The
    // group copies start at multiples of 256 bytes of k_new and v_new, whose
    // 16-byte alignment the C-ABI checks.
    static bool attr_set[64] = {};
    const int G = a.heads >= 32 ? 1 : 32 / a.heads;
    const int64_t groups = (a.tokens + G - 1) / G;
    const size_t smem = staged_smem_bytes(a.heads, G);
    int64_t grid = 0;
    const cudaError_t e = staged_grid((const void*)kv_append_int8_staged_kernel, attr_set, smem,
                                      staged_smem_bytes(kStagedMaxHeads, 1), groups, grid);
    if (e != cudaSuccess) return e;
    if (grid > 0) {
      kv_append_int8_staged_kernel<<<(unsigned)grid, 256, smem, s>>>(a, f, G, groups);
      return cudaGetLastError();
    }
  }
  const int64_t blocks = (a.tokens + kAppendTok - 1) / kAppendTok;
  kv_append_int8_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, f);
  return cudaGetLastError();
}

// RoPE fused into the e4m3 quantisation of the FP8 prefill's inputs.  Each
// (token, head) row of 128 values is rotated and rounded to bf16 exactly as
// rope_apply stores it, then quantised exactly as quant_fp8_rows /
// quant_fp8_heads quantise a bf16 row: scale = max|x| / 448, code =
// e4m3(x / scale) in fp32, ties to even, saturating; an all-zero group has
// scale 0 and codes 0.  The input is not modified.
//
// The kernels take rope_kernel's layout: a block holds NT tokens
// (their angles computed once, into shared memory) and a thread one 16-byte
// chunk c of the first half of a (token, head) row together with the partner
// chunk of the second half, so each RoPE pair is in one thread's registers.
// Eight consecutive lanes hold one row; its maximum takes three shuffles.
// NT * heads is a multiple of 4, so every warp covers whole rows and runs the
// loop the same number of times: rows past the last token load nothing and
// store nothing, but still take part in the shuffles.
__device__ __forceinline__ bool rope_chunk(const __nv_bfloat16* __restrict__ x, int64_t t0, int64_t tokens,
                                           int heads, const GridWalk& gw, const float (*cs_s)[64],
                                           const float (*sn_s)[64], RowChunk& r, int64_t& row) {
  const int c = gw.c, tt = gw.tt;
  const int64_t t = t0 + tt;
  row = t * heads + gw.h;
  const bool ok = t < tokens;
  load_chunk(x + row * 128, c, ok, r);
  rotate_chunk(r, cs_s[tt], sn_s[tt], c);
  return ok;
}

template <bool FAST>
__device__ __forceinline__ void chunk_codes(const RowChunk& r, float sc, float rc, uint2& a, uint2& b) {
  a.x = e4m3x4_div<FAST>(r.a[0], r.a[1], r.a[2], r.a[3], sc, rc);
  a.y = e4m3x4_div<FAST>(r.a[4], r.a[5], r.a[6], r.a[7], sc, rc);
  b.x = e4m3x4_div<FAST>(r.b[0], r.b[1], r.b[2], r.b[3], sc, rc);
  b.y = e4m3x4_div<FAST>(r.b[4], r.b[5], r.b[6], r.b[7], sc, rc);
}

__device__ __forceinline__ void chunk_store(const RowChunk& r, float sc, uint8_t* row_codes, int c) {
  uint2 a = make_uint2(0u, 0u), b = a;
  if (sc >= kFastDivMinScale)
    chunk_codes<true>(r, sc, __frcp_rn(sc), a, b);
  else if (sc != 0.0f)
    chunk_codes<false>(r, sc, 0.f, a, b);
  *reinterpret_cast<uint2*>(row_codes + 8 * c) = a;
  *reinterpret_cast<uint2*>(row_codes + 64 + 8 * c) = b;
}

// One scale per row (the queries).
template <int NT>
__global__ void __launch_bounds__(256) rope_quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens,
                                                              int heads, const int32_t* __restrict__ pos,
                                                              const InvFreq f, uint8_t* __restrict__ codes,
                                                              float* __restrict__ scales) {
  __shared__ __align__(16) float cs_s[NT][64], sn_s[NT][64];
  const int64_t t0 = (int64_t)blockIdx.x * NT;
  angle_tables<NT, 64>(cs_s, sn_s, t0, tokens, 64, pos, f);
  const int items = NT * heads * 8;
  GridWalk gw(threadIdx.x, blockDim.x, 8, heads);
#pragma unroll 2
  for (int it = threadIdx.x; it < items; it += blockDim.x, gw.next()) {
    RowChunk r;
    int64_t row;
    const bool ok = rope_chunk(x, t0, tokens, heads, gw, cs_s, sn_s, r, row);
    const float sc = chunk_amax(r) / 448.0f;
    if (ok) {
      chunk_store(r, sc, codes + row * 128, gw.c);
      if (gw.c == 0) scales[row] = sc;
    }
  }
}

// One scale per head over all tokens (the keys), pass 1: max |rotated x| per
// head, gathered in shared memory and folded into amax_bits[head] (the bits of
// a non-negative float order like the integers) with one atomic per block.
// The grid is persistent (a few blocks per SM, each taking groups of NT tokens
// in turn), so the global atomics number blocks x heads, not tokens.
template <int NT>
__global__ void __launch_bounds__(256) rope_amax_heads_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens,
                                                              int heads, const int32_t* __restrict__ pos,
                                                              const InvFreq f, unsigned* __restrict__ amax_bits) {
  __shared__ __align__(16) float cs_s[NT][64], sn_s[NT][64];
  __shared__ unsigned hmax[kMaxQuantHeads];
  for (int h = threadIdx.x; h < heads; h += blockDim.x) hmax[h] = 0u;
  const int items = NT * heads * 8;
  const int64_t groups = (tokens + NT - 1) / NT;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t t0 = g * NT;
    __syncthreads();  // the previous group's angles are no longer read
    angle_tables<NT, 64>(cs_s, sn_s, t0, tokens, 64, pos, f);  // its barrier also publishes hmax
    GridWalk gw(threadIdx.x, blockDim.x, 8, heads);
#pragma unroll 2
    for (int it = threadIdx.x; it < items; it += blockDim.x, gw.next()) {
      RowChunk r;
      int64_t row;
      const bool ok = rope_chunk(x, t0, tokens, heads, gw, cs_s, sn_s, r, row);
      const float m = chunk_amax(r);  // 0 for rows past the end
      if (ok && gw.c == 0) atomicMax(&hmax[gw.h], __float_as_uint(m));
    }
  }
  __syncthreads();
  for (int h = threadIdx.x; h < heads; h += blockDim.x)
    if (hmax[h]) atomicMax(amax_bits + h, hmax[h]);
}

// Pass 2: codes with the head's scale, row layout; block 0 also writes the scales.
template <int NT>
__global__ void __launch_bounds__(256) rope_quant_heads_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens,
                                                               int heads, const int32_t* __restrict__ pos,
                                                               const InvFreq f, const unsigned* __restrict__ amax_bits,
                                                               uint8_t* __restrict__ codes, float* __restrict__ scales) {
  __shared__ __align__(16) float cs_s[NT][64], sn_s[NT][64];
  const int64_t t0 = (int64_t)blockIdx.x * NT;
  angle_tables<NT, 64>(cs_s, sn_s, t0, tokens, 64, pos, f);
  if (blockIdx.x == 0)
    for (int h = threadIdx.x; h < heads; h += blockDim.x) scales[h] = __uint_as_float(amax_bits[h]) / 448.0f;
  const int items = NT * heads * 8;
  GridWalk gw(threadIdx.x, blockDim.x, 8, heads);
#pragma unroll 2
  for (int it = threadIdx.x; it < items; it += blockDim.x, gw.next()) {
    RowChunk r;
    int64_t row;
    if (rope_chunk(x, t0, tokens, heads, gw, cs_s, sn_s, r, row))
      chunk_store(r, __uint_as_float(__ldg(amax_bits + gw.h)) / 448.0f, codes + row * 128, gw.c);
  }
}

template <int NT>
static cudaError_t rope_quant_launch(const __nv_bfloat16* x, int64_t tokens, int heads, const int32_t* positions,
                                     const InvFreq& f, void* codes, float* scales, unsigned* amax_scratch,
                                     cudaStream_t s) {
  const unsigned blocks = (unsigned)((tokens + NT - 1) / NT);
  if (!amax_scratch) {
    rope_quant_rows_kernel<NT><<<blocks, 256, 0, s>>>(x, tokens, heads, positions, f, (uint8_t*)codes, scales);
    return cudaGetLastError();
  }
  cudaError_t e = cudaMemsetAsync(amax_scratch, 0, sizeof(unsigned) * heads, s);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned pblocks = (unsigned)std::min<int64_t>(blocks, 2 * std::max(sms, 1));
  rope_amax_heads_kernel<NT><<<pblocks, 256, 0, s>>>(x, tokens, heads, positions, f, amax_scratch);
  rope_quant_heads_kernel<NT><<<blocks, 256, 0, s>>>(x, tokens, heads, positions, f, amax_scratch,
                                                     (uint8_t*)codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_rope_quant_fp8(const void* x, int64_t tokens, int heads, const int32_t* positions, double base,
                                  void* codes, float* scales, unsigned* amax_scratch, cudaStream_t s) {
  const InvFreq f = make_inv_freq(base, 128);
  if (tokens == 0 || heads == 0) return cudaSuccess;
  const __nv_bfloat16* xb = (const __nv_bfloat16*)x;
  // blocks of 32-256 rows: few heads take more tokens per block
  if (heads >= 32) return rope_quant_launch<4>(xb, tokens, heads, positions, f, codes, scales, amax_scratch, s);
  if (heads >= 4) return rope_quant_launch<8>(xb, tokens, heads, positions, f, codes, scales, amax_scratch, s);
  return rope_quant_launch<32>(xb, tokens, heads, positions, f, codes, scales, amax_scratch, s);
}

// cos and sin of every (token, pair) angle, interleaved [tokens][d/2][2] fp32:
// the same numbers rope_kernel rotates with, for kernels that rotate on the fly.
__global__ void __launch_bounds__(256) rope_table_kernel(float2* __restrict__ cs_out, int64_t tokens, int d,
                                                         const int32_t* __restrict__ pos, const InvFreq f) {
  __shared__ float cs_s[kTok][128], sn_s[kTok][128];
  const int half = d / 2;
  const int64_t t0 = (int64_t)blockIdx.x * kTok;
  angle_tables(cs_s, sn_s, t0, tokens, half, pos, f);
  for (int i = threadIdx.x; i < kTok * half; i += blockDim.x) {
    const int tt = i / half, ii = i % half;
    const int64_t t = t0 + tt;
    if (t < tokens) cs_out[t * half + ii] = make_float2(cs_s[tt][ii], sn_s[tt][ii]);
  }
}

cudaError_t launch_rope_table(float* cs_out, int64_t tokens, int head_dim, const int32_t* positions, double base,
                              cudaStream_t s) {
  const InvFreq f = make_inv_freq(base, head_dim);
  if (tokens == 0) return cudaSuccess;
  const int64_t blocks = (tokens + kTok - 1) / kTok;
  rope_table_kernel<<<(unsigned)blocks, 256, 0, s>>>((float2*)cs_out, tokens, head_dim, positions, f);
  return cudaGetLastError();
}

cudaError_t launch_rope(const RopeLaunch& a, cudaStream_t s) {
  const InvFreq f = make_inv_freq(a.base, a.head_dim);
  if (a.tokens == 0 || a.heads + a.heads2 == 0) return cudaSuccess;
  // few heads: 16 tokens per block, so the angle tables are amortised over enough rows
  const bool few = a.heads + a.heads2 <= 16;
  const int nt = few ? 16 : kTok;
  const unsigned blocks = (unsigned)((a.tokens + nt - 1) / nt);
  if (a.dtype == 0) {
    auto* x = (__nv_bfloat16*)a.x;
    auto* x2 = (__nv_bfloat16*)a.x2;
    if (few)
      rope_kernel<__nv_bfloat16, 16><<<blocks, 256, 0, s>>>(x, a.tokens, a.heads, a.head_dim, a.stride_token, x2,
                                                            a.heads2, a.stride2, a.positions, f);
    else
      rope_kernel<__nv_bfloat16, kTok><<<blocks, 256, 0, s>>>(x, a.tokens, a.heads, a.head_dim, a.stride_token, x2,
                                                              a.heads2, a.stride2, a.positions, f);
  } else {
    auto* x = (float*)a.x;
    auto* x2 = (float*)a.x2;
    if (few)
      rope_kernel<float, 16><<<blocks, 256, 0, s>>>(x, a.tokens, a.heads, a.head_dim, a.stride_token, x2, a.heads2,
                                                    a.stride2, a.positions, f);
    else
      rope_kernel<float, kTok><<<blocks, 256, 0, s>>>(x, a.tokens, a.heads, a.head_dim, a.stride_token, x2, a.heads2,
                                                      a.stride2, a.positions, f);
  }
  return cudaGetLastError();
}

}  // namespace attn
