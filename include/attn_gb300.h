/*
 * attn_gb300.h -- C ABI of libattn_gb300.so: exact causal GQA attention for
 * LLM serving on GB300 (sm_103a).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor and table pointers are DEVICE pointers owned by the caller.
 *    The library never allocates or frees caller memory and keeps no state
 *    between calls apart from cached per-device constants -- except
 *    attn_decode_paged_noalloc, whose calls share one static scratch array per
 *    device and leave their partials in it.
 *  - Tensors are packed row-major with the head dimension contiguous:
 *    Q/K/V/O as [tokens][heads][head_dim] ("Ulysses sequence parallelism for
 *    inference", section 2.2: Q/K/V shaped [seq, heads, head_dim]).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call only
 *    enqueues work on it and returns; nothing synchronises.
 *  - Return value: ATTN_OK (0) or an ATTN_ERR_* code.  On an argument error
 *    nothing is launched; attn_last_error() describes the failure (thread-local).
 *  - Faults found on the device (a page id outside the cache, a pipeline wait
 *    that ran out of time) never trap: the kernel records a code that
 *    attn_device_status() returns after the work has finished.
 *  - Calls on different streams may run concurrently and share no scratch,
 *    except attn_decode_paged_noalloc: its calls share one static array per
 *    device, so overlapping calls of it must be serialised.
 *  - Cached per-device addresses (the device error word, the no-alloc scratch)
 *    are looked up once per device ordinal in the context current at the
 *    first call -- the device's primary context, under the CUDA runtime.
 *    cudaDeviceReset() or a switch to another context on that ordinal
 *    invalidates them; the library does not support either after its first
 *    call on a device.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_BF16 = 0, ATTN_FP32 = 1 } attn_dtype_t;

enum {
  ATTN_OK = 0,
  ATTN_ERR_ARG = 1,         /* null pointer, negative or inconsistent size */
  ATTN_ERR_SHAPE = 2,       /* head layout the kernels do not support */
  ATTN_ERR_ALIGN = 3,       /* a pointer or stride is not 16-byte aligned */
  ATTN_ERR_UNSUPPORTED = 4, /* dtype / option combination not built */
  ATTN_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed */
  ATTN_ERR_DEVICE = 6       /* a kernel recorded a device-side fault */
};

/* Message for the last non-zero status returned on this thread. */
ATTN_API const char *attn_last_error(void);

/* Synchronises the current device, then returns ATTN_OK, or ATTN_ERR_DEVICE if
 * a kernel recorded a fault since the last clear (the code is in the message),
 * or ATTN_ERR_CUDA if the synchronisation itself failed.  clear != 0 resets
 * the recorded code.  Device codes: 0x101-0x105 a pipeline wait ran out of
 * time (TMA producer, MMA issuer, softmax, decode, cache append); 0x201 a
 * page id outside [0, num_pages); 0x202 a cache slot outside the cache; 0x203
 * an INT8 decode operand beyond the fp16 range; 0x204 an FP8 prefill key
 * sequence not starting at a multiple of 16 tokens.  When several faults
 * happen, the first code recorded is kept. */
ATTN_API int attn_device_status(int clear);

/* A check of the device-error path that the kernels' bounded waits take, with
 * no fault: one block waits, through the wait helper `which` selects, on an
 * mbarrier that nothing completes.  The wait gives up after its limit (2 s)
 * and records its code: which = 0, the prefill and decode pipelines' wait
 * (code 0x102); which = 1, the staged cache appends' wait (code 0x105).  The
 * next attn_device_status() then reports ATTN_ERR_DEVICE with that code, and
 * the context stays usable.  The pipelines' wait also stops at once when a
 * code is already recorded (another CTA failed), so clear the status first.
 * Asynchronous on `stream`; the block runs for about 2 s. */
ATTN_API int attn_selftest_wait_timeout(int which, void *stream);

/*
 * rope_apply -- rotary position embedding at ABSOLUTE positions, in place.
 *
 * Defined by: Ulysses page, section 3.2 (each local token carries its absolute
 * position from a global token-index table and RoPE uses that position) and
 * section 5.3 (local indices must never be used).  The pages give no formula;
 * this library uses the half-split pairing: for i in [0, head_dim/2),
 *     a = positions[t] * base^(-2i/head_dim)
 *     x[i]          <- x[i] cos a - x[i + head_dim/2] sin a
 *     x[i + d/2]    <- x[i + d/2] cos a + x[i] sin a
 * The angle is reduced exactly: base^(-2i/d) / 2pi is held as a 64-bit
 * fixed-point fraction of a turn, the phase of position p is the low 64 bits
 * of the integer product p * theta_i, and its top 32 bits give the angle in
 * turns for sincospif.  The rotation itself is computed in fp32 and stored back
 * in the tensor's dtype (bf16: round to nearest even).
 *
 *  x            [tokens][heads][head_dim] of `dtype`, row t at x + t*stride_token
 *               elements; 16-byte aligned; rotated in place.
 *  positions    [tokens] int32 absolute positions (>= 0).
 *  stride_token elements between consecutive tokens (>= heads*head_dim, multiple
 *               of 8 for bf16 / 4 for fp32).
 *  head_dim     even, with head_dim/2 a multiple of 8 (bf16) or 4 (fp32).
 */
ATTN_API int rope_apply(void *x, attn_dtype_t dtype, int64_t tokens, int heads, int head_dim,
               int64_t stride_token, const int32_t *positions, double base, void *stream);

/*
 * rope_apply_qk -- rope_apply on a token's queries and keys in one launch: q
 * [tokens][q_heads][head_dim] (row t at q + t*q_stride_token) and k
 * [tokens][k_heads][head_dim] (row t at k + t*k_stride_token), both rotated in
 * place at the same absolute positions, bit for bit as two rope_apply calls
 * would rotate them (one angle table per token serves both).  Either head count
 * may be 0 (its pointer is then ignored).  Same dtype, head_dim, alignment and
 * error rules as rope_apply, for each tensor.
 */
ATTN_API int rope_apply_qk(void *q, int q_heads, int64_t q_stride_token, void *k, int k_heads,
                           int64_t k_stride_token, attn_dtype_t dtype, int64_t tokens, int head_dim,
                           const int32_t *positions, double base, void *stream);

/*
 * rope_table -- the cos and sin of every RoPE angle, for kernels that rotate on
 * the fly: cs_out[t][i] = (cos a, sin a), a = positions[t] * base^(-2i/head_dim),
 * i < head_dim/2, as fp32 pairs [tokens][head_dim/2][2] (16-byte aligned).  The
 * numbers are exactly those rope_apply rotates with (Ulysses page, sections
 * 3.2 and 5.3: absolute positions).  head_dim even, <= 256; base > 0.
 */
ATTN_API int rope_table(const int32_t *positions, int64_t tokens, int head_dim, double base, float *cs_out,
                        void *stream);

/*
 * attn_kv_append_paged -- write a chunk of new tokens' keys and values into the
 * head-major paged KV cache, rotating the keys (RoPE at their absolute
 * positions) on the way.
 *
 * Defined by: SGLang page, section 2.1 (every new token is given a cache slot
 * through a token-to-slot table before attention runs) and section 2.2 (a
 * prefill chunk's K/V join the cache, where the next chunk and the decode
 * steps read them); Ulysses page, section 2.3 (the cache is split by KV head)
 * and section 3.2 (keys are rotated at their absolute positions).  The
 * rotation is rope_apply's, bit for bit.
 *
 *  k_new, v_new  [tokens][num_kv_heads][head_dim] bf16, packed, 16-byte aligned;
 *                k_new holds unrotated keys and is not modified.
 *  positions     [tokens] int32 absolute position of each key (its RoPE angle).
 *  slots         [tokens] int32 cache slot of each token, page * page_size + offset
 *                in [0, num_pages * page_size); -1 skips the token (padding).
 *  k_cache, v_cache  [num_kv_heads][num_pages][page_size][head_dim] bf16: token t
 *                of KV head g goes to row g * num_pages * page_size + slots[t].
 *  k_rot_out     NULL, or [tokens][num_kv_heads][head_dim] bf16 that also receives
 *                the rotated keys (the chunk's own causal attention can read them
 *                contiguously).  Skipped tokens are not written here either.
 *  base          RoPE base (> 0), or 0 to copy the keys unrotated.
 *  head_dim      head_dim/2 a multiple of 8, at most 256.
 * Errors: argument errors return before launch.  A slot >= num_pages *
 * page_size or < -1 is not written; the kernel records it and
 * attn_device_status() reports ATTN_ERR_DEVICE.  Two tokens with the same slot
 * race; the caller assigns distinct slots.
 */
ATTN_API int attn_kv_append_paged(const void *k_new, const void *v_new, const int32_t *positions,
                                  const int32_t *slots, int64_t tokens, int num_kv_heads, int head_dim,
                                  void *k_cache, void *v_cache, int64_t num_pages, int page_size,
                                  void *k_rot_out, double base, void *stream);

/*
 * attn_kv_append_paged_int8 -- attn_kv_append_paged into an INT8 cache (the
 * cache attn_decode_paged_int8 reads).  Keys are rotated exactly as
 * attn_kv_append_paged rotates them and rounded to bf16; then every key and
 * value row of 128 values is quantised to symmetric int8 in fp32: scale =
 * max|x| / 127, code = x / scale rounded to nearest (ties to even), clamped
 * to [-127, 127]; an all-zero row gets scale 0 ("Flash Attention and
 * distributed parallelism", section 18.12; Ulysses page, section 5.4).
 *
 *  k_cache, v_cache  [num_kv_heads][num_pages][page_size][128] int8 codes.
 *  k_scale, v_scale  [num_kv_heads][num_pages][page_size] fp32 (16-byte aligned).
 *  k_rot_out         NULL, or the rotated bf16 keys [tokens][num_kv_heads][128].
 *  Everything else as attn_kv_append_paged (head_dim must be 128).
 */
ATTN_API int attn_kv_append_paged_int8(const void *k_new, const void *v_new, const int32_t *positions,
                                       const int32_t *slots, int64_t tokens, int num_kv_heads, int head_dim,
                                       void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                                       int64_t num_pages, int page_size, void *k_rot_out, double base,
                                       void *stream);

/*
 * quant_fp8_rows / quant_fp8_heads -- e4m3 codes for the FP8 prefill ("Flash
 * Attention and distributed parallelism", section 18.5: an FP8 mode with block
 * quantisation).  A group of values shares one fp32 scale = max|x| / 448; each
 * value is stored as e4m3(x / scale), rounded to nearest even with x / scale
 * in fp32 (saturating at +-448); an all-zero group has scale 0 and codes 0.
 * The value a code stands for is code * scale.
 *
 *  quant_fp8_rows:  x [tokens][heads][128] bf16 -> codes [tokens][heads][128]
 *                   e4m3, scales [tokens][heads] fp32; one group per row (the
 *                   queries).
 *  quant_fp8_heads: one group per head over all tokens (keys, values) ->
 *                   scales [heads]; codes [tokens][heads][128] (transposed = 0)
 *                   or [heads][128][t_stride] (transposed = 1, t_stride >= tokens
 *                   and a multiple of 16: the values, whose P V contraction reads
 *                   V^T rows; columns [tokens, t_stride) are written as zero
 *                   codes).  amax_scratch: caller-owned [heads] unsigned.
 * x and codes 16-byte aligned; head_dim must be 128.
 */
ATTN_API int quant_fp8_rows(const void *x, int64_t tokens, int heads, int head_dim, void *codes, float *scales,
                            void *stream);
ATTN_API int quant_fp8_heads(const void *x, int64_t tokens, int heads, int head_dim, void *codes, float *scales,
                             unsigned *amax_scratch, int transposed, int64_t t_stride, void *stream);

/*
 * rope_quant_fp8_rows / rope_quant_fp8_heads -- RoPE (as rope_apply) fused into
 * the e4m3 quantisation above, for unrotated queries and keys: each row is
 * rotated at its absolute position and rounded to bf16 exactly as rope_apply
 * stores it, then quantised exactly as quant_fp8_rows / quant_fp8_heads
 * quantise that bf16 row.  The result equals rope_apply (on a copy) followed by
 * quant_fp8_rows / quant_fp8_heads (row layout) bit for bit; x is not modified.
 *
 *  x          [tokens][heads][128] bf16, 16-byte aligned, unrotated.
 *  positions  [tokens] int32 absolute positions; base > 0 (e.g. 10000).
 *  codes      [tokens][heads][128] e4m3, 16-byte aligned.
 *  scales     rows: [tokens][heads] fp32; heads: [heads] fp32.
 *  amax_scratch (heads only): caller-owned [heads] unsigned; heads <= 256.
 * Reads x once (rows) or twice (heads: the per-head maximum, then the codes).
 */
ATTN_API int rope_quant_fp8_rows(const void *x, int64_t tokens, int heads, int head_dim, const int32_t *positions,
                                 double base, void *codes, float *scales, void *stream);
ATTN_API int rope_quant_fp8_heads(const void *x, int64_t tokens, int heads, int head_dim, const int32_t *positions,
                                  double base, void *codes, float *scales, unsigned *amax_scratch, void *stream);

/*
 * attn_prefill -- exact causal GQA attention, FlashAttention-style tiled.
 *
 * Computes, for every query row of every sequence and every query head h in
 * [h_lo, h_hi):  S = scale * q k^T over the visible keys, A = softmax(S), O = A V,
 * and LSE = ln sum_j exp(S_j)  ("Flash Attention and distributed parallelism",
 * section 18.2 for the definition; section 18.3 for the blockwise online
 * softmax with per-block rescaling by exp(m_old - m_new); section 18.4 for the
 * query-outer loop with normalisation deferred to the end).  The N x N score
 * matrix is never stored.  Key j is visible to query i iff (!causal or
 * kpos_j <= qpos_i) -- positions, not indices (Ulysses page, section 5.3).
 * Query head h reads KV head h / (num_q_heads / num_kv_heads) (GQA, Ulysses
 * page, section 3.2).  Heads outside [h_lo, h_hi) of out/lse are not touched,
 * so head slices of one problem put together equal the all-heads call
 * ("full sequence, some heads", Ulysses page, sections 2.1-2.2).
 *
 *  q          [Tq][num_q_heads][head_dim] (already rotated), Tq = cu_q[batch].
 *  cu_q       [batch+1] int32 prefix offsets of each sequence's query rows.
 *  q_pos      [Tq] int32 absolute query positions, non-decreasing within a sequence.
 *  total_q    Tq as a host value (sizes the TMA descriptor of q).
 *  max_seqlen_q  largest cu_q[b+1]-cu_q[b] (host value; sizes the grid).
 *  Contiguous key/value source (page_table == NULL):
 *    k, v     [Tk][num_kv_heads][head_dim], Tk = cu_k[batch]; cu_k [batch+1];
 *    k_pos    [Tk] absolute key positions, non-decreasing within a sequence;
 *    total_k  Tk as a host value.
 *  Paged key/value source (page_table != NULL; SGLang page, section 2.1:
 *  token-to-cache-slot indirection; Ulysses page, section 2.3: head-sharded cache):
 *    k, v     head-major caches [num_kv_heads][num_pages][page_size][head_dim];
 *    page_table [batch][max_pages] int32 physical page of each logical page;
 *    k_lens   [batch] int32 cached tokens of each request; cached token j of
 *             request b is page_table[b][j/page_size], slot j%page_size, and sits
 *             at position j.  cu_k and k_pos must be NULL, total_k is ignored.
 *             Unused slots of a request's last page must hold finite values.
 *  out        [Tq][num_q_heads][head_dim] of out_dtype.
 *  lse        [Tq][num_q_heads] fp32 natural-log LSE of the scaled scores, or NULL.
 *             A row with no visible key gets O = 0 and LSE = -inf.
 *  h_lo, h_hi query-head range; both multiples of num_q_heads/num_kv_heads.
 *  dtype      ATTN_BF16 (tensor-core path; head_dim 128 uses the tcgen05 kernel)
 *             or ATTN_FP32 (CUDA-core path).  head_dim: multiple of 32, <= 256.
 *             bf16 paged sources need page_size 64 for the tensor-core kernel.
 * All pointers 16-byte aligned.  Errors: ATTN_ERR_ARG / _SHAPE / _ALIGN / _CUDA.
 */
ATTN_API int attn_prefill(const void *q, const void *k, const void *v, void *out, attn_dtype_t out_dtype,
                 float *lse, attn_dtype_t dtype, int batch, const int32_t *cu_q,
                 const int32_t *q_pos, int64_t total_q, int max_seqlen_q, const int32_t *cu_k,
                 const int32_t *k_pos, int64_t total_k,
                 const int32_t *page_table, const int32_t *k_lens, int max_pages, int page_size,
                 int64_t num_pages, int num_q_heads, int num_kv_heads, int head_dim, int h_lo,
                 int h_hi, float scale, int causal, void *stream);

/*
 * attn_prefill_rope_q -- attn_prefill with the query's RoPE fused in: q holds
 * UNROTATED queries, and the kernel rotates each query row in on-chip memory,
 * with the cos/sin of q_rope_cs ([total_q][head_dim/2][2] fp32 from rope_table
 * over q_pos, 16-byte aligned), before its scores.  The result equals
 * rope_apply(q) followed by attn_prefill bit for bit; q itself is not
 * modified.  Keys must already be rotated (rope_apply or attn_kv_append_paged).
 * Only the tensor-core path takes it (bf16, head_dim 128); other shapes return
 * ATTN_ERR_UNSUPPORTED.  All other arguments as attn_prefill.
 */
ATTN_API int attn_prefill_rope_q(const void *q, const void *k, const void *v, void *out, attn_dtype_t out_dtype,
                                 float *lse, attn_dtype_t dtype, int batch, const int32_t *cu_q,
                                 const int32_t *q_pos, int64_t total_q, int max_seqlen_q, const int32_t *cu_k,
                                 const int32_t *k_pos, int64_t total_k, const int32_t *page_table,
                                 const int32_t *k_lens, int max_pages, int page_size, int64_t num_pages,
                                 int num_q_heads, int num_kv_heads, int head_dim, int h_lo, int h_hi, float scale,
                                 int causal, const float *q_rope_cs, void *stream);

/*
 * attn_prefill_fp8 -- attn_prefill (contiguous source) on e4m3 codes: the FP8
 * mode of "Flash Attention and distributed parallelism", section 18.5, with
 * block quantisation.  The attention computed is that of the values the codes
 * stand for: q = code * q_scale[row], k = code * k_scale[kv head], v = code *
 * v_scale[kv head] (quant_fp8_rows / quant_fp8_heads produce them).  Both
 * contractions run on e4m3 operands with fp32 accumulation; the softmax is
 * fp32 and the weights P are rounded to e4m3 for P V (P <= 256), so O carries
 * that rounding (relative 2^-4 per weight); LSE uses the unrounded weights.
 *
 *  q        [total_q][num_q_heads][128] e4m3;  q_scale [total_q][num_q_heads] fp32.
 *  k        [total_k][num_kv_heads][128] e4m3; k_scale [num_kv_heads] fp32.
 *  v_t      [num_kv_heads][128][v_t_stride] e4m3 (values transposed, keys
 *           contiguous; v_t_stride >= total_k, a multiple of 16); v_scale
 *           [num_kv_heads] fp32.
 *  Every key sequence must start at a multiple of 16 tokens (cu_k[b] % 16 == 0):
 *  a CTA whose sequence does not records a device error and writes nothing.
 *  Everything else as attn_prefill (head_dim 128; no paged source).
 */
ATTN_API int attn_prefill_fp8(const void *q, const float *q_scale, const void *k, const float *k_scale,
                              const void *v_t, const float *v_scale, int64_t v_t_stride, void *out,
                              attn_dtype_t out_dtype, float *lse, int batch, const int32_t *cu_q,
                              const int32_t *q_pos, int64_t total_q, int max_seqlen_q, const int32_t *cu_k,
                              const int32_t *k_pos, int64_t total_k, int num_q_heads, int num_kv_heads,
                              int head_dim, int h_lo, int h_hi, float scale, int causal, void *stream);

/*
 * attn_decode_paged -- split-KV decode over a head-major paged KV cache.
 *
 * One new query token per request at position ctx_lens[b]-1 attends to all
 * ctx_lens[b] cached tokens (its own K/V already written to the cache).  The
 * cached tokens are cut into num_splits partitions of whole pages; each
 * partition yields a partial (O_s, LSE_s) and the partials are combined by the
 * log-sum-exp merge of attn_lse_merge.  Defined by: Flash Attention page,
 * section 18.3 (partial softmax states over disjoint key blocks combine through
 * the rescale exp(m_old - m_new)) and section 18.4 (the key sequence as a
 * parallel axis); paged cache: SGLang page, section 2.1, and the PagedAttention
 * reference in section 18.12 of the Flash Attention page; head-major layout:
 * Ulysses page, section 2.3.  Split s covers logical pages
 * [s*pps, min((s+1)*pps, n_pages)) with n_pages = ceil(ctx/page_size) and
 * pps = ceil(n_pages/num_splits); an empty split has LSE_s = -inf.
 *
 *  q          [batch][num_q_heads][head_dim] bf16, already rotated.
 *  k_cache, v_cache  [num_kv_heads][num_pages][page_size][head_dim] bf16.
 *  page_table [batch][max_pages] int32; ctx_lens [batch] int32 (>= 0,
 *             <= max_pages*page_size).
 *  part_out   workspace [batch][num_q_heads][num_splits][head_dim] fp32 and
 *  part_lse   workspace [batch][num_q_heads][num_splits] fp32, written here.
 *  out        [batch][num_q_heads][head_dim] of out_dtype; lse [batch][num_q_heads]
 *             fp32 or NULL.  If out is NULL only the partials are written.
 *  Supported: bf16, head_dim 128, page_size 64, num_q_heads/num_kv_heads = 8,
 *  1 <= num_splits <= 256.  Errors: ATTN_ERR_ARG / _SHAPE / _ALIGN / _CUDA.
 */
ATTN_API int attn_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *page_table, const int32_t *ctx_lens, int batch,
                      int max_pages, int page_size, int64_t num_pages, int num_q_heads,
                      int num_kv_heads, int head_dim, int num_splits, float scale,
                      float *part_out, float *part_lse, void *out, attn_dtype_t out_dtype,
                      float *lse, void *stream);

/*
 * attn_decode_paged_noalloc -- attn_decode_paged without a caller workspace.
 *
 * The pages have no counterpart for this call: it exists for callers that
 * cannot allocate device memory -- e.g. a serving engine that gives all free
 * HBM to its KV-cache pool at start-up, a plugin inside a framework whose
 * caching allocator owns the device memory, or a latency-critical path where
 * cudaMalloc/cudaFree would synchronise the device.  It computes exactly what
 * attn_decode_paged computes, with the split partials kept in a scratch array
 * the library holds statically on each device (16.1 MiB, held until exit).
 * It calls no allocator.
 *
 *  Arguments as attn_decode_paged, minus part_out/part_lse; out must not be
 *  NULL.  batch * num_q_heads * num_splits must be <= 32768 (e.g. 32 requests
 *  x 64 heads x 16 splits), else ATTN_ERR_ARG and nothing is launched.
 *  All calls on a device share the scratch and it keeps the last call's
 *  contents (no part of it needs to start at zero); calls that overlap on the
 *  GPU race on it, so serialise them.  The first call on a device looks up the
 *  scratch's device address (cudaGetSymbolAddress) with that device current;
 *  make that first call before any stream capture.  The address found is that
 *  of the context current then (the primary context under the runtime API) and
 *  is kept for the device ordinal: after cudaDeviceReset(), or under another
 *  context on the same ordinal, it is stale, so neither is supported once this
 *  call has run on a device.
 */
ATTN_API int attn_decode_paged_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *page_table, const int32_t *ctx_lens, int batch,
                                       int max_pages, int page_size, int64_t num_pages,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int num_splits, float scale, void *out,
                                       attn_dtype_t out_dtype, float *lse, void *stream);

/*
 * attn_decode_paged_int8 -- attn_decode_paged over an INT8 KV cache.
 *
 * Defined by: the same attention as attn_decode_paged, over cached values
 * code * scale.  An INT8 cache halves the bytes per cached token ("Flash
 * Attention and distributed parallelism", section 18.12); a quantised cache
 * keeps grouped codes with their scales (Ulysses page, section 5.4).  Here the
 * codes are symmetric int8 and the group is one (KV head, cached token).
 *
 *  k_cache, v_cache  [num_kv_heads][num_pages][page_size][head_dim] int8 codes.
 *  k_scale, v_scale  [num_kv_heads][num_pages][page_size] fp32, 16-byte aligned:
 *                    the cached value is code * scale.
 *  Everything else as attn_decode_paged (head_dim 128, page_size 64, 8 query
 *  heads per KV head; same workspace, merge and outputs).
 * The group contraction runs with fp16 operands: a rotated query element or a
 * softmax weight times v_scale beyond 65504 in magnitude is recorded as a
 * device error (attn_device_status reports ATTN_ERR_DEVICE).
 */
ATTN_API int attn_decode_paged_int8(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                                    const float *v_scale, const int32_t *page_table, const int32_t *context_lens,
                                    int batch, int max_pages, int page_size, int64_t num_pages, int num_q_heads,
                                    int num_kv_heads, int head_dim, int num_splits, float scale, float *part_out,
                                    float *part_lse, void *out, attn_dtype_t out_dtype, float *lse, void *stream);

/*
 * attn_lse_merge -- combine partial attention results over disjoint key sets.
 *
 *   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s
 * Parts with LSE_s = -inf carry weight 0; if every part is -inf, O = 0 and
 * LSE = -inf.  Defined by: Flash Attention page, section 18.3 (merging the
 * running (m, l, O) state of one key block into another by exp(m_old - m_new)),
 * and the per-step accumulation of ring attention on the SGLang page,
 * section 3.5.  Used for split-KV decode and for a prefill chunk merged with
 * its cached prefix.
 *
 *  part_out   fp32, element (p, r, h, i) at
 *             part_out[p*o_stride_part + r*o_stride_row + h*o_stride_head + i]
 *  part_lse   fp32, element (p, r, h) at
 *             part_lse[p*l_stride_part + r*l_stride_row + h*l_stride_head]
 *  out        [rows][heads][head_dim] of out_dtype; lse_out [rows][heads] fp32 or NULL.
 *  Strides are in elements.  1 <= n_parts <= 1024.
 */
ATTN_API int attn_lse_merge(const float *part_out, const float *part_lse, int n_parts, int64_t rows,
                   int heads, int head_dim, int64_t o_stride_part, int64_t o_stride_row,
                   int64_t o_stride_head, int64_t l_stride_part, int64_t l_stride_row,
                   int64_t l_stride_head, void *out, attn_dtype_t out_dtype, float *lse_out,
                   void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
