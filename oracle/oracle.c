/*
 * CPU oracle for exact causal GQA attention with RoPE, paged decode and LSE merge.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
 * baseline use this file; the product library never links or calls it, and
 * it shares no code, header or table with the CUDA sources.
 *
 * Everything is plain fp64 and follows the definitions on the pages, with no
 * tiling, fusion or reordering beyond what those definitions state:
 *
 *   attention   S = Q K^T * scale, A = softmax(S), O = A V
 *               ("Flash Attention and distributed parallelism", section 18.2),
 *               evaluated as the three-pass softmax the same page describes in
 *               section 18.3 (max pass, denominator pass, output pass);
 *   causal mask key j is visible to query i iff pos_j <= pos_i, with pos the
 *               absolute token position ("Ulysses sequence parallelism for
 *               inference", section 5.3: a global mask, never a local one);
 *   GQA         query head h reads KV head h / (Hq / Hkv) (same page, 3.2);
 *   RoPE        rotation by the absolute position from the global token index
 *               table (same page, 3.2 and 5.3); half-split pairing, see below;
 *   paging      token j of request b lives in page page_table[b][j / P], slot
 *               j % P, of a head-major cache (same page, 2.3; SGLang page, 2.1);
 *   merge       parts over disjoint key sets combine through their log-sum-exp,
 *               the same rescale by exp(m_old - m_new) that section 18.3 of the
 *               Flash Attention page applies between K/V blocks.
 *
 * Readings where the pages are silent:
 *   - RoPE pairs element i with element i + d/2, angle pos * base^(-2i/d);
 *   - LSE is the natural log of sum_j exp(scale * q.k_j) over visible keys;
 *   - a query with no visible key has O = 0 and LSE = -inf, and such a part
 *     gets weight 0 in a merge;
 *   - a decode query sits at position ctx - 1 and sees all ctx cached keys.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ RoPE */

/* Rotate x[t][h][:] in place by the angles of absolute position pos[t]:
 *   theta_i = base^(-2i/d),  a = pos * theta_i,  i in [0, d/2)
 *   x'_i       = x_i cos a - x_{i+d/2} sin a
 *   x'_{i+d/2} = x_{i+d/2} cos a + x_i sin a                                  */
void oracle_rope(double *x, int64_t tokens, int heads, int d, const int32_t *pos, double base)
{
    const int half = d / 2;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < tokens; ++t) {
        for (int i = 0; i < half; ++i) {
            double theta = pow(base, -2.0 * (double)i / (double)d);
            double a = (double)pos[t] * theta;
            double c = cos(a), s = sin(a);
            for (int h = 0; h < heads; ++h) {
                double *r = x + (t * heads + h) * (int64_t)d;
                double x1 = r[i], x2 = r[i + half];
                r[i] = x1 * c - x2 * s;
                r[i + half] = x2 * c + x1 * s;
            }
        }
    }
}

/* ------------------------------------------------------- bf16 rounding */

/* Round to the nearest bf16 value (8 significant bits, exponent range of fp32),
 * ties to even.  Used where the path stores a result in bf16, e.g. the rotated
 * Q/K that the attention step then consumes. */
static double round_bf16_one(double x)
{
    if (!isfinite(x) || x == 0.0) return x;
    int e;
    (void)frexp(x, &e);          /* x = m * 2^e, 0.5 <= |m| < 1 */
    int q = e - 8;               /* exponent of one unit in the last place */
    if (q < -133) q = -133;      /* subnormal spacing 2^-133 */
    double r = ldexp(nearbyint(ldexp(x, -q)), q);
    if (fabs(r) > 3.3895313892515355e38) r = copysign(INFINITY, x);
    return r;
}

void oracle_round_bf16(double *x, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) x[i] = round_bf16_one(x[i]);
}

/* ------------------------------------------------------------ attention */

/* One query row against nk keys with stride kstride (elements between tokens).
 * Three passes over the scores: max, denominator, weighted sum of V. */
static void attend_row(const double *qv, const double *kb, const double *vb, int64_t kstride,
                       const int32_t *kpos, int64_t nk, int32_t qp, int causal, int d,
                       double scale, double *sc, double *out, double *lse)
{
    double M = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
        if (causal && kpos[j] > qp) continue;
        const double *kr = kb + j * kstride;
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += qv[i] * kr[i];
        s *= scale;
        sc[j] = s;
        if (s > M) M = s;
    }
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    if (M == -INFINITY) { *lse = -INFINITY; return; }
    double L = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
        if (causal && kpos[j] > qp) continue;
        L += exp(sc[j] - M);
    }
    for (int64_t j = 0; j < nk; ++j) {
        if (causal && kpos[j] > qp) continue;
        double w = exp(sc[j] - M) / L;
        const double *vr = vb + j * kstride;
        for (int i = 0; i < d; ++i) out[i] += w * vr[i];
    }
    *lse = M + log(L);
}

/* q      [nq][hq][d]   query rows (already rotated), row r belongs to sequence q_seq[r]
 *                      and sits at absolute position q_pos[r]
 * k, v   [Tk][hkv][d]  keys/values of all sequences, sequence b = rows cu_k[b]..cu_k[b+1]-1
 * k_pos  [Tk]          absolute key positions
 * out    [nq][hq][d], lse [nq][hq]: written for heads h_lo..h_hi-1 only.
 * Returns 0, or -1 on a bad argument. */
int oracle_attention(const double *q, int64_t nq, const int32_t *q_seq, const int32_t *q_pos,
                     const double *k, const double *v, int batch, const int32_t *cu_k,
                     const int32_t *k_pos, int hq, int hkv, int d, int h_lo, int h_hi,
                     double scale, int causal, double *out, double *lse)
{
    if (hkv <= 0 || hq % hkv != 0 || h_lo < 0 || h_hi > hq || h_lo > h_hi) return -1;
    const int G = hq / hkv;
    int64_t maxk = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t n = (int64_t)cu_k[b + 1] - cu_k[b];
        if (n < 0) return -1;
        if (n > maxk) maxk = n;
    }
    for (int64_t r = 0; r < nq; ++r)
        if (q_seq[r] < 0 || q_seq[r] >= batch) return -1;
    const int nh = h_hi - h_lo;
    const int64_t items = nq * (int64_t)nh;
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(maxk > 0 ? maxk : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t it = 0; it < items; ++it) {
            int64_t r = it / nh;
            int h = h_lo + (int)(it % nh);
            int b = q_seq[r];
            int g = h / G;
            int64_t k0 = cu_k[b], nk = (int64_t)cu_k[b + 1] - cu_k[b];
            attend_row(q + (r * hq + h) * (int64_t)d,
                       k + (k0 * hkv + g) * (int64_t)d, v + (k0 * hkv + g) * (int64_t)d,
                       (int64_t)hkv * d, k_pos + k0, nk, q_pos[r], causal, d, scale, sc,
                       out + (r * hq + h) * (int64_t)d, lse + r * hq + h);
        }
        free(sc);
    }
    return 0;
}

/* ------------------------------------------------------------ paged KV */

/* Copy the first ctx tokens of request b, KV head g, out of a head-major paged
 * cache [hkv][num_pages][page][d] into dst [ctx][d] in logical token order.
 * Returns 0, or -1 if a page id is outside [0, num_pages). */
int oracle_gather_pages(const double *cache, const int32_t *page_table, int max_pages,
                        int page, int64_t num_pages, int d, int g, int b, int32_t ctx,
                        double *dst)
{
    const int32_t *row = page_table + (int64_t)b * max_pages;
    for (int32_t j = 0; j < ctx; ++j) {
        int lp = j / page;
        if (lp >= max_pages) return -1;
        int32_t pid = row[lp];
        if (pid < 0 || pid >= num_pages) return -1;
        const double *src = cache + (((int64_t)g * num_pages + pid) * page + (j % page)) * (int64_t)d;
        memcpy(dst + (int64_t)j * d, src, sizeof(double) * (size_t)d);
    }
    return 0;
}

/* Append new tokens to the head-major paged cache (SGLang page, sections 2.1
 * and 2.2: each new token is given a cache slot, page * page_size + offset,
 * and its K/V are written there before attention reads them; Ulysses page,
 * section 2.3: one pool per KV head; section 3.2: keys rotated at their
 * absolute positions).
 *   k_new, v_new [tokens][heads][d]; pos [tokens]; slots [tokens]
 *   k_cache, v_cache [heads][rows][d], rows = num_pages * page_size
 * Key rows are rotated (when base > 0) and rounded to bf16, as the path stores
 * them; value rows are copied.  Slot -1 skips a token.  Returns the number of
 * tokens whose slot lies outside [-1, rows); those are skipped too. */
int oracle_kv_append(const double *k_new, const double *v_new, const int32_t *pos, const int32_t *slots,
                     int64_t tokens, int heads, int d, double *k_cache, double *v_cache, int64_t rows,
                     double base)
{
    int bad = 0;
    double *krow = malloc((size_t)d * sizeof(double));
    if (!krow) return -1;
    for (int64_t t = 0; t < tokens; ++t) {
        const int64_t s = slots[t];
        if (s == -1) continue;
        if (s < -1 || s >= rows) { ++bad; continue; }
        for (int h = 0; h < heads; ++h) {
            const double *src = k_new + (t * heads + h) * (int64_t)d;
            for (int i = 0; i < d; ++i) krow[i] = src[i];
            if (base > 0.0) {
                oracle_rope(krow, 1, 1, d, pos + t, base);
                oracle_round_bf16(krow, d);
            }
            double *kd = k_cache + ((int64_t)h * rows + s) * d;
            double *vd = v_cache + ((int64_t)h * rows + s) * d;
            const double *vs = v_new + (t * heads + h) * (int64_t)d;
            for (int i = 0; i < d; ++i) {
                kd[i] = krow[i];
                vd[i] = vs[i];
            }
        }
    }
    free(krow);
    return bad;
}

/* INT8 KV cache (Flash Attention page, section 18.12: an INT8 cache halves the
 * bytes per cached token; Ulysses page, section 5.4: a quantised cache stores
 * grouped codes with their scales).  Symmetric codes with one scale per (KV
 * head, cached token): the value is code * scale, computed here exactly.
 *   codes [rows][d] int8, scales [rows] fp32 -> out [rows][d] */
void oracle_dequant_int8(const int8_t *codes, const float *scales, int64_t rows, int d, double *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < d; ++i)
            out[r * d + i] = (double)codes[r * d + i] * (double)scales[r];
}

/* Symmetric INT8 quantisation of one cache row (the reading taken of the
 * Flash Attention page, section 18.12, and the Ulysses page, section 5.4:
 * grouped codes with a scale, the group being one (KV head, token) row).  In
 * fp32, as the path decides it: scale = max|x| / 127, code = x / scale rounded
 * to the nearest integer (ties to even), clamped to [-127, 127]; an all-zero
 * row has scale 0 and codes 0.  x holds d values that are exact in fp32. */
static void quant_row_int8(const double *x, int d, int8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
        float a = fabsf((float)x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    *scale = s;
    for (int i = 0; i < d; ++i) {
        if (s == 0.0f) { codes[i] = 0; continue; }
        float q = rintf((float)x[i] / s);
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        codes[i] = (int8_t)q;
    }
}

/* oracle_kv_append for an INT8 cache: keys rotated (base > 0) and rounded to
 * bf16, as the bf16 cache would hold them, then each key and value row is
 * quantised by quant_row_int8 into codes [heads][rows][d] and scales
 * [heads][rows].  Slot -1 skips a token; returns the number of tokens whose
 * slot lies outside [-1, rows), which are skipped too. */
int oracle_kv_append_int8(const double *k_new, const double *v_new, const int32_t *pos, const int32_t *slots,
                          int64_t tokens, int heads, int d, int8_t *k_codes, int8_t *v_codes, float *k_scale,
                          float *v_scale, int64_t rows, double base)
{
    int bad = 0;
    double *krow = malloc((size_t)d * sizeof(double));
    if (!krow) return -1;
    for (int64_t t = 0; t < tokens; ++t) {
        const int64_t s = slots[t];
        if (s == -1) continue;
        if (s < -1 || s >= rows) { ++bad; continue; }
        for (int h = 0; h < heads; ++h) {
            const double *src = k_new + (t * heads + h) * (int64_t)d;
            for (int i = 0; i < d; ++i) krow[i] = src[i];
            if (base > 0.0) {
                oracle_rope(krow, 1, 1, d, pos + t, base);
                oracle_round_bf16(krow, d);
            }
            const int64_t r = (int64_t)h * rows + s;
            quant_row_int8(krow, d, k_codes + r * d, k_scale + r);
            quant_row_int8(v_new + (t * heads + h) * (int64_t)d, d, v_codes + r * d, v_scale + r);
        }
    }
    free(krow);
    return bad;
}

/* ---------------------------------------------------------------- FP8 (e4m3) */

/* The nearest e4m3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, largest finite 448, subnormal spacing 2^-9), ties to even;
 * finite values beyond 448 saturate to +-448.  The FP8 path of the Flash
 * Attention page, section 18.5 (an FP8 mode with block quantisation). */
static double round_e4m3(double x)
{
    if (x != x || x == 0.0) return x;
    double a = fabs(x);
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1: binade [2^(e-1), 2^e) */
    int q = (e - 1) - 3;         /* 3 mantissa bits */
    if (q < -9) q = -9;          /* subnormal spacing */
    double r = rint(a / ldexp(1.0, q)) * ldexp(1.0, q);
    if (r > 448.0) r = 448.0;
    return copysign(r, x);
}

void oracle_round_e4m3(double *x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) x[i] = round_e4m3(x[i]);
}

/* Quantise groups of values to e4m3 with one fp32 scale per group: scale =
 * max|x| / 448, value = e4m3(x / scale) with x / scale in fp32 (as the path
 * decides it); an all-zero group gets scale 0 and values 0.  codes receives
 * the e4m3 VALUES (not their bit patterns).
 *   x [groups][n] (exact in fp32) -> codes [groups][n], scales [groups] */
void oracle_quant_e4m3(const double *x, int64_t groups, int64_t n, double *codes, float *scales)
{
    for (int64_t g = 0; g < groups; ++g) {
        const double *xg = x + g * n;
        float amax = 0.0f;
        for (int64_t i = 0; i < n; ++i) {
            float a = fabsf((float)xg[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 448.0f;
        scales[g] = s;
        for (int64_t i = 0; i < n; ++i)
            codes[g * n + i] = s == 0.0f ? 0.0 : round_e4m3((double)((float)xg[i] / s));
    }
}

/* Decode: q [B][hq][d] (already rotated, at position ctx_b - 1) against the
 * ctx_b cached tokens of request b.  out [B][hq][d], lse [B][hq]. */
int oracle_decode_paged(const double *q, const double *k_cache, const double *v_cache,
                        const int32_t *page_table, const int32_t *ctx_lens, int batch,
                        int max_pages, int page, int64_t num_pages, int hq, int hkv, int d,
                        double scale, double *out, double *lse)
{
    if (hkv <= 0 || hq % hkv != 0 || page <= 0) return -1;
    const int G = hq / hkv;
    int32_t maxc = 0;
    for (int b = 0; b < batch; ++b) {
        if (ctx_lens[b] < 0) return -1;
        if (ctx_lens[b] > maxc) maxc = ctx_lens[b];
    }
    int bad = 0;
#pragma omp parallel
    {
        size_t n = (size_t)(maxc > 0 ? maxc : 1);
        double *kb = (double *)malloc(sizeof(double) * n * (size_t)d);
        double *vb = (double *)malloc(sizeof(double) * n * (size_t)d);
        int32_t *kp = (int32_t *)malloc(sizeof(int32_t) * n);
        double *sc = (double *)malloc(sizeof(double) * n);
        for (int32_t j = 0; j < maxc; ++j) kp[j] = j;
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < (int64_t)batch * hkv; ++it) {
            int b = (int)(it / hkv), g = (int)(it % hkv);
            int32_t ctx = ctx_lens[b];
            if (oracle_gather_pages(k_cache, page_table, max_pages, page, num_pages, d, g, b, ctx, kb) ||
                oracle_gather_pages(v_cache, page_table, max_pages, page, num_pages, d, g, b, ctx, vb)) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int h = g * G; h < (g + 1) * G; ++h)
                attend_row(q + ((int64_t)b * hq + h) * d, kb, vb, d, kp, ctx, ctx - 1, 1, d,
                           scale, sc, out + ((int64_t)b * hq + h) * d, lse + (int64_t)b * hq + h);
        }
        free(kb); free(vb); free(kp); free(sc);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------ LSE merge */

/* part_o [n_parts][n][d], part_lse [n_parts][n] -> out [n][d], lse [n]:
 *   LSE* = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE*) O_s.
 * Parts with LSE = -inf carry weight 0; if every part is -inf, O = 0 and
 * LSE* = -inf.  The sum is evaluated relative to max_s LSE_s. */
void oracle_lse_merge(const double *part_o, const double *part_lse, int n_parts, int64_t n,
                      int d, double *out, double *lse)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double mx = -INFINITY;
        for (int s = 0; s < n_parts; ++s) {
            double l = part_lse[(int64_t)s * n + r];
            if (l > mx) mx = l;
        }
        double *o = out + r * (int64_t)d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (mx == -INFINITY) { lse[r] = -INFINITY; continue; }
        double S = 0.0;
        for (int s = 0; s < n_parts; ++s) {
            double l = part_lse[(int64_t)s * n + r];
            if (l != -INFINITY) S += exp(l - mx);
        }
        double L = mx + log(S);
        for (int s = 0; s < n_parts; ++s) {
            double l = part_lse[(int64_t)s * n + r];
            if (l == -INFINITY) continue;
            double w = exp(l - L);
            const double *po = part_o + ((int64_t)s * n + r) * d;
            for (int i = 0; i < d; ++i) o[i] += w * po[i];
        }
        lse[r] = L;
    }
}
