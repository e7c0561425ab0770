/*
 * csa_oracle.c -- plain, slow, fp64 CPU oracle for the CSA + HCA hybrid
 * compressed attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; both sides only read the same seeded inputs.
 *
 * Sources (cited by page title and section):
 *   [V4]   "DeepSeek-V4 core architecture" (gitcode.csdn.net article),
 *          §2.2 "CSA: compressed sparse attention" -- step 1 token-level
 *          compression, step 2 lightning indexer, step 3 shared-KV MQA;
 *          §2.3 "HCA: heavily compressed attention";
 *          §9 "key innovations summary" (table row 5: the indexer QK
 *          product is quantised);
 *   [DEBT] "DeepSeek V4's architecture debt chain" (vendordeep.com),
 *          "Constraint 1 -> Innovation 1: CSA+HCA hybrid attention"
 *          (128x fusion of many tokens' KV into one compressed token).
 *   [SWA]  the bjdmk.com.cn DeepSeek-V4 walkthrough, §3.2 "SWA
 *          sliding-window attention": each token attends only to the
 *          tokens of a fixed window before it (4096 in its example).
 *
 * Readings where the pages leave a step open (all listed in the design
 * notes):
 *   R1  indexer score s(t,j) = sum over indexer heads h of q_{t,h} . k_j
 *       (one key vector per compressed entry, shared by all heads); no
 *       ReLU, weight or scale.
 *   R2  a query also attends to the raw tokens of its own incomplete block.
 *   R3  a block's entry is visible only once the block is complete:
 *       entry j (tokens j*m .. j*m+m-1) is visible to position t iff
 *       (j+1)*m <= t+1.
 *   A1  blocks are non-overlapping and aligned at position 0.
 *   A2  one scalar gate logit per token, shared across the d channels;
 *       the block's weights are the softmax of its tokens' logits.
 *   A7  top-k order: higher score first, ties to the lower entry index;
 *       the selected indices are returned ascending, padded with -1.
 *   P1-P4 [DEBT]'s inverse-RoPE correction of the attention output (the
 *       pages give no convention; readings): P1 the rotated dims are the
 *       last d_rope of each head's d; P2 they pair as (2i, 2i+1) within that
 *       slice; P3 pair i turns at theta_i = base^(-2i/d_rope); P4 the output
 *       of the query at position t is turned by the angle -t * theta_i.
 *       Parity partly unpinned: the pins fix the direction, the pairing
 *       against the forward rotary embedding and the linearity in t, not
 *       the readings P1-P3 themselves.
 *   W1  [SWA] the window of a token at position t holds positions
 *       max(0, t - w + 1) .. t: the token itself and the w - 1 before it.
 *   R8  the low-precision indexer stores each key row as FP8 E4M3 codes
 *       scaled so the row's largest magnitude maps to 448, plus an fp32
 *       scale (see the FP8 section below).
 *
 * Everything is computed in double precision; bf16 and fp32 inputs
 * convert to double exactly.  Plain loops, no blocking or reordering
 * beyond the definitions.  OpenMP only splits independent queries/blocks.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double (exact: bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Token-level compression ([V4] §2.2 step 1: every m adjacent tokens' KV
 * become one entry, with learnable softmax-normalised weights; [V4] §2.3 and
 * [DEBT]: the same weighted fusion with m = 128 for HCA).
 *
 * Block j of one sequence holds tokens j*m .. j*m+m-1 (A1).  With the gate
 * logits z of those tokens (A2):
 *     w_t = exp(z_t) / sum_{s in block} exp(z_s)
 *     e_j = sum_{t in block} w_t * c_t
 * The largest logit is subtracted before exp (same value, no overflow).
 * ---------------------------------------------------------------------- */
static void compress_block(const uint16_t *c, const float *z, int d, int m,
                           int64_t j, double *e)
{
    const int64_t t0 = j * (int64_t)m;
    double zmax = -INFINITY;
    for (int i = 0; i < m; i++)
        if ((double)z[t0 + i] > zmax) zmax = (double)z[t0 + i];
    double denom = 0.0;
    for (int i = 0; i < m; i++) denom += exp((double)z[t0 + i] - zmax);
    for (int x = 0; x < d; x++) e[x] = 0.0;
    for (int i = 0; i < m; i++) {
        const double w = exp((double)z[t0 + i] - zmax) / denom;
        const uint16_t *row = c + (t0 + i) * (int64_t)d;
        for (int x = 0; x < d; x++) e[x] += w * bf16_to_double(row[x]);
    }
}

/* All complete blocks of one sequence of n_tok tokens: out[n_tok/m, d].
 * A trailing partial block gets no entry (R3). */
int orc_compress(const uint16_t *c, const float *z, int64_t n_tok, int d,
                 int m, double *out)
{
    if (!c || !z || !out || d <= 0 || m <= 0 || n_tok < 0) return 1;
    const int64_t n_blocks = n_tok / m;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n_blocks; j++)
        compress_block(c, z, d, m, j, out + j * (int64_t)d);
    return 0;
}

/* ------------------------------------------------------------------------
 * Lightning indexer scores ([V4] §2.2 step 2: a light scorer rates each
 * query against every compressed entry), in the form R1 fixes:
 *     s_j = sum_{h < HI} sum_{i < dI} qI[h, i] * kI[j, i]
 * qI: [HI, dI] one query's indexer heads; kI: [n, dI] one key per entry.
 * ---------------------------------------------------------------------- */
int orc_index_scores(const uint16_t *qI, const uint16_t *kI, int64_t n,
                     int HI, int dI, double *s)
{
    if (!qI || (!kI && n > 0) || (!s && n > 0) || HI <= 0 || dI <= 0) return 1;
    for (int64_t j = 0; j < n; j++) {
        double acc = 0.0;
        for (int h = 0; h < HI; h++)
            for (int i = 0; i < dI; i++)
                acc += bf16_to_double(qI[h * dI + i]) *
                       bf16_to_double(kI[j * (int64_t)dI + i]);
        s[j] = acc;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * FP8 indexer keys ([V4] §9 "key innovations summary", table row 5: the
 * indexer's QK product runs quantised).  Reading R8: each key row j is
 * scaled so its largest magnitude maps to 448, the largest finite FP8 E4M3
 * value, and stored as E4M3 codes plus one fp32 scale; the score is then
 * the R1 score on the dequantised keys.  The pages give no quantiser; the
 * tests pin these functions to the E4M3 format's definition instead.
 *
 * E4M3 ("e4m3fn"): sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * no infinities; exponent 15 with mantissa 7 is NaN, so the largest finite
 * value is 1.75 * 2^8 = 448; exponent 0 holds the subnormals m/8 * 2^-6.
 * ---------------------------------------------------------------------- */
double orc_e4m3_decode(uint8_t c)
{
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp(m / 8.0, -6);
    else        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round to the nearest finite E4M3 value, ties to the code with an even
 * mantissa, magnitudes above 448 saturate to 448 (the "satfinite" mode).
 * The sign is kept, so negative values that round to zero give -0 (0x80).
 * Plain scan over the 127 finite magnitudes 0x00 .. 0x7e, which ascend. */
uint8_t orc_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a >= 448.0) return sign | 0x7e;
    int lo = 0;
    while (lo + 1 <= 0x7e && orc_e4m3_decode((uint8_t)(lo + 1)) <= a) lo++;
    if (lo == 0x7e) return sign | 0x7e;
    const double dlo = a - orc_e4m3_decode((uint8_t)lo);
    const double dhi = orc_e4m3_decode((uint8_t)(lo + 1)) - a;
    int c;
    if (dlo < dhi)      c = lo;
    else if (dhi < dlo) c = lo + 1;
    else                c = (lo & 1) ? lo + 1 : lo;
    return sign | (uint8_t)c;
}

/* Quantise n key rows of width dI (bf16) to E4M3 codes and fp32 scales.
 * The scaling arithmetic is fp32 with IEEE rounding, as the format of the
 * stored scale fixes it: a = max |k|, inv = 448 / a, q = k * inv,
 * scale = a / 448; a row of zeros gets codes 0 and scale 0. */
int orc_quantize_index_keys(const uint16_t *kI, int64_t n, int dI,
                            uint8_t *codes, float *scale)
{
    if ((n > 0 && (!kI || !codes || !scale)) || dI <= 0) return 1;
    for (int64_t j = 0; j < n; j++) {
        float a = 0.0f;
        for (int i = 0; i < dI; i++) {
            const float v = (float)bf16_to_double(kI[j * (int64_t)dI + i]);
            if (fabsf(v) > a) a = fabsf(v);
        }
        if (a == 0.0f) {
            for (int i = 0; i < dI; i++) codes[j * (int64_t)dI + i] = 0;
            scale[j] = 0.0f;
            continue;
        }
        const float inv = 448.0f / a;
        for (int i = 0; i < dI; i++) {
            const float v = (float)bf16_to_double(kI[j * (int64_t)dI + i]);
            const float q = v * inv;
            codes[j * (int64_t)dI + i] = orc_e4m3_encode((double)q);
        }
        scale[j] = a / 448.0f;
    }
    return 0;
}

/* R1 score on the dequantised keys: s_j = sum_h sum_i qI[h,i] * kq[j,i]
 * with kq[j,i] = scale_j * e4m3(codes[j,i]) (exact in double). */
int orc_index_scores_fp8(const uint16_t *qI, const uint8_t *codes,
                         const float *scale, int64_t n, int HI, int dI,
                         double *s)
{
    if (!qI || (n > 0 && (!codes || !scale || !s)) || HI <= 0 || dI <= 0)
        return 1;
    for (int64_t j = 0; j < n; j++) {
        double acc = 0.0;
        for (int h = 0; h < HI; h++)
            for (int i = 0; i < dI; i++)
                acc += bf16_to_double(qI[h * dI + i]) *
                       ((double)scale[j] *
                        orc_e4m3_decode(codes[j * (int64_t)dI + i]));
        s[j] = acc;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Top-k ([V4] §2.2 step 2: keep only the k most relevant entries).
 * Order (A7): score descending, then index ascending.  The first min(k, n)
 * are returned in ascending index order, the rest of idx[0..k) is -1.
 * The library sort (qsort) is the selection step.
 * ---------------------------------------------------------------------- */
typedef struct { double s; int64_t j; } scored_t;

static int cmp_scored(const void *a, const void *b)
{
    const scored_t *x = (const scored_t *)a, *y = (const scored_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int cmp_i32(const void *a, const void *b)
{
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int orc_topk(const double *s, int64_t n, int k, int32_t *idx)
{
    if ((!s && n > 0) || !idx || k <= 0 || n < 0) return 1;
    scored_t *all = (scored_t *)malloc(sizeof(scored_t) * (size_t)(n > 0 ? n : 1));
    if (!all) return 2;
    for (int64_t j = 0; j < n; j++) { all[j].s = s[j]; all[j].j = j; }
    qsort(all, (size_t)n, sizeof(scored_t), cmp_scored);
    const int64_t take = n < k ? n : k;
    for (int64_t i = 0; i < take; i++) idx[i] = (int32_t)all[i].j;
    qsort(idx, (size_t)take, sizeof(int32_t), cmp_i32);
    for (int64_t i = take; i < k; i++) idx[i] = -1;
    free(all);
    return 0;
}

/* ------------------------------------------------------------------------
 * Multi-query attention with shared KV ([V4] §2.2 step 3: every selected
 * entry is both Key and Value, and all query heads share the same KV).
 * q: [H, d] bf16; keys: [nk, d] fp64.  Per head h:
 *     l_i = scale * q_h . x_i,  p = softmax(l),  o_h = sum_i p_i x_i,
 *     lse_h = log sum_i exp(l_i)   (natural log)
 * ---------------------------------------------------------------------- */
int orc_attend(const uint16_t *q, int H, int d, const double *keys, int64_t nk,
               double scale, double *o, double *lse)
{
    if (!q || !keys || !o || H <= 0 || d <= 0 || nk <= 0) return 1;
    double *l = (double *)malloc(sizeof(double) * (size_t)nk);
    if (!l) return 2;
    for (int h = 0; h < H; h++) {
        const uint16_t *qh = q + (int64_t)h * d;
        double lmax = -INFINITY;
        for (int64_t i = 0; i < nk; i++) {
            double acc = 0.0;
            for (int x = 0; x < d; x++)
                acc += bf16_to_double(qh[x]) * keys[i * (int64_t)d + x];
            l[i] = scale * acc;
            if (l[i] > lmax) lmax = l[i];
        }
        double denom = 0.0;
        for (int64_t i = 0; i < nk; i++) denom += exp(l[i] - lmax);
        double *oh = o + (int64_t)h * d;
        for (int x = 0; x < d; x++) oh[x] = 0.0;
        for (int64_t i = 0; i < nk; i++) {
            const double p = exp(l[i] - lmax) / denom;
            for (int x = 0; x < d; x++) oh[x] += p * keys[i * (int64_t)d + x];
        }
        if (lse) lse[h] = lmax + log(denom);
    }
    free(l);
    return 0;
}

/* ------------------------------------------------------------------------
 * Whole queries of a packed batch.
 *
 * Sequence b owns tokens cu_kv[b] .. cu_kv[b+1]-1 (length L_b), CSA entries
 * cu_csa[b] .. (floor(L_b/mC) of them) and queries cu_q[b] .. cu_q[b+1]-1;
 * its queries are its last n_q = cu_q[b+1]-cu_q[b] positions.  For a query
 * at position t (0-based within its sequence):
 *     n_C = floor((t+1)/mC),  r_C = (t+1) mod mC     (R3, R2)
 *     n_H = floor((t+1)/mH),  r_H = (t+1) mod mH
 * CSA ([V4] §2.2): scores over entries j < n_C (R1), top-k (A7), attention
 *   over the selected entries plus the r_C raw tokens t-r_C+1 .. t.
 * HCA ([V4] §2.3): attention over all n_H entries plus the r_H raw tokens.
 *
 * The CSA entries a query needs are compressed on demand from the raw
 * tokens; the HCA entries are taken from hca_entries (fp64, from
 * orc_compress with m = mH, packed by cu_hca).  When given_idx is not NULL
 * the CSA branch attends over those indices instead of its own top-k (to
 * check attention on another selection).  Outputs (per evaluated query):
 * idx[k] int32, oC[H,d], lseC[H], oH[H,d], lseH[H]; any output may be NULL
 * to skip that branch's output (the CSA branch still needs idx storage
 * internally).
 * ---------------------------------------------------------------------- */
static int64_t find_seq(int B, const int64_t *cu_q, int64_t qi)
{
    int64_t lo = 0, hi = B - 1;
    while (lo < hi) {
        int64_t mid = (lo + hi + 1) / 2;
        if (cu_q[mid] <= qi) lo = mid; else hi = mid - 1;
    }
    return lo;
}

int orc_hybrid_queries(int B, const int64_t *cu_kv, const int64_t *cu_q,
                       const int64_t *cu_csa, const int64_t *cu_hca,
                       const uint16_t *kv, const float *gate,
                       const uint16_t *qI, const uint16_t *kI,
                       const uint16_t *q, int d, int H, int HI, int dI,
                       int mC, int mH, int top_k, double scale,
                       const double *hca_entries, int64_t n_eval,
                       const int64_t *eval_q, const int32_t *given_idx,
                       int do_csa, int do_hca,
                       int32_t *idx_out, double *oC, double *lseC,
                       double *oH, double *lseH)
{
    if (B <= 0 || !cu_kv || !cu_q || !kv || !q || d <= 0 || H <= 0 ||
        mC <= 0 || mH <= 0 || top_k <= 0 || n_eval < 0 || !eval_q)
        return 1;
    if (do_csa && (!cu_csa || !gate || !qI || !kI)) return 1;
    if (do_hca && (!cu_hca || !hca_entries)) return 1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t e = 0; e < n_eval; e++) {
        const int64_t qi = eval_q[e];
        const int64_t b = find_seq(B, cu_q, qi);
        const int64_t L = cu_kv[b + 1] - cu_kv[b];
        const int64_t nq = cu_q[b + 1] - cu_q[b];
        const int64_t t = L - nq + (qi - cu_q[b]);
        const uint16_t *c_seq = kv + cu_kv[b] * (int64_t)d;
        const uint16_t *q_t = q + qi * (int64_t)H * d;
        if (t < 0 || t >= L) { err |= 1; continue; }

        if (do_csa) {
            const int64_t nC = (t + 1) / mC, rC = (t + 1) % mC;
            int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)top_k);
            if (!sel) { err |= 2; continue; }
            if (given_idx) {
                memcpy(sel, given_idx + e * (int64_t)top_k, sizeof(int32_t) * (size_t)top_k);
            } else {
                double *s = (double *)malloc(sizeof(double) * (size_t)(nC > 0 ? nC : 1));
                if (!s) { free(sel); err |= 2; continue; }
                err |= orc_index_scores(qI + qi * (int64_t)HI * dI,
                                        kI + cu_csa[b] * (int64_t)dI, nC, HI, dI, s);
                err |= orc_topk(s, nC, top_k, sel);
                free(s);
            }
            if (idx_out) memcpy(idx_out + e * (int64_t)top_k, sel, sizeof(int32_t) * (size_t)top_k);
            int64_t nsel = 0;
            for (int i = 0; i < top_k; i++) if (sel[i] >= 0) nsel++;
            const int64_t nk = nsel + rC;
            double *keys = (double *)malloc(sizeof(double) * (size_t)nk * d);
            if (!keys) { free(sel); err |= 2; continue; }
            int64_t w = 0;
            for (int i = 0; i < top_k; i++) {
                if (sel[i] < 0) continue;
                if (sel[i] >= nC) err |= 4;   /* not visible: invalid selection */
                else compress_block(c_seq, gate + cu_kv[b], d, mC, sel[i], keys + w * d);
                w++;
            }
            for (int64_t r = 0; r < rC; r++, w++) {
                const uint16_t *row = c_seq + (t - rC + 1 + r) * (int64_t)d;
                for (int x = 0; x < d; x++) keys[w * d + x] = bf16_to_double(row[x]);
            }
            if (oC)
                err |= orc_attend(q_t, H, d, keys, nk, scale,
                                  oC + e * (int64_t)H * d, lseC ? lseC + e * (int64_t)H : NULL);
            free(keys);
            free(sel);
        }
        if (do_hca) {
            const int64_t nH = (t + 1) / mH, rH = (t + 1) % mH;
            const int64_t nk = nH + rH;
            double *keys = (double *)malloc(sizeof(double) * (size_t)nk * d);
            if (!keys) { err |= 2; continue; }
            memcpy(keys, hca_entries + cu_hca[b] * (int64_t)d, sizeof(double) * (size_t)(nH * d));
            for (int64_t r = 0; r < rH; r++) {
                const uint16_t *row = c_seq + (t - rH + 1 + r) * (int64_t)d;
                for (int x = 0; x < d; x++) keys[(nH + r) * d + x] = bf16_to_double(row[x]);
            }
            if (oH)
                err |= orc_attend(q_t, H, d, keys, nk, scale,
                                  oH + e * (int64_t)H * d, lseH ? lseH + e * (int64_t)H : NULL);
            free(keys);
        }
    }
    return err;
}

/* Compress the blocks of every sequence of a packed batch (entries packed
 * by cu_out, floor(L_b/m) per sequence).  Used to build fp64 HCA entries. */
int orc_compress_packed(int B, const int64_t *cu_kv, const int64_t *cu_out,
                        const uint16_t *kv, const float *gate, int d, int m,
                        double *out)
{
    if (B <= 0 || !cu_kv || !cu_out || !kv || !gate || !out) return 1;
    int err = 0;
    for (int b = 0; b < B; b++) {
        const int64_t L = cu_kv[b + 1] - cu_kv[b];
        if (cu_out[b + 1] - cu_out[b] != L / m) return 3;
        err |= orc_compress(kv + cu_kv[b] * (int64_t)d, gate + cu_kv[b], L, d, m,
                            out + cu_out[b] * (int64_t)d);
    }
    return err;
}

/* Compress only the listed blocks (global entry indices into the packed
 * entry array), for sampled checks at full size. */
int orc_compress_selected(int B, const int64_t *cu_kv, const int64_t *cu_out,
                          const uint16_t *kv, const float *gate, int d, int m,
                          int64_t n_sel, const int64_t *entry, double *out)
{
    if (B <= 0 || !cu_kv || !cu_out || !kv || !gate || !out || !entry) return 1;
    int err = 0;
#pragma omp parallel for schedule(static) reduction(| : err)
    for (int64_t i = 0; i < n_sel; i++) {
        const int64_t g = entry[i];
        /* the last sequence whose first entry is <= g owns entry g */
        const int64_t bb = find_seq(B, cu_out, g);
        const int64_t j = g - cu_out[bb];
        const int64_t L = cu_kv[bb + 1] - cu_kv[bb];
        if (j < 0 || (j + 1) * m > L) { err |= 4; continue; }
        compress_block(kv + cu_kv[bb] * (int64_t)d, gate + cu_kv[bb], d, m, j,
                       out + i * (int64_t)d);
    }
    return err;
}

/* ------------------------------------------------------------------------
 * Sliding-window attention over the raw tokens ([SWA] §3.2, reading W1),
 * with the shared-KV MQA of [V4] §2.2 step 3: query qi at position t of its
 * sequence attends, with each of its H heads, over the raw token rows
 * max(0, t - w + 1) .. t of its sequence, each row its own key and value.
 * Per evaluated query: o [H, d], lse [H] (natural log).
 * ---------------------------------------------------------------------- */
int orc_swa_queries(int B, const int64_t *cu_kv, const int64_t *cu_q,
                    const uint16_t *kv, const uint16_t *q, int d, int H,
                    int64_t w, double scale, int64_t n_eval,
                    const int64_t *eval_q, double *o, double *lse)
{
    if (B <= 0 || !cu_kv || !cu_q || !kv || !q || d <= 0 || H <= 0 || w <= 0 ||
        n_eval < 0 || !eval_q || !o)
        return 1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int64_t e = 0; e < n_eval; e++) {
        const int64_t qi = eval_q[e];
        const int64_t b = find_seq(B, cu_q, qi);
        const int64_t L = cu_kv[b + 1] - cu_kv[b];
        const int64_t nq = cu_q[b + 1] - cu_q[b];
        const int64_t t = L - nq + (qi - cu_q[b]);
        if (t < 0 || t >= L) { err |= 1; continue; }
        const int64_t u0 = t - w + 1 > 0 ? t - w + 1 : 0;
        const int64_t nk = t - u0 + 1;
        double *keys = (double *)malloc(sizeof(double) * (size_t)nk * d);
        if (!keys) { err |= 2; continue; }
        for (int64_t r = 0; r < nk; r++) {
            const uint16_t *row = kv + (cu_kv[b] + u0 + r) * (int64_t)d;
            for (int x = 0; x < d; x++) keys[r * d + x] = bf16_to_double(row[x]);
        }
        err |= orc_attend(q + qi * (int64_t)H * d, H, d, keys, nk, scale,
                          o + e * (int64_t)H * d, lse ? lse + e * (int64_t)H : NULL);
        free(keys);
    }
    return err;
}

/* ------------------------------------------------------------------------
 * Inverse-RoPE correction of attention outputs ([DEBT] "Constraint 1 ->
 * Innovation 1": the attention output receives an inverse rotary
 * correction; readings P1-P4).  For the query qi at position t of its
 * sequence, each head h and pair i < d_rope / 2, with
 *     phi = t * base^(-2i / d_rope),
 *     (x, y) = (o[qi, h, d - d_rope + 2i], o[qi, h, d - d_rope + 2i + 1]),
 * the pair becomes (x cos phi + y sin phi, -x sin phi + y cos phi), the
 * rotation by -phi; every other dim is copied.  in, out: [nq_total, H, d].
 * ---------------------------------------------------------------------- */
int orc_inverse_rope(int B, const int64_t *cu_kv, const int64_t *cu_q, int H, int d,
                     int d_rope, double base, const double *in, double *out)
{
    if (B <= 0 || !cu_kv || !cu_q || !in || !out || H <= 0 || d <= 0 ||
        d_rope <= 0 || d_rope > d || (d_rope & 1) || !(base > 0.0))
        return 1;
    const int64_t nq_total = cu_q[B];
    int err = 0;
#pragma omp parallel for schedule(static) reduction(| : err)
    for (int64_t qi = 0; qi < nq_total; qi++) {
        const int64_t b = find_seq(B, cu_q, qi);
        const int64_t L = cu_kv[b + 1] - cu_kv[b];
        const int64_t t = L - (cu_q[b + 1] - cu_q[b]) + (qi - cu_q[b]);
        if (t < 0 || t >= L) { err |= 1; continue; }
        for (int h = 0; h < H; h++) {
            const double *x = in + (qi * H + h) * (int64_t)d;
            double *y = out + (qi * H + h) * (int64_t)d;
            for (int c = 0; c < d; c++) y[c] = x[c];
            for (int i = 0; i < d_rope / 2; i++) {
                const double phi = (double)t * pow(base, -2.0 * i / d_rope);
                const double c0 = cos(phi), s0 = sin(phi);
                const int j = d - d_rope + 2 * i;
                y[j] = x[j] * c0 + x[j + 1] * s0;
                y[j + 1] = -x[j] * s0 + x[j + 1] * c0;
            }
        }
    }
    return err;
}
