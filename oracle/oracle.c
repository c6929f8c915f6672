/*
 * oracle.c -- float64 CPU reference for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: it is used by tests/, by the smoke check in
 * __graft_entry__.py and by the cpu_baseline / reference arm of bench.py.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition, no splitting, no blocking):
 *
 *   For each sequence b, query position i in [0, Q) and query head h:
 *     kvh      = floor(h / g),  g = Hq / Hk          (contiguous GQA groups;
 *                the HRX issue page only states "32 query heads / 4 KV heads",
 *                "Other models / GQA configurations" disposition)
 *     T        = { t : 0 <= t < L_b, and t <= L_b - Q + i when causal }
 *                (bottom-right causal alignment for a multi-token query)
 *     K_t      = K_pool[ table[b][t / P], kvh, t mod P, : ]   (same for V)
 *     z_t      = scale * sum_d q[b,i,h,d] * K_t[d]             (in double)
 *     out      = sum_t exp(z_t - max z) V_t / sum_t exp(z_t - max z)
 *     lse      = max z + ln sum_t exp(z_t - max z)
 *   An empty T gives out = 0 and lse = -inf.
 *
 * This is softmax(q K^T * scale) V over the tokens gathered through the page
 * table: the "partial KV block" / normalisation-scratch machinery of the HRX
 * issue (root cause and multipass sections) and the "o and lse" outputs of the
 * FlashInfer PR ("What changed") reach exactly this result in exact arithmetic,
 * so the oracle has no splits.  K/V element (page, head, slot, dim) lives at
 * base + page*stride_page + head*stride_head + slot*stride_token + dim, which
 * covers the separate-pool, interleaved [pages,2,...] and [2,pages,...] forms
 * named in the FlashInfer PR's "Architecture / design notes" table.
 *
 * oracle_merge_states: the log-sum-exp combination of normalised (o, lse)
 * states (the merge/cascade operation the FlashInfer test plan names):
 *   lse = ln sum_i exp(lse_i),  o = sum_i exp(lse_i - lse) o_i,
 * with states whose lse is -inf contributing nothing.
 *
 * 16-bit storage is decoded to double exactly, from the IEEE 754 binary16
 * definition and from the bfloat16 definition (the top half of a binary32).
 *
 * Quantised caches: K and V may instead be stored as 8-bit E4M3 floating point
 * (the fp8 caches of the FlashInfer PR's AITER paged-attention notes, which
 * carry a k_scale and a v_scale).  Then the key and value of a token are
 *   K_t = k_scale * e4m3(K_stored),   V_t = v_scale * e4m3(V_stored)
 * and everything above applies unchanged to these K_t, V_t.  For 16-bit caches
 * the same scales apply (1 gives the plain definition).
 *
 * Or K and V may be stored as q8_0, the block format of the llama.cpp caches the
 * turboquant PR runs ("q8_0-K", and "KV cache types (q8_0 / q4_0)" in the HRX
 * issue); the pages name it without printing it, and its public definition is:
 * a row of d elements is d/32 blocks of 32 signed 8-bit codes, each block with one
 * binary16 scale, and element e of the row is scale[e / 32] * code[e].  The codes
 * live in the K / V pool at the addresses above (one byte each), the scales in a
 * pool of their own, scale j of (page, head, slot) at
 * base + page*stride_page + head*stride_head + slot*stride_token + j.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);             /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/2^10) * 2^(expo-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xff;
    int frac = bits & 0x7f;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -133);            /* frac * 2^-126 * 2^-7 */
    } else if (expo == 255) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(128 + frac), expo - 134); /* (1 + frac/2^7) * 2^(expo-127) */
    }
    return sign ? -mag : mag;
}

/* OCP 8-bit floating point E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits
 * (bias 7), 3 fraction bits; exponent 0 is subnormal; there is no infinity and
 * only S.1111.111 is NaN, so the largest magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int expo = (bits >> 3) & 0xf;
    int frac = bits & 0x7;
    double mag;
    if (expo == 0xf && frac == 0x7) {
        mag = NAN;
    } else if (expo == 0) {
        mag = ldexp((double)frac, -9);              /* frac/8 * 2^-6 */
    } else {
        mag = ldexp((double)(8 + frac), expo - 10); /* (1 + frac/8) * 2^(expo-7) */
    }
    return sign ? -mag : mag;
}

typedef double (*decode_fn)(uint16_t);

/* Storage formats of a K or V pool. */
#define ORACLE_KV_16BIT 0
#define ORACLE_KV_E4M3 1
#define ORACLE_KV_Q8_0 2

/* Element e of a K or V row whose first element is pool[idx]: 16-bit (decoded by
 * dec), E4M3, or q8_0 with the row's scales at scales[sidx ...]. */
static double kv_elem(const void* pool, int64_t idx, int e, int kv_fmt, decode_fn dec, const uint16_t* scales,
                      int64_t sidx) {
    if (kv_fmt == ORACLE_KV_E4M3) return oracle_e4m3_to_double(((const uint8_t*)pool)[idx + e]);
    if (kv_fmt == ORACLE_KV_Q8_0)
        return oracle_f16_to_double(scales[sidx + e / 32]) * (double)((const int8_t*)pool)[idx + e];
    return dec(((const uint16_t*)pool)[idx + e]);
}

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_PAGE (-2)

int oracle_paged_attention(
    const uint16_t* q, int64_t q_off, int64_t q_stride_tok, int64_t q_stride_head,
    const void* k, int64_t k_off, int64_t k_pages, int64_t k_sp, int64_t k_sh, int64_t k_st,
    const void* v, int64_t v_off, int64_t v_pages, int64_t v_sp, int64_t v_sh, int64_t v_st,
    const int32_t* table, int64_t table_stride, const int32_t* seq_lens,
    int batch, int q_len, int hq, int hk, int d, int page_size, int is_bf16, int causal,
    double scale, int kv_fmt, double k_scale, double v_scale,
    const uint16_t* ksc, int64_t ksc_off, int64_t ksc_sp, int64_t ksc_sh, int64_t ksc_st,
    const uint16_t* vsc, int64_t vsc_off, int64_t vsc_sp, int64_t vsc_sh, int64_t vsc_st,
    const int64_t* rows, int64_t n_rows, double* out, double* lse, int n_threads)
{
    if (batch < 0 || q_len < 1 || hq < 1 || hk < 1 || hq % hk != 0 || d < 1 || page_size < 1)
        return ORACLE_BAD_ARG;
    if (kv_fmt < ORACLE_KV_16BIT || kv_fmt > ORACLE_KV_Q8_0) return ORACLE_BAD_ARG;
    if (kv_fmt == ORACLE_KV_Q8_0 && (d % 32 != 0 || ksc == NULL || vsc == NULL)) return ORACLE_BAD_ARG;
    const int g = hq / hk;
    const decode_fn dec = is_bf16 ? oracle_bf16_to_double : oracle_f16_to_double;
    const int64_t total_rows = (int64_t)batch * q_len * hq;
    const int64_t nr = rows ? n_rows : total_rows;
    int status = ORACLE_OK;
    int64_t max_len = 0;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[b] > max_len) max_len = seq_lens[b];

#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < nr; ++n) {
            const int64_t row = rows ? rows[n] : n;        /* row = (b*Q + i)*Hq + h */
            double* o_row = out + n * d;
            if (row < 0 || row >= total_rows) {
#pragma omp atomic write
                status = ORACLE_BAD_ARG;
                continue;
            }
            const int h = (int)(row % hq);
            const int64_t tok = row / hq;                   /* b*Q + i */
            const int i = (int)(tok % q_len);
            const int b = (int)(tok / q_len);
            const int kvh = h / g;
            const int64_t L = seq_lens[b];
            int64_t n_vis = L;                              /* tokens 0 .. n_vis-1 are visible */
            if (causal) {
                int64_t last = L - q_len + i;               /* bottom-right alignment */
                n_vis = last + 1 < L ? last + 1 : L;
            }
            if (n_vis < 0) n_vis = 0;

            const uint16_t* qp = q + q_off + tok * q_stride_tok + (int64_t)h * q_stride_head;
            for (int e = 0; e < d; ++e) qd[e] = dec(qp[e]);

            /* scores over the gathered keys */
            double zmax = -INFINITY;
            for (int64_t t = 0; t < n_vis; ++t) {
                const int64_t page = table[(int64_t)b * table_stride + t / page_size];
                const int64_t slot = t % page_size;
                if (page < 0 || page >= k_pages || page >= v_pages) {
#pragma omp atomic write
                    status = ORACLE_BAD_PAGE;
                    z[t] = -INFINITY;
                    continue;
                }
                const int64_t kp = k_off + page * k_sp + (int64_t)kvh * k_sh + slot * k_st;
                const int64_t ks = ksc_off + page * ksc_sp + (int64_t)kvh * ksc_sh + slot * ksc_st;
                double s = 0.0;
                for (int e = 0; e < d; ++e) s += qd[e] * (k_scale * kv_elem(k, kp, e, kv_fmt, dec, ksc, ks));
                z[t] = scale * s;
                if (z[t] > zmax) zmax = z[t];
            }

            /* softmax-weighted sum of the gathered values */
            for (int e = 0; e < d; ++e) acc[e] = 0.0;
            double denom = 0.0;
            for (int64_t t = 0; t < n_vis; ++t) {
                const int64_t page = table[(int64_t)b * table_stride + t / page_size];
                if (page < 0 || page >= k_pages || page >= v_pages) continue;
                const int64_t slot = t % page_size;
                const int64_t vp = v_off + page * v_sp + (int64_t)kvh * v_sh + slot * v_st;
                const int64_t vs = vsc_off + page * vsc_sp + (int64_t)kvh * vsc_sh + slot * vsc_st;
                const double w = exp(z[t] - zmax);
                denom += w;
                for (int e = 0; e < d; ++e) acc[e] += w * (v_scale * kv_elem(v, vp, e, kv_fmt, dec, vsc, vs));
            }
            if (n_vis == 0 || denom == 0.0) {
                for (int e = 0; e < d; ++e) o_row[e] = 0.0;
                lse[n] = -INFINITY;
            } else {
                for (int e = 0; e < d; ++e) o_row[e] = acc[e] / denom;
                lse[n] = zmax + log(denom);
            }
        }
        free(z);
        free(qd);
        free(acc);
    }
    return status;
}

/* Merge n_states normalised attention states, each [rows][d] with lse [rows]. */
int oracle_merge_states(const double* o, const double* lse, int n_states, int64_t rows, int d,
                        double* o_out, double* lse_out)
{
    if (n_states < 0 || rows < 0 || d < 1) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < n_states; ++s) {
            const double x = lse[(int64_t)s * rows + r];
            if (x > m) m = x;
        }
        double* orow = o_out + r * d;
        for (int e = 0; e < d; ++e) orow[e] = 0.0;
        if (m == -INFINITY) {
            lse_out[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int s = 0; s < n_states; ++s) sum += exp(lse[(int64_t)s * rows + r] - m);
        const double total = m + log(sum);
        for (int s = 0; s < n_states; ++s) {
            const double w = exp(lse[(int64_t)s * rows + r] - total);
            const double* os = o + ((int64_t)s * rows + r) * d;
            for (int e = 0; e < d; ++e) orow[e] += w * os[e];
        }
        lse_out[r] = total;
    }
    return ORACLE_OK;
}
