/*
 * bsa_oracle.c -- plain, slow CPU oracle for block-sparse attention (long prefill).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  The CUDA library never links
 * it, includes it or falls back to it, and this file includes nothing from the CUDA
 * library: the two implementations share no code, header, table or helper.
 *
 * Source of the method.  The post "CUDA inference engine for running Qwen3.5/3.6 hybrid
 * models on mining cards (CMP 100-210)" (news.hada.io topic 29953, feature list) speeds up
 * long prefill with MInference-style block-sparse attention: each block of queries attends
 * only to a chosen set of key blocks.  The post gives no more; the readings:
 *   A1 causal self-attention of a prefill: query t of head h sees keys j <= t, and among
 *      them only those whose 64-token key block is listed as active for the query's
 *      64-token block (a CSR list per head and query block, ascending, blocks <= the
 *      query block).  Blocks and the choice of blocks come from outside (the pattern
 *      search of MInference is not part of this step).
 *   A2 grouped-query attention: H query heads share Hkv key/value heads, head h reading
 *      key/value head h / (H / Hkv).
 *   A3 o_t = sum_j p_j v_j, p = softmax over the visible keys of (q_t . k_j) / sqrt(d);
 *      bf16 inputs widened exactly; evaluated in binary64, rounded once to binary32.  A
 *      query that sees no key gets o_t = 0.
 *   A4 layouts: q [H][T][d], k and v [Hkv][T][d] (d = 128 contiguous), o [H][T][d];
 *      T a multiple of 64.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math -pthread
 *        bsa_oracle.c -o libobsa.so -lm      (oracle/build.py does this)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OBSA_B 64

static double obsa_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* o_t of one query (head h, token t), in binary64, into out[d]. */
void obsa_one_query(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t H,
                    int64_t Hkv, int64_t T, int64_t d, const int32_t *row_ptr,
                    const int32_t *col_idx, int64_t h, int64_t t, double *out)
{
    int64_t nqb = T / OBSA_B;
    int64_t hk = h / (H / Hkv);
    int64_t qb = t / OBSA_B;
    const uint16_t *qt = q + (h * T + t) * d;
    double *s = malloc(sizeof(double) * (size_t)T);
    int64_t *idx = malloc(sizeof(int64_t) * (size_t)T);
    int64_t n = 0;
    double mx = -INFINITY;
    for (int32_t e = row_ptr[h * nqb + qb]; e < row_ptr[h * nqb + qb + 1]; ++e) {
        int64_t kb = col_idx[e];
        for (int64_t j = kb * OBSA_B; j < (kb + 1) * OBSA_B && j <= t; ++j) {
            const uint16_t *kj = k + (hk * T + j) * d;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += obsa_bf16(qt[c]) * obsa_bf16(kj[c]);
            s[n] = dot / sqrt((double)d);
            idx[n] = j;
            if (s[n] > mx)
                mx = s[n];
            ++n;
        }
    }
    for (int64_t c = 0; c < d; ++c)
        out[c] = 0.0;
    if (n > 0) {
        double l = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            s[i] = exp(s[i] - mx);
            l += s[i];
        }
        for (int64_t i = 0; i < n; ++i) {
            const uint16_t *vj = v + (hk * T + idx[i]) * d;
            double p = s[i] / l;
            for (int64_t c = 0; c < d; ++c)
                out[c] += p * obsa_bf16(vj[c]);
        }
    }
    free(s);
    free(idx);
}

/* The whole output o [H][T][d] binary32 (every query of every head). */
void obsa_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t H,
                    int64_t Hkv, int64_t T, int64_t d, const int32_t *row_ptr,
                    const int32_t *col_idx, float *o)
{
    double *out = malloc(sizeof(double) * (size_t)d);
    for (int64_t h = 0; h < H; ++h)
        for (int64_t t = 0; t < T; ++t) {
            obsa_one_query(q, k, v, H, Hkv, T, d, row_ptr, col_idx, h, t, out);
            for (int64_t c = 0; c < d; ++c)
                o[(h * T + t) * d + c] = (float)out[c];
        }
    free(out);
}

/* Sampled queries: o_s = o[heads[s]][tokens[s]][:], for s < n. */
void obsa_attention_at(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t H,
                       int64_t Hkv, int64_t T, int64_t d, const int32_t *row_ptr,
                       const int32_t *col_idx, const int64_t *heads, const int64_t *tokens,
                       int64_t n, float *o)
{
    double *out = malloc(sizeof(double) * (size_t)d);
    for (int64_t s = 0; s < n; ++s) {
        obsa_one_query(q, k, v, H, Hkv, T, d, row_ptr, col_idx, heads[s], tokens[s], out);
        for (int64_t c = 0; c < d; ++c)
            o[s * d + c] = (float)out[c];
    }
    free(out);
}
