/*
 * q8_oracle.c -- plain, slow CPU oracle for the Q8_0 block-quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  The CUDA library never
 * links it, includes it or falls back to it, and this file includes nothing from the
 * CUDA library: the two implementations share no code, header, table or helper.
 *
 * Source of the method.  The post "CUDA inference engine for running Qwen3.5/3.6
 * hybrid models on mining cards (CMP 100-210)" (news.hada.io topic 29953) runs its
 * GEMMs as an int8 DP4A kernel (list of un-throttled paths) and supports only Q8_0
 * weights ("Limitations" list).  The Q8_0 block format this library implements is:
 *   - K is cut into blocks of 32 consecutive elements;
 *   - per block, amax = max |v_j|, scale d = amax / 127, codes q_j = round(v_j / d);
 *   - weight scales are stored as IEEE binary16, activation scales as binary32;
 *   - y[m,n] = sum over blocks b of d_w[n,b] * d_x[m,b] * (sum_j xq[m,32b+j] * wq[n,32b+j]).
 *
 * Readings taken where the definition leaves a step open (each is a reading, and the
 * GPU library takes the same one):
 *   R1  codes are computed from the binary32 scale d32 = fl32(amax / 127), not from its
 *       binary16 rounding; binary16 is only how weight scales are stored.
 *   R2  v / d is one IEEE binary32 division (round to nearest even).
 *   R3  round() is half away from zero (C roundf).
 *   R4  binary32 -> binary16 is IEEE round-to-nearest-even with subnormals; a scale that
 *       underflows to 0 is stored as 0 and its codes are kept.
 *   R5  activation scales stay binary32 (never rounded to binary16).
 *   R6  an all-zero block, or a block whose d32 underflows to 0, gets scale 0 and codes 0.
 *   R7  codes are clamped to [-127, 127]; with a normal d32 the clamp never acts because
 *       |v / d32| <= 127 * (1 + 2^-23) rounds to at most 127.  It acts only when d32 is a
 *       binary32 subnormal (amax below about 2^-119), where d32 carries few bits.
 *   R8  bf16 activations are widened to binary32 exactly before quantization.
 *   R9  y is accumulated in binary64 and rounded once to binary32 (the order of the
 *       floating-point sum is not fixed by the method, so y is compared within a
 *       tolerance; codes, scales and block sums are compared bit for bit).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math -pthread
 *        q8_oracle.c -o liboq8.so -lm      (oracle/build.py does this)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OQ8_QK 32 /* elements per Q8_0 block */

/* ------------------------------------------------------------------------- */
/* IEEE 754 conversions, written from the format definitions.                 */
/* ------------------------------------------------------------------------- */

/* binary32 -> binary16 bits, round to nearest, ties to even, with subnormals.
 * Works in binary64, where every step below is exact except nearbyint(), which
 * rounds to nearest-even in the default floating-point environment. */
uint16_t oq8_f32_to_f16(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    /* 65504 is the largest finite binary16; the midpoint to the next (2^16) is 65520,
     * and a tie there goes to the even neighbour, which is 2^16 = infinity. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7c00u);
    if (a < 0x1p-14) {
        /* subnormal range (or zero): the value is an integer count of 2^-24 */
        double units = nearbyint(a * 0x1p24);
        return (uint16_t)(sign | (uint16_t)units); /* 1024 units is the smallest normal */
    }
    int e;
    double fr = frexp(a, &e); /* a = fr * 2^e, fr in [0.5, 1) */
    int E = e - 1;            /* a = (2 fr) * 2^E, 2 fr in [1, 2) */
    double mant = nearbyint((2.0 * fr - 1.0) * 1024.0);
    if (mant == 1024.0) {
        mant = 0.0;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)mant);
}

/* binary16 bits -> exact binary64 value */
double oq8_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

/* bfloat16 bits -> binary32 (exact: bf16 is the top half of a binary32) */
float oq8_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------- */
/* Quantization of one 32-element block (readings R1-R3, R6, R7).             */
/* ------------------------------------------------------------------------- */

/* Quantizes v[0..31]; writes codes q[0..31] and the binary32 scale *d32. */
void oq8_quantize_block(const float *v, int8_t *q, float *d32)
{
    float amax = 0.0f;
    for (int j = 0; j < OQ8_QK; ++j) {
        float a = fabsf(v[j]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    if (d == 0.0f) {
        *d32 = 0.0f;
        for (int j = 0; j < OQ8_QK; ++j)
            q[j] = 0;
        return;
    }
    for (int j = 0; j < OQ8_QK; ++j) {
        float r = roundf(v[j] / d);
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        q[j] = (int8_t)r;
    }
    *d32 = d;
}

/* W[N,K] binary32 row-major -> Wq[N,K] int8 codes and Wd[N,K/32] binary16 scale bits. */
void oq8_quantize_weights(const float *W, int64_t N, int64_t K, int8_t *Wq, uint16_t *Wd)
{
    int64_t nb = K / OQ8_QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) {
            float d;
            oq8_quantize_block(W + n * K + b * OQ8_QK, Wq + n * K + b * OQ8_QK, &d);
            Wd[n * nb + b] = oq8_f32_to_f16(d);
        }
}

/* x[M,K] binary32 -> xq[M,K] int8 codes and xd[M,K/32] binary32 scales. */
void oq8_quantize_act_f32(const float *x, int64_t M, int64_t K, int8_t *xq, float *xd)
{
    int64_t nb = K / OQ8_QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b)
            oq8_quantize_block(x + m * K + b * OQ8_QK, xq + m * K + b * OQ8_QK, xd + m * nb + b);
}

/* x[M,K] bfloat16 bits -> xq, xd as above (reading R8: widen exactly, then quantize). */
void oq8_quantize_act_bf16(const uint16_t *x, int64_t M, int64_t K, int8_t *xq, float *xd)
{
    int64_t nb = K / OQ8_QK;
    float v[OQ8_QK];
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            for (int j = 0; j < OQ8_QK; ++j)
                v[j] = oq8_bf16_to_f32(x[m * K + b * OQ8_QK + j]);
            oq8_quantize_block(v, xq + m * K + b * OQ8_QK, xd + m * nb + b);
        }
}

/* ------------------------------------------------------------------------- */
/* Per-block integer dot products and the rescaled sum.                       */
/* ------------------------------------------------------------------------- */

/* isum[m,n,b] = sum_{j<32} xq[m,32b+j] * Wq[n,32b+j], exact (|isum| <= 32*127*127). */
void oq8_block_sums(const int8_t *xq, const int8_t *Wq, int64_t M, int64_t N, int64_t K,
                    int32_t *isum)
{
    int64_t nb = K / OQ8_QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b) {
                int64_t s = 0;
                for (int j = 0; j < OQ8_QK; ++j)
                    s += (int64_t)xq[m * K + b * OQ8_QK + j] * (int64_t)Wq[n * K + b * OQ8_QK + j];
                isum[(m * N + n) * nb + b] = (int32_t)s;
            }
}

/* One output: y[m,n] = fl32( sum_b f16(Wd[n,b]) * xd[m,b] * isum[m,n,b] ) in binary64. */
/* One output before its final rounding: sum over blocks of d_w * d_x * isum in binary64. */
static double oq8_one_output_f64(const int8_t *xq_row, const float *xd_row, const int8_t *wq_row,
                                 const uint16_t *wd_row, int64_t K)
{
    int64_t nb = K / OQ8_QK;
    double acc = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t s = 0;
        for (int j = 0; j < OQ8_QK; ++j)
            s += (int64_t)xq_row[b * OQ8_QK + j] * (int64_t)wq_row[b * OQ8_QK + j];
        acc += oq8_f16_to_f64(wd_row[b]) * (double)xd_row[b] * (double)s;
    }
    return acc;
}

static float oq8_one_output(const int8_t *xq_row, const float *xd_row, const int8_t *wq_row,
                            const uint16_t *wd_row, int64_t K)
{
    return (float)oq8_one_output_f64(xq_row, xd_row, wq_row, wd_row, K);
}

typedef struct {
    const int8_t *xq;
    const float *xd;
    const int8_t *Wq;
    const uint16_t *Wd;
    int64_t M, N, K, begin, end; /* flat output index range [begin, end) over M*N */
    float *y;
} oq8_job;

static void *oq8_linear_worker(void *arg)
{
    oq8_job *j = (oq8_job *)arg;
    int64_t nb = j->K / OQ8_QK;
    for (int64_t i = j->begin; i < j->end; ++i) {
        int64_t m = i / j->N, n = i % j->N;
        j->y[i] = oq8_one_output(j->xq + m * j->K, j->xd + m * nb, j->Wq + n * j->K,
                                 j->Wd + n * nb, j->K);
    }
    return NULL;
}

/* y[M,N] from codes and scales.  nthreads <= 1 runs on the calling thread; otherwise
 * the flat output range is cut into nthreads contiguous pieces (the arithmetic of each
 * output is the same either way). */
void oq8_linear_codes(const int8_t *xq, const float *xd, const int8_t *Wq, const uint16_t *Wd,
                      int64_t M, int64_t N, int64_t K, float *y, int nthreads)
{
    int64_t total = M * N;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > total)
        nthreads = (int)(total > 0 ? total : 1);
    oq8_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (oq8_job){xq, xd, Wq, Wd, M, N, K, total * t / nthreads,
                            total * (t + 1) / nthreads, y};
    }
    if (nthreads == 1) {
        oq8_linear_worker(&jobs[0]);
        return;
    }
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, oq8_linear_worker, &jobs[t]) != 0)
            break;
        ++started;
    }
    for (int t = started; t < nthreads; ++t) /* could not start a thread: do it here */
        oq8_linear_worker(&jobs[t]);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
}

/* Sampled outputs: out[i] = y[rows[i], cols[i]], for checks at sizes where the full
 * product is too slow on the CPU. */
void oq8_linear_codes_at(const int8_t *xq, const float *xd, const int8_t *Wq,
                         const uint16_t *Wd, int64_t K, const int64_t *rows,
                         const int64_t *cols, int64_t count, float *out)
{
    int64_t nb = K / OQ8_QK;
    for (int64_t i = 0; i < count; ++i)
        out[i] = oq8_one_output(xq + rows[i] * K, xd + rows[i] * nb, Wq + cols[i] * K,
                                Wd + cols[i] * nb, K);
}

/* The whole linear layer from raw activations: quantize x (dtype 0 = binary32,
 * 1 = bfloat16 bits), then y = the rescaled block sums.  xq/xd are caller scratch of
 * M*K bytes and M*(K/32) floats. */
void oq8_linear(const void *x, int dtype, const int8_t *Wq, const uint16_t *Wd, float *y,
                int64_t M, int64_t N, int64_t K, int8_t *xq, float *xd, int nthreads)
{
    if (dtype == 0)
        oq8_quantize_act_f32((const float *)x, M, K, xq, xd);
    else
        oq8_quantize_act_bf16((const uint16_t *)x, M, K, xq, xd);
    oq8_linear_codes(xq, xd, Wq, Wd, M, N, K, y, nthreads);
}

/* ---------------------------------------------------------------------------------- */
/* The layer's neighbours fused into its output (epilogue): y = op(x . W^T, aux).       */
/* The post runs its Q8_0 linears inside GDN + attention blocks whose FFN multiplies     */
/* SiLU(gate) by up and adds residuals; these readings define that step:                 */
/*   E1 op 0: y = acc;  op 1 (residual): y = acc + aux;  op 2 (gated unit):               */
/*      y = silu(aux) * acc with silu(g) = g / (1 + exp(-g)), aux being the gate          */
/*      projection's output and acc the up projection's.                                 */
/*   E2 acc, aux and op are evaluated in binary64 and rounded once, to binary32 or to     */
/*      bfloat16 (round to nearest even, subnormals kept, overflow to infinity).          */
/* ---------------------------------------------------------------------------------- */

/* binary64 -> bfloat16 bits, round to nearest even (8-bit significand, binary32 range). */
uint16_t oq8_f64_to_bf16(double v)
{
    if (v != v)
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;           /* a = (2m) * 2^E, 2m in [1, 2) */
    if (E < -126) {          /* subnormal: multiples of 2^-133 */
        double q = nearbyint(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)q); /* q == 128 is the smallest normal */
    }
    double q = nearbyint(ldexp(2.0 * m, 7)); /* 8 significant bits: [128, 256] */
    if (q == 256.0) {
        q = 128.0;
        E += 1;
    }
    if (E > 127)
        return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | ((uint16_t)(E + 127) << 7) | (uint16_t)((int)q - 128));
}

double oq8_silu(double g) { return g / (1.0 + exp(-g)); }

static double oq8_epilogue_f64(double acc, int op, const float *aux, int64_t i)
{
    if (op == 1)
        return acc + (double)aux[i];
    if (op == 2)
        return oq8_silu((double)aux[i]) * acc;
    return acc;
}

/* y[M,N] = op(rowscale[m] * rescaled block sums, aux), stored as binary32 (ytype 0) or
 * bfloat16 bits (ytype 1).  aux is [M,N] binary32 (unused for op 0); rowscale is [M]
 * binary64, or NULL for 1 (it carries the RMSNorm factor r, reading N1).
 * Single-threaded. */
void oq8_linear_epilogue(const int8_t *xq, const float *xd, const int8_t *Wq, const uint16_t *Wd,
                         int64_t M, int64_t N, int64_t K, const double *rowscale, const float *aux,
                         int op, int ytype, void *y)
{
    int64_t nb = K / OQ8_QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t i = m * N + n;
            double acc = oq8_one_output_f64(xq + m * K, xd + m * nb, Wq + n * K, Wd + n * nb, K);
            if (rowscale != NULL)
                acc = acc * rowscale[m];
            double v = oq8_epilogue_f64(acc, op, aux, i);
            if (ytype == 1)
                ((uint16_t *)y)[i] = oq8_f64_to_bf16(v);
            else
                ((float *)y)[i] = (float)v;
        }
}

/* ---------------------------------------------------------------------------------- */
/* RMSNorm fused into the activation quantizer (the layer's prologue).                  */
/* In these hybrid blocks a projection's input is the RMS-normalised hidden state       */
/* (root mean square layer normalisation, Zhang and Sennrich, NeurIPS 2019):             */
/*   z[m,k] = x[m,k] * r[m] * gamma[k],   r[m] = 1 / sqrt(mean over k of x[m,k]^2 + eps). */
/* Readings:                                                                             */
/*   N1 r[m] is one factor per row, so it rides on the row's block scales: the codes    */
/*      are those of u[m,k] = fl32(x[m,k] * gamma[k]) (R1-R8 applied to u) and the       */
/*      activation scale is d_u[m,b] * r[m].  In exact arithmetic this is the            */
/*      quantization of z itself (amax and every ratio u / d scale by r alike); it       */
/*      keeps every code independent of how r is rounded.                               */
/*   N2 the oracle evaluates r in binary64 from the exactly widened x and applies it to  */
/*      y in binary64 before the one rounding (the kernels: binary32).                  */
/*   N3 eps > 0 (the entry point rejects anything else), so r is finite; rows whose sum  */
/*      of squares leaves the binary32 range are outside the domain, like NaN and Inf.   */
/* ---------------------------------------------------------------------------------- */

static float oq8_act_value(const void *x, int dtype, int64_t i)
{
    return dtype == 1 ? oq8_bf16_to_f32(((const uint16_t *)x)[i]) : ((const float *)x)[i];
}

/* x[M,K] (binary32, or bfloat16 bits for dtype 1), gamma[K] binary32 ->
 * xq[M,K] codes of u, xd_u[M,K/32] binary32 scales of u, r[M] binary64. */
void oq8_rmsnorm_quantize_act(const void *x, int dtype, const float *gamma, double eps, int64_t M,
                              int64_t K, int8_t *xq, float *xd_u, double *r)
{
    int64_t nb = K / OQ8_QK;
    float u[OQ8_QK];
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = (double)oq8_act_value(x, dtype, m * K + k);
            ss += a * a;
        }
        double mean = K > 0 ? ss / (double)K : 0.0;
        r[m] = 1.0 / sqrt(mean + eps);
        for (int64_t b = 0; b < nb; ++b) {
            for (int j = 0; j < OQ8_QK; ++j) {
                int64_t k = b * OQ8_QK + j;
                u[j] = oq8_act_value(x, dtype, m * K + k) * gamma[k];
            }
            oq8_quantize_block(u, xq + m * K + b * OQ8_QK, xd_u + m * nb + b);
        }
    }
}
