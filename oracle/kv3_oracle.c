/*
 * kv3_oracle.c -- plain, slow CPU oracle for the 3-bit KV-cache codec (WHT + Lloyd-Max).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  The CUDA library never links
 * it, includes it or falls back to it, and this file includes nothing from the CUDA
 * library: the two implementations share no code, header, table or helper.
 *
 * Source of the method.  The post "CUDA inference engine for running Qwen3.5/3.6 hybrid
 * models on mining cards (CMP 100-210)" (news.hada.io topic 29953, feature list) runs a
 * 256K-token context with a 3-bit KV cache built from a Walsh-Hadamard transform (WHT) and
 * a Lloyd-Max quantizer, which takes the cache from 17 GB to 3.5 GB.  The post names the
 * two parts and the sizes; every other step below is a reading (the GPU library takes the
 * same one):
 *   K1 groups of d = 128 consecutive elements of a key or value vector (half of a 256-wide
 *      head); per group 128 three-bit codes and one binary32 scale, 3.25 bits per element
 *      (a 17.2 GB bf16 cache becomes 3.49 GB).
 *   K2 rotation: the unnormalised fast Walsh-Hadamard transform in Sylvester order, in
 *      binary32: stages h = 1, 2, 4, ..., 64, each pairing j with j + h (j with bit h clear)
 *      as (a, b) -> (a + b, a - b).  It spreads outlier channels over the whole group, so
 *      the rotated values are close to Gaussian.
 *   K3 scale: s = sqrt(ss / 128) in binary32, ss the pairwise sum (balanced binary tree
 *      over the natural order, Higham 1993) of the binary32 squares u_i * u_i of the
 *      rotated group u: the RMS of u.
 *   K4 codebook: the 8-level Lloyd-Max quantizer of the unit Gaussian as tabulated by Max
 *      (1960): levels +-0.2451, +-0.7560, +-1.3440, +-2.1520 and decision thresholds
 *      0.5006, 1.0500, 1.7480 (binary32 constants).  The decision u/s against a threshold t
 *      is taken as |u| >= fl32(t * s): code = 4 * (u < 0) + #{t : |u| >= fl32(t * s)}.
 *      A group with s == 0 (all zero) gets codes 0.
 *   K5 bit layout: the code of element i at bits [3i, 3i + 3) of a little-endian bit
 *      stream, 12 uint32 words (48 bytes) per group; scales in their own array.
 *   K6 decode: w_i = fl32(s * (+-level)), then x_i = WHT(w)_i / 128 (an exact scaling, as
 *      the unnormalised WHT applied twice is 128 times the identity), rounded to bfloat16
 *      (nearest even) when the output is bfloat16.
 *   K7 domain: finite groups whose sum of squares stays inside the binary32 range
 *      (|x| below about 1e18); beyond it s overflows and the decoder meets inf - inf.  Like
 *      NaN and Inf inputs, such groups are outside the domain.  A sum that underflows to 0
 *      is inside it (s == 0: codes 0, decoded to 0).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math kv3_oracle.c
 *        -o libokv3.so -lm      (oracle/build.py does this)
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OKV3_D 128
#define OKV3_WORDS 12

static const float okv3_level[4] = {0.2451f, 0.7560f, 1.3440f, 2.1520f};
static const float okv3_threshold[3] = {0.5006f, 1.0500f, 1.7480f};

/* K2: in-place unnormalised fast Walsh-Hadamard transform of 128 binary32 values. */
void okv3_fwht(float *a)
{
    for (int h = 1; h < OKV3_D; h <<= 1)
        for (int i = 0; i < OKV3_D; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float x = a[j], y = a[j + h];
                a[j] = x + y;
                a[j + h] = x - y;
            }
}

/* K3: pairwise (balanced tree) sum of n binary32 values, n a power of two. */
static float okv3_pairwise(const float *v, int n)
{
    if (n == 1)
        return v[0];
    return okv3_pairwise(v, n / 2) + okv3_pairwise(v + n / 2, n / 2);
}

static float okv3_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* One group: 128 values -> 12 code words and the scale. */
void okv3_encode_group(const float *x, uint32_t *words, float *scale)
{
    float u[OKV3_D], sq[OKV3_D];
    memcpy(u, x, sizeof u);
    okv3_fwht(u);
    for (int i = 0; i < OKV3_D; ++i)
        sq[i] = u[i] * u[i];
    float ss = okv3_pairwise(sq, OKV3_D);
    float s = sqrtf(ss / 128.0f);
    *scale = s;
    memset(words, 0, OKV3_WORDS * sizeof(uint32_t));
    if (s == 0.0f)
        return;
    float T[3];
    for (int k = 0; k < 3; ++k)
        T[k] = okv3_threshold[k] * s;
    for (int i = 0; i < OKV3_D; ++i) {
        float a = fabsf(u[i]);
        uint32_t m = 0;
        for (int k = 0; k < 3; ++k)
            m += (a >= T[k]) ? 1u : 0u;
        uint32_t code = (u[i] < 0.0f ? 4u : 0u) | m;
        int bit = 3 * i;
        words[bit / 32] |= code << (bit % 32);
        if (bit % 32 > 29) /* the code crosses into the next word */
            words[bit / 32 + 1] |= code >> (32 - bit % 32);
    }
}

/* One group: 12 code words and the scale -> 128 binary32 values. */
void okv3_decode_group(const uint32_t *words, float scale, float *out)
{
    float w[OKV3_D];
    for (int i = 0; i < OKV3_D; ++i) {
        int bit = 3 * i;
        uint32_t code = words[bit / 32] >> (bit % 32);
        if (bit % 32 > 29)
            code |= words[bit / 32 + 1] << (32 - bit % 32);
        code &= 7u;
        float level = okv3_level[code & 3u];
        w[i] = scale * ((code & 4u) ? -level : level);
    }
    okv3_fwht(w);
    for (int i = 0; i < OKV3_D; ++i)
        out[i] = w[i] / 128.0f;
}

/* x [n][128] binary32 (dtype 0) or bfloat16 bits (dtype 1) -> words [n][12], scales [n]. */
void okv3_encode(const void *x, int dtype, int64_t n, uint32_t *words, float *scales)
{
    float v[OKV3_D];
    for (int64_t g = 0; g < n; ++g) {
        for (int i = 0; i < OKV3_D; ++i)
            v[i] = dtype == 1 ? okv3_bf16_to_f32(((const uint16_t *)x)[g * OKV3_D + i])
                              : ((const float *)x)[g * OKV3_D + i];
        okv3_encode_group(v, words + g * OKV3_WORDS, scales + g);
    }
}

/* words [n][12], scales [n] -> out [n][128] binary32. */
void okv3_decode(const uint32_t *words, const float *scales, int64_t n, float *out)
{
    for (int64_t g = 0; g < n; ++g)
        okv3_decode_group(words + g * OKV3_WORDS, scales[g], out + g * OKV3_D);
}
