// q8_kv3.cu -- 3-bit KV-cache codec: Walsh-Hadamard rotation + Lloyd-Max quantizer.
//
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, feature list) keeps a 256K-token context in a
// 3-bit KV cache built from a Walsh-Hadamard transform (WHT) and a Lloyd-Max quantizer,
// 17 GB -> 3.5 GB.  The codec here (readings of the post):
//   * groups of 128 consecutive elements of a key or value vector; per group 128 three-bit
//     codes (a little-endian bit stream, 12 uint32 words) and one binary32 scale:
//     3.25 bits per element;
//   * encode: u = unnormalised fast WHT of the group (Sylvester order, binary32, stages
//     h = 1 .. 64, (a, b) -> (a + b, a - b)); s = sqrt(ss / 128), ss the pairwise (balanced
//     tree) sum of the squares u_i^2: the RMS of u; code_i = 4 * (u_i < 0) + the number of
//     thresholds t of the 8-level unit-Gaussian Lloyd-Max quantizer (Max 1960: 0.5006,
//     1.0500, 1.7480) with |u_i| >= fl32(t * s); s == 0 gives codes 0;
//   * decode: w_i = s * (+-level), levels 0.2451, 0.7560, 1.3440, 2.1520; x = WHT(w) / 128.
//
// Layout on the GPU: four lanes per group, eight groups per warp.  Lane t of a group holds
// the elements j = 32 c + 8 t + e (c, e = 0..3, 0..7), so each load instruction moves 64
// contiguous bytes of a group.  WHT stages h = 1, 2, 4 (bits of e) and 32, 64 (bits of c)
// are register butterflies; h = 8, 16 exchange with lanes t ^ 1, t ^ 2.  The stages run in
// the order h = 1, 2, ..., 64 and the sum of squares follows the pairwise tree over the
// natural order (e bits, then t bits across lanes, then c bits), so every rounding is the
// oracle's.  The 24 code bits of (c, t) sit at stream bits 96 c + 24 t: lanes t < 3 each
// form one of the three words of block c from their chunk and the next lane's.
// The butterflies, the sums and the threshold differences run on packed binary32 pairs
// (add / fma .f32x2, one rounding per element as the scalar operations): element e of chunk c
// shares a register pair with element e of chunk c + 2, so one instruction does two chunks';
// a - b is fma(-1, b, a), whose product is exact.  Products that feed additions stay scalar
// (__fmul_rn is never fused into an FMA; a packed product was measured being fused).
#include <cuda_bf16.h>

#include <algorithm>

#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int kD = 128;
constexpr int kWords = 12;
constexpr unsigned kFull = 0xFFFFFFFFu;

// +-level of each 3-bit code (bit 2: the sign, bits 0-1: the magnitude cell); the decoder
// copies it to shared memory and looks codes up there (one load in place of a chain of
// selects on the integer pipe)
__constant__ float kLevel[8] = {0.2451f,  0.7560f,  1.3440f,  2.1520f,
                                -0.2451f, -0.7560f, -1.3440f, -2.1520f};

constexpr int kE = 8;  // elements of a (c, t) chunk

// a - b with one rounding (the product with -1 is exact)
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  return __ffma2_rn(make_float2(-1.0f, -1.0f), b, a);
}

// Unnormalised WHT of a group held by four lanes: w[c][e] = (element 32 c + 8 t + e,
// element 32 (c + 2) + 8 t + e), c = 0, 1.
__device__ __forceinline__ void fwht_group(float2 (&w)[2][kE], int t) {
#pragma unroll
  for (int h = 1; h < kE; h <<= 1)  // h = 1, 2, 4: inside a chunk
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e = 0; e < kE; ++e)
        if ((e & h) == 0) {
          const float2 a = w[c][e], b = w[c][e + h];
          w[c][e] = __fadd2_rn(a, b);
          w[c][e + h] = sub2(a, b);
        }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {  // h = 8, 16: the lane t ^ o; the upper lane takes a - b
    // q + (+-1) v in one rounding: the product with +-1 is exact, so this is q +- v
    const float sg = (t & o) ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const float2 q = make_float2(__shfl_xor_sync(kFull, w[c][e].x, o), __shfl_xor_sync(kFull, w[c][e].y, o));
        w[c][e] = __ffma2_rn(sg2, w[c][e], q);
      }
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) {  // h = 32: chunk 0 with 1 and 2 with 3, i.e. w[0] with w[1]
    const float2 a = w[0][e], b = w[1][e];
    w[0][e] = __fadd2_rn(a, b);
    w[1][e] = sub2(a, b);
  }
#pragma unroll
  for (int c = 0; c < 2; ++c)  // h = 64: chunk c with c + 2, the two halves of a pair
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const float a = w[c][e].x, b = w[c][e].y;
      w[c][e] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
    }
}

struct Kv3Params {
  const void* x;      // [n][128] bf16 bits or f32 (encode input)
  int xtype;          // 0 f32, 1 bf16
  uint32_t* codes;    // [n][12]
  float* scales;      // [n]
  const uint32_t* codes_in;
  const float* scales_in;
  void* out;          // [n][128] (decode output)
  int otype;          // 0 f32, 1 bf16
  int64_t n;
};

// binary32 input: the lane's four 8-element chunks of group g (zeros past the end), paired
// chunk c with c + 2
template <int kXType>
__device__ __forceinline__ void load_group(const void* x, int64_t g, int64_t n, int t,
                                           float2 (&w)[2][kE]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int64_t off = g * kD + 32 * c + 8 * t;
    float v[kE];
    if (g >= n) {
#pragma unroll
      for (int e = 0; e < kE; ++e) v[e] = 0.0f;
    } else {
      const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
      const float4 a = __ldcs(f), b = __ldcs(f + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      if (c < 2)
        w[c][e].x = v[e];
      else
        w[c - 2][e].y = v[e];
    }
  }
}

// bfloat16 input: the lane's four 16-byte pieces of group g (zeros past the end), and their
// values paired chunk c with c + 2
__device__ __forceinline__ void load_raw_bf16(const void* x, int64_t g, int64_t n, int t, uint4 (&raw)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    raw[c] = g < n ? __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + g * kD + 32 * c + 8 * t))
                   : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void unpack_bf16(const uint4 (&raw)[4], float2 (&w)[2][kE]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xFFFF0000u);
      if (c < 2) {
        w[c][2 * i].x = lo;
        w[c][2 * i + 1].x = hi;
      } else {
        w[c - 2][2 * i].y = lo;
        w[c - 2][2 * i + 1].y = hi;
      }
    }
  }
}

template <int kXType>
__global__ void __launch_bounds__(256) kv3_encode_kernel(const Kv3Params p) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  const int64_t team = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
  const int64_t nteams = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 2;
  const int64_t rounds = (p.n + nteams - 1) / nteams;  // the same for every lane of the grid
  // bfloat16 input: the next group's bytes are in flight while this one is encoded
  uint4 raw[4];
  if constexpr (kXType == 1) load_raw_bf16(p.x, team, p.n, t, raw);
  for (int64_t it = 0; it < rounds; ++it) {
    const int64_t g = it * nteams + team;
    float2 w[2][kE];
    if constexpr (kXType == 1) {
      unpack_bf16(raw, w);
      load_raw_bf16(p.x, g + nteams, p.n, t, raw);
    } else {
      load_group<kXType>(p.x, g, p.n, t, w);
    }
    fwht_group(w, t);
    // pairwise sum of the squares: e levels in the lane, t levels across lanes, then c
    float2 sc[2];  // (chunk c, chunk c + 2)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float2 q[kE];
#pragma unroll
      for (int e = 0; e < kE; ++e)  // scalar products: a packed one may be fused into the adds
        q[e] = make_float2(__fmul_rn(w[c][e].x, w[c][e].x), __fmul_rn(w[c][e].y, w[c][e].y));
      sc[c] = __fadd2_rn(__fadd2_rn(__fadd2_rn(q[0], q[1]), __fadd2_rn(q[2], q[3])),
                         __fadd2_rn(__fadd2_rn(q[4], q[5]), __fadd2_rn(q[6], q[7])));
#pragma unroll
      for (int o = 1; o < 4; o <<= 1)
        sc[c] = __fadd2_rn(sc[c], make_float2(__shfl_xor_sync(kFull, sc[c].x, o), __shfl_xor_sync(kFull, sc[c].y, o)));
    }
    const float2 s01 = __fadd2_rn(sc[0], sc[1]);  // (chunks 0 + 1, chunks 2 + 3)
    const float ss = __fadd_rn(s01.x, s01.y);
    const float s = __fsqrt_rn(__fmul_rn(ss, 0.0078125f));  // ss / 128, exact
    const float t0 = __fmul_rn(0.5006f, s), t1 = __fmul_rn(1.0500f, s), t2 = __fmul_rn(1.7480f, s);
    const float2 t02 = make_float2(t0, t0), t12 = make_float2(t1, t1), t22 = make_float2(t2, t2);
    uint32_t chunk[4];  // 24 code bits of (c, t): element 32 c + 8 t + e at bit 3 e
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t lo = 0, hi = 0;  // chunks c and c + 2
#pragma unroll
      for (int e = kE - 1; e >= 0; --e) {
        // the three bits of the code from sign bits, each shifted in at the bottom (element
        // 7 first): the sign of v + 0 (v < 0; -0 + 0 is +0), the sign of a - t1 (a < t1),
        // and the parity of the signs of a - t0, a - t1, a - t2 (the thresholds not passed;
        // a - t is +0 when they are equal, so a >= t is a clear sign bit).  m counts the
        // thresholds passed, so its bits are the complements of the last two: inverted below.
        const float2 a = make_float2(fabsf(w[c][e].x), fabsf(w[c][e].y));
        const float2 sg = __fadd2_rn(w[c][e], make_float2(0.0f, 0.0f));
        const float2 d0 = sub2(a, t02), d1 = sub2(a, t12), d2 = sub2(a, t22);
        lo = __funnelshift_l(__float_as_uint(sg.x), lo, 1);
        lo = __funnelshift_l(__float_as_uint(d1.x), lo, 1);
        lo = __funnelshift_l(__float_as_uint(d0.x) ^ __float_as_uint(d1.x) ^ __float_as_uint(d2.x), lo, 1);
        hi = __funnelshift_l(__float_as_uint(sg.y), hi, 1);
        hi = __funnelshift_l(__float_as_uint(d1.y), hi, 1);
        hi = __funnelshift_l(__float_as_uint(d0.y) ^ __float_as_uint(d1.y) ^ __float_as_uint(d2.y), hi, 1);
      }
      chunk[c] = s == 0.0f ? 0u : lo ^ 0x6DB6DBu;  // bits 3 e and 3 e + 1 of each code
      chunk[c + 2] = s == 0.0f ? 0u : hi ^ 0x6DB6DBu;
    }
    // stream bits 96 c + 24 t: lane t < 3 forms word 3 c + t from its chunk and lane t + 1's
    const int next = (lane & ~3) | ((t + 1) & 3);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t up = __shfl_sync(kFull, chunk[c], next);
      const uint32_t word = (chunk[c] >> (8 * t)) | (up << (24 - 8 * t));
      if (g < p.n && t < 3) p.codes[g * kWords + 3 * c + t] = word;
    }
    if (g < p.n && t == 0) p.scales[g] = s;
  }
}

// the lane's four 24-bit code chunks of group g: bits [96 c + 24 t, + 24) of its stream,
// i.e. word 3 c + (3 t) / 4 from bit (24 t) % 32, and the next word when they cross
__device__ __forceinline__ void load_chunks(const uint32_t* codes, int64_t g, int64_t n, int t,
                                            uint32_t (&lo)[4], uint32_t (&hi)[4]) {
  const int bit = 24 * t, w0 = bit >> 5, off = bit & 31;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    lo[c] = 0u;
    hi[c] = 0u;
    if (g < n) {
      const uint32_t* w = codes + g * kWords + 3 * c;
      lo[c] = __ldg(w + w0);
      if (off > 8) hi[c] = __ldg(w + w0 + 1);
    }
  }
}

template <int kOType>
__global__ void __launch_bounds__(256) kv3_decode_kernel(const Kv3Params p) {
  __shared__ float level[8];
  if (threadIdx.x < 8) level[threadIdx.x] = kLevel[threadIdx.x];
  __syncthreads();
  const int lane = threadIdx.x & 31, t = lane & 3;
  const int64_t team = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
  const int64_t nteams = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 2;
  const int64_t rounds = (p.n + nteams - 1) / nteams;
  const int off = (24 * t) & 31;
  // software pipeline: the next group's code words and scale are in flight while this
  // group is transformed
  uint32_t lo[4], hi[4];
  load_chunks(p.codes_in, team, p.n, t, lo, hi);
  float s = team < p.n ? __ldg(p.scales_in + team) : 0.0f;
  for (int64_t it = 0; it < rounds; ++it) {
    const int64_t g = it * nteams + team;
    const int64_t gn = g + nteams;
    uint32_t nlo[4], nhi[4];
    load_chunks(p.codes_in, gn, p.n, t, nlo, nhi);
    const float ns = gn < p.n ? __ldg(p.scales_in + gn) : 0.0f;
    float2 w[2][kE];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t ca = ((lo[c] >> off) | (off > 8 ? hi[c] << (32 - off) : 0u)) & 0xFFFFFFu;
      const uint32_t cb = ((lo[c + 2] >> off) | (off > 8 ? hi[c + 2] << (32 - off) : 0u)) & 0xFFFFFFu;
#pragma unroll
      for (int e = 0; e < kE; ++e)  // scalar products: a packed one may be fused into the adds
        w[c][e] = make_float2(__fmul_rn(s, level[(ca >> (3 * e)) & 7u]), __fmul_rn(s, level[(cb >> (3 * e)) & 7u]));
    }
    fwht_group(w, t);
    if (g < p.n) {
      const float2 inv2 = make_float2(0.0078125f, 0.0078125f);  // / 128, exact
      float out[4][kE];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < kE; ++e) {
          const float2 pr = __fmul2_rn(w[c][e], inv2);
          out[c][e] = pr.x;
          out[c + 2][e] = pr.y;
        }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float* o = out[c];
        const int64_t eo = g * kD + 32 * c + 8 * t;
        if constexpr (kOType == 1) {
          uint32_t u[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
            u[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + eo), make_uint4(u[0], u[1], u[2], u[3]));
        } else {
          float4* f = reinterpret_cast<float4*>(static_cast<float*>(p.out) + eo);
          __stcs(f, make_float4(o[0], o[1], o[2], o[3]));
          __stcs(f + 1, make_float4(o[4], o[5], o[6], o[7]));
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      lo[c] = nlo[c];
      hi[c] = nhi[c];
    }
    s = ns;
  }
}

int kv3_grid(int64_t n, const DeviceInfo& dev) {
  const int64_t blocks = (n + 63) / 64;  // 64 groups per 256-thread block
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
  return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

}  // namespace

cudaError_t launch_kv3_encode(const void* x, int xtype, uint32_t* codes, float* scales, int64_t n,
                              const DeviceInfo& dev, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  Kv3Params p = {};
  p.x = x;
  p.xtype = xtype;
  p.codes = codes;
  p.scales = scales;
  p.n = n;
  const int grid = kv3_grid(n, dev);
  if (xtype == 1)
    kv3_encode_kernel<1><<<grid, 256, 0, stream>>>(p);
  else
    kv3_encode_kernel<0><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv3_decode(const uint32_t* codes, const float* scales, void* out, int otype,
                              int64_t n, const DeviceInfo& dev, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  Kv3Params p = {};
  p.codes_in = codes;
  p.scales_in = scales;
  p.out = out;
  p.otype = otype;
  p.n = n;
  const int grid = kv3_grid(n, dev);
  if (otype == 1)
    kv3_decode_kernel<1><<<grid, 256, 0, stream>>>(p);
  else
    kv3_decode_kernel<0><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace q8
