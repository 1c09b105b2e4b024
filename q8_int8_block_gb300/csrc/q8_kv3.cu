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

// Unnormalised WHT of a group held by four lanes (v[c][e] = element 32 c + 8 t + e).
__device__ __forceinline__ void fwht_group(float (&v)[4][kE], int t) {
#pragma unroll
  for (int h = 1; h < kE; h <<= 1)  // h = 1, 2, 4: inside a chunk
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e = 0; e < kE; ++e)
        if ((e & h) == 0) {
          const float a = v[c][e], b = v[c][e + h];
          v[c][e] = __fadd_rn(a, b);
          v[c][e + h] = __fsub_rn(a, b);
        }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {  // h = 8, 16: the lane t ^ o; the upper lane takes a - b
    // q + (+-1) v in one rounding: the product with +-1 is exact, so this is q +- v
    const float sg = (t & o) ? -1.0f : 1.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const float q = __shfl_xor_sync(kFull, v[c][e], o);
        v[c][e] = __fmaf_rn(sg, v[c][e], q);
      }
  }
#pragma unroll
  for (int hc = 1; hc < 4; hc <<= 1)  // h = 32, 64: across chunks of the lane
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if ((c & hc) == 0)
#pragma unroll
        for (int e = 0; e < kE; ++e) {
          const float a = v[c][e], b = v[c + hc][e];
          v[c][e] = __fadd_rn(a, b);
          v[c + hc][e] = __fsub_rn(a, b);
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

// the lane's four 8-element chunks of group g (zeros past the end)
template <int kXType>
__device__ __forceinline__ void load_group(const void* x, int64_t g, int64_t n, int t,
                                           float (&v)[4][kE]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int64_t off = g * kD + 32 * c + 8 * t;
    if (g >= n) {
#pragma unroll
      for (int e = 0; e < kE; ++e) v[c][e] = 0.0f;
    } else if constexpr (kXType == 1) {
      const uint4 w = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off));
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[c][2 * i] = __uint_as_float(u[i] << 16);
        v[c][2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    } else {
      const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
      const float4 a = __ldcs(f), b = __ldcs(f + 1);
      v[c][0] = a.x; v[c][1] = a.y; v[c][2] = a.z; v[c][3] = a.w;
      v[c][4] = b.x; v[c][5] = b.y; v[c][6] = b.z; v[c][7] = b.w;
    }
  }
}

template <int kXType>
__global__ void __launch_bounds__(256) kv3_encode_kernel(const Kv3Params p) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  const int64_t team = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
  const int64_t nteams = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 2;
  const int64_t rounds = (p.n + nteams - 1) / nteams;  // the same for every lane of the grid
  for (int64_t it = 0; it < rounds; ++it) {
    const int64_t g = it * nteams + team;
    float v[4][kE];
    load_group<kXType>(p.x, g, p.n, t, v);
    fwht_group(v, t);
    // pairwise sum of the squares: e levels in the lane, t levels across lanes, then c
    float sc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float q[kE];
#pragma unroll
      for (int e = 0; e < kE; ++e) q[e] = __fmul_rn(v[c][e], v[c][e]);
      sc[c] = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                        __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) sc[c] = __fadd_rn(sc[c], __shfl_xor_sync(kFull, sc[c], o));
    }
    const float ss = __fadd_rn(__fadd_rn(sc[0], sc[1]), __fadd_rn(sc[2], sc[3]));
    const float s = __fsqrt_rn(__fmul_rn(ss, 0.0078125f));  // ss / 128, exact
    const float t0 = __fmul_rn(0.5006f, s), t1 = __fmul_rn(1.0500f, s), t2 = __fmul_rn(1.7480f, s);
    uint32_t chunk[4];  // 24 code bits of (c, t): element 32 c + 8 t + e at bit 3 e
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t bits = 0;
#pragma unroll
      for (int e = kE - 1; e >= 0; --e) {
        // the three bits of the code from sign bits, each shifted in at the bottom (element
        // 7 first): the sign of v + 0 (v < 0; -0 + 0 is +0), the sign of a - t1 (a < t1),
        // and the parity of the signs of a - t0, a - t1, a - t2 (the thresholds not passed;
        // a - t is +0 when they are equal, so a >= t is a clear sign bit).  m counts the
        // thresholds passed, so its bits are the complements of the last two: inverted below.
        const float a = fabsf(v[c][e]);
        const uint32_t sg = __float_as_uint(__fadd_rn(v[c][e], 0.0f));
        const uint32_t d0 = __float_as_uint(__fsub_rn(a, t0));
        const uint32_t d1 = __float_as_uint(__fsub_rn(a, t1));
        const uint32_t d2 = __float_as_uint(__fsub_rn(a, t2));
        bits = __funnelshift_l(sg, bits, 1);
        bits = __funnelshift_l(d1, bits, 1);
        bits = __funnelshift_l(d0 ^ d1 ^ d2, bits, 1);
      }
      chunk[c] = s == 0.0f ? 0u : bits ^ 0x6DB6DBu;  // bits 3 e and 3 e + 1 of each code
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
    float v[4][kE];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t chunk = ((lo[c] >> off) | (off > 8 ? hi[c] << (32 - off) : 0u)) & 0xFFFFFFu;
#pragma unroll
      for (int e = 0; e < kE; ++e) v[c][e] = __fmul_rn(s, level[(chunk >> (3 * e)) & 7u]);
    }
    fwht_group(v, t);
    if (g < p.n) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[kE];
#pragma unroll
        for (int e = 0; e < kE; ++e) o[e] = __fmul_rn(v[c][e], 0.0078125f);  // / 128, exact
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
