// q8_quant.cu -- Q8_0 quantization kernels (weights and activations).
//
// Q8_0 block quantizer of the int8 GEMM in "CUDA inference engine for running
// Qwen3.5/3.6 hybrid models on mining cards (CMP 100-210)" (news.hada.io topic 29953;
// un-throttled-paths list: the DP4A int8 GEMM; "Limitations": Q8_0 only): per 32-element
// block, d = amax / 127 (IEEE binary32 division), q = round(v / d) with ties away from
// zero, clamped to [-127, 127]; d == 0 gives codes 0.  Weight scales are then rounded to
// binary16 (nearest even), activation scales stay binary32.
//
// Mapping: 4 consecutive lanes own one block (8 values each, one 16-byte load for bf16,
// two for f32), combine amax with two xor-shuffles, and each writes its 8 codes with one
// vector store.  Grid-stride over blocks, so any number of rows works.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q8_internal.h"
#include "q8_quant_dev.cuh"

namespace q8 {
namespace {

template <typename InT>
struct Loader;

template <>
struct Loader<float> {
  static __device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

template <>
struct Loader<uint16_t> {  // bfloat16 bit patterns: widening is a 16-bit shift, exact
  static __device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
    bf16x8_to_f32(__ldcs(reinterpret_cast<const uint4*>(p)), v);
  }
};

// gamma / r: the RMSNorm prologue (nullptr: none).  Codes are those of fl32(v * gamma);
// the stored scale is d * r[row].
template <typename InT, bool kF16Codes, bool kF16Scale>
__global__ void __launch_bounds__(256) quantize_kernel(const InT* __restrict__ x,
                                                       void* __restrict__ codes,
                                                       void* __restrict__ scales,
                                                       int64_t nblocks, int64_t nb,
                                                       const float* __restrict__ gamma,
                                                       const float* __restrict__ r) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const unsigned group_mask = 0xFu << (lane & ~3);
  const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 2;
  for (int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
       blk < nblocks; blk += stride) {
    const int64_t off = blk * kQK + sub * 8;
    float v[8];
    Loader<InT>::load8(x + off, v);
    const int64_t m = blk / nb;
    if (gamma != nullptr) {
      const int64_t k = (blk - m * nb) * kQK + sub * 8;
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma + k));
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma + k) + 1);
      const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], g[i]);
    }
    int q[8];
    float d = quantize_block_x4(v, group_mask, q);
    if (r != nullptr) d = __fmul_rn(d, __ldg(r + m));
    if constexpr (kF16Codes) {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = __half_as_ushort(__int2half_rn(q[2 * i]));
        const uint32_t hi = __half_as_ushort(__int2half_rn(q[2 * i + 1]));
        h[i] = lo | (hi << 16);
      }
      reinterpret_cast<uint4*>(static_cast<uint16_t*>(codes) + off)[0] =
          make_uint4(h[0], h[1], h[2], h[3]);
    } else {
      reinterpret_cast<uint2*>(static_cast<int8_t*>(codes) + off)[0] = pack_codes_i8(q);
    }
    if (sub == 0) {
      if constexpr (kF16Scale)
        static_cast<uint16_t*>(scales)[blk] = __half_as_ushort(__float2half_rn(d));
      else
        static_cast<float*>(scales)[blk] = d;
    }
  }
}

__global__ void __launch_bounds__(256) codes_to_f16_kernel(const int8_t* __restrict__ q,
                                                           uint16_t* __restrict__ out,
                                                           int64_t n16) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride) {
    const int4 c = reinterpret_cast<const int4*>(q)[i];
    const int w[4] = {c.x, c.y, c.z, c.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int b0 = static_cast<int8_t>((w[k] >> (16 * j)) & 0xFF);
        const int b1 = static_cast<int8_t>((w[k] >> (16 * j + 8)) & 0xFF);
        h[2 * k + j] = static_cast<uint32_t>(__half_as_ushort(__int2half_rn(b0))) |
                       (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(b1))) << 16);
      }
    }
    uint4* o = reinterpret_cast<uint4*>(out) + 2 * i;
    o[0] = make_uint4(h[0], h[1], h[2], h[3]);
    o[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// One CTA per row (grid-stride): thread t sums the squares of its 8-element pieces
// t, t + 256, ... in order; the warps' sums meet by a fixed xor tree, then thread 0 adds
// the eight warp sums in order.  The result does not depend on timing.
template <typename InT>
__global__ void __launch_bounds__(256) row_rms_kernel(const InT* __restrict__ x, int64_t M,
                                                      int64_t K, float eps, float* __restrict__ r) {
  // the next kernel (an activation quantizer launched as its programmatic dependent)
  // reads x at once and waits for this grid only before it reads r
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float part[8];
  const int t = threadIdx.x;
  const int64_t npieces = K / 8;
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    float ss = 0.0f;
    for (int64_t p = t; p < npieces; p += 256) {
      float v[8];
      Loader<InT>::load8(x + m * K + 8 * p, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((t & 31) == 0) part[t >> 5] = ss;
    __syncthreads();
    if (t == 0) {
      float s = 0.0f;
      for (int w = 0; w < 8; ++w) s += part[w];
      r[m] = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(s, static_cast<float>(K)), eps)));
    }
    __syncthreads();
  }
}

int grid_for(int64_t work_threads, const DeviceInfo& dev) {
  const int64_t want = (work_threads + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_quantize(const void* x, int xtype, void* codes, bool codes_f16, void* scales,
                            bool scale_f16, int64_t rows, int64_t K, const DeviceInfo& dev,
                            cudaStream_t stream, const Prologue& pro) {
  const int64_t nblocks = rows * (K / kQK);
  if (nblocks == 0) return cudaSuccess;
  const int grid = grid_for(nblocks * 4, dev);
#define Q8_LAUNCH(IN, C16, S16)                                                             \
  quantize_kernel<IN, C16, S16><<<grid, 256, 0, stream>>>(                                  \
      static_cast<const IN*>(x), codes, scales, nblocks, K / kQK, pro.gamma, pro.r)
  if (xtype == 0) {
    if (codes_f16) {
      if (scale_f16) Q8_LAUNCH(float, true, true); else Q8_LAUNCH(float, true, false);
    } else {
      if (scale_f16) Q8_LAUNCH(float, false, true); else Q8_LAUNCH(float, false, false);
    }
  } else {
    if (codes_f16) {
      if (scale_f16) Q8_LAUNCH(uint16_t, true, true); else Q8_LAUNCH(uint16_t, true, false);
    } else {
      if (scale_f16) Q8_LAUNCH(uint16_t, false, true); else Q8_LAUNCH(uint16_t, false, false);
    }
  }
#undef Q8_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_codes_to_f16(const int8_t* q, uint16_t* out, int64_t n, const DeviceInfo& dev,
                                cudaStream_t stream) {
  const int64_t n16 = n / 16;
  if (n16 == 0) return cudaSuccess;
  codes_to_f16_kernel<<<grid_for(n16, dev), 256, 0, stream>>>(q, out, n16);
  return cudaGetLastError();
}

cudaError_t launch_row_rms(const void* x, int xtype, int64_t M, int64_t K, float eps, float* r,
                           const DeviceInfo& dev, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int grid = static_cast<int>(M < static_cast<int64_t>(dev.sm_count) * 8 ? M : dev.sm_count * 8);
  if (xtype == 0)
    row_rms_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), M, K, eps, r);
  else
    row_rms_kernel<uint16_t><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), M, K, eps, r);
  return cudaGetLastError();
}

}  // namespace q8
