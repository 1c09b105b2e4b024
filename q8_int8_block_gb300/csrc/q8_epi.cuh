// q8_epi.cuh -- the layer's neighbours fused into every kernel's output store:
// y = op(acc, aux), stored as binary32 or bfloat16.
//
// The post runs its Q8_0 linears inside GDN + attention blocks ("CUDA inference engine for
// running Qwen3.5/3.6 hybrid models on mining cards (CMP 100-210)", news.hada.io topic
// 29953, feature list), whose FFN gates the up projection by SiLU of the gate projection and
// whose blocks add residuals.  Readings: op 1 adds a residual (y = acc + aux), op 2 is the
// gated unit (y = silu(aux) * acc, aux = the gate projection's output, silu(g) =
// g / (1 + e^-g)); binary32 arithmetic, then round-to-nearest-even to bfloat16 if asked.
//
// aux never overlaps y (the entry point's contract), so it is read through the read-only
// data path.  The kernels load aux early (or prefetch it to L2) and apply the epilogue at
// the store, so that the load latency is not paid once per output.
#pragma once
#include <cuda_bf16.h>

#include "q8_internal.h"

namespace q8 {

// aux value of output i (0 when the epilogue takes none)
__device__ __forceinline__ float epi_aux(const Epilogue& e, int64_t i) {
  return e.op == kEpiNone ? 0.0f : __ldg(e.aux + i);
}

// aux values of outputs i .. i + 3 (i a multiple of 4: aux is 16-byte aligned)
__device__ __forceinline__ float4 epi_aux4(const Epilogue& e, int64_t i) {
  return e.op == kEpiNone ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                          : __ldg(reinterpret_cast<const float4*>(e.aux + i));
}

__device__ __forceinline__ float epi_apply(const Epilogue& e, float v, float a) {
  if (e.op == kEpiAdd) return v + a;
  if (e.op == kEpiSiluMul) return v * (a / (1.0f + expf(-a)));
  return v;
}

__device__ __forceinline__ float4 epi_apply4(const Epilogue& e, float4 v, float4 a) {
  return make_float4(epi_apply(e, v.x, a.x), epi_apply(e, v.y, a.y), epi_apply(e, v.z, a.z),
                     epi_apply(e, v.w, a.w));
}

__device__ __forceinline__ void epi_put(const Epilogue& e, float* y, int64_t i, float v) {
  if (e.bf16)
    reinterpret_cast<__nv_bfloat16*>(y)[i] = __float2bfloat16_rn(v);
  else
    y[i] = v;
}

// outputs i .. i + 3, i a multiple of 4 (y is 16-byte aligned: 8 bytes of bfloat16)
__device__ __forceinline__ void epi_put4(const Epilogue& e, float* y, int64_t i, float4 v) {
  if (e.bf16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(y) + i) = u;
  } else {
    *reinterpret_cast<float4*>(y + i) = v;
  }
}

__device__ __forceinline__ void epi_store(const Epilogue& e, float* y, int64_t i, float v) {
  epi_put(e, y, i, epi_apply(e, v, epi_aux(e, i)));
}

// bring aux[i .. i + n) towards L2 ahead of its use (one prefetch per 128-byte line)
__device__ __forceinline__ void epi_prefetch(const Epilogue& e, int64_t i, int n) {
  if (e.op == kEpiNone) return;
  const char* a = reinterpret_cast<const char*>(e.aux + i);
  const char* end = reinterpret_cast<const char*>(e.aux + i + n);
  for (const char* l = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(127));
       l < end; l += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(l));
}

}  // namespace q8
