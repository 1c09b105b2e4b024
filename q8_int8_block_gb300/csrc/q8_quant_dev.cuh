// q8_quant_dev.cuh -- the Q8_0 block quantizer as a device function, shared by the
// standalone quantization kernel and the decode kernel's fused activation quantizer, so
// both produce the same codes and scales bit for bit.
//
// Four consecutive lanes own one 32-element block, 8 values each.  d = amax / 127 (IEEE
// binary32 division); q = round(v / d), ties away from zero (roundf), clamped to
// [-127, 127]; d == 0 gives codes 0.
#pragma once
#include <cstdint>

namespace q8 {

// v: this lane's 8 values of the block; group_mask: the 4 lanes of the block.
// Returns d; writes the 8 codes into q.
__device__ __forceinline__ float quantize_block_x4(const float (&v)[8], unsigned group_mask,
                                                   int (&q)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(group_mask, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(group_mask, amax, 2));
  const float d = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = 0.0f;
    if (d != 0.0f) r = fminf(fmaxf(roundf(__fdiv_rn(v[i], d)), -127.0f), 127.0f);
    q[i] = static_cast<int>(r);
  }
  return d;
}

// 8 int codes -> 8 packed int8 bytes (lo = codes 0..3, hi = codes 4..7).
__device__ __forceinline__ uint2 pack_codes_i8(const int (&q)[8]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo |= (static_cast<uint32_t>(q[i]) & 0xFFu) << (8 * i);
    hi |= (static_cast<uint32_t>(q[4 + i]) & 0xFFu) << (8 * i);
  }
  return make_uint2(lo, hi);
}

// 8 bf16 bit patterns (one 16-byte vector) -> 8 floats (exact widening).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 a, float (&v)[8]) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

}  // namespace q8
