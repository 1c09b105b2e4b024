// bench_rates.cu -- per-SM rate microbenchmarks behind the secondary rooflines of bench.py
// and the Q8_0 GEMM's analysis.  Every kernel runs one CTA per SM; each timed warp measures
// its own loop with clock64, and a rate is (operations of the SM) / (cycles of its slowest
// timed warp).  Built and run by bench_rates.py; the results are a JSON line.
//
//   ffma      binary32 fused multiply-adds per clock per SM (scalar FFMA)
//   ffma2     the same with the packed f32x2 form (fma.rn.f32x2)
//   dp4a      4-way int8 dot products per clock per SM
//   hmma      mma.sync m16n8k16 f16 x f16 -> f32 multiply-adds per clock per SM
//   imma      mma.sync m16n8k32 s8 x s8 -> s32 multiply-adds per clock per SM
//   umma      tcgen05.mma kind::f16 M128 N256 K16: multiply-adds per clock per SM, one thread
//             issuing back to back into two TMEM buffers
//   lds_bcast 16-byte shared-memory loads with one address per warp (the GEMM drain's
//             column-scale loads), warp instructions per clock per SM
//   commit_rt tcgen05.commit + mbarrier wait round trip after an M128 N256 K16 pair, cycles
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "q8_int8_block_gb300/csrc/q8_ptx.cuh"

using namespace q8;

namespace {

constexpr int kIters = 4096;

// 8 independent chains per thread so that the pipe, not latency, is the limit
__global__ void __launch_bounds__(512) ffma_kernel(float* out, long long* cyc) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = threadIdx.x * 1e-3f + i;
  const float b = 0.999f, c = 1e-4f;
  const long long t0 = clock64();
#pragma unroll 4
  for (int it = 0; it < kIters; ++it)
#pragma unroll
    for (int i = 0; i < 8; ++i) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a[i]) : "f"(b), "f"(c));
  const long long t1 = clock64();
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if ((threadIdx.x & 31) == 0) cyc[blockIdx.x * 16 + (threadIdx.x >> 5)] = t1 - t0;
}

__global__ void __launch_bounds__(512) ffma2_kernel(float* out, long long* cyc) {
  float2 a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = make_float2(threadIdx.x * 1e-3f + i, i + 0.5f);
  const float2 b = make_float2(0.999f, 0.998f), c = make_float2(1e-4f, 2e-4f);
  const long long t0 = clock64();
#pragma unroll 4
  for (int it = 0; it < kIters; ++it)
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = __ffma2_rn(a[i], b, c);
  const long long t1 = clock64();
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) s += a[i].x + a[i].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if ((threadIdx.x & 31) == 0) cyc[blockIdx.x * 16 + (threadIdx.x >> 5)] = t1 - t0;
}

__global__ void __launch_bounds__(512) dp4a_kernel(int* out, long long* cyc) {
  int a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = threadIdx.x + i;
  const int b = 0x01FF7F80, c = 0x7F01FF02;
  const long long t0 = clock64();
#pragma unroll 4
  for (int it = 0; it < kIters; ++it)
#pragma unroll
    for (int i = 0; i < 8; ++i) asm volatile("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(a[i]) : "r"(b), "r"(c));
  const long long t1 = clock64();
  int s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if ((threadIdx.x & 31) == 0) cyc[blockIdx.x * 16 + (threadIdx.x >> 5)] = t1 - t0;
}

// 4 independent accumulators of one m16n8k16 (f16 in, f32 accumulate) per warp
__global__ void __launch_bounds__(512) hmma_kernel(float* out, long long* cyc) {
  uint32_t a[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
  uint32_t b[2] = {0x3C003C00u, 0x3C003C00u};
  float d[4][4] = {};
  const long long t0 = clock64();
#pragma unroll 2
  for (int it = 0; it < kIters; ++it)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(d[k][0]), "+f"(d[k][1]), "+f"(d[k][2]), "+f"(d[k][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  const long long t1 = clock64();
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) s += d[k][0] + d[k][1] + d[k][2] + d[k][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if ((threadIdx.x & 31) == 0) cyc[blockIdx.x * 16 + (threadIdx.x >> 5)] = t1 - t0;
}

// 4 independent accumulators of one m16n8k32 (s8 in, s32 accumulate) per warp
__global__ void __launch_bounds__(512) imma_kernel(int* out, long long* cyc) {
  uint32_t a[4] = {0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u};
  uint32_t b[2] = {0x01010101u, 0x01010101u};
  int d[4][4] = {};
  const long long t0 = clock64();
#pragma unroll 2
  for (int it = 0; it < kIters; ++it)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+r"(d[k][0]), "+r"(d[k][1]), "+r"(d[k][2]), "+r"(d[k][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  const long long t1 = clock64();
  int s = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) s += d[k][0] + d[k][1] + d[k][2] + d[k][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if ((threadIdx.x & 31) == 0) cyc[blockIdx.x * 16 + (threadIdx.x >> 5)] = t1 - t0;
}

// Broadcast 16-byte shared-memory loads: every lane of a warp reads the same address.
__global__ void __launch_bounds__(256) lds_kernel(float* out, long long* cyc) {
  __shared__ float4 tab[1024];
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) tab[i] = make_float4(i, i + 1, i + 2, i + 3);
  __syncthreads();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int warp = threadIdx.x >> 5;
  const long long t0 = clock64();
#pragma unroll 8
  for (int it = 0; it < kIters; ++it) {
    const float4 v = tab[(it * 8 + warp) & 1023];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const long long t1 = clock64();
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc.x + acc.y + acc.z + acc.w;
  if ((threadIdx.x & 31) == 0) cyc[blockIdx.x * 16 + warp] = t1 - t0;
}

// tcgen05 kind::f16 M128 N256 K16 back to back (mode 0: pairs into alternating buffers,
// commit every 8 pairs; mode 1: one pair, commit, wait -- the round trip).
template <int kMode>
__global__ void __launch_bounds__(128, 1) umma_kernel(int iters, long long* cyc, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ uint64_t bar;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023) & ~1023u) - raw);
  for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(base)[i] = 0x3C003C00u;
  fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  if (threadIdx.x == 32) {
    constexpr uint32_t idesc = idesc_f16_f32(128, 256);
    const uint32_t a0 = smem_u32(base), b0 = smem_u32(base + 16384);
    int phase = 0;
    const long long t0 = clock64();
    for (int p = 0; p < iters; ++p) {
      const uint32_t d = tmem_base + static_cast<uint32_t>((p & 1) * 256);
      mma_f16_ss(d, sdesc_k_sw128(a0), sdesc_k_sw128(b0), idesc, 0u);
      mma_f16_ss(d, sdesc_k_sw128(a0 + 32), sdesc_k_sw128(b0 + 32), idesc, 1u);
      if (kMode == 1 || (p & 7) == 7) {
        mma_commit(&bar);
        if (!mbar_wait(&bar, phase & 1, nullptr)) {
          atomicOr(err, 1u);
          break;
        }
        ++phase;
      }
    }
    // every MMA issued is finished before TMEM is freed
    mma_commit(&bar);
    if (!mbar_wait(&bar, phase & 1, nullptr)) atomicOr(err, 1u);
    const long long t1 = clock64();
    cyc[blockIdx.x] = (t1 - t0) / iters;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// tcgen05 kind::f16 (bfloat16) chains of the block-sparse attention kernel's shapes.  One
// thread per CTA issues dependent K=16 MMAs into one accumulator (commit + wait every 64).
// kMix = 0: M x N MMAs only; kMix = 1: per "block" 8 x M64 N64 (S) + 4 x M64 N128 (O), the
// attention kernel's per-key-block work.  Shared memory is sized for at most two CTAs per SM.
template <int M, int N, int kMix>
__global__ void __launch_bounds__(128) umma_chain_kernel(int iters, long long* cyc, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ uint64_t bar;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023) & ~1023u) - raw);
  for (int i = threadIdx.x; i < 49152 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(base)[i] = 0x3F803F80u;
  fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  if (threadIdx.x == 32) {
    const uint32_t a0 = smem_u32(base), b0 = smem_u32(base + 16384);
    constexpr uint32_t kBf16 = (1u << 7) | (1u << 10);
    int phase = 0;
    const long long t0 = clock64();
    for (int p = 0; p < iters; ++p) {
      if (kMix == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          mma_f16_ss(tmem_base, sdesc_k_sw128(a0 + (q & 3) * 32), sdesc_k_sw128(b0 + (q & 3) * 32),
                     idesc_f16_f32(M, N) | kBf16, (p | q) ? 1u : 0u);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          mma_f16_ss(tmem_base + (p & 1) * 64, sdesc_k_sw128(a0 + (q & 3) * 32),
                     sdesc_k_sw128(b0 + (q & 3) * 32), idesc_f16_f32(64, 64) | kBf16, q > 0 ? 1u : 0u);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          mma_f16_ss(tmem_base + 128, sdesc_k_sw128(a0 + (q & 3) * 32), sdesc_k_sw128(b0 + (q & 3) * 32),
                     idesc_f16_f32(64, 128) | kBf16, 1u);
      }
      if ((p & 7) == 7) {
        mma_commit(&bar);
        if (!mbar_wait(&bar, phase & 1, nullptr)) {
          atomicOr(err, 1u);
          break;
        }
        ++phase;
      }
    }
    // every MMA issued is finished before TMEM is freed
    mma_commit(&bar);
    if (!mbar_wait(&bar, phase & 1, nullptr)) atomicOr(err, 1u);
    cyc[blockIdx.x] = (clock64() - t0) / iters;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

double max_cycles(const long long* h, int n) {
  double m = 0;
  for (int i = 0; i < n; ++i) m = h[i] > m ? static_cast<double>(h[i]) : m;
  return m;
}

}  // namespace

// Runs every benchmark on `sms` SMs; fills res[] (see the names in bench_rates.py).
extern "C" int q8_rates(int sms, double* res) {
  float* fout = nullptr;
  long long* cyc = nullptr;
  uint32_t* err = nullptr;
  if (cudaMalloc(&fout, sizeof(float) * sms * 512) != cudaSuccess) return -1;
  if (cudaMalloc(&cyc, sizeof(long long) * sms * 16) != cudaSuccess) return -1;
  if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return -1;
  cudaMemset(err, 0, sizeof(uint32_t));
  long long* h = new long long[sms * 16];
  // slowest timed warp of the last launch; the slots are cleared before each measurement
  auto clear = [&]() { cudaMemset(cyc, 0, sizeof(long long) * sms * 16); };
  auto get = [&](int n) {
    cudaMemcpy(h, cyc, sizeof(long long) * n, cudaMemcpyDeviceToHost);
    return max_cycles(h, n);
  };
  // per SM: 512 threads x kIters x 8 chains
  clear();
  ffma_kernel<<<sms, 512>>>(fout, cyc);
  ffma_kernel<<<sms, 512>>>(fout, cyc);
  res[0] = 512.0 * kIters * 8 / get(sms * 16);  // FMA per clock per SM
  clear();
  ffma2_kernel<<<sms, 512>>>(fout, cyc);
  ffma2_kernel<<<sms, 512>>>(fout, cyc);
  res[1] = 512.0 * kIters * 8 / get(sms * 16);  // FMA per clock per SM (2 per instruction)
  clear();
  dp4a_kernel<<<sms, 512>>>(reinterpret_cast<int*>(fout), cyc);
  dp4a_kernel<<<sms, 512>>>(reinterpret_cast<int*>(fout), cyc);
  res[2] = 512.0 * kIters * 8 / get(sms * 16);  // dp4a per clock per SM
  clear();
  hmma_kernel<<<sms, 512>>>(fout, cyc);
  hmma_kernel<<<sms, 512>>>(fout, cyc);
  res[3] = 16.0 * kIters * 4 * (16 * 8 * 16) / get(sms * 16);  // MACs per clock per SM
  clear();
  imma_kernel<<<sms, 512>>>(reinterpret_cast<int*>(fout), cyc);
  imma_kernel<<<sms, 512>>>(reinterpret_cast<int*>(fout), cyc);
  res[4] = 16.0 * kIters * 4 * (16 * 8 * 32) / get(sms * 16);  // MACs per clock per SM
  clear();
  lds_kernel<<<sms, 256>>>(fout, cyc);
  lds_kernel<<<sms, 256>>>(fout, cyc);
  res[5] = 8.0 * kIters / get(sms * 16);  // warp-wide broadcast LDS.128 per clock per SM
  const int smem = 160 * 1024;  // one CTA per SM (the TMEM allocation is the whole SM's)
  cudaFuncSetAttribute(umma_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(umma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  clear();
  umma_kernel<0><<<sms, 128, smem>>>(8000, cyc, err);
  umma_kernel<0><<<sms, 128, smem>>>(8000, cyc, err);
  res[6] = 2.0 * (128 * 256 * 16) / get(sms);  // MACs per clock per SM
  clear();
  umma_kernel<1><<<sms, 128, smem>>>(2000, cyc, err);
  umma_kernel<1><<<sms, 128, smem>>>(2000, cyc, err);
  res[7] = get(sms);  // cycles per pair + commit + wait
  // attention shapes: per-CTA cycles of the slowest CTA, two CTAs (or one) per SM
  const int smem2 = 80 * 1024;  // at most two CTAs per SM (49 KB used)
  cudaFuncSetAttribute(umma_chain_kernel<64, 64, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
  cudaFuncSetAttribute(umma_chain_kernel<128, 64, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
  cudaFuncSetAttribute(umma_chain_kernel<64, 64, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
  clear();
  umma_chain_kernel<64, 64, 0><<<sms, 128, smem2>>>(1024, cyc, err);
  umma_chain_kernel<64, 64, 0><<<sms, 128, smem2>>>(1024, cyc, err);
  res[8] = get(sms) / 8.0;  // cycles per M64 N64 MMA, one CTA per SM
  clear();
  umma_chain_kernel<64, 64, 0><<<2 * sms, 128, smem2>>>(1024, cyc, err);
  umma_chain_kernel<64, 64, 0><<<2 * sms, 128, smem2>>>(1024, cyc, err);
  res[9] = 2.0 * 8 * (64 * 64 * 16) / get(2 * sms);  // MACs per clock per SM
  clear();
  umma_chain_kernel<128, 64, 0><<<2 * sms, 128, smem2>>>(1024, cyc, err);
  umma_chain_kernel<128, 64, 0><<<2 * sms, 128, smem2>>>(1024, cyc, err);
  res[10] = 2.0 * 8 * (128 * 64 * 16) / get(2 * sms);  // MACs per clock per SM
  clear();
  umma_chain_kernel<64, 64, 1><<<2 * sms, 128, smem2>>>(1024, cyc, err);
  umma_chain_kernel<64, 64, 1><<<2 * sms, 128, smem2>>>(1024, cyc, err);
  res[11] = get(2 * sms);  // cycles per attention key block per CTA
  uint32_t e = 0;
  cudaMemcpy(&e, err, sizeof e, cudaMemcpyDeviceToHost);
  const cudaError_t st = cudaDeviceSynchronize();
  delete[] h;
  cudaFree(fout);
  cudaFree(cyc);
  cudaFree(err);
  return (st == cudaSuccess && e == 0) ? 12 : -2;
}
