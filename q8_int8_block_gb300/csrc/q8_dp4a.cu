// q8_dp4a.cu -- the Q8_0 int8 GEMM as the post builds it: dp4a on CUDA cores.
//
// Operation: y[m,n] = sum_b Wd[n,b] * xd[m,b] * isum[m,n,b], the Q8_0 int8 GEMM of
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, list of un-throttled paths: the DP4A int8
// GEMM, "int8, 17 TFLOP" on the mining cards).  There the tensor cores are throttled, so
// the post forms the int8 dot products with the 4-way dp4a instruction; this kernel is that
// design on GB300, kept as the prior-art comparison for the tensor-core path (q8_gemm.cu).
// It is exact in the same way: each 32-element block sum is 8 dp4a into an int32.
//
// Design (tile of 64 tokens x 128 weight rows, 256 threads, 2 CTAs per SM):
//   * 64-wide K chunks (two Q8_0 blocks) of the int8 activation codes (64 x 64 bytes) and
//     weight codes (128 x 64 bytes) are copied into shared memory with 16-byte cp.async,
//     double-buffered; rows are 80 bytes apart so that the 16-byte loads of 8 consecutive
//     weight rows fall in 8 distinct bank groups;
//   * thread (ty, tx) owns tokens ty + 16 i (i < 4) and weight rows tx + 16 j (j < 8): per
//     block it loads the 32 codes of each, forms the 32 block sums with 8 dp4a each, and
//     adds (xd * Wd) * isum to binary32 accumulators;
//   * block-sum mode (for checking) stores the int32 sums instead.
#include <cuda_fp16.h>

#include <algorithm>

#include "q8_epi.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int TM = 64;         // tokens per CTA
constexpr int TN = 128;        // weight rows per CTA
constexpr int TK = 64;         // K per chunk (two Q8_0 blocks)
constexpr int kPitch = 80;     // bytes per shared-memory row (64 + 16 padding)
constexpr int kThreads = 256;
constexpr int kTileA = TM * kPitch;  // 5120 bytes
constexpr int kTileB = TN * kPitch;  // 10240 bytes

struct Dp4aParams {
  const int8_t* xq;    // [M, K]
  const float* xd;     // [M, nb]
  const int8_t* Wq;    // [N, K]
  const uint16_t* Wd;  // [N, nb]
  float* y;            // [M, N]
  int32_t* isum;       // [M, N, nb] (block-sum mode)
  int M, N, K;
  Epilogue epi;        // fused output step
};

// 16-byte global -> shared copy; src_bytes 0 fills zeros (rows or K past the ends).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kBlockSums>
__global__ void __launch_bounds__(kThreads, 2) dp4a_gemm_kernel(const Dp4aParams p) {
  __shared__ __align__(16) uint8_t sA[2][kTileA];
  __shared__ __align__(16) uint8_t sB[2][kTileB];
  const int t = threadIdx.x;
  const int tx = t & 15, ty = t >> 4;
  const int n0 = blockIdx.x * TN, m0 = blockIdx.y * TM;
  const int M = p.M, N = p.N, K = p.K;
  const int nb = K / 32;
  const int nchunk = (K + TK - 1) / TK;

  // one chunk: A 64 rows x 4 pieces (1 per thread), B 128 rows x 4 pieces (2 per thread)
  auto load_chunk = [&](int c, int buf) {
    const int k0 = c * TK;
    {
      const int r = t >> 2, q = t & 3;
      const int m = m0 + r, k = k0 + 16 * q;
      const bool ok = m < M && k < K;
      cp_async16(&sA[buf][r * kPitch + 16 * q], ok ? p.xq + static_cast<int64_t>(m) * K + k : p.xq,
                 ok ? 16 : 0);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int idx = t + kThreads * h;
      const int r = idx >> 2, q = idx & 3;
      const int n = n0 + r, k = k0 + 16 * q;
      const bool ok = n < N && k < K;
      cp_async16(&sB[buf][r * kPitch + 16 * q], ok ? p.Wq + static_cast<int64_t>(n) * K + k : p.Wq,
                 ok ? 16 : 0);
    }
    cp_async_commit();
  };

  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  load_chunk(0, 0);
  for (int c = 0; c < nchunk; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunk) {
      load_chunk(c + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // the chunk's two Q8_0 blocks
      const int b = 2 * c + h;
      if (b >= nb) break;
      // block sums in two 16-byte halves (keeps the codes of one half in registers)
      int sum[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) sum[i][j] = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        int4 a[4], w[8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          a[i] = *reinterpret_cast<const int4*>(&sA[buf][(ty + 16 * i) * kPitch + 32 * h + 16 * q]);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          w[j] = *reinterpret_cast<const int4*>(&sB[buf][(tx + 16 * j) * kPitch + 32 * h + 16 * q]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            int s4 = __dp4a(a[i].x, w[j].x, sum[i][j]);
            s4 = __dp4a(a[i].y, w[j].y, s4);
            s4 = __dp4a(a[i].z, w[j].z, s4);
            sum[i][j] = __dp4a(a[i].w, w[j].w, s4);
          }
      }
      if constexpr (kBlockSums) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
            if (m < M && n < N) p.isum[(static_cast<int64_t>(m) * N + n) * nb + b] = sum[i][j];
          }
      } else {
        float dx[4], dw[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = m0 + ty + 16 * i;
          dx[i] = m < M ? __ldg(p.xd + static_cast<int64_t>(m) * nb + b) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = n0 + tx + 16 * j;
          dw[j] = n < N ? __half2float(__ushort_as_half(__ldg(p.Wd + static_cast<int64_t>(n) * nb + b)))
                        : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            acc[i][j] = fmaf(dx[i] * dw[j], static_cast<float>(sum[i][j]), acc[i][j]);
      }
    }
    __syncthreads();  // the buffer is refilled by the next iteration's copies
  }
  if constexpr (!kBlockSums) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + ty + 16 * i;
      if (m >= M) continue;
      float a[8];  // the row's aux loads in flight together
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = n0 + tx + 16 * j;
        a[j] = n < N ? epi_aux(p.epi, static_cast<int64_t>(m) * N + n) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = n0 + tx + 16 * j;
        if (n < N) epi_put(p.epi, p.y, static_cast<int64_t>(m) * N + n, epi_apply(p.epi, acc[i][j], a[j]));
      }
    }
  }
}

}  // namespace

cudaError_t launch_dp4a_gemm(const int8_t* xq, const float* xd, const int8_t* Wq,
                             const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                             int64_t K, cudaStream_t stream, const Epilogue& epi) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0) return cudaErrorInvalidValue;  // the API handles K == 0 without a launch
  const int64_t gx = (N + TN - 1) / TN, gy = (M + TM - 1) / TM;
  if (gx > 0x7FFFFFFF || gy > 65535) return cudaErrorInvalidValue;
  Dp4aParams p;
  p.xq = xq;
  p.xd = xd;
  p.Wq = Wq;
  p.Wd = Wd;
  p.y = y;
  p.isum = isum;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.epi = epi;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  if (isum)
    dp4a_gemm_kernel<true><<<grid, kThreads, 0, stream>>>(p);
  else
    dp4a_gemm_kernel<false><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace q8
