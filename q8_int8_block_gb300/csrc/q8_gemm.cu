// q8_gemm.cu -- prefill Q8_0 linear on the 5th-generation tensor cores (tcgen05).
//
// Operation: y[m,n] = sum_b Wd[n,b] * xd[m,b] * isum[m,n,b], the Q8_0 int8 GEMM of
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, list of un-throttled paths: the DP4A int8
// GEMM), for prefill-sized M, where the layer is a dense int8 contraction.
//
// Exact integer block sums on the f16 tensor pipe.  sm_103a has no tcgen05 int8 MMA
// kind, so the int8 codes enter the MMA as binary16 values (|q| <= 127 is exact in
// binary16, every product |q_x q_w| <= 16129 is exact, and every partial sum of one
// 32-element block is an integer of magnitude <= 516128 < 2^24, exact in the binary32
// accumulator).  Each Q8_0 block gets its own TMEM accumulator (two K=16 MMAs starting
// from zero), so the value read back is exactly the int32 block sum isum[m,n,b].
//
// Design (one CTA per 128 x 256 output tile, 320 threads):
//   warp 0     TMA producer: A (activation codes, 128 x 64 binary16) and B (weight codes,
//              256 x 64 binary16) tiles with 128-byte swizzle into a 4-stage ring;
//   warp 1     TMEM owner and MMA issuer: per 32-K block, 2 x tcgen05.mma
//              (M=128, N=256, K=16) into one of two 256-column TMEM buffers, then
//              tcgen05.commit to that buffer's "full" barrier;
//   warps 2-9  rescale drain, two warpgroups of 128 columns each: tcgen05.ld the block
//              sums of their TMEM lanes, y_acc += (Wd * xd) * isum in binary32
//              registers, release the TMEM buffer; finally store y.
// Block-sum mode (for checking) stores the TMEM block sums as int32 instead.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "q8_internal.h"
#include "q8_ptx.cuh"

namespace q8 {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // two Q8_0 blocks per pipeline stage (one 128-byte swizzle row)
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kDrainWarps = 8;
constexpr uint32_t kStageA = BM * BK * 2;   // 16 KB
constexpr uint32_t kStageB = BN * BK * 2;   // 32 KB
constexpr uint32_t kTmemCols = 2 * BN;      // two accumulation buffers
constexpr size_t kSmemBytes = 1024 /*align*/ + kStages * (kStageA + kStageB) +
                              2 /*wg*/ * 2 /*buf*/ * 128 * sizeof(float);

struct GemmParams {
  const float* xd;     // [M, nb]
  const uint16_t* Wd;  // [N, nb]
  float* y;            // [M, N]
  int32_t* isum;       // [M, N, nb] (block-sum mode)
  int M, N, K;
  uint32_t* err;
};

template <bool kBlockSums>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = p.M, N = p.N, K = p.K;
  const int nb = K / kQK;
  const int nk = (K + BK - 1) / BK;
  const int mtiles = (M + BM - 1) / BM;
  const int m0 = (blockIdx.x % mtiles) * BM;
  const int n0 = (blockIdx.x / mtiles) * BN;

  // 1024-byte aligned carve-up (128-byte swizzle atoms must sit on 1024-byte boundaries)
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023) & ~1023u) - raw);
  uint8_t* sA = base;
  uint8_t* sB = base + kStages * kStageA;
  float* sDw = reinterpret_cast<float*>(sB + kStages * kStageB);  // [wg][buf][128]

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kDrainWarps);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(&tmem_base_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;

  if (warp == 0) {
    // ------------------------------- TMA producer -------------------------------------
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&empty_bar[s], ((kb / kStages) & 1) ^ 1, &abort_flag)) {
          report_error(p.err, kErrWaitTimeout, &abort_flag);
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], kStageA + kStageB);
        tma_load_2d(sA + s * kStageA, &tmA, &full_bar[s], kb * BK, m0);
        tma_load_2d(sB + s * kStageB, &tmB, &full_bar[s], kb * BK, n0);
        ++issued;
      }
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
        if (!mbar_wait(&full_bar[kb % kStages], (kb / kStages) & 1, nullptr)) {
          report_error(p.err, kErrWaitTimeout, nullptr);
          break;
        }
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer ---------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      int last_stage = -1;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&full_bar[s], (kb / kStages) & 1, &abort_flag)) {
          report_error(p.err, kErrWaitTimeout, &abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kStageA);
        const uint32_t b0 = smem_u32(sB + s * kStageB);
        const int nblk = (nb - 2 * kb) < 2 ? (nb - 2 * kb) : 2;
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
          const int blk = 2 * kb + j;
          const int buf = blk & 1;
          if (!mbar_wait(&tempty_bar[buf], ((blk >> 1) & 1) ^ 1, &abort_flag)) {
            report_error(p.err, kErrWaitTimeout, &abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((2 * j + kk) * 32);  // 16 f16 = 32 B
            mma_f16_ss(d, sdesc_k_sw128(a0 + koff), sdesc_k_sw128(b0 + koff), idesc,
                       kk > 0 ? 1u : 0u);
          }
          mma_commit(&tfull_bar[buf]);
        }
        mma_commit(&empty_bar[s]);
        last_stage = kb;
        if (!ok) break;
      }
      // do not leave while MMAs are still reading shared memory / writing TMEM
      if (last_stage >= 0 &&
          !mbar_wait(&empty_bar[last_stage % kStages], (last_stage / kStages) & 1, nullptr))
        report_error(p.err, kErrWaitTimeout, nullptr);
    }
  } else {
    // ------------------------------- rescale drain ------------------------------------
    const int dw_idx = warp - 2;            // 0..7
    const int wg = dw_idx >> 2;             // column half of the tile
    const int quad = warp & 3;              // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;       // tile row = TMEM lane
    const int m = m0 + row;
    const int wg_tid = (dw_idx & 3) * 32 + lane;  // 0..127 within the warpgroup
    const int n_load = n0 + wg * 128 + wg_tid;    // the column whose scale this thread stages
    const bool m_ok = m < M;
    float acc[kBlockSums ? 1 : 128];
    if constexpr (!kBlockSums) {
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
    }
    float dw_next = (!kBlockSums && n_load < N) ? __half2float(__ushort_as_half(p.Wd[static_cast<int64_t>(n_load) * nb])) : 0.0f;
    float dx_next = (!kBlockSums && m_ok) ? p.xd[static_cast<int64_t>(m) * nb] : 0.0f;
    for (int blk = 0; blk < nb; ++blk) {
      const int buf = blk & 1;
      float* dws = sDw + (wg * 2 + buf) * 128;
      float dx = 0.0f;
      if constexpr (!kBlockSums) {
        dws[wg_tid] = dw_next;
        dx = dx_next;
      }
      const bool ok = mbar_wait(&tfull_bar[buf], (blk >> 1) & 1, &abort_flag);
      // Warpgroup barrier that also ORs the failures: the 128 threads leave together, and
      // the staged scales are visible to all of them.
      if (wg_barrier_any(2 + wg, !ok)) {
        if (lane == 0) report_error(p.err, kErrWaitTimeout, &abort_flag);
        break;
      }
      if constexpr (!kBlockSums) {
        if (blk + 1 < nb) {
          dw_next = n_load < N ? __half2float(__ushort_as_half(p.Wd[static_cast<int64_t>(n_load) * nb + blk + 1])) : 0.0f;
          dx_next = m_ok ? p.xd[static_cast<int64_t>(m) * nb + blk + 1] : 0.0f;
        }
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(buf * BN + wg * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
        if constexpr (kBlockSums) {
          if (m_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int n = n0 + wg * 128 + c * 32 + i;
              if (n < N)
                p.isum[(static_cast<int64_t>(m) * N + n) * nb + blk] =
                    __float2int_rn(__uint_as_float(r[i]));
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(dws + c * 32 + i);
            acc[c * 32 + i + 0] = fmaf(dx * w4.x, __uint_as_float(r[i + 0]), acc[c * 32 + i + 0]);
            acc[c * 32 + i + 1] = fmaf(dx * w4.y, __uint_as_float(r[i + 1]), acc[c * 32 + i + 1]);
            acc[c * 32 + i + 2] = fmaf(dx * w4.z, __uint_as_float(r[i + 2]), acc[c * 32 + i + 2]);
            acc[c * 32 + i + 3] = fmaf(dx * w4.w, __uint_as_float(r[i + 3]), acc[c * 32 + i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[buf]);
    }
    if constexpr (!kBlockSums) {
      if (m_ok) {
        float* yrow = p.y + static_cast<int64_t>(m) * N;
        const int nbase = n0 + wg * 128;
        if ((N & 3) == 0 && nbase + 128 <= N) {
#pragma unroll
          for (int i = 0; i < 128; i += 4)
            *reinterpret_cast<float4*>(yrow + nbase + i) =
                make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (nbase + i < N) yrow[nbase + i] = acc[i];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---- host: tensor maps ------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D binary16 matrix [rows, cols] (cols contiguous), box = box_rows x 64 columns, 128B swizzle.
bool make_tmap_f16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBS>
cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, int grid,
                        cudaStream_t stream) {
  auto fn = gemm_tc_kernel<kBS>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  fn<<<grid, kThreads, kSmemBytes, stream>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(const uint16_t* A16, const uint16_t* B16, const float* xd,
                           const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                           int64_t K, const DeviceInfo& dev, cudaStream_t stream) {
  (void)dev;
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0) return cudaErrorInvalidValue;  // the API handles K == 0 without a launch
  CUtensorMap ta, tb;
  if (!make_tmap_f16(&ta, A16, static_cast<uint64_t>(M), static_cast<uint64_t>(K), BM) ||
      !make_tmap_f16(&tb, B16, static_cast<uint64_t>(N), static_cast<uint64_t>(K), BN))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.xd = xd;
  p.Wd = Wd;
  p.y = y;
  p.isum = isum;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.err = dev.err_word;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  return isum ? launch_impl<true>(ta, tb, p, static_cast<int>(tiles), stream)
              : launch_impl<false>(ta, tb, p, static_cast<int>(tiles), stream);
}

}  // namespace q8
