// q8_decode.cu -- small-M (decode) Q8_0 linear: streams the weight codes from HBM once,
// at the memory's rate, and forms every block sum with dp4a.
//
// Operation: y[m,n] = sum_b Wd[n,b] * xd[m,b] * isum[m,n,b], the Q8_0 int8 GEMM of
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, list of un-throttled paths: the DP4A int8
// GEMM), at decode batch sizes (M <= 8), where the layer is bound by reading the weights.
//
// Design (one CTA per SM, persistent):
//   * CTA c owns the contiguous rows [r0, r1) of W; their codes form one contiguous byte
//     range, streamed row by row through a ring of shared-memory stages with bulk async
//     copies (one elected producer thread, one mbarrier per stage).  A row's binary16
//     scales ride in the same stage when the row of scales is 16-byte sized (K % 256 == 0),
//     else they are read from global memory.
//   * While the first rows are in flight, the consumer warps quantize the M activation
//     rows into shared memory (fused activation quantizer: the same device function as
//     the standalone quantizer, so codes and scales are identical).
//   * Each consumer warp takes whole rows: lane l handles the 16-byte pieces l, l+32, ...
//     of the row, 4 dp4a per piece and token; an xor-shuffle joins the two halves of each
//     32-element block into the exact int32 block sum, the even lane rescales it by
//     Wd*xd in binary32, and a warp reduction finishes the row.
//   * Block-sum mode (for checking) takes int8 codes instead of x and writes the raw
//     block sums instead of y.
#include <cuda_fp16.h>

#include "q8_internal.h"
#include "q8_ptx.cuh"
#include "q8_quant_dev.cuh"

namespace q8 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxStages = 32;

struct DecodeParams {
  const void* x;       // [M,K] bf16 bits or f32 (fused quantization)
  int xtype;           // 0 f32, 1 bf16
  const int8_t* xq;    // [M,K] int8 codes (block-sum mode)
  const int8_t* Wq;    // [N,K]
  const uint16_t* Wd;  // [N,K/32]
  float* y;            // [M,N]
  int32_t* isum;       // [M,N,K/32] (block-sum mode)
  int M, N, K;
  int stages;
  uint32_t* err;
};

__device__ __forceinline__ int4 lds128(const void* p) {
  return *reinterpret_cast<const int4*>(p);
}

template <int MT, bool kBlockSums, bool kScalesInStage>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full_bar[kMaxStages];
  __shared__ uint64_t empty_bar[kMaxStages];
  __shared__ int abort_flag;

  const int K = p.K, N = p.N, M = p.M;
  const int nb = K / kQK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * N / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * N / gridDim.x;
  const int nrows = static_cast<int>(r1 - r0);
  const int S = p.stages;

  // shared memory carve-up: [x codes MT*K][x scales MT*nb f32][stages]
  int8_t* xs = reinterpret_cast<int8_t*>(smem);
  float* xds = reinterpret_cast<float*>(smem + MT * K);
  const uint32_t scale_bytes = kScalesInStage ? static_cast<uint32_t>(nb * 2) : 0u;
  const uint32_t stage_bytes = static_cast<uint32_t>(K) + scale_bytes;
  uint8_t* ring = smem + ((MT * K + MT * nb * 4 + 127) & ~127);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer: one thread streams the rows through the ring ----------
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nrows; ++j) {
        const int s = j % S;
        if (!mbar_wait(&empty_bar[s], ((j / S) & 1) ^ 1, &abort_flag)) {
          report_error(p.err, kErrWaitTimeout, &abort_flag);
          break;
        }
        uint8_t* st = ring + static_cast<size_t>(s) * stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
        bulk_load(st, p.Wq + (r0 + j) * static_cast<int64_t>(K), static_cast<uint32_t>(K),
                  &full_bar[s]);
        if constexpr (kScalesInStage)
          bulk_load(st + K, p.Wd + (r0 + j) * static_cast<int64_t>(nb), scale_bytes,
                    &full_bar[s]);
        ++issued;
      }
      // Never leave with copies in flight: wait for the last stages issued.
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
        if (!mbar_wait(&full_bar[j % S], (j / S) & 1, nullptr)) {
          report_error(p.err, kErrWaitTimeout, nullptr);
          break;
        }
    }
  } else {
    // ---------------- consumers ----------------------------------------------------------
    const int cw = warp - 1;                   // consumer warp index
    const int ct = threadIdx.x - 32;           // consumer thread index
    constexpr int kCT = 32 * kConsumerWarps;   // consumer threads
    // 1) activation codes and scales into shared memory
    if constexpr (kBlockSums) {
      const int n16 = M * K / 16;
      for (int i = ct; i < n16; i += kCT)
        reinterpret_cast<int4*>(xs)[i] = reinterpret_cast<const int4*>(p.xq)[i];
    } else {
      const int nblk = M * nb;
      const int sub = lane & 3;
      const unsigned gmask = 0xFu << (lane & ~3);
      // every group of 4 lanes of every warp runs the same number of iterations
      const int iters = (nblk + kCT / 4 - 1) / (kCT / 4);
      for (int it = 0; it < iters; ++it) {
        const int blk = it * (kCT / 4) + (ct >> 2);
        if (blk < nblk) {
          float v[8];
          const int64_t off = static_cast<int64_t>(blk) * kQK + sub * 8;
          if (p.xtype == 1) {
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + off),
                          v);
          } else {
            const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off);
            const float4 a = f[0], b = f[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
          }
          int q[8];
          const float d = quantize_block_x4(v, gmask, q);
          *reinterpret_cast<uint2*>(xs + off) = pack_codes_i8(q);
          if (sub == 0) xds[blk] = d;
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory");

    // 2) rows
    const int npieces = K >> 4;  // 16-byte pieces per row (even, since K % 32 == 0)
    const int iters = (npieces + 31) >> 5;
    for (int j = cw; j < nrows; j += kConsumerWarps) {
      const int s = j % S;
      // every lane waits (and so observes the copied bytes); the warp leaves together
      const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full_bar[s], (j / S) & 1, &abort_flag));
      if (!ok) {
        if (lane == 0) report_error(p.err, kErrWaitTimeout, &abort_flag);
        break;
      }
      const uint8_t* st = ring + static_cast<size_t>(s) * stage_bytes;
      const uint16_t* wd_row = kScalesInStage
                                   ? reinterpret_cast<const uint16_t*>(st + K)
                                   : p.Wd + (r0 + j) * static_cast<int64_t>(nb);
      const int64_t n = r0 + j;
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
#pragma unroll 2
      for (int i = 0; i < iters; ++i) {
        const int pc = lane + (i << 5);
        const bool valid = pc < npieces;
        const int blk = pc >> 1;
        int4 w = make_int4(0, 0, 0, 0);
        float dw = 0.0f;
        if (valid) {
          w = lds128(st + 16 * pc);
          if constexpr (!kBlockSums) dw = __half2float(__ushort_as_half(wd_row[blk]));
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          int sum = 0;
          if (t < M && valid) {
            const int4 xv = lds128(xs + t * K + 16 * pc);
            sum = __dp4a(w.x, xv.x, sum);
            sum = __dp4a(w.y, xv.y, sum);
            sum = __dp4a(w.z, xv.z, sum);
            sum = __dp4a(w.w, xv.w, sum);
          }
          sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);  // exact int32 block sum
          if constexpr (kBlockSums) {
            if (t < M && valid && !(lane & 1))
              p.isum[(static_cast<int64_t>(t) * N + n) * nb + blk] = sum;
          } else {
            if (t < M && valid && !(lane & 1))
              acc[t] = fmaf(dw * xds[t * nb + blk], static_cast<float>(sum), acc[t]);
          }
        }
      }
      if constexpr (!kBlockSums) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          float a = acc[t];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
          if (lane == 0 && t < M) p.y[static_cast<int64_t>(t) * N + n] = a;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
  }
  __syncthreads();
}

template <int MT, bool kBS, bool kSc>
cudaError_t launch_one(const DecodeParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto fn = decode_kernel<MT, kBS, kSc>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  fn<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int MT>
cudaError_t launch_mt(const DecodeParams& p, bool bs, bool sc, int grid, size_t smem,
                      cudaStream_t stream) {
  if (bs) return sc ? launch_one<MT, true, true>(p, grid, smem, stream)
                    : launch_one<MT, true, false>(p, grid, smem, stream);
  return sc ? launch_one<MT, false, true>(p, grid, smem, stream)
            : launch_one<MT, false, false>(p, grid, smem, stream);
}

int mt_for(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

size_t fixed_bytes(int MT, int64_t K) {
  const int64_t nb = K / kQK;
  return static_cast<size_t>((MT * K + MT * nb * 4 + 127) & ~static_cast<int64_t>(127));
}

}  // namespace

size_t decode_smem_bytes(int64_t M, int64_t K, const DeviceInfo& dev) {
  if (M < 1 || M > kDecodeMaxM || K < kQK) return 0;
  const int MT = mt_for(M);
  const size_t stage = static_cast<size_t>(K) + ((K % 256 == 0) ? static_cast<size_t>(K / 16) : 0);
  const size_t fixed = fixed_bytes(MT, K);
  const size_t budget = static_cast<size_t>(dev.max_smem_optin) - 2048;  // static smem headroom
  if (fixed + 2 * stage > budget) return 0;
  size_t stages = (budget - fixed) / stage;
  if (stages > kMaxStages) stages = kMaxStages;
  // enough stages to keep ~96 KB in flight; more only costs shared memory
  size_t want = (96 * 1024 + stage - 1) / stage;
  if (want < 2) want = 2;
  if (stages > want) stages = want;
  return fixed + stages * stage;
}

cudaError_t launch_decode(const void* x, int xtype, const int8_t* xq_in, const int8_t* Wq,
                          const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                          int64_t K, const DeviceInfo& dev, cudaStream_t stream) {
  if (M == 0 || N == 0) return cudaSuccess;
  const size_t smem = decode_smem_bytes(M, K, dev);
  if (smem == 0) return cudaErrorInvalidValue;
  const int MT = mt_for(M);
  // block-sum mode reads no scales
  const bool scales_in_stage = (K % 256) == 0 && isum == nullptr;
  const size_t stage = static_cast<size_t>(K) + (scales_in_stage ? static_cast<size_t>(K / 16) : 0);
  DecodeParams p;
  p.x = x;
  p.xtype = xtype;
  p.xq = xq_in;
  p.Wq = Wq;
  p.Wd = Wd;
  p.y = y;
  p.isum = isum;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  const size_t stages = (smem - fixed_bytes(MT, K)) / stage;
  p.stages = static_cast<int>(stages < kMaxStages ? stages : kMaxStages);
  p.err = dev.err_word;
  const int grid = static_cast<int>(N < dev.sm_count ? N : dev.sm_count);
  const bool bs = isum != nullptr;
  switch (MT) {
    case 1: return launch_mt<1>(p, bs, scales_in_stage, grid, smem, stream);
    case 2: return launch_mt<2>(p, bs, scales_in_stage, grid, smem, stream);
    case 4: return launch_mt<4>(p, bs, scales_in_stage, grid, smem, stream);
    default: return launch_mt<8>(p, bs, scales_in_stage, grid, smem, stream);
  }
}

}  // namespace q8
