// q8_decode.cu -- small-M (decode) Q8_0 linear: streams the weight codes from HBM once,
// at the memory's rate, and forms every block sum with dp4a.
//
// Operation: y[m,n] = sum_b Wd[n,b] * xd[m,b] * isum[m,n,b], the Q8_0 int8 GEMM of
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, list of un-throttled paths: the DP4A int8
// GEMM), at decode batch sizes (M <= 8), where the layer is bound by reading the weights.
//
// Design (one CTA per SM, 1 producer warp + 16 consumer warps):
//   * CTA c owns the contiguous rows [r0, r1) of W.  Their codes (and, when a row of scales
//     is a multiple of 16 bytes, their binary16 scales) are contiguous, and stream through a
//     ring of shared-memory stages of R whole rows (about 24 KB; 192 KB in flight per SM)
//     by bulk asynchronous copies that one elected thread issues; each stage completes on
//     its own mbarrier.  Large copies keep the per-copy overhead of the copy engine small
//     (4 KB copies ran at a third of the bandwidth).
//   * Programmatic dependent launch: the kernel lets the next kernel in the stream start as
//     soon as it begins, and its producer fills the ring before anything waits for the
//     previous kernel.  Only the consumers wait (griddepcontrol.wait) before they read x and
//     write y.  So the weights, which are read before that wait, must not be written by a
//     kernel that triggers its dependents early (no kernel of this library does).  The next
//     kernel's CTAs start streaming their first stages as soon as this kernel's CTAs exit.
//   * Fused activation quantizer: after the wait, the consumers quantize the M activation
//     rows into shared memory with the same device function as the standalone quantizer.
//   * Consumer warp w takes rows w, w + 16, ...: lane l handles the 16-byte pieces
//     l + 32 i of the row, 4 dp4a per piece and token; an xor-shuffle joins the two halves
//     of each 32-element block into the exact int32 block sum; the even lane rescales it by
//     Wd * xd in binary32; a warp reduction finishes the row.
//   * Block-sum mode (for checking) takes int8 codes instead of x and writes the raw block
//     sums instead of y.
#include <cuda_fp16.h>

#include "q8_epi.cuh"
#include "q8_internal.h"
#include "q8_ptx.cuh"
#include "q8_quant_dev.cuh"

namespace q8 {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxStages = 32;
// Stage and ring sizes (measured on GB300 for the M=1 decode workload, graph replays with
// programmatic dependent launch): 24 KB stages in a 192 KB ring beat 16 KB stages in a
// ring small enough for two CTAs per SM (9.3 us vs 10.5 us per 53.5 MB call).
constexpr int kStageTarget = 24 * 1024;  // bytes of codes per stage (whole rows)
constexpr int kRingTarget = 192 * 1024;  // bytes of codes and scales in flight per CTA
constexpr int kXRegPieces = 8;           // one token with K <= 4096: codes in registers

struct DecodeParams {
  const void* x;       // [M,K] bf16 bits or f32 (fused quantization)
  int xtype;           // 0 f32, 1 bf16
  const int8_t* xq;    // [M,K] int8 codes (block-sum mode)
  const int8_t* Wq;    // [N,K]
  const uint16_t* Wd;  // [N,K/32]
  float* y;            // [M,N]
  int32_t* isum;       // [M,N,K/32] (block-sum mode)
  int M, N, K;
  int rows_per_stage;  // R
  int stages;          // S
  uint32_t* err;
  Epilogue epi;        // fused output step
  Prologue pro;        // fused RMSNorm (gamma, eps): r is computed here and scales y
};

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int4 lds128(const void* p) { return *reinterpret_cast<const int4*>(p); }

// kXP > 0: one token, K <= 512 * kXP; each lane always covers the same K positions, so it
// keeps its activation codes and scales in registers instead of reading shared memory.
// kFused: the fused neighbours (RMSNorm in the quantize pass, epilogue at the store); the
// plain layer is a separate instantiation so that it carries none of that code.
template <int MT, bool kBlockSums, bool kScalesInStage, int kXP, bool kFused>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[kMaxStages];
  __shared__ uint64_t empty_bar[kMaxStages];
  __shared__ int abort_flag;
  // Stages issued so far.  A consumer waits for its stage's ticket before the parity wait
  // on the stage's barrier: once stage st is issued, the barrier of its slot has finished
  // every phase before st's, so the parity names st's phase exactly, whatever the number
  // of stages and consumers.
  __shared__ volatile int issued;
  __shared__ float rs_part[kConsumerWarps][8];  // RMSNorm: per-warp sums of squares

  const int K = p.K, N = p.N, M = p.M, R = p.rows_per_stage, S = p.stages;
  const int nb = K / kQK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * N / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * N / gridDim.x;
  const int nrows = static_cast<int>(r1 - r0);
  const int nstages = (nrows + R - 1) / R;
  const uint32_t code_bytes = static_cast<uint32_t>(R) * K;
  const uint32_t scale_bytes = kScalesInStage ? static_cast<uint32_t>(R) * nb * 2 : 0u;
  const uint32_t stage_bytes = code_bytes + scale_bytes;
  // carve-up: [x codes MT*K][x scales MT*nb f32][ring S*stage_bytes]
  int8_t* xs = reinterpret_cast<int8_t*>(smem);
  float* xds = reinterpret_cast<float*>(smem + MT * K);
  uint8_t* ring = smem + ((MT * K + MT * nb * 4 + 127) & ~127);

  if (S > kMaxStages || S < 2) {  // the launcher never does this
    if (threadIdx.x == 0) report_error(p.err, kErrBadLaunch, nullptr);
    return;
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    issued = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], static_cast<uint32_t>(R));
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer: weights only, so it does not wait for the previous kernel
    if (lane == 0) {
      for (int st = 0; st < nstages; ++st) {
        const int s = st % S;
        if (!mbar_wait(&empty_bar[s], ((st / S) & 1) ^ 1, &abort_flag)) {
          report_error(p.err, kErrWaitTimeout, &abort_flag);
          break;
        }
        const int64_t ra = r0 + static_cast<int64_t>(st) * R;
        const int rows = static_cast<int>((r1 - ra) < R ? (r1 - ra) : R);
        uint8_t* dst = ring + static_cast<size_t>(s) * stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(rows) * (K + (kScalesInStage ? nb * 2 : 0)));
        bulk_load(dst, p.Wq + ra * K, static_cast<uint32_t>(rows) * K, &full_bar[s]);
        if constexpr (kScalesInStage)
          bulk_load(dst + code_bytes, p.Wd + ra * nb, static_cast<uint32_t>(rows) * nb * 2, &full_bar[s]);
        issued = st + 1;
      }
      // never leave with copies in flight
      const int n_issued = issued;
      for (int st = (n_issued > S ? n_issued - S : 0); st < n_issued; ++st)
        if (!mbar_wait(&full_bar[st % S], (st / S) & 1, nullptr)) {
          report_error(p.err, kErrWaitTimeout, nullptr);
          break;
        }
    }
  } else {
    // ---------------- consumers ---------------------------------------------------------
    const int cw = warp - 1;
    const int ct = threadIdx.x - 32;
    constexpr int kCT = 32 * kConsumerWarps;
    pdl_wait();  // x, y: wait for the previous kernel in the stream
    // RMSNorm: the quantize pass below also sums each token's squares (thread ct adds its
    // blocks' in order; a fixed xor tree per warp; the warps' sums are added in order
    // after the pass), and r scales the token's outputs at the store
    const bool norm = kFused && !kBlockSums && p.pro.gamma != nullptr;
    float ss[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) ss[t] = 0.0f;
    if constexpr (kBlockSums) {
      const int n16 = M * K / 16;
      for (int i = ct; i < n16; i += kCT)
        reinterpret_cast<int4*>(xs)[i] = reinterpret_cast<const int4*>(p.xq)[i];
    } else {
      const int nblk = M * nb;
      const int sub = lane & 3;
      const unsigned gmask = 0xFu << (lane & ~3);
      const int iters = (nblk + kCT / 4 - 1) / (kCT / 4);
      for (int it = 0; it < iters; ++it) {
        const int blk = it * (kCT / 4) + (ct >> 2);
        if (blk < nblk) {  // the 4 lanes of a group agree on this
          float v[8];
          const int64_t off = static_cast<int64_t>(blk) * kQK + sub * 8;
          if (p.xtype == 1) {
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + off), v);
          } else {
            const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off);
            const float4 a = f[0], b = f[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
          }
          if (norm) {  // codes of x * gamma
            float s2 = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s2 = fmaf(v[i], v[i], s2);
            const int tb = blk / nb;
#pragma unroll
            for (int t = 0; t < MT; ++t)
              if (t == tb) ss[t] += s2;
            const int k = (blk % nb) * kQK + sub * 8;
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.pro.gamma + k));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.pro.gamma + k) + 1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], g[i]);
          }
          int q[8];
          const float d = quantize_block_x4(v, gmask, q);
          *reinterpret_cast<uint2*>(xs + off) = pack_codes_i8(q);
          if (sub == 0) xds[blk] = d;
        }
      }
    }
    if (norm) {
#pragma unroll
      for (int t = 0; t < MT; ++t) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss[t] += __shfl_xor_sync(0xFFFFFFFFu, ss[t], o);
        if (lane == 0) rs_part[cw][t] = ss[t];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory");
    float rt = 1.0f;  // lane t < M: the RMSNorm factor of token t
    if (norm && lane < M) {
      float s = 0.0f;
      for (int w = 0; w < kConsumerWarps; ++w) s += rs_part[w][lane];
      rt = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(s, static_cast<float>(K)), p.pro.eps)));
    }

    const int npieces = K >> 4;  // even, since K % 32 == 0
    const int iters = (npieces + 31) >> 5;
    int4 xr[kXP > 0 ? kXP : 1];
    float xdr[kXP > 0 ? kXP : 1];
    if constexpr (kXP > 0) {
#pragma unroll
      for (int i = 0; i < kXP; ++i) {
        const int pc = lane + 32 * i;
        xr[i] = pc < npieces ? lds128(xs + 16 * pc) : make_int4(0, 0, 0, 0);
        xdr[i] = pc < npieces ? xds[pc >> 1] : 0.0f;
      }
    }
    for (int j = cw; j < nrows; j += kConsumerWarps) {
      const int64_t n = r0 + j;
      float ax = 0.0f;  // lane t < M: aux of output (t, n), loaded before the row's weights land
      if constexpr (!kBlockSums && kFused) {
        if (lane < M) ax = epi_aux(p.epi, static_cast<int64_t>(lane) * N + n);
      }
      const int st = j / R;
      const int s = st % S;
      bool ticket = issued > st;
      if (!ticket) {
        const long long t0 = clock64();
        while (!(ticket = issued > st) && !*reinterpret_cast<volatile int*>(&abort_flag) &&
               clock64() - t0 < kWaitBudgetCycles)
          __nanosleep(64);
      }
      // every lane waits (and so observes the copied bytes); the warp leaves together
      const bool ok =
          __all_sync(0xFFFFFFFFu, ticket && mbar_wait(&full_bar[s], (st / S) & 1, &abort_flag));
      if (!ok) {
        if (lane == 0) report_error(p.err, kErrWaitTimeout, &abort_flag);
        break;
      }
      const uint8_t* stage = ring + static_cast<size_t>(s) * stage_bytes;
      const int jr = j - st * R;  // row within the stage
      const uint8_t* wrow = stage + static_cast<size_t>(jr) * K;
      const uint16_t* wd_row = kScalesInStage
                                   ? reinterpret_cast<const uint16_t*>(stage + code_bytes) + jr * nb
                                   : p.Wd + n * nb;
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
      if constexpr (kXP > 0) {
#pragma unroll
        for (int i = 0; i < kXP; ++i) {
          const int pc = lane + 32 * i;
          const bool valid = pc < npieces;  // the same on both lanes of a block
          int4 w = make_int4(0, 0, 0, 0);
          float dw = 0.0f;
          if (valid) {
            w = lds128(wrow + 16 * pc);
            if constexpr (!kBlockSums) dw = __half2float(__ushort_as_half(wd_row[pc >> 1]));
          }
          int sum = __dp4a(w.x, xr[i].x, 0);
          sum = __dp4a(w.y, xr[i].y, sum);
          sum = __dp4a(w.z, xr[i].z, sum);
          sum = __dp4a(w.w, xr[i].w, sum);
          sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);  // exact int32 block sum
          if (valid && !(lane & 1)) {
            if constexpr (kBlockSums)
              p.isum[n * nb + (pc >> 1)] = sum;
            else
              acc[0] = fmaf(dw * xdr[i], static_cast<float>(sum), acc[0]);
          }
        }
      } else
#pragma unroll 4
      for (int i = 0; i < iters; ++i) {
        const int pc = lane + (i << 5);
        const bool valid = pc < npieces;  // the same on both lanes of a block
        const int blk = pc >> 1;
        int4 w = make_int4(0, 0, 0, 0);
        float dw = 0.0f;
        if (valid) {
          w = lds128(wrow + 16 * pc);
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
          if (t < M && valid && !(lane & 1)) {
            if constexpr (kBlockSums)
              p.isum[(static_cast<int64_t>(t) * N + n) * nb + blk] = sum;
            else
              acc[t] = fmaf(dw * xds[t * nb + blk], static_cast<float>(sum), acc[t]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);  // the row's bytes are no longer needed
      if constexpr (!kBlockSums) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          float a = acc[t];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
          if constexpr (kFused) {
            // the butterfly leaves the same sum on every lane: lane t stores output t
            if (lane == t && t < M)
              epi_put(p.epi, p.y, static_cast<int64_t>(t) * N + n, epi_apply(p.epi, norm ? a * rt : a, ax));
          } else {
            if (lane == 0 && t < M) p.y[static_cast<int64_t>(t) * N + n] = a;
          }
        }
      }
    }
  }
  __syncthreads();
}

struct Plan {
  int R = 0, S = 0;
  bool scales_in_stage = false;
  size_t smem = 0;
};

int mt_for(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

Plan plan_for(int64_t M, int64_t K, bool block_sums, const DeviceInfo& dev) {
  Plan pl;
  if (M < 1 || M > kDecodeMaxM || K < kQK) return pl;
  const int MT = mt_for(M);
  const int64_t nb = K / kQK;
  pl.scales_in_stage = !block_sums && (nb % 8 == 0);
  pl.R = static_cast<int>(K >= kStageTarget ? 1 : kStageTarget / K);
  const size_t stage = static_cast<size_t>(pl.R) * (K + (pl.scales_in_stage ? nb * 2 : 0));
  const size_t fixed = static_cast<size_t>((MT * K + MT * nb * 4 + 127) & ~static_cast<int64_t>(127));
  const int smin = 2;
  int want = static_cast<int>((kRingTarget + stage - 1) / stage);
  if (want < smin) want = smin;
  if (want > kMaxStages) want = kMaxStages;
  const size_t budget = static_cast<size_t>(dev.max_smem_optin) - 2048;  // static smem headroom
  if (fixed + smin * stage > budget) return Plan{};
  int S = want;
  while (S > smin && fixed + S * stage > budget) --S;
  pl.S = S;
  pl.smem = fixed + S * stage;
  return pl;
}

template <int MT, bool kBS, bool kSc, int kXP = 0, bool kFused = false>
cudaError_t launch_one(const DecodeParams& p, int grid, size_t smem, cudaStream_t stream,
                       int dev_id) {
  auto fn = decode_kernel<MT, kBS, kSc, kXP, kFused>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(fn), smem, dev_id);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <int MT, bool kFused>
cudaError_t launch_y(const DecodeParams& p, bool sc, int grid, size_t smem, cudaStream_t stream,
                     int dev_id) {
  if constexpr (MT == 1) {
    if (p.K <= 512 * kXRegPieces)  // activation codes in registers
      return sc ? launch_one<1, false, true, kXRegPieces, kFused>(p, grid, smem, stream, dev_id)
                : launch_one<1, false, false, kXRegPieces, kFused>(p, grid, smem, stream, dev_id);
  }
  return sc ? launch_one<MT, false, true, 0, kFused>(p, grid, smem, stream, dev_id)
            : launch_one<MT, false, false, 0, kFused>(p, grid, smem, stream, dev_id);
}

template <int MT>
cudaError_t launch_mt(const DecodeParams& p, bool bs, bool sc, int grid, size_t smem,
                      cudaStream_t stream, int dev_id) {
  if (bs) {
    if constexpr (MT == 1) {
      if (p.K <= 512 * kXRegPieces) return launch_one<1, true, false, kXRegPieces>(p, grid, smem, stream, dev_id);
    }
    return launch_one<MT, true, false>(p, grid, smem, stream, dev_id);
  }
  if (!p.epi.plain() || p.pro.on()) return launch_y<MT, true>(p, sc, grid, smem, stream, dev_id);
  return launch_y<MT, false>(p, sc, grid, smem, stream, dev_id);
}

}  // namespace

size_t decode_smem_bytes(int64_t M, int64_t K, const DeviceInfo& dev) {
  return plan_for(M, K, false, dev).smem;
}

cudaError_t launch_decode(const void* x, int xtype, const int8_t* xq_in, const int8_t* Wq,
                          const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                          int64_t K, const DeviceInfo& dev, cudaStream_t stream,
                          const Epilogue& epi, const Prologue& pro) {
  if (M == 0 || N == 0) return cudaSuccess;
  const bool bs = isum != nullptr;
  const Plan pl = plan_for(M, K, bs, dev);
  if (pl.smem == 0) return cudaErrorInvalidValue;
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
  p.rows_per_stage = pl.R;
  p.stages = pl.S;
  p.err = dev.err_word;
  p.epi = epi;
  p.pro = pro;
  const int grid = static_cast<int>(N < dev.sm_count ? N : dev.sm_count);
  switch (mt_for(M)) {
    case 1: return launch_mt<1>(p, bs, pl.scales_in_stage, grid, pl.smem, stream, dev.device);
    case 2: return launch_mt<2>(p, bs, pl.scales_in_stage, grid, pl.smem, stream, dev.device);
    case 4: return launch_mt<4>(p, bs, pl.scales_in_stage, grid, pl.smem, stream, dev.device);
    default: return launch_mt<8>(p, bs, pl.scales_in_stage, grid, pl.smem, stream, dev.device);
  }
}

}  // namespace q8
