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
// Design (384 threads = 3 warpgroups per CTA, one CTA per SM; the control warpgroup hands
// registers to the two drain warpgroups with setmaxnreg).  A CTA works through one to three
// segments, each a 128 x 256 output tile over a range of K: a whole tile, a split-K range
// of one, or (stream-K, for a partial last wave) an equal run of scale windows that may
// cross tile boundaries (see gemm_schedule).  The pipelines run on across segments.
//   warp 0     TMA producer: A (activation codes, 128 x 64 binary16) and B (weight codes,
//              256 x 64 binary16) tiles with 128-byte swizzle into a 3-stage ring;
//   warp 1     TMEM owner and MMA issuer: per 32-K block, 2 x tcgen05.mma
//              (M=128, N=256, K=16) into one of two 256-column TMEM buffers, then
//              tcgen05.commit to that buffer's "full" barrier;
//   warps 2-3  scale producer: windows of 16 blocks of Wd (the tile's columns) and xd (its
//              rows), widened to binary32 into a 2-slot shared-memory ring;
//   warps 4-11 rescale drain, two warpgroups of 128 columns each: per block, tcgen05.ld
//              the block sums of their TMEM lanes 16 columns at a time and the column
//              scales from shared memory, both one chunk ahead, then
//              y_acc += (xd * Wd) * isum in binary32 registers (packed f32x2 multiply,
//              scalar fused multiply-add); release the TMEM buffer; at a segment's end
//              store y, or a partial tile that a reduction kernel adds.  The CTA's last
//              segment is staged in the then idle operand ring and written by TMA stores.
// Block-sum mode (for checking) stores the TMEM block sums as int32 instead.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>

#include "q8_epi.cuh"
#include "q8_internal.h"
#include "q8_ptx.cuh"

namespace q8 {
namespace {

// ---- TMA stores and named barriers (used by this file only) ------------------------
// 2-D / 3-D tile store from shared memory, completed through the issuing thread's bulk
// groups; the parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src,
                                             int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src,
                                             int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Brings a whole 2-D box of the tensor towards L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until this thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}


constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // two Q8_0 blocks per pipeline stage (one 128-byte swizzle row)
constexpr int kStages = 3;
constexpr int kThreads = 384;               // 3 warpgroups
// Register split (setmaxnreg): the kernel is compiled for kLaunchRegs per thread; the
// control warpgroup gives registers back, the two drain warpgroups take them.  Per SM
// sub-partition (one warp of each warpgroup) and in total the split equals the launch.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 56;
constexpr int kDrainRegs = 224;
static_assert(128 * kCtrlRegs + 256 * kDrainRegs == kThreads * kLaunchRegs, "register split");
static_assert(32 * (kCtrlRegs + 2 * kDrainRegs) <= 16384, "registers per sub-partition");
constexpr int kDrainWarps = 8;
constexpr int kScaleThreads = 64;           // warps 2-3 stage the scales
constexpr uint32_t kStageA = BM * BK * 2;   // 16 KB
constexpr uint32_t kStageB = BN * BK * 2;   // 32 KB
constexpr uint32_t kTmemCols = 2 * BN;      // two accumulation buffers
constexpr int kWin = 16;                    // Q8_0 blocks per window of staged scales
constexpr int kWinSlots = 2;                // windows in the scale ring
constexpr uint32_t kWinDw = kWin * BN * 4;  // Wd of the tile's columns, f32   (16 KB)
constexpr uint32_t kWinDx = kWin * BM * 4;  // xd of the tile's rows, f32      (8 KB)
constexpr size_t kSmemBytes = 1024 /*align*/ + kStages * (kStageA + kStageB) +
                              kWinSlots * (kWinDw + kWinDx);
// int8-weight variant (kConv): the weight codes arrive by TMA as int8 ([256 rows][64 bytes]
// per stage) and the scale warps widen them into a 2-slot ring of binary16 B tiles in the
// MMA's layout.  A keeps its kStages ring.
constexpr uint32_t kStageB8 = BN * BK;      // 16 KB of int8 codes
constexpr int kFSlots = 2;                  // binary16 B tiles ready for the MMA
constexpr size_t kSmemBytesConv = 1024 + kStages * (kStageA + kStageB8) + kFSlots * kStageB +
                                  kWinSlots * (kWinDw + kWinDx);
static_assert(kSmemBytesConv <= 232448, "shared memory per CTA (int8-weight variant)");
static_assert(kDrainWarps * 32 * 128 * 4 <= kStages * (kStageA + kStageB8) + kFSlots * kStageB,
              "output staging (int8-weight variant)");
// The CTA's last results are staged in the operand ring, 16 KB per drain warp.
static_assert(kDrainWarps * 32 * 128 * 4 <= kStages * (kStageA + kStageB), "output staging");

// Output tile t -> its first row (token) and column (weight row): token tile fastest, so the
// CTAs resident at one time share a few weight slabs of B.  (A grouped order that keeps A
// in L2 as well cut the 27B up-projection's DRAM reads from 2.8 GB to a fraction, but ran
// about 1 % slower on every prefill shape: the kernel is bound on chip, not by DRAM.)
__host__ __device__ __forceinline__ void tile_origin(int t, int mtiles, int* m0, int* n0) {
  *m0 = (t % mtiles) * BM;
  *n0 = (t / mtiles) * BN;
}

struct GemmParams {
  const float* xd;     // [M, nb]
  const uint16_t* Wd;  // [N, nb]
  float* y;            // [M, N]
  float* part;         // split-K partial outputs: [splits, M, N]; stream-K: [2 sk_ctas, BM, BN]
  int splits;          // K split into this many ranges of whole scale windows (blockIdx.y)
  // Stream-K (sk_ctas > 0): the scale windows of tiles [0, sk_tiles), sk_windows of them in
  // tile order, are cut into sk_ctas equal contiguous runs, one per CTA [0, sk_ctas) (see
  // cta_segments); the CTAs after them take one whole tile each, tiles [sk_tiles, ...).  A
  // run that covers only part of a tile stores a partial tile, and reduce_sk_kernel adds a
  // tile's partials.  The runs come first so that they start together on an idle GPU and the
  // whole tiles after them even out the SMs' finishing times.
  int sk_ctas;
  int sk_tiles;
  int sk_windows;
  int32_t* isum;       // [M, N, nb] (block-sum mode)
  int M, N, K;
  int tma_y;           // whole-K tiles are stored through tmY (binary32 y, box 32 x 32)
  int tma_aux;         // fused epilogue: tmP maps aux (box 128 rows x 256 columns), prefetched
                       // to L2 while a whole tile's last window is loaded
  int tma_part;        // partial tiles are stored through tmP (binary32, 3-D, box 32 x 32 x 1):
                       // stream-K [2 sk_ctas][BM][BN] at (column, row, slot), split-K
                       // [splits][M][N] at (n, m, split)
  uint32_t* err;
  Epilogue epi;        // fused output step (applied by the reduction where K is split)
};

// A CTA's work: up to kMaxSegs segments, each one output tile over a range of its scale
// windows.  A stream-K run is shorter than two tiles, so it touches at most three.
constexpr int kMaxSegs = 3;
struct Seg {
  int tile;
  int w0, w1;  // scale windows [w0, w1) of the tile's K
  int slot;    // >= 0: partial tile slot of a stream-K run; -1: whole K of the tile
};

// Stream-K: run j of G covers windows [start(j), start(j + 1)) of the W in the stream-K
// tiles, start(j) = floor(j W / G).  A partial first segment of run j takes partial-tile
// slot 2 j, a partial last one slot 2 j + 1.
__host__ __device__ __forceinline__ int sk_start(int j, int W, int G) {
  return static_cast<int>(static_cast<int64_t>(j) * W / G);
}

__device__ int cta_segments(const GemmParams& p, int nwin, Seg* seg) {
  const int bid = static_cast<int>(blockIdx.x);
  if (bid >= p.sk_ctas) {
    const int s = static_cast<int>(blockIdx.y), ns = p.splits;  // split-K range s of ns
    seg[0].tile = p.sk_tiles + (bid - p.sk_ctas);
    seg[0].w0 = static_cast<int>(static_cast<int64_t>(s) * nwin / ns);
    seg[0].w1 = static_cast<int>(static_cast<int64_t>(s + 1) * nwin / ns);
    seg[0].slot = -1;
    return 1;
  }
  const int j = bid;
  const int a = sk_start(j, p.sk_windows, p.sk_ctas);
  const int e = sk_start(j + 1, p.sk_windows, p.sk_ctas);
  int n = 0;
  for (int t = a / nwin; t * nwin < e && n < kMaxSegs; ++t, ++n) {
    const int w0 = max(a, t * nwin) - t * nwin;
    const int w1 = min(e, (t + 1) * nwin) - t * nwin;
    seg[n].tile = t;
    seg[n].w0 = w0;
    seg[n].w1 = w1;
    seg[n].slot = (w0 == 0 && w1 == nwin) ? -1 : (n == 0 ? 2 * j : 2 * j + 1);
  }
  return n;
}

// 16 int8 codes -> 16 binary16 values, exactly: a byte biased to u = q + 128 becomes the low
// byte of the binary16 pattern 0x64uu, whose value is 1024 + u, and 1024 + u - 1152 = q.
__device__ __forceinline__ void codes16_to_f16(uint4 in, uint4* lo, uint4* hi) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[8];
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = w[i] ^ 0x80808080u;
    uint32_t a = __byte_perm(t, 0x64646464u, 0x5150);  // codes 0, 1 of the word
    uint32_t b = __byte_perm(t, 0x64646464u, 0x5352);  // codes 2, 3
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    o[2 * i] = *reinterpret_cast<uint32_t*>(&ha);
    o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&hb);
  }
  *lo = make_uint4(o[0], o[1], o[2], o[3]);
  *hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Fill one window of scales: Wd of the tile's 256 columns and xd of its 128 rows, blocks
// [16 w, 16 w + 16) (zero past the ends), as f32 [block][column] and [block][row].
__device__ __forceinline__ void stage_scales(const GemmParams& p, int w, int m0, int n0, int nb,
                                             float* dws, float* dxs, int t) {
  const int b0 = w * kWin;
  const bool vec_w = (nb % 8) == 0;   // 8 binary16 scales of a row are one 16-byte load
  const bool vec_x = (nb % 4) == 0;
#pragma unroll 1
  for (int q = 0; q < BN / kScaleThreads; ++q) {
    const int col = t + kScaleThreads * q;
    const int n = n0 + col;
#pragma unroll
    for (int h = 0; h < kWin; h += 8) {
      float f[8];
      if (n < p.N && vec_w && b0 + h + 8 <= nb) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.Wd + static_cast<int64_t>(n) * nb + b0 + h));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 g = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
          f[2 * i] = g.x;
          f[2 * i + 1] = g.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          f[i] = (n < p.N && b0 + h + i < nb)
                     ? __half2float(__ushort_as_half(p.Wd[static_cast<int64_t>(n) * nb + b0 + h + i]))
                     : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) dws[(h + i) * BN + col] = f[i];
    }
  }
#pragma unroll 1
  for (int q = 0; q < BM / kScaleThreads; ++q) {
    const int row = t + kScaleThreads * q;
    const int m = m0 + row;
#pragma unroll
    for (int h = 0; h < kWin; h += 4) {
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (m < p.M && vec_x && b0 + h + 4 <= nb) {
        v = __ldg(reinterpret_cast<const float4*>(p.xd + static_cast<int64_t>(m) * nb + b0 + h));
      } else if (m < p.M) {
        const float* src = p.xd + static_cast<int64_t>(m) * nb + b0 + h;
        if (b0 + h + 0 < nb) v.x = src[0];
        if (b0 + h + 1 < nb) v.y = src[1];
        if (b0 + h + 2 < nb) v.z = src[2];
        if (b0 + h + 3 < nb) v.w = src[3];
      }
      dxs[(h + 0) * BM + row] = v.x;
      dxs[(h + 1) * BM + row] = v.y;
      dxs[(h + 2) * BM + row] = v.z;
      dxs[(h + 3) * BM + row] = v.w;
    }
  }
}

// kFused: the drain's final store applies the epilogue (residual, SiLU gate, bfloat16 y);
// the plain layer is a separate instantiation so that it carries none of that code.
// kSK: the launch has stream-K runs, whose CTAs walk several segments; without it every CTA
// has exactly one, known at compile time.  kConv: B is given as the int8 weight codes
// (tmB over Wq [N, K] bytes) and widened in shared memory by the scale warps.
template <bool kBlockSums, bool kFused, bool kSK, bool kConv>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmP,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2];
  __shared__ uint64_t sfull_bar[kWinSlots], sempty_bar[kWinSlots];
  __shared__ uint64_t cfull_bar[kFSlots], cempty_bar[kFSlots];  // kConv: widened B tiles
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;
  __shared__ Seg segs[kMaxSegs];
  __shared__ int nseg_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = p.M, N = p.N, K = p.K;
  const int nb = K / kQK;
  const int nwin = (nb + kWin - 1) / kWin;
  const int mtiles = (M + BM - 1) / BM;
  // Every role walks the CTA's segments in order.  Segment s covers Q8_0 blocks
  // [16 w0, min(16 w1, nb)) of its tile, i.e. 64-wide stages [8 w0, (b_end + 1) / 2); the
  // operand ring, the TMEM buffers, the scale ring and their barrier phases count on across
  // segments, so the pipelines do not drain between them.

  // 1024-byte aligned carve-up (128-byte swizzle atoms must sit on 1024-byte boundaries)
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023) & ~1023u) - raw);
  uint8_t* sA = base;
  uint8_t* sB = base + kStages * kStageA;  // kConv: the int8 tiles, [stage][BN][BK bytes]
  uint8_t* sF = sB + kStages * kStageB8;   // kConv: the widened binary16 tiles
  float* sW = reinterpret_cast<float*>(kConv ? sF + kFSlots * kStageB
                                             : sB + kStages * kStageB);  // [slot][kWin][BN]
  float* sX = sW + kWinSlots * kWin * BN;                          // [slot][kWin][BM]

  if (threadIdx.x == 0) {
    abort_flag = 0;
    nseg_s = cta_segments(p, nwin, segs);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      // kConv: a stage is free once the MMA has read A (commit) and both scale warps have
      // read the int8 codes
      mbar_init(&empty_bar[s], kConv ? 3 : 1);
    }
    if constexpr (kConv) {
      for (int f = 0; f < kFSlots; ++f) {
        mbar_init(&cfull_bar[f], 2);
        mbar_init(&cempty_bar[f], 1);
      }
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kDrainWarps);
    }
    for (int b = 0; b < kWinSlots; ++b) {
      mbar_init(&sfull_bar[b], kScaleThreads);
      mbar_init(&sempty_bar[b], kDrainWarps);
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
  const int nseg = kSK ? nseg_s : 1;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (warp == 0) {
      // ------------------------------- TMA producer -----------------------------------
      if (lane == 0) {
        int issued = 0;  // stages, all segments
        bool ok = true;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          const Seg S = segs[sg];
          int m0, n0;
          tile_origin(S.tile, mtiles, &m0, &n0);
          const int kb_end = (min(S.w1 * kWin, nb) + 1) / 2;
          for (int kb = S.w0 * (kWin / 2); kb < kb_end; ++kb) {
            if constexpr (kFused) {
              // the epilogue's aux tile, towards L2 a window ahead of its use
              if (p.tma_aux && S.slot < 0 && kb == (S.w1 - 1) * (kWin / 2)) tma_prefetch_l2_2d(&tmP, n0, m0);
            }
            const int s = issued % kStages;
            if (!mbar_wait(&empty_bar[s], ((issued / kStages) & 1) ^ 1, &abort_flag)) {
              report_error(p.err, kErrWaitTimeout, &abort_flag);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_bar[s], kStageA + (kConv ? kStageB8 : kStageB));
            tma_load_2d(sA + s * kStageA, &tmA, &full_bar[s], kb * BK, m0);
            tma_load_2d(sB + s * (kConv ? kStageB8 : kStageB), &tmB, &full_bar[s], kb * BK, n0);
            ++issued;
          }
        }
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
          if (!mbar_wait(&full_bar[i % kStages], (i / kStages) & 1, nullptr)) {
            report_error(p.err, kErrWaitTimeout, nullptr);
            break;
          }
      }
    } else if (warp == 1) {
      // ------------------------------- MMA issuer -------------------------------------
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
        int i = 0;  // stages consumed, all segments
        int g = 0;  // blocks issued, all segments: TMEM buffer g & 1, phase (g >> 1) & 1
        int last_stage = -1;
        bool ok = true;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          const Seg S = segs[sg];
          const int b_end = min(S.w1 * kWin, nb);
          for (int kb = S.w0 * (kWin / 2); kb < (b_end + 1) / 2 && ok; ++kb, ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&full_bar[s], (i / kStages) & 1, &abort_flag)) {
              report_error(p.err, kErrWaitTimeout, &abort_flag);
              ok = false;
              break;
            }
            const int f = i % kFSlots;
            if constexpr (kConv) {
              if (!mbar_wait(&cfull_bar[f], (i / kFSlots) & 1, &abort_flag)) {
                report_error(p.err, kErrWaitTimeout, &abort_flag);
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * kStageA);
            const uint32_t b0 = kConv ? smem_u32(sF + f * kStageB) : smem_u32(sB + s * kStageB);
            const int nblk = min(b_end - 2 * kb, 2);
            for (int j = 0; j < nblk; ++j, ++g) {
              const int buf = g & 1;
              if (!mbar_wait(&tempty_bar[buf], ((g >> 1) & 1) ^ 1, &abort_flag)) {
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
            if constexpr (kConv) mma_commit(&cempty_bar[f]);
            last_stage = i;
          }
        }
        // do not leave while MMAs are still reading shared memory / writing TMEM
        if (last_stage >= 0 &&
            !mbar_wait(&empty_bar[last_stage % kStages], (last_stage / kStages) & 1, nullptr))
          report_error(p.err, kErrWaitTimeout, nullptr);
      }
    } else if constexpr (!kBlockSums) {
      // ------------------------------- scale producer (warps 2-3) ---------------------
      const int t = threadIdx.x - 64;  // 0..63
      int u = 0;   // windows staged, all segments
      int ci = 0;  // kConv: stages widened, all segments
      bool ok = true;
      for (int sg = 0; sg < nseg && ok; ++sg) {
        const Seg S = segs[sg];
        int m0, n0;
        tile_origin(S.tile, mtiles, &m0, &n0);
        for (int w = S.w0; w < S.w1 && ok; ++w, ++u) {
          const int slot = u % kWinSlots;
          if (!mbar_wait(&sempty_bar[slot], ((u / kWinSlots) & 1) ^ 1, &abort_flag)) {
            report_error(p.err, kErrWaitTimeout, &abort_flag);
            ok = false;
            break;
          }
          stage_scales(p, w, m0, n0, nb, sW + slot * kWin * BN, sX + slot * kWin * BM, t);
          mbar_arrive(&sfull_bar[slot]);  // release: the stores above are visible to waiters
          if constexpr (kConv) {
            // Widen the window's stages of int8 weight codes into binary16 B tiles in the
            // MMA's 128-byte swizzled layout (row r at 128 r, 16-byte chunk j at j ^ (r % 8)).
            // Thread t takes 16-byte chunk t % 4 of rows t / 4, t / 4 + 16, ...: the 8 threads
            // of a quarter warp read 128 contiguous bytes and write 8 distinct bank groups.
            const int kb_end = min((w + 1) * (kWin / 2), (min(S.w1 * kWin, nb) + 1) / 2);
            for (int kb = w * (kWin / 2); kb < kb_end; ++kb, ++ci) {
              const int s8 = ci % kStages, f = ci % kFSlots;
              if (!mbar_wait(&full_bar[s8], (ci / kStages) & 1, &abort_flag) ||
                  !mbar_wait(&cempty_bar[f], ((ci / kFSlots) & 1) ^ 1, &abort_flag)) {
                report_error(p.err, kErrWaitTimeout, &abort_flag);
                ok = false;
                break;
              }
              const uint8_t* src = sB + s8 * kStageB8;
              uint8_t* dst = sF + f * kStageB;
              const int c = t & 3;
#pragma unroll 2
              for (int r = t >> 2; r < BN; r += kScaleThreads / 4) {
                uint4 lo, hi;
                codes16_to_f16(*reinterpret_cast<const uint4*>(src + r * BK + c * 16), &lo, &hi);
                *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * c) ^ (r & 7)) * 16)) = lo;
                *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * c + 1) ^ (r & 7)) * 16)) = hi;
              }
              fence_proxy_async_smem();  // the tensor core reads these stores
              __syncwarp();
              if (lane == 0) {
                mbar_arrive(&cfull_bar[f]);
                mbar_arrive(&empty_bar[s8]);  // the int8 codes of the stage are read
              }
            }
          }
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kDrainRegs));
    // ------------------------------- rescale drain ------------------------------------
    // Warp w (4..11) may read TMEM lanes 32*(w%4)..+31 (its quadrant); warpgroup wg owns
    // tile columns [128 wg, 128 wg + 128).  Each thread owns one row m and 128 columns:
    // per block b, acc[n] += (xd[m,b] * Wd[n,b]) * isum[m,n,b] in binary32.  Per block:
    // 8 chunks of 16 columns; the TMEM load and the shared-memory scale load of chunk
    // c + 1 are in flight while chunk c is computed.
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    float2 acc[kBlockSums ? 1 : 64];
    bool failed = false;
    int u = 0;  // windows consumed, all segments
    int g = 0;  // blocks drained, all segments
    for (int sg = 0; sg < nseg && !failed; ++sg) {
      // (the segment's fields are read from shared memory where they are used, so that
      // the tile's origin is not held in registers through the accumulation)
      const int w1 = segs[sg].w1;
      if constexpr (!kBlockSums) {
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);
      }
      for (int w = segs[sg].w0; w < w1 && !failed; ++w, ++u) {
        const int slot = u % kWinSlots;
        const float* dws = sW + slot * kWin * BN + wg * 128;
        const float* dxs = sX + slot * kWin * BM;
        if constexpr (!kBlockSums) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sfull_bar[slot], (u / kWinSlots) & 1, &abort_flag))) {
            if (lane == 0) report_error(p.err, kErrWaitTimeout, &abort_flag);
            failed = true;
            break;
          }
        }
        const int nbw = min(nb - w * kWin, kWin);
#pragma unroll 1
        for (int bb = 0; bb < nbw; ++bb, ++g) {
          const int blk = w * kWin + bb;  // block of the tile's K (block-sum output index)
          const int buf = g & 1;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull_bar[buf], (g >> 1) & 1, &abort_flag))) {
            if (lane == 0) report_error(p.err, kErrWaitTimeout, &abort_flag);
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                 static_cast<uint32_t>(buf * BN + wg * 128);
          const float* dwb = dws + bb * BN;
          float dx = 0.0f;
          if constexpr (!kBlockSums) dx = dxs[bb * BM + row];
          const float2 dx2 = make_float2(dx, dx);
          uint32_t r[2][16];
          float4 wv[2][4];
          tmem_ld_32x32b_x16(taddr, r[0]);
          if constexpr (!kBlockSums) {
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[0][i] = *reinterpret_cast<const float4*>(dwb + 4 * i);
          }
          tmem_ld_wait_regs(r[0]);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (c + 1 < 8) {
              tmem_ld_32x32b_x16(taddr + (c + 1) * 16, r[(c + 1) & 1]);
              if constexpr (!kBlockSums) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  wv[(c + 1) & 1][i] = *reinterpret_cast<const float4*>(dwb + (c + 1) * 16 + 4 * i);
              }
            }
            const uint32_t* rc = r[c & 1];
            if constexpr (kBlockSums) {
              int m0, n0;
              tile_origin(segs[sg].tile, mtiles, &m0, &n0);
              const int m = m0 + row;
              if (m < M) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int n = n0 + wg * 128 + c * 16 + i;
                  if (n < N)
                    p.isum[(static_cast<int64_t>(m) * N + n) * nb + blk] =
                        __float2int_rn(__uint_as_float(rc[i]));
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 w4 = wv[c & 1][i];
                const float2 c0 = __fmul2_rn(dx2, make_float2(w4.x, w4.y));
                const float2 c1 = __fmul2_rn(dx2, make_float2(w4.z, w4.w));
                const int a = (c * 16 + 4 * i) >> 1;
                acc[a].x = fmaf(c0.x, __uint_as_float(rc[4 * i]), acc[a].x);
                acc[a].y = fmaf(c0.y, __uint_as_float(rc[4 * i + 1]), acc[a].y);
                acc[a + 1].x = fmaf(c1.x, __uint_as_float(rc[4 * i + 2]), acc[a + 1].x);
                acc[a + 1].y = fmaf(c1.y, __uint_as_float(rc[4 * i + 3]), acc[a + 1].y);
              }
            }
            if (c + 1 < 8) tmem_ld_wait_regs(r[(c + 1) & 1]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[buf]);
        }
        if constexpr (!kBlockSums) {
          __syncwarp();
          if (lane == 0 && !failed) mbar_arrive(&sempty_bar[slot]);
        }
      }
      if constexpr (!kBlockSums) {
        const Seg S = segs[sg];
        int m0, n0;
        tile_origin(S.tile, mtiles, &m0, &n0);
        const int m = m0 + row;
        const bool m_ok = m < M;
        // this segment stores final outputs (else partial sums for a reduction kernel)
        const bool direct = S.slot < 0 && p.splits == 1;
        // The CTA's last segment is stored by TMA: y of a whole-K tile (plain output), or a
        // partial tile.  The operand ring is idle by then (every MMA has completed and no load
        // is left), so each drain warp stages its 32 rows x 128 columns there as four 32 x 32
        // boxes in the 128-byte swizzled layout (16-byte chunk c of row r at position
        // c ^ (r % 8): the warp's shared-memory stores hit distinct banks), and one lane
        // writes them as whole 128-byte lines, instead of 32 rows' scattered 16-byte pieces.
        // (partial tiles take this path only without stream-K: with it, the extra code in
        // the drain measurably slowed the accumulation loop of the stream-K kernels)
        const bool tma = sg + 1 == nseg && (direct ? (!kFused && p.tma_y) : (!kSK && p.tma_part));
        if (tma && !failed) {
          float* stg = reinterpret_cast<float*>(base) + (warp - 4) * (32 * 128);
          // box origin: (column, row[, plane]) in the target tensor
          int x = n0 + wg * 128, yr = m0 + quad * 32, z = static_cast<int>(blockIdx.y);
          bool rows_in = yr < M;
          if (S.slot >= 0) {
            x = wg * 128;
            yr = quad * 32;
            z = S.slot;
            rows_in = true;
          }
          const int x_end = S.slot >= 0 ? BN : N;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int i = 16 * q + 2 * k;
              *reinterpret_cast<float4*>(stg + q * 1024 + lane * 32 + ((k ^ (lane & 7)) * 4)) =
                  make_float4(acc[i].x, acc[i].y, acc[i + 1].x, acc[i + 1].y);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && rows_in) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (x + 32 * q < x_end) {
                if (direct)
                  tma_store_2d(&tmY, stg + q * 1024, x + 32 * q, yr);
                else
                  tma_store_3d(&tmP, stg + q * 1024, x + 32 * q, yr, z);
              }
            }
            bulk_commit_group();
          }
        } else if (m_ok && !failed && S.slot >= 0) {
          // a stream-K partial tile, compact: [slot][BM][BN], no bounds past N to mind
          float* dst = p.part + (static_cast<int64_t>(S.slot) * BM + row) * BN + wg * 128;
#pragma unroll
          for (int i = 0; i < 64; i += 2)
            *reinterpret_cast<float4*>(dst + 2 * i) = make_float4(acc[i].x, acc[i].y, acc[i + 1].x, acc[i + 1].y);
        } else if (m_ok && !failed) {
          float* yrow = (p.splits > 1 ? p.part + static_cast<int64_t>(blockIdx.y) * M * N : p.y) +
                        static_cast<int64_t>(m) * N;
          const int nbase = n0 + wg * 128;
          if (kFused && direct) {
            const int64_t r0 = static_cast<int64_t>(m) * N + nbase;
            if ((N & 3) == 0 && nbase + 128 <= N) {
              // 4 chunks of 32 columns; the 8 aux loads of chunk h + 1 are in flight while
              // chunk h is computed and stored
              float4 a[2][8];
#pragma unroll
              for (int q = 0; q < 8; ++q) a[0][q] = epi_aux4(p.epi, r0 + 4 * q);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                if (h + 1 < 4) {
#pragma unroll
                  for (int q = 0; q < 8; ++q) a[(h + 1) & 1][q] = epi_aux4(p.epi, r0 + 32 * (h + 1) + 4 * q);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const int i = 16 * h + 2 * q;  // columns 2i .. 2i + 3 of the slice
                  const float4 v = make_float4(acc[i].x, acc[i].y, acc[i + 1].x, acc[i + 1].y);
                  epi_put4(p.epi, p.y, r0 + 32 * h + 4 * q, epi_apply4(p.epi, v, a[h & 1][q]));
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 64; ++i) {
                if (nbase + 2 * i < N) epi_store(p.epi, p.y, r0 + 2 * i, acc[i].x);
                if (nbase + 2 * i + 1 < N) epi_store(p.epi, p.y, r0 + 2 * i + 1, acc[i].y);
              }
            }
          } else if ((N & 3) == 0 && nbase + 128 <= N) {
#pragma unroll
            for (int i = 0; i < 64; i += 2)
              *reinterpret_cast<float4*>(yrow + nbase + 2 * i) =
                  make_float4(acc[i].x, acc[i].y, acc[i + 1].x, acc[i + 1].y);
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              if (nbase + 2 * i < N) yrow[nbase + 2 * i] = acc[i].x;
              if (nbase + 2 * i + 1 < N) yrow[nbase + 2 * i + 1] = acc[i].y;
            }
          }
        }
      }
    }
  }

  if (warp >= 4 && lane == 0) bulk_wait_all();  // this warp's TMA stores have completed
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

// The kinds of tensor map the GEMM uses, all [planes][rows][cols] with cols contiguous: the
// binary16 operands (2-D, box box_rows x 64 columns, 128-byte swizzle), the int8 weight codes
// (2-D, box box_rows x 64 bytes, unswizzled: the widening warps read them in row order), the
// binary32 outputs the drain stores from its staged boxes (box 32 x 32, 128-byte swizzle:
// y 2-D, partial tiles 3-D), and the fused epilogue's aux (2-D, a whole 128 x 256 tile,
// unswizzled, only ever prefetched to L2).
enum TmapKind : uint32_t { kTmapF16Operand = 0, kTmapF32Out = 1, kTmapF32Planes = 2, kTmapU8Operand = 3,
                          kTmapF32Tile = 4 };

bool encode_tmap(CUtensorMap* map, TmapKind kind, const void* ptr, uint64_t planes, uint64_t rows,
                 uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  const bool operand = kind == kTmapF16Operand || kind == kTmapU8Operand;
  const uint64_t esz = kind == kTmapU8Operand ? 1 : kind == kTmapF16Operand ? 2 : 4;
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {cols * esz, rows * cols * esz};
  const cuuint32_t box[3] = {operand ? static_cast<cuuint32_t>(BK) : kind == kTmapF32Tile ? static_cast<cuuint32_t>(BN) : 32u,
                             box_rows, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = kind == kTmapU8Operand    ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : kind == kTmapF16Operand ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return enc(map, dt, kind == kTmapF32Planes ? 3 : 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             (kind == kTmapU8Operand || kind == kTmapF32Tile) ? CU_TENSOR_MAP_SWIZZLE_NONE
                                                              : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps, keyed by everything the encoding depends on (kind, address, shape,
// box), so a cached map is always the one a fresh encoding would give.  Bounded: cleared
// when full.
struct TmapKey {
  uint32_t kind;
  const void* ptr;
  uint64_t planes, rows, cols;
  uint32_t box_rows;
  bool operator<(const TmapKey& o) const {
    if (kind != o.kind) return kind < o.kind;
    if (ptr != o.ptr) return ptr < o.ptr;
    if (planes != o.planes) return planes < o.planes;
    if (rows != o.rows) return rows < o.rows;
    if (cols != o.cols) return cols < o.cols;
    return box_rows < o.box_rows;
  }
};
std::mutex g_tmap_mu;
std::map<TmapKey, CUtensorMap> g_tmaps;
constexpr size_t kTmapCacheMax = 4096;

bool make_tmap(CUtensorMap* map, TmapKind kind, const void* ptr, uint64_t planes, uint64_t rows,
               uint64_t cols, uint32_t box_rows) {
  const TmapKey key{kind, ptr, planes, rows, cols, box_rows};
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    auto it = g_tmaps.find(key);
    if (it != g_tmaps.end()) {
      *map = it->second;
      return true;
    }
  }
  if (!encode_tmap(map, kind, ptr, planes, rows, cols, box_rows)) return false;
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  if (g_tmaps.size() >= kTmapCacheMax) g_tmaps.clear();
  g_tmaps[key] = *map;
  return true;
}

// y = sum over s of part[s] (fixed order: the result does not depend on timing).
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float4* __restrict__ part,
                                                            float4* __restrict__ y, int64_t n4,
                                                            int splits, const Epilogue epi) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = part[static_cast<int64_t>(s) * n4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if (epi.plain())
      y[i] = a;
    else
      epi_put4(epi, reinterpret_cast<float*>(y), 4 * i, epi_apply4(epi, a, epi_aux4(epi, 4 * i)));
  }
}

__global__ void __launch_bounds__(256) reduce_splits_scalar_kernel(const float* __restrict__ part,
                                                                   float* __restrict__ y, int64_t n,
                                                                   int splits, const Epilogue epi) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float a = part[i];
    for (int s = 1; s < splits; ++s) a += part[static_cast<int64_t>(s) * n + i];
    epi_store(epi, y, i, a);
  }
}

// Stream-K fix-up.  The stream-K region holds more tiles than there are runs, so every run
// is longer than a tile, run boundaries are at least a tile apart, and a tile holds at most
// one of them: a split tile has exactly two partials, the end of run j - 1 and the start of
// run j.  CTA (j - 1, r) takes the boundary between runs j - 1 and j and, if that boundary
// falls inside a tile, adds the tile's two partials (in that order: the result does not
// depend on timing) for its rows [32 r, 32 r + 32) and stores them through the epilogue.
constexpr int kFixRows = 32;
__global__ void __launch_bounds__(256) reduce_sk_kernel(const float* __restrict__ part, float* y,
                                                        int M, int N, int mtiles, int nwin, int G,
                                                        int W, const Epilogue epi) {
  const int j = static_cast<int>(blockIdx.x) + 1;
  const int w = sk_start(j, W, G);
  if (w % nwin == 0) return;  // on a tile boundary: both tiles were stored whole
  const int ts = w / nwin;
  const int s_lo = (sk_start(j - 1, W, G) / nwin == ts) ? 2 * (j - 1) : 2 * (j - 1) + 1;
  const int s_hi = 2 * j;
  int m0, n0;
  tile_origin(ts, mtiles, &m0, &n0);
  const float* lo = part + static_cast<int64_t>(s_lo) * BM * BN;
  const float* hi = part + static_cast<int64_t>(s_hi) * BM * BN;
#pragma unroll 4
  for (int k = 0; k < kFixRows * (BN / 4) / 256; ++k) {
    const int idx = k * 256 + static_cast<int>(threadIdx.x);
    const int row = static_cast<int>(blockIdx.y) * kFixRows + idx / (BN / 4);
    const int col = 4 * (idx % (BN / 4));
    const int m = m0 + row, n = n0 + col;
    if (m >= M || n >= N) continue;
    const float4 a = *reinterpret_cast<const float4*>(lo + row * BN + col);
    const float4 b = *reinterpret_cast<const float4*>(hi + row * BN + col);
    const float4 v = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    const int64_t o = static_cast<int64_t>(m) * N + n;
    if ((N & 3) == 0 && n + 4 <= N) {
      if (epi.plain())
        *reinterpret_cast<float4*>(y + o) = v;
      else
        epi_put4(epi, y, o, epi_apply4(epi, v, epi_aux4(epi, o)));
    } else {
      const float e[4] = {v.x, v.y, v.z, v.w};
      for (int c = 0; c < 4 && n + c < N; ++c) epi_store(epi, y, o + c, e[c]);
    }
  }
}

template <bool kBS, bool kFused = false, bool kSK = false, bool kConv = false>
cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& yt,
                        const CUtensorMap& pt, const GemmParams& p, int grid, cudaStream_t stream,
                        int dev_id) {
  auto fn = gemm_tc_kernel<kBS, kFused, kSK, kConv>;
  constexpr size_t smem = kConv ? kSmemBytesConv : kSmemBytes;
  // setmaxnreg.inc waits until the registers exist: the split above is exact only if the
  // kernel was compiled for kLaunchRegs per thread.  Refuse to launch otherwise.
  int regs = 0;
  cudaError_t e = kernel_regs(reinterpret_cast<const void*>(fn), dev_id, &regs);
  if (e != cudaSuccess) return e;
  if (regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  e = ensure_smem(reinterpret_cast<const void*>(fn), smem, dev_id);
  if (e != cudaSuccess) return e;
  fn<<<dim3(grid, p.splits), kThreads, smem, stream>>>(a, b, yt, pt, p);
  return cudaGetLastError();
}

}  // namespace

void forget_tensor_maps() {
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  g_tmaps.clear();
}

namespace {
// How the output tiles are spread over the GPU's SMs (one CTA per SM at a time):
//  - fewer tiles than SMs: every tile is split along K into `splits` ranges of whole scale
//    windows, one CTA each (uniform split-K, partials [splits, M, N]);
//  - a whole number of waves: one CTA per tile;
//  - otherwise stream-K: the tiles of one full wave plus the partial one (sk_tiles, fewer
//    than two waves) are shared out as equal runs of scale windows over one CTA per SM,
//    launched first; the other waves' tiles (dp_tiles) follow as whole tiles.
struct Schedule {
  int splits = 1;
  int64_t dp_tiles = 0;
  int sk_ctas = 0;
  int64_t sk_tiles = 0;
  int64_t nwin = 0;
};

Schedule gemm_schedule(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  Schedule sc;
  if (M <= 0 || N <= 0 || K <= 0 || dev.sm_count <= 0) return sc;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int64_t G = dev.sm_count;
  sc.nwin = (K / kQK + kWin - 1) / kWin;
  sc.dp_tiles = tiles;
  if (tiles < G) {
    sc.splits = static_cast<int>(std::max<int64_t>(1, std::min(G / tiles, sc.nwin)));
  } else if (tiles % G != 0) {
    sc.sk_tiles = G + tiles % G;
    sc.dp_tiles = tiles - sc.sk_tiles;
    sc.sk_ctas = static_cast<int>(G);
  }
  return sc;
}
}  // namespace

int gemm_splits(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  return gemm_schedule(M, N, K, dev).splits;
}

size_t gemm_part_bytes(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  const Schedule sc = gemm_schedule(M, N, K, dev);
  if (sc.splits > 1) return static_cast<size_t>(sc.splits) * M * N * 4;
  return static_cast<size_t>(2) * sc.sk_ctas * BM * BN * 4;
}

cudaError_t launch_gemm_tc(const uint16_t* A16, const void* B, bool b_int8, const float* xd,
                           const uint16_t* Wd, float* y, int32_t* isum, float* part, int splits,
                           int64_t M, int64_t N, int64_t K, const DeviceInfo& dev,
                           cudaStream_t stream, const Epilogue& epi) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0) return cudaErrorInvalidValue;  // the API handles K == 0 without a launch
  if (b_int8 && isum != nullptr) return cudaErrorInvalidValue;  // block sums: binary16 B only
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, kTmapF16Operand, A16, 1, static_cast<uint64_t>(M), static_cast<uint64_t>(K), BM) ||
      !make_tmap(&tb, b_int8 ? kTmapU8Operand : kTmapF16Operand, B, 1, static_cast<uint64_t>(N),
                 static_cast<uint64_t>(K), BN))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.xd = xd;
  p.Wd = Wd;
  p.y = y;
  p.isum = isum;
  if (isum != nullptr || splits < 1 || part == nullptr) splits = 1;  // block sums: one range
  p.splits = splits;
  p.part = splits > 1 ? part : nullptr;
  // stream-K needs the caller's partial buffer (sized by gemm_part_bytes); y only
  const Schedule sc = gemm_schedule(M, N, K, dev);
  const bool sk = isum == nullptr && splits == 1 && part != nullptr && sc.sk_ctas > 0;
  const int64_t mtiles = (M + BM - 1) / BM;
  const int64_t tiles0 = mtiles * ((N + BN - 1) / BN);
  p.sk_ctas = sk ? sc.sk_ctas : 0;
  p.sk_tiles = static_cast<int>(sk ? sc.sk_tiles : 0);
  p.sk_windows = static_cast<int>(sk ? sc.sk_tiles * sc.nwin : 0);
  if (sk) p.part = part;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.err = dev.err_word;
  p.epi = epi;
  // TMA stores: y (plain binary32 output) and the partial tiles, where the rows are 16-byte
  // multiples on 16-byte aligned bases
  CUtensorMap ty, tp;
  std::memset(&ty, 0, sizeof(ty));
  std::memset(&tp, 0, sizeof(tp));
  const bool rows16 = (N % 4) == 0;
  p.tma_y = isum == nullptr && splits == 1 && epi.plain() && rows16 &&
            (reinterpret_cast<uintptr_t>(y) % 16) == 0 &&
            make_tmap(&ty, kTmapF32Out, y, 1, static_cast<uint64_t>(M), static_cast<uint64_t>(N), 32);
  const bool part_ok = part != nullptr && (reinterpret_cast<uintptr_t>(part) % 16) == 0;
  p.tma_aux = 0;
  if (!epi.plain() && splits == 1 && isum == nullptr) {
    // the fused kernel: tmP maps aux instead (its partial tiles are never stored by TMA)
    p.tma_part = 0;
    p.tma_aux = epi.aux != nullptr && rows16 && (reinterpret_cast<uintptr_t>(epi.aux) % 16) == 0 &&
                make_tmap(&tp, kTmapF32Tile, epi.aux, 1, static_cast<uint64_t>(M), static_cast<uint64_t>(N), BM);
  } else if (sk)
    p.tma_part = part_ok && make_tmap(&tp, kTmapF32Planes, part, 2 * static_cast<uint64_t>(sc.sk_ctas), BM, BN, 32);
  else
    p.tma_part = splits > 1 && part_ok && rows16 &&
                 make_tmap(&tp, kTmapF32Planes, part, static_cast<uint64_t>(splits),
                           static_cast<uint64_t>(M), static_cast<uint64_t>(N), 32);
  const int64_t ctas = sk ? sc.dp_tiles + sc.sk_ctas : tiles0;
  if (tiles0 > 0x7FFFFFFF || (sk && sc.sk_tiles * sc.nwin > 0x7FFFFFFF)) return cudaErrorInvalidValue;
  if (isum) return launch_impl<true>(ta, tb, ty, tp, p, static_cast<int>(ctas), stream, dev.device);
  // the epilogue runs in the drain unless split-K partials take the reduce kernel's
  const int grid = static_cast<int>(ctas);
  cudaError_t e;
  if (splits == 1 && !epi.plain())
    e = b_int8 ? (sk ? launch_impl<false, true, true, true>(ta, tb, ty, tp, p, grid, stream, dev.device)
                     : launch_impl<false, true, false, true>(ta, tb, ty, tp, p, grid, stream, dev.device))
               : (sk ? launch_impl<false, true, true>(ta, tb, ty, tp, p, grid, stream, dev.device)
                     : launch_impl<false, true, false>(ta, tb, ty, tp, p, grid, stream, dev.device));
  else
    e = b_int8 ? (sk ? launch_impl<false, false, true, true>(ta, tb, ty, tp, p, grid, stream, dev.device)
                     : launch_impl<false, false, false, true>(ta, tb, ty, tp, p, grid, stream, dev.device))
               : (sk ? launch_impl<false, false, true>(ta, tb, ty, tp, p, grid, stream, dev.device)
                     : launch_impl<false, false, false>(ta, tb, ty, tp, p, grid, stream, dev.device));
  if (e != cudaSuccess) return e;
  if (sk && sc.sk_ctas > 1) {
    reduce_sk_kernel<<<dim3(sc.sk_ctas - 1, BM / kFixRows), 256, 0, stream>>>(
        part, y, static_cast<int>(M), static_cast<int>(N), static_cast<int>(mtiles),
        static_cast<int>(sc.nwin), sc.sk_ctas, p.sk_windows, epi);
    return cudaGetLastError();
  }
  if (splits == 1) return e;
  const int64_t n = M * N;
  const int blocks = static_cast<int>(std::min<int64_t>((n / 4 + 255) / 256, 4 * dev.sm_count)) + 1;
  if (n % 4 == 0)
    reduce_splits_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(part),
                                                     reinterpret_cast<float4*>(y), n / 4, splits, epi);
  else
    reduce_splits_scalar_kernel<<<blocks, 256, 0, stream>>>(part, y, n, splits, epi);
  return cudaGetLastError();
}

namespace {
__global__ void __launch_bounds__(256) epilogue_only_kernel(const Epilogue epi, float* y, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    epi_store(epi, y, i, 0.0f);
}
}  // namespace

cudaError_t launch_epilogue_only(const Epilogue& epi, float* y, int64_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  epilogue_only_kernel<<<blocks, 256, 0, stream>>>(epi, y, n);
  return cudaGetLastError();
}

}  // namespace q8
