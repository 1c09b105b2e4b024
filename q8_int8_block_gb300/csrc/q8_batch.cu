// q8_batch.cu -- batched-decode Q8_0 linear (2 <= M <= 64 tokens): streams the weights from
// HBM once, forms the exact int32 block sums on the mma.sync tensor path, rescales in
// registers.
//
// Operation: y[m,n] = sum_b Wd[n,b] * xd[m,b] * isum[m,n,b], the Q8_0 int8 GEMM of
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, list of un-throttled paths: the DP4A int8
// GEMM), at batched-decode sizes, where reading the weights still dominates but one dp4a
// per 4 MACs and token is too slow.
//
// Exact block sums.  The int8 codes enter mma.sync.m16n8k16 (binary16 in, binary32
// accumulate) as binary16 values: |q| <= 127 is exact, each product is exact, and every
// partial sum of one 32-element block is an integer below 2^24, exact in binary32.  Two
// MMAs from zero (one per 16-wide half) and their sum give the block sum.  The K order inside a block does not matter for an
// exact sum, so A and B only have to agree on it: lane (g, c) of the warp (g = lane / 4,
// c = lane % 4) supplies K positions {4c..4c+3} to the first MMA and {16+4c..16+4c+3} to
// the second, in fragment slots (2c, 2c+1) and (2c+8, 2c+9).
//
// Design (one CTA per 16 * RG weight rows, 1 producer warp + 15 consumer warps, so that
// 16 warps with up to 128 registers each fill an SM):
//   * the CTA's weight rows stream through a ring of K chunks, 512 wide where K and the ring
//     allow (else 256): one TMA box of 16 RG rows x 128 int8 codes per 4 blocks, with
//     128-byte swizzle (so ldmatrix reads them without bank conflicts), one box of the
//     rows' binary16 scales, and the chunk's activation codes and scales by bulk copies.
//     A chunk costs the consumers a fixed latency besides its work (measured: ~0.5 us per
//     256-wide chunk at M = 4), which the wider chunk spreads over twice the weights;
//   * the activations arrive from quantize_batch_kernel in a fragment-ordered layout,
//     xb[b][t][32] binary16 (for each 16-byte piece c: K 4c..4c+3 then K 16+4c..16+4c+3)
//     and xbd[b][t] binary32, tokens padded with zeros to whole groups of 8, so each lane's
//     B fragments of one block are one 16-byte load;
//   * consumer warp w works on row group rg = w % RG (16 rows) and a share of the token
//     groups (8 tokens each); when token groups are fewer than the warps of a row group,
//     the warps split the chunk's 8 blocks instead and their partial sums are added in
//     shared memory at the end;
//   * a warp takes its blocks of a chunk up to 4 at a time: ldmatrix.x4 of the weight codes
//     (shared by the warp's token groups), widening to binary16, one 16-byte load of
//     activation codes and two MMAs per token group and block, all issued before the
//     rescale y_acc += (Wd * xd) * S in packed binary32 (f32x2) registers;
//   * programmatic dependent launch: the producer loads the first stages' weights before
//     waiting for the previous kernel (the activation quantizer), then their activations.
//   * Block-sum mode (for checking) stores the MMA results as int32 instead.
//
// Measured limits (GB300, 12288 x 4096 weights): weight streaming alone runs at the HBM
// rate (9 us); the separate quantizer kernel costs ~4 us of each call; at large M the
// activation chunks (32 KB per 256-wide chunk at M = 64) outweigh the weights in the ring.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "q8_epi.cuh"
#include "q8_internal.h"
#include "q8_ptx.cuh"
#include "q8_quant_dev.cuh"

namespace q8 {
namespace {

// K per stage: 512 (16 Q8_0 blocks) where K allows, else 256.  A chunk costs the consumer
// warps a fixed latency (their dependent chains of shared-memory loads, widening, MMAs and
// rescale) besides its work, so the wider chunk halves that cost per weight byte.
constexpr int kChunkK = 256;                 // the narrow chunk: K % 256 == 0 is required
constexpr int kChunkBlocks = kChunkK / kQK;  // 8 Q8_0 blocks
constexpr int kMaxChunkBlocks = 16;
constexpr int kConsumerWarps = 15;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxRG = kConsumerWarps;       // every row group needs a warp (16 * RG <= 256 rows)
constexpr int kMaxStages = 8;
constexpr int kRingTarget = 192 * 1024;
// 16 warps, 4 per SM sub-partition: 4 x 32 x 128 registers fill a sub-partition's 16384
constexpr int kMaxRegs = 128;
static_assert((kConsumerWarps + 1 + 3) / 4 * 32 * kMaxRegs <= 16384, "registers per sub-partition");

struct BatchParams {
  const uint16_t* xb;   // [nb][TP][32] binary16 codes, fragment order
  const float* xbd;     // [nb][TP] scales
  float* y;             // [M,N]
  int32_t* isum;        // [M,N,nb] (block-sum mode)
  int M, N, K;
  int RG;               // row groups of 16 per CTA
  int KPall;            // partial-sum layers (block splits) of the busiest row group
  int stages;
  int cb;               // Q8_0 blocks per chunk (8 or 16)
  uint32_t stage_bytes;
  uint32_t off_w1, off_wd, off_x, off_xd;  // offsets inside a stage (off_w1: one 128-byte weight box)
  uint32_t* err;
  Epilogue epi;         // fused output step
};

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 4 int8 codes -> 2 half2 (bytes 0,1 and bytes 2,3), exactly: byte b = q + 128 goes under
// the binary16 exponent of 1024 (0x6400 | b = 1024 + b), then 1152 = 1024 + 128 is
// subtracted; all values are small integers, nothing rounds.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t magic = 0x64646464u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(u), "r"(magic));
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(b) : "r"(u), "r"(magic));
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// Not volatile: the compiler may schedule it freely after the point where `addr` is known
// (the callers derive `addr` from a value laundered after the stage's barrier wait).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

// Shared-memory loads by 32-bit shared address (not volatile: callers derive the address
// from a value laundered after the stage's barrier wait).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t a) {
  float2 v;
  asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f16(uint32_t a) {
  unsigned short h;
  asm("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
  return __half2float(__ushort_as_half(h));
}

// D = A (16 x 16, row) * B (16 x 8, col) + C, binary16 in, binary32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// kNTG: the most token groups one warp handles (a warp handles ntg <= kNTG of them).
// kFused: the output store applies the epilogue (residual, SiLU gate, bfloat16 y); the
// plain layer is a separate instantiation so that it carries none of that code.
template <bool kBlockSums, int kNTG, bool kFused>
__global__ void __maxnreg__(kMaxRegs)
    batch_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                 const BatchParams p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = p.M, N = p.N, K = p.K, RG = p.RG, S = p.stages;
  const int nb = K / kQK;
  const int cbk = p.cb;           // blocks per chunk
  const int nchunks = cbk > 0 ? K / (kQK * cbk) : 0;
  const int rows = 16 * RG;
  const int row0 = blockIdx.x * rows;
  const int TG = (M + 7) >> 3;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023) & ~1023u) - raw);

  if (S > kMaxStages || S < 2 || RG < 1 || RG > kMaxRG || M < 1 || M > kBatchMaxM ||
      (cbk != kChunkBlocks && cbk != kMaxChunkBlocks)) {
    if (threadIdx.x == 0) report_error(p.err, kErrBadLaunch, nullptr);  // the launcher never does this
    return;
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmS);
  }
  __syncthreads();

  const uint32_t wbytes = static_cast<uint32_t>(rows) * (kQK * cbk + cbk * 2);
  const uint32_t xbytes = static_cast<uint32_t>(cbk * 8 * TG) * (64 + 4);

  if (warp == 0) {
    // ---------------- producer ---------------------------------------------------------
    if (lane == 0) {
      auto load_w = [&](int st) {
        uint8_t* stg = ring + static_cast<size_t>(st % S) * p.stage_bytes;
        uint64_t* bar = &full_bar[st % S];
        for (int bx = 0; bx < cbk / 4; ++bx)  // 128-byte boxes of 4 blocks
          tma_load_2d(stg + bx * p.off_w1, &tmW, bar, st * kQK * cbk + 128 * bx, row0);
        tma_load_2d(stg + p.off_wd, &tmS, bar, st * cbk, row0);
      };
      auto load_x = [&](int st) {
        uint8_t* stg = ring + static_cast<size_t>(st % S) * p.stage_bytes;
        uint64_t* bar = &full_bar[st % S];
        const size_t blk0 = static_cast<size_t>(st) * cbk * (8 * TG);
        bulk_load(stg + p.off_x, p.xb + blk0 * 32, static_cast<uint32_t>(cbk * 8 * TG) * 64, bar);
        bulk_load(stg + p.off_xd, p.xbd + blk0, static_cast<uint32_t>(cbk * 8 * TG) * 4, bar);
      };
      // weights of the first stages before waiting for the previous kernel, activations after
      const int pre = nchunks < S ? nchunks : S;
      for (int st = 0; st < pre; ++st) {
        mbar_arrive_expect_tx(&full_bar[st], wbytes + xbytes);
        load_w(st);
      }
      pdl_wait();
      for (int st = 0; st < pre; ++st) load_x(st);
      int issued = pre;
      for (int st = pre; st < nchunks; ++st) {
        const int s = st % S;
        if (!mbar_wait_sleep(&empty_bar[s], ((st / S) & 1) ^ 1, &abort_flag)) {
          report_error(p.err, kErrWaitTimeout, &abort_flag);
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], wbytes + xbytes);
        load_w(st);
        load_x(st);
        issued = st + 1;
      }
      // never leave with copies in flight
      for (int st = (issued > S ? issued - S : 0); st < issued; ++st)
        if (!mbar_wait(&full_bar[st % S], (st / S) & 1, nullptr)) {
          report_error(p.err, kErrWaitTimeout, nullptr);
          break;
        }
    }
  } else {
    // ---------------- consumers --------------------------------------------------------
    const int cw = warp - 1;
    pdl_wait();  // x, y / isum: wait for the previous kernel before reading or writing
    if constexpr (!kBlockSums && kFused) {
      // this CTA's aux rows (one per token) towards L2 for the epilogue
      const int nrow = (N - row0) < rows ? (N - row0) : rows;
      for (int t = cw; t < M; t += kConsumerWarps)
        if (lane == 0) epi_prefetch(p.epi, static_cast<int64_t>(t) * N + row0, nrow);
    }
    const int rg = cw % RG;
    const int idx = cw / RG;
    const int nw = (kConsumerWarps - 1 - rg) / RG + 1;  // warps of this row group
    // token groups tg0, tg0 + tgstep, ... (ntg of them); blocks b' = kp (mod KP) of a chunk
    int tg0, tgstep, ntg, kp, KP;
    if (TG >= nw) {
      KP = 1;
      kp = 0;
      tg0 = idx;
      tgstep = nw;
      ntg = (TG - idx + nw - 1) / nw;
    } else {
      KP = nw / TG;
      if (KP > cbk) KP = cbk;
      tg0 = idx % TG;
      tgstep = TG;
      kp = idx / TG;
      ntg = kp < KP ? 1 : 0;
    }
    const int g = lane >> 2, c = lane & 3;
    // ldmatrix row address of this lane: matrix mi = lane / 8 (0: rows 0-7, 1: rows 8-15 of
    // the group; 2, 3: the same rows, next 16-byte chunk), row r = lane % 8
    const int mi = lane >> 3, lr = lane & 7;
    const int lrow = 16 * rg + lr + 8 * (mi & 1);
    bool failed = false;
    const int TP = 8 * TG;  // tokens padded to whole groups of 8
    float2 acc[kNTG][2];    // (row g, tokens t0, t0+1), (row g+8, tokens t0, t0+1)
#pragma unroll
    for (int i = 0; i < kNTG; ++i) acc[i][0] = acc[i][1] = make_float2(0.0f, 0.0f);
    if (ntg > kNTG) {  // the launcher never does this
      if (lane == 0) report_error(p.err, kErrBadLaunch, &abort_flag);
      failed = true;
    }
    // per-lane byte offsets inside a stage
    const uint32_t a_lane = static_cast<uint32_t>(lrow * 128);
    const uint32_t x_lane = static_cast<uint32_t>(p.off_x + g * 64 + 16 * c);
    const uint32_t x_block = static_cast<uint32_t>(TP * 64);
    const uint32_t dx_lane = static_cast<uint32_t>(p.off_xd + 8 * c);
    const uint32_t wd_lane = static_cast<uint32_t>(p.off_wd + (16 * rg + g) * cbk * 2);
    int s = 0;
    uint32_t phase = 0;  // slot s and parity of stage st, kept without divisions
    for (int st = 0; st < nchunks && !failed; ++st, s = (s + 1 == S ? 0 : s + 1), phase ^= (s == 0)) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_sleep(&full_bar[s], phase, &abort_flag))) {
        if (lane == 0) report_error(p.err, kErrWaitTimeout, &abort_flag);
        failed = true;
        break;
      }
      const uint8_t* stg = ring + static_cast<size_t>(s) * p.stage_bytes;
      // the stage's shared-memory address, passed through an empty asm after the wait so
      // that no load of the stage can be scheduled before the wait
      uint32_t stg32 = smem_u32(stg);
      asm volatile("" : "+r"(stg32)::"memory");
      if (ntg > 0) {
        // this warp's blocks of the chunk: kp, kp + KP, ...; two at a time, so that the
        // shared-memory loads and MMAs of both are in flight together
        const int nmine = (cbk - kp + KP - 1) / KP;
        // kGB of this warp's blocks at a time: all their shared-memory loads and MMAs are
        // issued before any result is used (the chains are long-latency: ldmatrix, MMA, FMA);
        // slots past the last block repeat it and are not accumulated
        constexpr int kGB = kNTG <= 2 ? 4 : 2;
        for (int j0 = 0; j0 < nmine; j0 += kGB) {
          int bps[kGB];
#pragma unroll
          for (int k = 0; k < kGB; ++k) bps[k] = kp + (j0 + k < nmine ? j0 + k : nmine - 1) * KP;
          uint32_t wa[kGB][4];
#pragma unroll
          for (int k = 0; k < kGB; ++k) {
            const int bp = bps[k];
            const uint32_t chunk = static_cast<uint32_t>(2 * (bp & 3) + (mi >> 1));
            ldmatrix_x4(stg32 + static_cast<uint32_t>(bp >> 2) * p.off_w1 + a_lane + ((chunk ^ lr) << 4), wa[k][0],
                        wa[k][1], wa[k][2], wa[k][3]);
          }
          float dw0[kGB], dw1[kGB];  // Wd of rows g and g + 8
#pragma unroll
          for (int k = 0; k < kGB; ++k) {
            dw0[k] = dw1[k] = 0.0f;
            if constexpr (!kBlockSums) {
              const uint32_t wda = stg32 + wd_lane + 2 * bps[k];
              dw0[k] = lds_f16(wda);
              dw1[k] = lds_f16(wda + 8 * cbk * 2);
            }
          }
          {
            uint32_t a1[kGB][4], a2[kGB][4];
#pragma unroll
            for (int k = 0; k < kGB; ++k) {
              widen4(wa[k][0], a1[k][0], a1[k][2]);  // row g,     K 4c..4c+3 of the block's first half
              widen4(wa[k][1], a1[k][1], a1[k][3]);  // row g + 8
              widen4(wa[k][2], a2[k][0], a2[k][2]);  // row g,     K 16+4c..
              widen4(wa[k][3], a2[k][1], a2[k][3]);  // row g + 8
            }
#pragma unroll
            for (int i = 0; i < kNTG; ++i) {
              if (i < ntg) {
                const int tg = tg0 + i * tgstep;
                uint4 xv[kGB];
                float d[kGB][4];
#pragma unroll
                for (int k = 0; k < kGB; ++k)  // B fragments of token 8 tg + g (tokens padded to TP)
                  xv[k] = lds128(stg32 + x_lane + bps[k] * x_block + tg * 512);
#pragma unroll
                for (int k = 0; k < kGB; ++k) {
                  if (j0 + k < nmine) {
                    const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    float h[4];
                    mma_16816(h, a1[k], xv[k].x, xv[k].y, z);
                    mma_16816(d[k], a2[k], xv[k].z, xv[k].w, h);  // exact: integers below 2^24
                  }
                }
#pragma unroll
                for (int k = 0; k < kGB; ++k) {
                  if (j0 + k < nmine) {
                    if constexpr (kBlockSums) {
                      const int b = st * cbk + bps[k];
                      const int n0 = row0 + 16 * rg + g;
                      const int t0 = 8 * tg + 2 * c;
#pragma unroll
                      for (int e = 0; e < 4; ++e) {
                        const int t = t0 + (e & 1), n = n0 + 8 * (e >> 1);
                        if (t < M && n < N)
                          p.isum[(static_cast<int64_t>(t) * N + n) * nb + b] = __float2int_rn(d[k][e]);
                      }
                    } else {
                      const float2 dx = lds64f(stg32 + dx_lane + (bps[k] * TP + 8 * tg) * 4);
                      acc[i][0] = __ffma2_rn(__fmul2_rn(make_float2(dw0[k], dw0[k]), dx),
                                             make_float2(d[k][0], d[k][1]), acc[i][0]);
                      acc[i][1] = __ffma2_rn(__fmul2_rn(make_float2(dw1[k], dw1[k]), dx),
                                             make_float2(d[k][2], d[k][3]), acc[i][1]);
                    }
                  }
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);  // this warp no longer reads the stage
    }
    if constexpr (!kBlockSums) {
      // partial sums [kp][token][row] in the ring (every copy has landed: the consumers
      // waited for the last stage), then one coalesced pass adds the layers and writes y
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
      const bool any_fail = wg_barrier_any<32 * kConsumerWarps>(2, failed);
      if (!any_fail) {
        float* red = reinterpret_cast<float*>(ring);
        const int layer = rows * TP;
        for (int i = threadIdx.x - 32; i < p.KPall * layer; i += 32 * kConsumerWarps) red[i] = 0.0f;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
#pragma unroll
        for (int i = 0; i < kNTG; ++i) {
          if (i < ntg) {
            const int t0 = 8 * (tg0 + i * tgstep) + 2 * c;
            float* l = red + kp * layer + t0 * rows + 16 * rg + g;
            l[0] = acc[i][0].x;
            l[rows] = acc[i][0].y;
            l[8] = acc[i][1].x;
            l[rows + 8] = acc[i][1].y;
          }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
        if constexpr (kFused) {
          constexpr int kT = 32 * kConsumerWarps;
          constexpr int kU = 4;  // outputs per thread whose aux loads are in flight together
          for (int i0 = threadIdx.x - 32; i0 < M * rows; i0 += kU * kT) {
            float a[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const int i = i0 + u * kT;
              const int t = i / rows, n = row0 + (i - t * rows);
              a[u] = (i < M * rows && n < N) ? epi_aux(p.epi, static_cast<int64_t>(t) * N + n) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const int i = i0 + u * kT;
              const int t = i / rows, r = i - t * rows;
              const int n = row0 + r;
              if (i < M * rows && n < N) {
                float v = 0.0f;
                for (int k = 0; k < p.KPall; ++k) v += red[k * layer + t * rows + r];
                epi_put(p.epi, p.y, static_cast<int64_t>(t) * N + n, epi_apply(p.epi, v, a[u]));
              }
            }
          }
        } else {  // the plain layer: binary32 y
          for (int i = threadIdx.x - 32; i < M * rows; i += 32 * kConsumerWarps) {
            const int t = i / rows, r = i - t * rows;
            const int n = row0 + r;
            if (n < N) {
              float v = 0.0f;
              for (int k = 0; k < p.KPall; ++k) v += red[k * layer + t * rows + r];
              p.y[static_cast<int64_t>(t) * N + n] = v;
            }
          }
        }
      }
    }
  }
  __syncthreads();
}

// Activations -> xb [nb][M][32] binary16 codes in fragment order and xbd [nb][M] scales.
// Four lanes own one block of one row (8 values each); lane sub holds K 8 sub..8 sub+7 and
// writes them as two 8-byte halves: K 8 sub..+3 to piece 2 (sub & 1), K 8 sub+4..+7 to
// piece 2 (sub & 1) + 1, in the piece's first half for sub < 2, second half otherwise.
// kCodes: the input is int8 codes already (block-sum mode); no scales.
// gamma / r: the RMSNorm prologue (nullptr: none): codes of fl32(x * gamma), scale d * r[m].
template <typename InT, bool kCodes>
__global__ void __launch_bounds__(256) quantize_batch_kernel(const InT* __restrict__ x,
                                                             uint16_t* __restrict__ xb,
                                                             float* __restrict__ xbd, int M,
                                                             int TP, int nb,
                                                             const float* __restrict__ gamma,
                                                             const float* __restrict__ r) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const unsigned group_mask = 0xFu << (lane & ~3);
  const int64_t nblocks = static_cast<int64_t>(TP) * nb;  // rows M..TP-1 are zero padding
  const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 2;
  for (int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
       blk < nblocks; blk += stride) {
    const int m = static_cast<int>(blk / nb);
    const int b = static_cast<int>(blk - static_cast<int64_t>(m) * nb);
    const int64_t off = blk * kQK + sub * 8;
    int q[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float d = 0.0f;
    if (m >= M) {
      // padding token: zero codes and scale
    } else if constexpr (kCodes) {
      const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const int8_t*>(x) + off);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        q[i] = static_cast<int8_t>((v.x >> (8 * i)) & 0xFFu);
        q[4 + i] = static_cast<int8_t>((v.y >> (8 * i)) & 0xFFu);
      }
    } else {
      float v[8];
      if constexpr (sizeof(InT) == 2) {
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + off), v);
      } else {
        const float4 a = reinterpret_cast<const float4*>(x + off)[0];
        const float4 c = reinterpret_cast<const float4*>(x + off)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
      }
      if (gamma != nullptr) {
        const int k = b * kQK + sub * 8;
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma + k));
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma + k) + 1);
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], g[i]);
      }
      d = quantize_block_x4(v, group_mask, q);
      if (r != nullptr) {
        pdl_wait();  // r comes from the row-RMS kernel this one may overlap
        d = __fmul_rn(d, r[m]);
      }
    }
    const int p0 = 2 * (sub & 1);
    {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 t = __halves2half2(__int2half_rn(q[2 * i]), __int2half_rn(q[2 * i + 1]));
        h[i] = *reinterpret_cast<const uint32_t*>(&t);
      }
      uint16_t* dst = xb + (static_cast<int64_t>(b) * TP + m) * 32;
      const int hoff = (sub >> 1) * 4;  // halves: piece p at 8 p, second half +4
      *reinterpret_cast<uint2*>(dst + 8 * p0 + hoff) = make_uint2(h[0], h[1]);
      *reinterpret_cast<uint2*>(dst + 8 * (p0 + 1) + hoff) = make_uint2(h[2], h[3]);
    }
    if constexpr (!kCodes)
      if (sub == 0) xbd[static_cast<int64_t>(b) * TP + m] = d;
  }
}

// ---- host ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

struct BatchPlan {
  int RG = 0, S = 0, grid = 0, KPall = 1, cb = kChunkBlocks;
  uint32_t stage = 0, off_w1 = 0, off_wd = 0, off_x = 0, off_xd = 0;
  size_t smem = 0;
};

uint32_t up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// The consumers' block split: a row group served by more warps than it has token groups
// splits each chunk's blocks among them (kp layers).  Must match the kernel's mapping.
int kp_layers(int RG, int TG, int cb) {
  int all = 1;
  for (int r = 0; r < RG; ++r) {
    const int nwr = (kConsumerWarps - 1 - r) / RG + 1;
    if (TG < nwr) {
      int k = nwr / TG;
      if (k > cb) k = cb;
      if (k > all) all = k;
    }
  }
  return all;
}

// The plan for chunks of cb blocks (empty: the shape or the ring does not fit).
BatchPlan batch_plan_cb(int64_t M, int64_t N, int64_t K, int cb_blocks, const DeviceInfo& dev) {
  BatchPlan pl;
  if (M < 1 || M > kBatchMaxM || N < 1 || K < kQK * cb_blocks || K % (kQK * cb_blocks) != 0 ||
      dev.sm_count < 1)
    return pl;
  const int64_t groups = (N + 15) / 16;
  const int64_t RG = (groups + dev.sm_count - 1) / dev.sm_count;
  if (RG > kMaxRG) return pl;
  const uint32_t rows = static_cast<uint32_t>(16 * RG);
  const uint32_t m = static_cast<uint32_t>(M);
  pl.RG = static_cast<int>(RG);
  pl.grid = static_cast<int>((groups + RG - 1) / RG);
  pl.cb = cb_blocks;
  const uint32_t cb = static_cast<uint32_t>(cb_blocks);
  pl.off_w1 = rows * 128;                               // multiple of 2048: swizzle atoms aligned
  pl.off_wd = cb / 4 * rows * 128;                      // after the chunk's 128-byte weight boxes
  pl.off_x = pl.off_wd + rows * cb * 2;                 // 16-byte aligned
  const uint32_t tp = 8 * ((m + 7) / 8);  // tokens padded to whole groups of 8
  pl.off_xd = pl.off_x + cb * tp * 64;
  pl.stage = up(pl.off_xd + cb * tp * 4, 1024);
  pl.KPall = kp_layers(pl.RG, static_cast<int>((M + 7) / 8), pl.cb);
  const size_t red = static_cast<size_t>(pl.KPall) * rows * tp * 4;  // partial-sum layers
  const size_t budget = static_cast<size_t>(dev.max_smem_optin) - 2048 - 1024;
  int S = static_cast<int>((kRingTarget + pl.stage - 1) / pl.stage);
  if (S < 2) S = 2;
  if (S > kMaxStages) S = kMaxStages;
  while (S > 2 && static_cast<size_t>(S) * pl.stage > budget) --S;
  size_t ring = static_cast<size_t>(S) * pl.stage;
  if (ring > budget) return BatchPlan{};
  if (ring < red) ring = red;
  if (ring > budget) return BatchPlan{};
  pl.S = S;
  pl.smem = ring + 1024;
  return pl;
}

// Chunks of 16 blocks where K allows and the ring still holds 3 stages, else of 8.
BatchPlan batch_plan(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  if (K % (kQK * kMaxChunkBlocks) == 0) {
    const BatchPlan wide = batch_plan_cb(M, N, K, kMaxChunkBlocks, dev);
    if (wide.smem != 0 && wide.S >= 3) return wide;
  }
  return batch_plan_cb(M, N, K, kChunkBlocks, dev);
}

template <bool kBS, int kNTG, bool kFused = false>
cudaError_t launch_batch_kernel(const CUtensorMap& tw, const CUtensorMap& ts, const BatchParams& p,
                                int grid, size_t smem, cudaStream_t stream, int dev_id) {
  auto fn = batch_kernel<kBS, kNTG, kFused>;
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
  return cudaLaunchKernelEx(&cfg, fn, tw, ts, p);
}

}  // namespace

bool batch_supported(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  return batch_plan(M, N, K, dev).smem != 0;
}

size_t batch_ws_bytes(int64_t M, int64_t K) {
  const size_t nbm = static_cast<size_t>(K / kQK) * static_cast<size_t>((M + 7) / 8 * 8);
  return ((nbm * 64 + 255) & ~static_cast<size_t>(255)) + ((nbm * 4 + 255) & ~static_cast<size_t>(255));
}

cudaError_t launch_batch(const void* x, int xtype, const int8_t* xq_in, const int8_t* Wq,
                         const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                         int64_t K, void* ws, const DeviceInfo& dev, cudaStream_t stream,
                         const Epilogue& epi, const Prologue& pro) {
  if (M == 0 || N == 0) return cudaSuccess;
  const BatchPlan pl = batch_plan(M, N, K, dev);
  if (pl.smem == 0 || ws == nullptr) return cudaErrorInvalidValue;
  const bool bs = isum != nullptr;
  const int64_t nb = K / kQK;
  const int64_t TP = (M + 7) / 8 * 8;
  const size_t nbm = static_cast<size_t>(nb) * static_cast<size_t>(TP);
  uint16_t* xb = static_cast<uint16_t*>(ws);
  float* xbd = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                        ((nbm * 64 + 255) & ~static_cast<size_t>(255)));
  // 1. activations -> fragment-ordered binary16 codes and scales
  {
    const int64_t threads = static_cast<int64_t>(nbm) * 4;  // 4 lanes per block
    int blocks = static_cast<int>((threads + 255) / 256);
    const int cap = 8 * dev.sm_count;
    if (blocks > cap) blocks = cap;
    if (bs)
      quantize_batch_kernel<int8_t, true><<<blocks, 256, 0, stream>>>(
          xq_in, xb, xbd, static_cast<int>(M), static_cast<int>(TP), static_cast<int>(nb), nullptr,
          nullptr);
    else if (pro.r == nullptr && xtype == 1)
      quantize_batch_kernel<uint16_t, false><<<blocks, 256, 0, stream>>>(
          static_cast<const uint16_t*>(x), xb, xbd, static_cast<int>(M), static_cast<int>(TP),
          static_cast<int>(nb), pro.gamma, nullptr);
    else if (pro.r == nullptr)
      quantize_batch_kernel<float, false><<<blocks, 256, 0, stream>>>(
          static_cast<const float*>(x), xb, xbd, static_cast<int>(M), static_cast<int>(TP),
          static_cast<int>(nb), pro.gamma, nullptr);
    else {
      // after the row-RMS kernel (a normal launch, so x is complete when it starts): start
      // early and wait for it only before reading r
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(blocks);
      cfg.blockDim = dim3(256);
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const int iM = static_cast<int>(M), iTP = static_cast<int>(TP), inb = static_cast<int>(nb);
      cudaError_t e =
          xtype == 1
              ? cudaLaunchKernelEx(&cfg, quantize_batch_kernel<uint16_t, false>,
                                   static_cast<const uint16_t*>(x), xb, xbd, iM, iTP, inb, pro.gamma, pro.r)
              : cudaLaunchKernelEx(&cfg, quantize_batch_kernel<float, false>,
                                   static_cast<const float*>(x), xb, xbd, iM, iTP, inb, pro.gamma, pro.r);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2. tensor maps of the weight codes and scales; box = the CTA's 16 RG rows
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorInvalidValue;
  const cuuint32_t rows = static_cast<cuuint32_t>(16 * pl.RG);
  CUtensorMap tw, ts;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {128, rows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(Wq), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(pl.cb), rows};
    const cuuint32_t es[2] = {1, 1};
    // block-sum mode reads no scales; the map still needs a valid address
    const void* base = bs ? static_cast<const void*>(Wq) : static_cast<const void*>(Wd);
    if (enc(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  BatchParams p;
  p.xb = xb;
  p.xbd = xbd;
  p.y = y;
  p.isum = isum;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.RG = pl.RG;
  p.KPall = pl.KPall;
  p.stages = pl.S;
  p.cb = pl.cb;
  p.stage_bytes = pl.stage;
  p.off_w1 = pl.off_w1;
  p.off_wd = pl.off_wd;
  p.off_x = pl.off_x;
  p.off_xd = pl.off_xd;
  p.err = dev.err_word;
  p.epi = epi;
  // token groups per warp: at most ceil(TG / warps of a row group)
  const int TG = static_cast<int>((M + 7) / 8);
  int ntg_max = 1;
  for (int r = 0; r < pl.RG; ++r) {
    const int nwr = (kConsumerWarps - 1 - r) / pl.RG + 1;
    if (TG >= nwr && (TG + nwr - 1) / nwr > ntg_max) ntg_max = (TG + nwr - 1) / nwr;
  }
  if (bs) {
    if (ntg_max <= 1) return launch_batch_kernel<true, 1>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
    if (ntg_max <= 2) return launch_batch_kernel<true, 2>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
    if (ntg_max <= 4) return launch_batch_kernel<true, 4>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
    return launch_batch_kernel<true, 8>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
  }
  if (!epi.plain()) {
    if (ntg_max <= 1) return launch_batch_kernel<false, 1, true>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
    if (ntg_max <= 2) return launch_batch_kernel<false, 2, true>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
    if (ntg_max <= 4) return launch_batch_kernel<false, 4, true>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
    return launch_batch_kernel<false, 8, true>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
  }
  if (ntg_max <= 1) return launch_batch_kernel<false, 1>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
  if (ntg_max <= 2) return launch_batch_kernel<false, 2>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
  if (ntg_max <= 4) return launch_batch_kernel<false, 4>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
  return launch_batch_kernel<false, 8>(tw, ts, p, pl.grid, pl.smem, stream, dev.device);
}

}  // namespace q8
