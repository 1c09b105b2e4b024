// q8_bsa.cu -- block-sparse causal attention for long prefill (MInference-style) on the
// fifth-generation tensor cores.
//
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, feature list) speeds up long prefill with
// MInference-style block-sparse attention.  The operation here (readings of the post):
// query t of head h attends, causally, to the keys of the 64-token key blocks listed for
// its 64-token query block (CSR per head and query block); H query heads share Hkv
// key/value heads (head h reads h / (H / Hkv)); o_t = softmax(q_t . k / sqrt(d)) v over the
// visible keys, d = 128; a query that sees no key gets 0.
//
// Design (one CTA per head and query block, 64 query rows, two CTAs per SM):
//  - warp 0 (one thread) loads the Q tile once and, per listed key block, the K tile
//    (64 x 128 bfloat16, two 64-column boxes with 128-byte swizzle) by TMA into a two-stage
//    ring; warp 6 (one thread) loads the V tiles into another two-stage ring;
//  - warp 1 (one thread) issues the tcgen05 MMAs: S_j = Q K_j^T (M = 64, N = 64, eight
//    K = 16 steps) into one of two S buffers in TMEM, and O += P_j V_j (M = 64, N = 128,
//    four K = 16 steps, V read in place as an MN-major operand) into the O accumulator in
//    TMEM.  One group per key block: once the softmax warps have written P_j (so they have
//    read S_j), S_{j+2} (into S_j's buffer) and PV_j are issued together and committed to one
//    of two alternating barriers; S_{j+2} is then ready a whole block ahead of its use;
//  - warps 2-5 (the four TMEM lane quarters; an M = 64 accumulator keeps rows 16q .. 16q+15
//    in the first 16 lanes of quarter q) run the online softmax, waiting once per block: each
//    row is split over two threads (32 keys each), base-2 exponentials, P rounded to bfloat16
//    into one of two swizzled shared-memory tiles that the PV MMA reads as its A operand.
//    The running maximum used as the exponent reference moves only when a row's maximum
//    rises by more than 2^8; then that warp waits for the previous PV and rescales its rows
//    of O in TMEM, so most blocks need no correction of O at all; the weights stay <= 2^8
//    and the final o = O / l is unchanged.
// The grid runs key/value head by key/value head, and within one the query blocks from the
// last (most key blocks) to the first, the heads of a group side by side: the K and V tiles
// of the key/value head in flight (16 MB at 32K tokens) stay in L2 across the query blocks
// and heads that list them.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <mutex>

#include "q8_internal.h"
#include "q8_ptx.cuh"

namespace q8 {
namespace {

constexpr int kBlk = 64;     // tokens per query and key block
constexpr int kD = 128;      // head dim
constexpr int kThreads = 224;  // warps: 0 K/Q loads, 1 MMA, 2-5 softmax, 6 V loads
constexpr uint32_t kTileBytes = kBlk * kD * 2;  // 16 KB: two 64 x 64 swizzled boxes
constexpr uint32_t kBoxBytes = kTileBytes / 2;
constexpr uint32_t kPBytes = kBlk * kBlk * 2;   // 8 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + 2 * kTileBytes;  // two stages each
constexpr uint32_t kOffP = kOffV + 2 * kTileBytes;  // two buffers
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
constexpr uint32_t kSmemBytes = kOffBar + 128;  // barriers, TMEM address, abort flag
// two CTAs (and the runtime's 1 KB each) in the SM's 228 KB; the kernel checks that its
// dynamic shared memory starts on a 1024-byte boundary (the 128-byte swizzle atoms of the
// TMA tiles and MMA operands need it)
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t kTmemCols = 256;  // S buffers at columns 0 and 64, O at 128 .. 255
constexpr uint32_t kColO = 128;
constexpr float kRescaleLog2 = 8.0f;  // move the exponent reference when the max gains > 2^8
constexpr uint32_t kErrBadBlock = 1u << 8;  // a listed key block outside [0, query block]

struct BsaParams {
  const int32_t* row_ptr;  // [H * nqb + 1]
  const int32_t* col_idx;  // [nnz]
  int64_t nnz;
  void* o;             // [H][T][d] f32 or bf16
  int otype;
  int H, Hkv, T;
  float scale_log2;    // log2(e) / sqrt(d)
  uint32_t* err;
};

// tcgen05 instruction descriptor, kind::f16 with bfloat16 A and B, f32 D; A and B K-major,
// or (a_mn, b_mn) MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// Shared-memory descriptor of an MN-major operand with 128-byte swizzle: 64-element-wide
// atoms of 8 K rows (1024 bytes); lbo = byte stride between atoms along MN, sbo = between
// 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 16 TMEM lanes x 32 columns, twice: thread i < 16 gets lane (base + i), columns
// col .. col+31; thread i >= 16 gets lane (base + i - 16), columns col+kSplit .. +31.
template <int kSplit>
__device__ __forceinline__ void tmem_ld_16x32bx2_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32], %33;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr), "n"(kSplit)
      : "memory");
}

template <int kSplit>
__device__ __forceinline__ void tmem_st_16x32bx2_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, "
      "{%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, "
      "%18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33};" ::"r"(taddr),
      "n"(kSplit), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
      "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
      "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the special-function unit (hardware approximation, subnormals flushed; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// the i-th listed key block of a row, or -1 if it lies outside [0, qb]
__device__ __forceinline__ int listed_block(const int32_t* col_idx, int64_t e, int qb) {
  const int kb = __ldg(col_idx + e);
  return (kb >= 0 && kb <= qb) ? kb : -1;
}

// every lane of the warp waits; the warp leaves together if any lane's wait gave up
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag));
}

__global__ void __launch_bounds__(kThreads, 2)
    bsa_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const BsaParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  if ((smem_u32(sm) & 1023u) != 0) {  // the whole CTA leaves before touching anything
    if (threadIdx.x == 0 && p.err != nullptr) atomicOr(p.err, kErrBadLaunch);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2] K tile landed
  uint64_t* v_full = bars + 3;   // [2] V tile landed
  uint64_t* grp = bars + 5;      // [2] MMA group c done (c = 0: S_0, S_1; c = j + 1: S_{j+2}, PV_j)
  uint64_t* p_full = bars + 7;   // [2] P_j written (S_j read, O rescaled if needed): 4 arrivals
  uint64_t* end_bar = bars + 9;
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(sm + kOffBar + 96);
  int& abort_flag = *reinterpret_cast<int*>(sm + kOffBar + 100);

  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int nqb = p.T / kBlk, G = p.H / p.Hkv;
  const int per_kv = G * nqb;
  const int bid = static_cast<int>(blockIdx.x);
  const int hk = bid / per_kv, rem = bid - hk * per_kv;
  const int qb = nqb - 1 - rem / G;
  const int h = hk * G + rem % G;
  const int64_t rowi = static_cast<int64_t>(h) * nqb + qb;
  const int64_t e0 = p.row_ptr[rowi];
  int64_t e1 = p.row_ptr[rowi + 1];
  if (e1 > p.nnz) e1 = p.nnz;
  const int64_t eend = (e1 > e0 && e0 >= 0) ? e1 : e0;  // a malformed row lists nothing

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&grp[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(end_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  // MMA group c completes grp[c % 2] for the (c / 2)-th time
  auto grp_wait = [&](int c, bool warp_wide) -> bool {
    uint64_t* b = &grp[c & 1];
    const uint32_t par = static_cast<uint32_t>(c >> 1) & 1;
    return warp_wide ? warp_wait(b, par, &abort_flag) : mbar_wait(b, par, &abort_flag);
  };

  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers: warp 0 Q and K, warp 6 V ----------------
    if (lane == 0) {
      const bool isK = warp == 0;
      const CUtensorMap* map = isK ? &tmK : &tmV;
      uint64_t* full = isK ? k_full : v_full;
      uint8_t* ring = sm + (isK ? kOffK : kOffV);
      tma_prefetch_desc(map);
      if (isK) {
        tma_prefetch_desc(&tmQ);
        const int32_t qrow = h * p.T + qb * kBlk;
        mbar_arrive_expect_tx(q_full, kTileBytes);
        tma_load_2d(sm + kOffQ, &tmQ, q_full, 0, qrow);
        tma_load_2d(sm + kOffQ + kBoxBytes, &tmQ, q_full, 64, qrow);
      }
      int lastpar[2] = {-1, -1};
      bool ok = true;
      int j = 0;
      for (int64_t e = e0; e < eend; ++e) {
        const int kb = listed_block(p.col_idx, e, qb);
        if (kb < 0) {
          if (isK && p.err != nullptr) atomicOr(p.err, kErrBadBlock);
          continue;
        }
        const int st = j & 1;
        // the stage's previous tile (j - 2) is used: S_{j-2} is in group max(j - 3, 0), PV_{j-2}
        // in group j - 1
        if (j >= 2 && !grp_wait(isK ? (j >= 4 ? j - 3 : 0) : j - 1, false)) {
          ok = false;
          break;
        }
        const int32_t krow = hk * p.T + kb * kBlk;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        tma_load_2d(ring + st * kTileBytes, map, &full[st], 0, krow);
        tma_load_2d(ring + st * kTileBytes + kBoxBytes, map, &full[st], 64, krow);
        lastpar[st] = (j >> 1) & 1;
        ++j;
      }
      if (!ok) report_error(p.err, kErrWaitTimeout, &abort_flag);
      // no copy may still be landing in shared memory when the CTA ends
      if (isK) mbar_wait(q_full, 0, nullptr);
      for (int st = 0; st < 2; ++st)
        if (lastpar[st] >= 0) mbar_wait(&full[st], static_cast<uint32_t>(lastpar[st]), nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int n = 0;
      for (int64_t e = e0; e < eend; ++e) n += listed_block(p.col_idx, e, qb) >= 0 ? 1 : 0;
      const uint32_t sQ = smem_u32(sm + kOffQ), sP = smem_u32(sm + kOffP);
      // S = Q K^T: M = 64 queries, N = 64 keys.  O += P V: M = 64, N = 128 (head dim), V read
      // in place as the MN-major B operand.
      constexpr uint32_t idS = idesc_bf16(kBlk, kBlk, 0, 0), idO = idesc_bf16(kBlk, kD, 0, 1);
      // Operand descriptors are built once: a K step or another stage only moves the start
      // address, which the descriptor holds in 16-byte units in its low bits (shared-memory
      // addresses stay below 256 KB, so the sum never carries out of that field).
      const uint64_t dQ = sdesc_k_sw128(sQ), dK0 = sdesc_k_sw128(smem_u32(sm + kOffK));
      const uint64_t dP0 = sdesc_k_sw128(sP);
      const uint64_t dV0 = sdesc_mn_sw128(smem_u32(sm + kOffV), kBoxBytes, 1024);
      auto issue_s = [&](int i) -> bool {  // S_i into S buffer i % 2 (K_i in stage i % 2)
        const int st = i & 1;
        if (!mbar_wait(&k_full[st], static_cast<uint32_t>(i >> 1) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint64_t dK = dK0 + static_cast<uint64_t>(st) * (kTileBytes >> 4);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t off = static_cast<uint64_t>(((s >> 2) * kBoxBytes + (s & 3) * 32) >> 4);
          mma_f16_ss(tbase + static_cast<uint32_t>(st * kBlk), dQ + off, dK + off, idS, s > 0 ? 1u : 0u);
        }
        return true;
      };
      bool ok = true;
      if (n > 0) {
        ok = mbar_wait(q_full, 0, &abort_flag) && issue_s(0) && (n < 2 || issue_s(1));
        if (ok) mma_commit(&grp[0]);  // group 0
      }
      for (int j = 0; ok && j < n; ++j) {
        // P_j is written, so S_j has been read: its buffer takes S_{j+2}
        const int b = j & 1;
        const uint32_t par = static_cast<uint32_t>(j >> 1) & 1;
        if (!mbar_wait(&p_full[b], par, &abort_flag) || (j + 2 < n && !issue_s(j + 2)) ||
            !mbar_wait(&v_full[b], par, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dV = dV0 + static_cast<uint64_t>(b) * (kTileBytes >> 4);
        const uint64_t dP = dP0 + static_cast<uint64_t>(b) * (kPBytes >> 4);
#pragma unroll
        for (int s = 0; s < 4; ++s)  // 16 keys per step: 32 bytes along a P row, 16 rows of V
          mma_f16_ss(tbase + kColO, dP + static_cast<uint64_t>(s * 2), dV + static_cast<uint64_t>(s * 128), idO,
                     (j > 0 || s > 0) ? 1u : 0u);
        mma_commit(&grp[(j + 1) & 1]);  // group j + 1
      }
      if (!ok) report_error(p.err, kErrWaitTimeout, &abort_flag);
      // every MMA issued has finished before the CTA frees TMEM and shared memory
      mma_commit(end_bar);
      mbar_wait(end_bar, 0, nullptr);
    }
  } else {
    // ---------------- online softmax, O correction, output ----------------
    const int qd = warp & 3;              // TMEM lane quarter this warp may access
    const int hf = lane >> 4;             // keys 32 hf .. +31, output columns 64 hf .. +63
    const int r = 16 * qd + (lane & 15);  // query row within the block
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * qd) << 16);
    const float sl2 = p.scale_log2;
    float ref = -INFINITY, l = 0.0f;
    bool ok = true;
    int j = 0;
    for (int64_t e = e0; e < eend; ++e) {
      const int kb = listed_block(p.col_idx, e, qb);
      if (kb < 0) continue;
      const int sb = j & 1;
      // S_j is in group max(j - 1, 0), which also finished PV_{j-2} with P buffer j % 2
      if (!grp_wait(j > 0 ? j - 1 : 0, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld_16x32bx2_x32<32>(tl + static_cast<uint32_t>(sb * kBlk), sr);
      tmem_ld_wait();
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(sr[i]);
      if (kb == qb) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (32 * hf + i > r) x[i] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int i = 1; i < 32; ++i) mx = fmaxf(mx, x[i]);
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
      const float mn = mx * sl2;
      const bool resc = mn > ref + kRescaleLog2;  // always on a row's first block
      float alpha = 1.0f;
      if (resc) {
        alpha = ex2(ref - mn);  // 0 on the first block
        ref = mn;
      }
      float sum = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = ex2(fmaf(x[i], sl2, -ref));
        sum += x[i];
      }
      l = fmaf(l, alpha, sum);
      uint8_t* prow = sm + kOffP + sb * kPBytes + r * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int chunk = 4 * hf + c;
        uint4 v;
        v.x = pack_bf16(x[8 * c + 0], x[8 * c + 1]);
        v.y = pack_bf16(x[8 * c + 2], x[8 * c + 3]);
        v.z = pack_bf16(x[8 * c + 4], x[8 * c + 5]);
        v.w = pack_bf16(x[8 * c + 6], x[8 * c + 7]);
        *reinterpret_cast<uint4*>(prow + ((chunk ^ (r & 7)) << 4)) = v;
      }
      if (j > 0 && __any_sync(0xFFFFFFFFu, resc)) {
        // a row's reference moved: once PV_{j-1} (group j) is in, scale its O by alpha (rows
        // that kept theirs have alpha 1)
        if (!grp_wait(j, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t o[32];
          tmem_ld_16x32bx2_x32<64>(tl + kColO + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_16x32bx2_x32<64>(tl + kColO + c0, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
      ++j;
    }
    if (!ok) report_error(p.err, kErrWaitTimeout, &abort_flag);
    const float lt = l + __shfl_xor_sync(0xFFFFFFFFu, l, 16);
    bool have = false;
    if (ok && j > 0) {
      have = grp_wait(j, true);  // group j holds the last PV
      if (!have) report_error(p.err, kErrWaitTimeout, &abort_flag);
      tc_fence_after();
    }
    const float inv = (have && lt > 0.0f) ? 1.0f / lt : 0.0f;
    const int64_t orow = static_cast<int64_t>(h) * p.T + static_cast<int64_t>(qb) * kBlk + r;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t o[32];
      if (have) {
        tmem_ld_16x32bx2_x32<64>(tl + kColO + c0, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;  // no visible key (or an abandoned wait): 0
      }
      const int col = 64 * hf + c0;
      if (p.otype == 1) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow * kD + col);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
          v.y = pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
          v.z = pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
          v.w = pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
          dst[c] = v;
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * kD + col);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_float4(__uint_as_float(o[4 * c + 0]) * inv, __uint_as_float(o[4 * c + 1]) * inv,
                               __uint_as_float(o[4 * c + 2]) * inv, __uint_as_float(o[4 * c + 3]) * inv);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

// ---- host ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn bsa_encode_fn() {
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

// [rows][128] bfloat16, loaded as 64 x 64 boxes with 128-byte swizzle
bool encode_head_rows(CUtensorMap* map, const void* ptr, uint64_t rows) {
  EncodeTiledFn enc = bsa_encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlk)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_bsa(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* row_ptr, const int32_t* col_idx, int64_t nnz, void* o,
                       int otype, int64_t H, int64_t Hkv, int64_t T, const DeviceInfo& dev,
                       cudaStream_t stream) {
  if (H == 0 || T == 0) return cudaSuccess;
  // TMA row coordinates are 32-bit
  if (H * T > 0x7FFFFFFF || Hkv * T > 0x7FFFFFFF) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (!encode_head_rows(&mq, q, static_cast<uint64_t>(H * T)) ||
      !encode_head_rows(&mk, k, static_cast<uint64_t>(Hkv * T)) ||
      !encode_head_rows(&mv, v, static_cast<uint64_t>(Hkv * T)))
    return cudaErrorInvalidValue;
  BsaParams p;
  p.row_ptr = row_ptr;
  p.col_idx = col_idx;
  p.nnz = nnz;
  p.o = o;
  p.otype = otype;
  p.H = static_cast<int>(H);
  p.Hkv = static_cast<int>(Hkv);
  p.T = static_cast<int>(T);
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  p.err = dev.err_word;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(bsa_tc_kernel), kSmemBytes, dev.device);
  if (e != cudaSuccess) return e;
  const int64_t grid = H * (T / kBlk);
  bsa_tc_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace q8
