// q8_bsa.cu -- block-sparse causal attention for long prefill (MInference-style).
//
// "CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
// (CMP 100-210)" (news.hada.io topic 29953, feature list) speeds up long prefill with
// MInference-style block-sparse attention.  The operation here (readings of the post):
// query t of head h attends, causally, to the keys of the 64-token key blocks listed for
// its 64-token query block (CSR per head and query block); H query heads share Hkv
// key/value heads (head h reads h / (H / Hkv)); o_t = softmax(q_t . k / sqrt(d)) v over the
// visible keys, d = 128; a query that sees no key gets 0.
//
// Design: one CTA of four warps per (head, query block); warp w owns query rows
// 16 w .. 16 w + 15.  The Q tile stays in registers as mma.sync A fragments; each listed
// key block's K and V tiles (64 x 128 bf16 each) are copied into shared memory with
// cp.async, double-buffered, rows XOR-swizzled in 16-byte chunks so ldmatrix reads are
// conflict-free.  Per key block: S = Q K^T (64 mma.sync m16n8k16 per warp, fp32), causal
// mask on the diagonal block, online softmax in base 2 (running max and sum per row),
// then O += P V with P rounded to bf16 (64 more mma.sync per warp).  Query blocks are
// scheduled from the last (most key blocks) to the first.
#include <cuda_bf16.h>

#include <cstdint>

#include "q8_internal.h"
#include "q8_ptx.cuh"

namespace q8 {
namespace {

constexpr int kBlk = 64;     // tokens per query and key block
constexpr int kD = 128;      // head dim
constexpr int kRowBytes = kD * 2;
constexpr int kTile = kBlk * kRowBytes;  // 16 KB
constexpr int kThreads = 128;
constexpr uint32_t kErrBadBlock = 1u << 8;  // a listed key block outside [0, query block]

struct BsaParams {
  const uint16_t* q;   // [H][T][d]
  const uint16_t* k;   // [Hkv][T][d]
  const uint16_t* v;
  const int32_t* row_ptr;  // [H * nqb + 1]
  const int32_t* col_idx;  // [nnz]
  int64_t nnz;
  void* o;             // [H][T][d] f32 or bf16
  int otype;
  int H, Hkv, T;
  float scale_log2;    // log2(e) / sqrt(d)
  uint32_t* err;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a tile
  return static_cast<uint32_t>(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// a 64 x 128 bf16 tile (rows of 256 bytes) into shared memory, swizzled
__device__ __forceinline__ void load_tile(uint32_t smem, const uint16_t* g, int tid) {
#pragma unroll
  for (int i = 0; i < (kBlk * 16) / kThreads; ++i) {
    const int idx = tid + kThreads * i;
    const int row = idx >> 4, chunk = idx & 15;
    cp_async16(smem + swz(row, chunk), g + row * kD + chunk * 8);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 2) bsa_kernel(const BsaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int nqb = p.T / kBlk;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x / p.H);  // most key blocks first
  const int h = static_cast<int>(blockIdx.x % p.H);
  const int hk = h / (p.H / p.Hkv);
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + kTile;  // [2][K tile, V tile]

  const int64_t e0 = p.row_ptr[static_cast<int64_t>(h) * nqb + qb];
  int64_t e1 = p.row_ptr[static_cast<int64_t>(h) * nqb + qb + 1];
  if (e1 > p.nnz) e1 = p.nnz;
  const int64_t nlist = e1 > e0 && e0 >= 0 ? e1 - e0 : 0;

  const uint16_t* kbase = p.k + static_cast<int64_t>(hk) * p.T * kD;
  const uint16_t* vbase = p.v + static_cast<int64_t>(hk) * p.T * kD;
  // the i-th listed key block, or -1 if the entry is outside [0, qb] (then skipped)
  auto listed = [&](int64_t i) -> int {
    const int kb = p.col_idx[e0 + i];
    return (kb >= 0 && kb <= qb) ? kb : -1;
  };

  // Q tile -> shared -> A fragments (rows 16 warp .. +15, all of d)
  load_tile(sQ, p.q + (static_cast<int64_t>(h) * p.T + static_cast<int64_t>(qb) * kBlk) * kD, tid);
  asm volatile("cp.async.commit_group;" ::: "memory");
  if (nlist > 0) {
    const int kb = listed(0);
    if (kb >= 0) {
      load_tile(sKV, kbase + static_cast<int64_t>(kb) * kBlk * kD, tid);
      load_tile(sKV + kTile, vbase + static_cast<int64_t>(kb) * kBlk * kD, tid);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 1;" ::: "memory");
  __syncthreads();
  uint32_t qa[8][4];
#pragma unroll
  for (int kc = 0; kc < 8; ++kc) {
    const int row = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
    const int chunk = 2 * kc + (lane >> 4);
    ldsm_x4(sQ + swz(row, chunk), qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3]);
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // rows g and g + 8
  const int qrow0 = 16 * warp + g, qrow1 = qrow0 + 8;         // rows within the block

  for (int64_t it = 0; it < nlist; ++it) {
    const int buf = static_cast<int>(it & 1);
    const int kb = listed(it);
    if (it + 1 < nlist) {  // next block's tiles while this one is used
      const int kn = listed(it + 1);
      const uint32_t nb = sKV + static_cast<uint32_t>((buf ^ 1) * 2 * kTile);
      if (kn >= 0) {
        load_tile(nb, kbase + static_cast<int64_t>(kn) * kBlk * kD, tid);
        load_tile(nb + kTile, vbase + static_cast<int64_t>(kn) * kBlk * kD, tid);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    if (kb < 0) {
      if (tid == 0 && p.err != nullptr) atomicOr(p.err, kErrBadBlock);
      __syncthreads();
      continue;
    }
    const uint32_t sK = sKV + static_cast<uint32_t>(buf * 2 * kTile), sV = sK + kTile;

    // S = Q K^T: 8 key n-tiles of 8 keys, 8 d chunks of 16
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int kc = 0; kc < 8; kc += 2) {
        uint32_t b0, b1, b2, b3;  // d chunks kc and kc + 1 of keys 8 nt .. 8 nt + 7
        ldsm_x4(sK + swz(8 * nt + (lane & 7), 2 * kc + (lane >> 3)), b0, b1, b2, b3);
        mma_bf16(s[nt], qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b0, b1);
        mma_bf16(s[nt], qa[kc + 1][0], qa[kc + 1][1], qa[kc + 1][2], qa[kc + 1][3], b2, b3);
      }
    }
    // scale to base 2; causal mask on the diagonal block
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = 8 * nt + 2 * tig + j;
        float a = s[nt][j] * p.scale_log2, b = s[nt][2 + j] * p.scale_log2;
        if (kb == qb && key > qrow0) a = -INFINITY;
        if (kb == qb && key > qrow1) b = -INFINITY;
        s[nt][j] = a;
        s[nt][2 + j] = b;
        mx0 = fmaxf(mx0, a);
        mx1 = fmaxf(mx1, b);
      }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    // rows that have seen no key yet keep a finite reference (their terms are all zero)
    const float ref0 = mn0 == -INFINITY ? 0.0f : mn0, ref1 = mn1 == -INFINITY ? 0.0f : mn1;
    const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);  // exp2(-inf) = 0
    m0 = mn0;
    m1 = mn1;
    float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - ref0);
      s[nt][1] = exp2f(s[nt][1] - ref0);
      s[nt][2] = exp2f(s[nt][2] - ref1);
      s[nt][3] = exp2f(s[nt][3] - ref1);
      sum0 += s[nt][0] + s[nt][1];
      sum1 += s[nt][2] + s[nt][3];
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      sum0 += __shfl_xor_sync(0xFFFFFFFFu, sum0, off);
      sum1 += __shfl_xor_sync(0xFFFFFFFFu, sum1, off);
    }
    l0 = l0 * al0 + sum0;
    l1 = l1 * al1 + sum1;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      o[dn][0] *= al0;
      o[dn][1] *= al0;
      o[dn][2] *= al1;
      o[dn][3] *= al1;
    }
    // O += P V: 4 key chunks of 16, 16 d n-tiles of 8
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t a0 = pack_bf16(s[2 * j][0], s[2 * j][1]);
      const uint32_t a1 = pack_bf16(s[2 * j][2], s[2 * j][3]);
      const uint32_t a2 = pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]);
      const uint32_t a3 = pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3]);
#pragma unroll
      for (int dn = 0; dn < 16; dn += 2) {
        uint32_t b0, b1, b2, b3;  // keys 16 j .. +15 of d n-tiles dn and dn + 1
        const int row = 16 * j + (lane & 7) + 8 * ((lane >> 3) & 1);
        ldsm_x4_t(sV + swz(row, dn + (lane >> 4)), b0, b1, b2, b3);
        mma_bf16(o[dn], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[dn + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();  // this buffer is refilled two iterations on
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // O / l -> output (rows without any visible key stay 0)
  const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
  const int64_t t0 = static_cast<int64_t>(qb) * kBlk + qrow0, t1 = t0 + 8;
  const int64_t base0 = (static_cast<int64_t>(h) * p.T + t0) * kD, base1 = (static_cast<int64_t>(h) * p.T + t1) * kD;
#pragma unroll
  for (int dn = 0; dn < 16; ++dn) {
    const int col = 8 * dn + 2 * tig;
    if (p.otype == 1) {
      uint16_t* out = static_cast<uint16_t*>(p.o);
      *reinterpret_cast<uint32_t*>(out + base0 + col) = pack_bf16(o[dn][0] * inv0, o[dn][1] * inv0);
      *reinterpret_cast<uint32_t*>(out + base1 + col) = pack_bf16(o[dn][2] * inv1, o[dn][3] * inv1);
    } else {
      float* out = static_cast<float*>(p.o);
      *reinterpret_cast<float2*>(out + base0 + col) = make_float2(o[dn][0] * inv0, o[dn][1] * inv0);
      *reinterpret_cast<float2*>(out + base1 + col) = make_float2(o[dn][2] * inv1, o[dn][3] * inv1);
    }
  }
}

}  // namespace

size_t bsa_smem_bytes() { return static_cast<size_t>(kTile) * 5; }

cudaError_t launch_bsa(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* row_ptr, const int32_t* col_idx, int64_t nnz, void* o,
                       int otype, int64_t H, int64_t Hkv, int64_t T, const DeviceInfo& dev,
                       cudaStream_t stream) {
  if (H == 0 || T == 0) return cudaSuccess;
  BsaParams p;
  p.q = q;
  p.k = k;
  p.v = v;
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
  const size_t smem = bsa_smem_bytes();
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(bsa_kernel), smem, dev.device);
  if (e != cudaSuccess) return e;
  const int64_t grid = H * (T / kBlk);
  bsa_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace q8
