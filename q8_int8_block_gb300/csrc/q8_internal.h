// q8_internal.h -- launchers shared between the translation units of libq8 (not part of
// the public ABI; include/q8.h is).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace q8 {

constexpr int kQK = 32;  // elements per Q8_0 block

// Fused output step y = op(acc, aux) (see q8_epi.cuh); the default stores acc as binary32.
enum : int { kEpiNone = 0, kEpiAdd = 1, kEpiSiluMul = 2 };
struct Epilogue {
  const float* aux = nullptr;  // [M,N] binary32: the residual (add) or the gate (silu_mul)
  int op = kEpiNone;
  int bf16 = 0;                // 1: y holds bfloat16 bits
#ifdef __CUDACC__
  __host__ __device__
#endif
  bool plain() const { return op == kEpiNone && bf16 == 0; }
};

// RMSNorm fused into the activation quantizer: the codes are those of fl32(x * gamma),
// and the row's scales carry r = 1 / sqrt(mean(x^2) + eps).  gamma == nullptr: no norm.
// r: [M] factors computed beforehand (launch_row_rms), or nullptr where the kernel computes
// them itself (decode kernel).
struct Prologue {
  const float* gamma = nullptr;  // [K] binary32
  const float* r = nullptr;      // [M] binary32
  float eps = 0.0f;
#ifdef __CUDACC__
  __host__ __device__
#endif
  bool on() const { return gamma != nullptr; }
};

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_optin = 0;
  uint32_t* err_word = nullptr;  // device address of the library's error word
};

// ---- q8_api.cu --------------------------------------------------------------------
// Raises kernel `fn`'s dynamic shared-memory limit on `device` (the current device) to at
// least `bytes`, remembering what was set so that repeated launches skip the driver call.
cudaError_t ensure_smem(const void* fn, size_t bytes, int device);
// The kernel's register count per thread (cudaFuncGetAttributes, cached per kernel/device).
cudaError_t kernel_regs(const void* fn, int device, int* regs);
// Drops both caches (q8_release: a later context starts afresh).
void forget_kernel_attributes();
// The current device's checked info (compute capability 10.3, SM count, shared-memory
// limit, the device address of the library's error word), filled on first use per device.
// Returns 0 (Q8_OK) or a q8_status code.
int device_info(DeviceInfo* out);

// ---- q8_noalloc.cu ----------------------------------------------------------------
// Drops the cached device addresses of the static scratch array (q8_release).
void forget_noalloc_scratch();

// ---- q8_quant.cu ------------------------------------------------------------------
// Quantizes `rows` rows of K values (xtype 0 = f32, 1 = bf16 bits) into codes and scales.
//   codes_f16 == false: int8 codes;  true: binary16 codes (exact small integers).
//   scale_f16 == false: binary32 scales;  true: binary16 scale bits.
cudaError_t launch_quantize(const void* x, int xtype, void* codes, bool codes_f16, void* scales,
                            bool scale_f16, int64_t rows, int64_t K, const DeviceInfo& dev,
                            cudaStream_t stream, const Prologue& pro = Prologue());
// r[m] = 1 / sqrt(sum_k x[m,k]^2 / K + eps) in binary32, summed in a fixed order.
cudaError_t launch_row_rms(const void* x, int xtype, int64_t M, int64_t K, float eps, float* r,
                           const DeviceInfo& dev, cudaStream_t stream);

// int8 codes -> binary16 codes (n a multiple of 16).
cudaError_t launch_codes_to_f16(const int8_t* q, uint16_t* out, int64_t n, const DeviceInfo& dev,
                                cudaStream_t stream);

// ---- q8_decode.cu -----------------------------------------------------------------
// Largest M the decode kernel takes.
constexpr int kDecodeMaxM = 8;
// Shared memory the decode kernel needs for M tokens of K (0 if it cannot run).
size_t decode_smem_bytes(int64_t M, int64_t K, const DeviceInfo& dev);
// y = linear(x) (fused activation quantization) or, when isum != nullptr, the raw
// block sums of given codes xq (x ignored; xd ignored).
cudaError_t launch_decode(const void* x, int xtype, const int8_t* xq_in, const int8_t* Wq,
                          const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                          int64_t K, const DeviceInfo& dev, cudaStream_t stream,
                          const Epilogue& epi = Epilogue(), const Prologue& pro = Prologue());

// ---- q8_batch.cu ------------------------------------------------------------------
// Batched decode (2..kBatchMaxM tokens): weight streaming with mma.sync block sums.
constexpr int kBatchMaxM = 64;
// True if the batched kernel can run this shape (K % 256 == 0, N small enough, smem).
bool batch_supported(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
// Scratch: fragment-ordered binary16 activation codes and their scales.
size_t batch_ws_bytes(int64_t M, int64_t K);
// y = linear(x), or (isum != nullptr) the raw block sums of the codes xq_in.
cudaError_t launch_batch(const void* x, int xtype, const int8_t* xq_in, const int8_t* Wq,
                         const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                         int64_t K, void* ws, const DeviceInfo& dev, cudaStream_t stream,
                         const Epilogue& epi = Epilogue(), const Prologue& pro = Prologue());

// ---- q8_dp4a.cu -------------------------------------------------------------------
// The post's design: dp4a int8 GEMM on CUDA cores (prior-art comparison).  xq [M,K] int8,
// xd [M,K/32] f32 from launch_quantize; y [M,N], or isum [M,N,K/32] when isum != nullptr.
cudaError_t launch_dp4a_gemm(const int8_t* xq, const float* xd, const int8_t* Wq,
                             const uint16_t* Wd, float* y, int32_t* isum, int64_t M, int64_t N,
                             int64_t K, cudaStream_t stream, const Epilogue& epi = Epilogue());

// ---- q8_kv3.cu -------------------------------------------------------------------
// 3-bit KV-cache codec (Walsh-Hadamard rotation + Lloyd-Max), 128-element groups.
cudaError_t launch_kv3_encode(const void* x, int xtype, uint32_t* codes, float* scales, int64_t n,
                              const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_kv3_decode(const uint32_t* codes, const float* scales, void* out, int otype,
                              int64_t n, const DeviceInfo& dev, cudaStream_t stream);

// ---- q8_bsa.cu -------------------------------------------------------------------
// Block-sparse causal attention (64-token blocks, head dim 128, CSR block lists).
cudaError_t launch_bsa(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* row_ptr, const int32_t* col_idx, int64_t nnz, void* o,
                       int otype, int64_t H, int64_t Hkv, int64_t T, const DeviceInfo& dev,
                       cudaStream_t stream);

// ---- q8_gemm.cu -------------------------------------------------------------------
// Tensor-core GEMM on binary16 codes: A16 [M,K] activation codes, B16 [N,K] weight codes,
// xd [M,K/32] f32, Wd [N,K/32] binary16 bits.  Writes y [M,N] (rescaled sum) or, when
// isum != nullptr, the raw block sums isum [M,N,K/32].
// K ranges (of whole 16-block scale windows) the GEMM splits into when the output has fewer
// 128 x 256 tiles than the GPU has SMs; 1 otherwise.
int gemm_splits(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
// Bytes of partial outputs launch_gemm_tc needs in `part` (uniform split-K, or the stream-K
// runs' partial tiles), 0 if none.
size_t gemm_part_bytes(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
// With splits > 1, part [splits, M, N] f32 receives the partial outputs and a second kernel
// adds them (in a fixed order) into y.  B is the weight codes [N, K]: binary16 (B16), or with
// b_int8 the int8 codes themselves (widened inside the GEMM; not with isum).
cudaError_t launch_gemm_tc(const uint16_t* A16, const void* B, bool b_int8, const float* xd,
                           const uint16_t* Wd, float* y, int32_t* isum, float* part, int splits,
                           int64_t M, int64_t N, int64_t K, const DeviceInfo& dev,
                           cudaStream_t stream, const Epilogue& epi = Epilogue());
// Drops the cache of encoded TMA tensor maps (q8_release).
void forget_tensor_maps();
// y = op(0, aux) for K == 0 (an empty sum), M*N outputs.
cudaError_t launch_epilogue_only(const Epilogue& epi, float* y, int64_t n, cudaStream_t stream);

}  // namespace q8
