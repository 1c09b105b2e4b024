/*
 * q8.h -- C ABI of libq8: the Q8_0 block-quantized linear layer on GB300 (sm_103a).
 *
 * The operation.  The post "CUDA inference engine for running Qwen3.5/3.6 hybrid models
 * on mining cards (CMP 100-210)" (news.hada.io topic 29953) runs the linear layers of its
 * dense GDN + attention models as an int8 GEMM over Q8_0 weights (list of un-throttled
 * paths: the DP4A int8 GEMM; "Limitations" list: Q8_0 is the only supported type).
 * This library computes that layer with this Q8_0 definition:
 *   - K is cut into blocks of 32 consecutive elements (K must be a multiple of 32);
 *   - per block: amax = max |v|, d = amax / 127 in IEEE binary32, codes
 *     q = round(v / d) (one IEEE binary32 division, ties away from zero, clamped to
 *     [-127, 127]); an all-zero block (or one whose d underflows to 0) gets d = 0 and
 *     codes 0;
 *   - weight scales are stored as IEEE binary16 (round to nearest even), activation
 *     scales as binary32;
 *   - y[m,n] = sum_b Wd[n,b] * xd[m,b] * isum[m,n,b], with the exact integer block dot
 *     isum[m,n,b] = sum_{j<32} xq[m,32b+j] * Wq[n,32b+j]  (|isum| <= 516128).
 * Codes, scales and block sums are exact; y is a binary32 sum whose order is not fixed.
 *
 * Layouts (row-major, K contiguous, nn.Linear orientation y = x W^T):
 *   W  float   [N, K]          Wq int8  [N, K]      Wd uint16 [N, K/32]  (binary16 bits)
 *   x  bf16/f32 [M, K]         xq int8  [M, K]      xd float  [M, K/32]
 *   y  float   [M, N]          isum int32 [M, N, K/32]
 *
 * Conventions for every entry point:
 *   - all array pointers are DEVICE pointers owned by the caller; the library never
 *     frees or keeps them; every array pointer must be 16-byte aligned unless its entry
 *     point says otherwise; the pointer of an empty array (zero elements) may be NULL;
 *   - an output array must not overlap any input or other output of the same call (the
 *     kernels read inputs while other blocks write outputs); only aux against y is checked;
 *   - calls are asynchronous on `stream` (0 = the legacy default stream); inputs must
 *     stay valid and outputs untouched until the stream passes the call;
 *   - arguments are checked on the host before anything is launched; on any error
 *     nothing is launched and the status says why; Q8_ERR_CUDA reports a failed CUDA
 *     runtime call (its text: q8_last_cuda_error());
 *   - the current CUDA device must be a compute capability 10.3 GPU (GB300);
 *   - inputs must be finite (NaN / Inf are outside the domain and not checked).
 */
#ifndef Q8_H
#define Q8_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum q8_status {
    Q8_OK = 0,
    Q8_ERR_NULL = 1,     /* a required pointer is NULL                                 */
    Q8_ERR_SHAPE = 2,    /* M, N or K < 0, K not a multiple of 32, or a size overflows  */
    Q8_ERR_ALIGN = 3,    /* an array pointer is not aligned as required (16 bytes mostly) */
    Q8_ERR_DTYPE = 4,    /* unknown activation type or path selector                    */
    Q8_ERR_NOMEM = 5,    /* workspace too small, or the library could not allocate one  */
    Q8_ERR_CUDA = 6,     /* a CUDA runtime call failed                                  */
    Q8_ERR_DEVICE = 7,   /* the current device is not compute capability 10.3           */
    Q8_ERR_CAPTURE = 8,  /* the call would allocate while its stream is being captured  */
    Q8_ERR_VALUE = 9     /* an argument outside its domain (eps <= 0, aux overlapping y) */
} q8_status;

typedef enum q8_dtype {
    Q8_F32 = 0,          /* IEEE binary32 activations                                   */
    Q8_BF16 = 1          /* bfloat16 activations (uint16 bit patterns)                  */
} q8_dtype;

/* Which kernel family computes the product.  AUTO picks by M (decode kernel for one
 * token, batched-decode kernel for a few tokens, tensor-core GEMM otherwise); the explicit
 * choices exist for tests and benchmarks. */
typedef enum q8_path {
    Q8_PATH_AUTO = 0,
    Q8_PATH_DECODE = 1,  /* weight-streaming kernel (int8 dot products, fused act-quant);
                            M <= 8                                                        */
    Q8_PATH_TENSOR = 2,  /* tcgen05 tensor-core GEMM with per-block rescale               */
    Q8_PATH_BATCH = 3,   /* weight-streaming kernel with mma.sync block sums; 1 <= M <= 64,
                            K % 256 == 0                                                  */
    Q8_PATH_DP4A = 4     /* the post's own design: dp4a int8 GEMM on CUDA cores, kept as a
                            prior-art comparison; never chosen by AUTO                     */
} q8_path;

/*
 * q8_quantize_weights -- Q8_0 weight quantizer (one-off, per weight matrix).
 *   W  [N,K] float in;  Wq [N,K] int8 out;  Wd [N,K/32] binary16 bits out.
 *   N, K >= 0 (zero sizes launch nothing), K % 32 == 0.
 */
q8_status q8_quantize_weights(const float* W, int8_t* Wq, uint16_t* Wd, int64_t N, int64_t K,
                              cudaStream_t stream);

/*
 * q8_quantize_act -- Q8_0 activation quantizer.
 *   x [M,K] of type xtype in;  xq [M,K] int8 out;  xd [M,K/32] float out.
 */
q8_status q8_quantize_act(const void* x, q8_dtype xtype, int8_t* xq, float* xd, int64_t M,
                          int64_t K, cudaStream_t stream);

/*
 * q8_linear -- y = Q8_0 linear layer of bf16 activations x:  y[M,N] = x[M,K] . W^T through
 * the codes above (activations are quantized per call, inside the library).
 *   x [M,K] bf16 in;  Wq, Wd from q8_quantize_weights;  y [M,N] float out (overwritten).
 * Scratch memory (quantized activations, at most 2*M*K + 4*M*(K/32) bytes plus 2*N*K for
 * the tensor-core path) is owned by the library, one buffer per (device, stream); it
 * grows on demand with cudaMalloc, which is not allowed while the stream is captured:
 * make the first call with the largest shape before capturing (else Q8_ERR_CAPTURE).
 * q8_release() frees it.
 */
q8_status q8_linear(const void* x, const int8_t* Wq, const uint16_t* Wd, float* y, int64_t M,
                    int64_t N, int64_t K, cudaStream_t stream);

/*
 * q8_linear_ex -- q8_linear with the activation type, the kernel family and the scratch
 * memory chosen by the caller.  workspace may be NULL only if workspace_bytes is 0 and
 * q8_linear_workspace_size() returns 0 for the chosen path; never allocates.
 */
q8_status q8_linear_ex(const void* x, q8_dtype xtype, const int8_t* Wq, const uint16_t* Wd,
                       float* y, int64_t M, int64_t N, int64_t K, q8_path path,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * q8_quantize_act_rmsnorm -- RMSNorm fused into the Q8_0 activation quantizer.
 * The layer's input in a transformer block is the RMS-normalised hidden state
 * z = x * r * gamma, r = 1 / sqrt(mean_k x^2 + eps) (root mean square layer normalisation,
 * Zhang and Sennrich, 2019).  r is one factor per row, so it rides on the row's block
 * scales: xq holds the Q8_0 codes of fl32(x * gamma) and xd their binary32 scales times r
 * (in exact arithmetic the quantization of z itself; the codes do not depend on how r is
 * rounded).  r is summed in binary32 in a fixed order and also returned.
 *   x [M,K] of type xtype, gamma [K] float in;  xq [M,K] int8, xd [M,K/32] float,
 *   r [M] float out.  eps finite and > 0 (else Q8_ERR_VALUE).
 */
q8_status q8_quantize_act_rmsnorm(const void* x, q8_dtype xtype, const float* gamma, float eps,
                                  int8_t* xq, float* xd, float* r, int64_t M, int64_t K,
                                  cudaStream_t stream);

/*
 * q8_linear_fused -- the linear layer with its neighbours in the surrounding block fused
 * into it.  The post runs its Q8_0 linears inside GDN + attention blocks
 * ("CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
 * (CMP 100-210)", news.hada.io topic 29953, feature list).  Before the product:
 *   norm_weight != NULL: x is the un-normalised hidden state and the layer's input is its
 *                    RMSNorm with weight norm_weight [K] float and norm_eps (as
 *                    q8_quantize_act_rmsnorm, inside the layer's own quantizer);
 *                    norm_weight NULL: x is the input itself.
 * After it, in the output store:
 *   Q8_EPI_NONE      y = x . W^T
 *   Q8_EPI_ADD       y = x . W^T + aux              (residual add; aux [M,N] float)
 *   Q8_EPI_SILU_MUL  y = silu(aux) * (x . W^T)      (gated FFN unit: aux is the gate
 *                    projection's output [M,N] float, W the up projection;
 *                    silu(g) = g / (1 + e^-g))
 * y is [M,N] float (ytype Q8_F32) or bfloat16 bits (Q8_BF16, round to nearest even).
 * aux may be NULL for Q8_EPI_NONE, else it is 16-byte aligned and must not overlap y (the
 * kernels read it through the read-only data path; an in-place residual add needs a
 * separate output buffer).  x, Wq, Wd, M, N, K, path and stream as q8_linear_ex;
 * workspace NULL with workspace_bytes 0 uses the library-owned scratch of q8_linear (same
 * growth and capture rules), otherwise the caller's.  With K == 0 the sum is empty and y is
 * the epilogue of zero.
 * Errors: Q8_ERR_DTYPE for an unknown epilogue, output or activation type; Q8_ERR_NULL for
 * a NULL aux with an epilogue that reads it; Q8_ERR_ALIGN for aux or norm_weight not
 * 16-byte aligned; Q8_ERR_VALUE for a norm_eps that is not finite and > 0, or for an aux
 * whose M*N floats overlap the bytes of y; the rest as q8_linear_ex.
 */
typedef enum q8_epilogue {
    Q8_EPI_NONE = 0,
    Q8_EPI_ADD = 1,
    Q8_EPI_SILU_MUL = 2
} q8_epilogue;
q8_status q8_linear_fused(const void* x, q8_dtype xtype, const float* norm_weight,
                          float norm_eps, const int8_t* Wq, const uint16_t* Wd, q8_epilogue epi,
                          const float* aux, void* y, q8_dtype ytype, int64_t M, int64_t N,
                          int64_t K, q8_path path, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * 3-bit KV-cache codec: Walsh-Hadamard rotation + Lloyd-Max quantizer.  The post keeps a
 * 256K-token context in a 3-bit KV cache built from these two parts, 17 GB -> 3.5 GB
 * ("CUDA inference engine for running Qwen3.5/3.6 hybrid models on mining cards
 * (CMP 100-210)", news.hada.io topic 29953, feature list).
 * A group is 128 consecutive elements of a key or value vector (a 256-wide head is two
 * groups).  Per group: codes[12] uint32, the 128 three-bit codes as a little-endian bit
 * stream (element i at bits [3i, 3i + 3)), and one float scale: 52 bytes instead of 256
 * (bf16), 3.25 bits per element.
 *   encode: u = unnormalised Walsh-Hadamard transform of the group (binary32); s = the RMS
 *           of u (pairwise sum of the squares); code_i = 4 * (u_i < 0) + the number of
 *           thresholds t in (0.5006, 1.0500, 1.7480) with |u_i| >= t * s (the 8-level
 *           unit-Gaussian Lloyd-Max quantizer, Max 1960); s == 0 gives codes 0.
 *   decode: w_i = s * (+-level), levels (0.2451, 0.7560, 1.3440, 2.1520);
 *           out = WHT(w) / 128, binary32 or bfloat16 (round to nearest even).
 *   x [ngroups][128] of type xtype; codes [ngroups][12]; scales [ngroups];
 *   out [ngroups][128] of type otype.  ngroups >= 0; device pointers, 16-byte aligned.
 *   Domain: finite groups whose sum of squares stays within binary32 (|x| below ~1e18).
 */
q8_status q8_kv3_encode(const void* x, q8_dtype xtype, uint32_t* codes, float* scales,
                        int64_t ngroups, cudaStream_t stream);
q8_status q8_kv3_decode(const uint32_t* codes, const float* scales, void* out, q8_dtype otype,
                        int64_t ngroups, cudaStream_t stream);

/*
 * q8_bsa_attention -- block-sparse causal attention for long prefill.  The post speeds up
 * long prefill with MInference-style block-sparse attention ("CUDA inference engine for
 * running Qwen3.5/3.6 hybrid models on mining cards (CMP 100-210)", news.hada.io topic
 * 29953, feature list).  Query t of head h attends to the keys j <= t of the 64-token key
 * blocks listed for its 64-token query block; H query heads share Hkv key/value heads
 * (head h reads h / (H / Hkv)); o_t = softmax(q_t . k_j / sqrt(d)) weighted sum of v_j; a
 * query that sees no key gets 0.
 *   q [H][T][d], k and v [Hkv][T][d]: bfloat16 bits; d = 128; T a multiple of 64;
 *     H * T below 2^31 (else Q8_ERR_SHAPE).
 *   row_ptr [H * T/64 + 1], col_idx [nnz]: int32 CSR over (head, query block) rows; the
 *     key blocks of a row ascending, each in [0, query block] (others are skipped and set
 *     bit 8 of the device error word).
 *   o [H][T][d]: binary32 (otype Q8_F32) or bfloat16 (Q8_BF16).
 *   q, k, v and o 16-byte aligned, row_ptr and col_idx 4-byte aligned (else Q8_ERR_ALIGN).
 * Softmax in binary32 (base-2 exponentials), products on the tensor cores with the weights
 * rounded to bfloat16, as in FlashAttention.
 */
q8_status q8_bsa_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const int32_t* row_ptr, const int32_t* col_idx, int64_t nnz, void* o,
                           q8_dtype otype, int64_t H, int64_t Hkv, int64_t T, int64_t d,
                           cudaStream_t stream);

/*
 * Prepared weights for the tensor-core path.  The tensor path feeds the MMA binary16
 * copies of the int8 codes (exact: |q| <= 127); q8_linear / q8_linear_ex / q8_linear_fused
 * widen the codes on every call (read N*K bytes, write and re-read 2*N*K).  For weights
 * used by many prefill or medium-batch calls, widen them once and keep the copy:
 *   q8_weights_to_f16: Wq [N,K] int8 -> B16 [N,K] binary16 bits (2 bytes per weight).
 *   q8_linear_prepared: q8_linear_fused on the tensor-core path (any M; the batched and
 *     decode kernels, which read the int8 codes, are faster for M <= 64) with B16 in place
 *     of Wq; the same kernels and the same results as q8_linear_fused with
 *     Q8_PATH_TENSOR.  workspace: NULL with workspace_bytes 0 for the library-owned
 *     scratch, else at least q8_linear_prepared_workspace_size() bytes.
 */
q8_status q8_weights_to_f16(const int8_t* Wq, uint16_t* B16, int64_t N, int64_t K,
                            cudaStream_t stream);
q8_status q8_linear_prepared(const void* x, q8_dtype xtype, const float* norm_weight,
                             float norm_eps, const uint16_t* B16, const uint16_t* Wd,
                             q8_epilogue epi, const float* aux, void* y, q8_dtype ytype,
                             int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);
size_t q8_linear_prepared_workspace_size(int64_t M, int64_t N, int64_t K);

/* Bytes of scratch q8_linear_ex and q8_linear_fused need for this shape and path (0 if
 * none): the path's own arrays, the GEMM's partial outputs when it splits K, and a slot
 * for the rows' RMSNorm factors. */
size_t q8_linear_workspace_size(int64_t M, int64_t N, int64_t K, q8_path path);

/*
 * q8_block_sums -- the exact int32 block dot products isum[M,N,K/32] of given codes,
 * computed by the same kernel code as q8_linear on the chosen path (TENSOR: the tcgen05
 * MMAs whose binary32 TMEM results the rescale reads; DECODE: the dp4a kernel).  Meant
 * for checking; scratch as for q8_linear (library-owned).
 */
q8_status q8_block_sums(const int8_t* xq, const int8_t* Wq, int32_t* isum, int64_t M, int64_t N,
                        int64_t K, q8_path path, cudaStream_t stream);

/*
 * q8_device_error -- synchronizes the current device, then returns (and clears) the
 * library's device error word: bit 0 = a bounded device-side wait gave up (the results
 * of that call are undefined), bit 1 = a kernel met launch parameters it cannot handle.
 * 0 means no error.  Returns Q8_ERR_CUDA through *status if the sync itself failed.
 */
uint32_t q8_device_error(q8_status* status);

/*
 * q8_linear_noalloc -- the tensor-core Q8_0 linear layer (the same kernels as q8_linear_ex
 * with Q8_PATH_TENSOR, without its split of K on small outputs, so results agree within the
 * library's tolerance) for callers that cannot allocate device memory during
 * a call: a host framework that owns every device allocation through its own fixed pool,
 * or a serving loop where cudaMalloc's implicit device synchronization, or running out of
 * memory in the middle of a step, is not acceptable.  The post has no counterpart of this
 * entry point; it exists for such callers only.
 *   x [M,K] of type xtype, Wq/Wd from q8_quantize_weights, y [M,N] float out.
 * Scratch lives in one static device array of Q8_NOALLOC_SCRATCH_BYTES bytes that every
 * GPU loading the library holds until the process exits; this call allocates and frees
 * nothing.  A shape whose scratch (2*M*K + 4*M*(K/32) + 2*N*K bytes, each part rounded up
 * to 256) exceeds the array is rejected with Q8_ERR_NOMEM before anything runs.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current: make that first call before any stream capture.
 * All calls on a device share the one array, and its contents stay from the last call
 * (each call writes all the scratch it reads, so nothing needs clearing): calls that
 * overlap on the GPU -- on different streams, or from different threads -- race, so
 * serialize them.
 */
#define Q8_NOALLOC_SCRATCH_BYTES (64u << 20)
q8_status q8_linear_noalloc(const void* x, q8_dtype xtype, const int8_t* Wq, const uint16_t* Wd,
                            float* y, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * q8_set_timing_events -- timing hook for benchmarks.  With count > 0, each later
 * q8_linear / q8_linear_ex call records starts[i] on its stream right before the launch
 * of its main kernel (the decode kernel, or the tensor-core GEMM) and stops[i] right after
 * it, i = 0, 1, ..., count-1, count, ... taken modulo count (i restarts at 0 on every call
 * of this function).  Under stream capture the records become graph event nodes
 * (cudaEventRecordExternal).  The arrays are copied; the events must outlive their use.
 * count == 0 (or NULL arrays) switches the hook off.  Process-wide; calls that race with
 * this one may or may not see the change.  Returns Q8_ERR_NULL if count > 0 and an array
 * is NULL.
 */
q8_status q8_set_timing_events(cudaEvent_t* starts, cudaEvent_t* stops, int count);

/* Human-readable text of a status code (static storage). */
const char* q8_status_string(q8_status status);

/* Text of the last CUDA error seen by the calling thread in this library (static/TLS). */
const char* q8_last_cuda_error(void);

/* Frees library-owned scratch memory on every device and forgets the per-kernel launch
 * attributes the library has set (shared-memory limits, register counts), so that a new
 * CUDA context, e.g. after cudaDeviceReset, starts afresh.  Not thread-safe against calls in
 * flight: call it when no q8_linear / q8_block_sums call is running. */
void q8_release(void);

/* Library version, e.g. "0.1.0". */
const char* q8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* Q8_H */
