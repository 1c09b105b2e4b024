// q8_api.cu -- the C ABI of libq8 (declared in include/q8.h): host-side argument
// checks, device checks, scratch management and dispatch to the kernels.
//
// Nothing is launched unless every check passes.  Every launch is asynchronous on the
// caller's stream; the library holds no lock while kernels run.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/q8.h"
#include "q8_internal.h"

namespace q8 {
namespace {

// The library's device error word (one per device that loads the library).  Kernels
// get its address as a parameter and atomically OR error bits into it.
__device__ uint32_t g_err_word;

thread_local char g_last_cuda_error[256] = "no error";

q8_status cuda_fail(cudaError_t e) {
  std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return Q8_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// Checks the current device and fills its info on first use.
q8_status current_device(DeviceInfo* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return Q8_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.device < 0) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) return Q8_ERR_DEVICE;
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, g_err_word)) != cudaSuccess) return cuda_fail(e);
    d.sm_count = sms;
    d.max_smem_optin = smem;
    d.err_word = static_cast<uint32_t*>(addr);
    d.device = dev;
  }
  *out = d;
  return Q8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// M, N, K in [0, 2^31), K % 32 == 0, and byte sizes that fit comfortably in 64 bits.
q8_status check_shape(int64_t M, int64_t N, int64_t K) {
  const int64_t lim = static_cast<int64_t>(0x7FFFFFFF);
  if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim) return Q8_ERR_SHAPE;
  if (K % kQK != 0) return Q8_ERR_SHAPE;
  // every array the library touches is below 2^48 bytes
  const double big = 281474976710656.0;
  if (static_cast<double>(M) * K * 4 > big || static_cast<double>(N) * K * 4 > big ||
      static_cast<double>(M) * N * 4 > big)
    return Q8_ERR_SHAPE;
  return Q8_OK;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Resolves AUTO; returns Q8_ERR_SHAPE if the requested path cannot run this shape.
q8_status resolve_path(int64_t M, int64_t N, int64_t K, q8_path req, const DeviceInfo& dev,
                       q8_path* out) {
  const bool decode_ok = decode_smem_bytes(M < 1 ? 1 : M, K, dev) != 0 && M <= kDecodeMaxM;
  const bool batch_ok = batch_supported(M < 1 ? 1 : M, N < 1 ? 1 : N, K, dev);
  switch (req) {
    case Q8_PATH_AUTO:
      // the decode kernel (one dp4a per 4 MACs and token) streams faster than the batched
      // mma.sync kernel up to 2 tokens (measured on the 9B and sweep shapes)
      if (M <= 2 && decode_ok) *out = Q8_PATH_DECODE;
      else if (batch_ok) *out = Q8_PATH_BATCH;
      else if (decode_ok) *out = Q8_PATH_DECODE;
      else *out = Q8_PATH_TENSOR;
      return Q8_OK;
    case Q8_PATH_DECODE:
      if (!decode_ok) return Q8_ERR_SHAPE;
      *out = req;
      return Q8_OK;
    case Q8_PATH_BATCH:
      if (!batch_ok) return Q8_ERR_SHAPE;
      *out = req;
      return Q8_OK;
    case Q8_PATH_DP4A:
      if (M > static_cast<int64_t>(65535) * 64) return Q8_ERR_SHAPE;  // grid rows of 64 tokens
      *out = req;
      return Q8_OK;
    case Q8_PATH_TENSOR:
      *out = req;
      return Q8_OK;
    default:
      return Q8_ERR_DTYPE;
  }
}

// Scratch of the tensor path: A16 [M,K] f16 codes, xd [M,K/32] f32, B16 [N,K] f16 codes, and
// the GEMM's partial outputs (split-K, or its stream-K partial tiles: gemm_part_bytes).
// With prepared weights (q8_linear_prepared) the B16 region is not needed, nor up to
// kInt8WeightsMaxM tokens, where the GEMM reads the int8 codes and widens them itself.
constexpr int64_t kInt8WeightsMaxM = 128;
bool tensor_widens(int64_t M, bool prepared) { return !prepared && M > kInt8WeightsMaxM; }
size_t tensor_ws_bytes(int64_t M, int64_t N, int64_t K, size_t part_bytes, bool with_b16 = true) {
  return align256(static_cast<size_t>(M) * K * 2) + align256(static_cast<size_t>(M) * (K / kQK) * 4) +
         (with_b16 ? align256(static_cast<size_t>(N) * K * 2) : 0) + align256(part_bytes);
}

// Scratch of the dp4a path: int8 activation codes [M,K] and their scales [M,K/32].
size_t dp4a_ws_bytes(int64_t M, int64_t K) {
  return align256(static_cast<size_t>(M) * K) + align256(static_cast<size_t>(M) * (K / kQK) * 4);
}

// Scratch of a path: its own arrays, then a slot of M binary32 RMSNorm factors (used only
// when the call normalises its input).
size_t norm_slot_offset(q8_path p, int64_t M, int64_t N, int64_t K, size_t part_bytes,
                        bool with_b16 = true) {
  return p == Q8_PATH_BATCH  ? batch_ws_bytes(M, K)
         : p == Q8_PATH_DP4A ? dp4a_ws_bytes(M, K)
                             : tensor_ws_bytes(M, N, K, part_bytes, with_b16);
}
size_t path_ws_bytes(q8_path p, int64_t M, int64_t N, int64_t K, size_t part_bytes,
                     bool with_b16 = true) {
  if (p == Q8_PATH_DECODE || M == 0 || N == 0 || K == 0) return 0;
  return norm_slot_offset(p, M, N, K, part_bytes, with_b16) + align256(static_cast<size_t>(M) * 4);
}

// Library-owned scratch for (current device, stream), grown on demand.
q8_status library_workspace(const DeviceInfo& dev, cudaStream_t stream, size_t bytes, void** out) {
  *out = nullptr;
  if (bytes == 0) return Q8_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_ws[{dev.device, stream}];
  if (w.bytes >= bytes) {
    *out = w.ptr;
    return Q8_OK;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e);
  if (cap != cudaStreamCaptureStatusNone) return Q8_ERR_CAPTURE;
  void* p = nullptr;
  e = cudaMallocAsync(&p, bytes, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? Q8_ERR_NOMEM : cuda_fail(e);
  }
  if (w.ptr != nullptr) cudaFreeAsync(w.ptr, stream);  // stream-ordered: after prior users
  w.ptr = p;
  w.bytes = bytes;
  *out = p;
  return Q8_OK;
}

q8_status launch_status(cudaError_t e) { return e == cudaSuccess ? Q8_OK : cuda_fail(e); }

// ---- timing hook (q8_set_timing_events) ----------------------------------------------
std::mutex g_timing_mu;
std::vector<cudaEvent_t> g_t_start, g_t_stop;
size_t g_t_next = 0;

// Picks the event pair for the next main-kernel launch (false if the hook is off).
bool timing_pair(cudaEvent_t* a, cudaEvent_t* b) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (g_t_start.empty()) return false;
  const size_t i = g_t_next++ % g_t_start.size();
  *a = g_t_start[i];
  *b = g_t_stop[i];
  return true;
}

cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  if (cap == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
  return cudaEventRecord(ev, stream);
}

// Runs `launch` (the main kernel of a call) between the hook's events, if the hook is on.
template <typename F>
cudaError_t timed_launch(cudaStream_t stream, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool on = timing_pair(&a, &b);
  cudaError_t e = on ? record_event(a, stream) : cudaSuccess;
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess && on) e = record_event(b, stream);
  return e;
}

q8_status linear_impl(const void* x, q8_dtype xtype, const int8_t* Wq, const uint16_t* Wd,
                      float* y, int64_t M, int64_t N, int64_t K, q8_path path, void* ws,
                      size_t ws_bytes, bool library_ws, cudaStream_t stream,
                      const Epilogue& epi = Epilogue(), Prologue pro = Prologue(),
                      const uint16_t* B16_pre = nullptr) {
  if (xtype != Q8_F32 && xtype != Q8_BF16) return Q8_ERR_DTYPE;
  if (path != Q8_PATH_AUTO && path != Q8_PATH_DECODE && path != Q8_PATH_TENSOR &&
      path != Q8_PATH_BATCH && path != Q8_PATH_DP4A)
    return Q8_ERR_DTYPE;
  q8_status st = check_shape(M, N, K);
  if (st != Q8_OK) return st;
  // pointers of empty arrays may be NULL
  if ((M * K > 0 && x == nullptr) || (N * K > 0 && (Wq == nullptr || Wd == nullptr)) ||
      (M * N > 0 && y == nullptr))
    return Q8_ERR_NULL;
  if (!aligned16(x) || !aligned16(Wq) || !aligned16(Wd) || !aligned16(y)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != Q8_OK) return st;
  q8_path p;
  if ((st = resolve_path(M, N, K, path, dev, &p)) != Q8_OK) return st;
  if (M == 0 || N == 0) return Q8_OK;
  if (K == 0) {  // an empty sum
    if (epi.plain()) return launch_status(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 4, stream));
    return launch_status(launch_epilogue_only(epi, y, M * N, stream));
  }
  if (p == Q8_PATH_DECODE)
    return launch_status(timed_launch(stream, [&] {
      return launch_decode(x, static_cast<int>(xtype), nullptr, Wq, Wd, y, nullptr, M, N, K, dev,
                           stream, epi, pro);
    }));
  const int splits = gemm_splits(M, N, K, dev);
  const size_t part_bytes = gemm_part_bytes(M, N, K, dev);
  // Up to one 128-token tile the GEMM reads each weight once: it takes the int8 codes and
  // widens them in shared memory, in place of a separate pass that reads N K bytes and
  // writes and re-reads 2 N K.  Larger M widens once per call (the in-GEMM widening costs
  // more there than the pass).  Prepared weights need neither.
  const bool b8 = B16_pre == nullptr && !tensor_widens(M, false);
  const bool with_b16 = tensor_widens(M, B16_pre != nullptr);
  const size_t need = path_ws_bytes(p, M, N, K, part_bytes, with_b16);
  if (library_ws) {
    if ((st = library_workspace(dev, stream, need, &ws)) != Q8_OK) return st;
  } else {
    if (ws == nullptr) return Q8_ERR_NULL;
    if (!aligned16(ws)) return Q8_ERR_ALIGN;
    if (ws_bytes < need) return Q8_ERR_NOMEM;
  }
  if (pro.on()) {  // the rows' RMSNorm factors, read by the activation quantizer
    float* r = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                        norm_slot_offset(p, M, N, K, part_bytes, with_b16));
    cudaError_t e = launch_row_rms(x, static_cast<int>(xtype), M, K, pro.eps, r, dev, stream);
    if (e != cudaSuccess) return launch_status(e);
    pro.r = r;
  }
  if (p == Q8_PATH_BATCH)
    return launch_status(timed_launch(stream, [&] {
      return launch_batch(x, static_cast<int>(xtype), nullptr, Wq, Wd, y, nullptr, M, N, K, ws, dev,
                          stream, epi, pro);
    }));
  if (p == Q8_PATH_DP4A) {
    int8_t* xq = static_cast<int8_t*>(ws);
    float* xdq = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                          align256(static_cast<size_t>(M) * K));
    cudaError_t e =
        launch_quantize(x, static_cast<int>(xtype), xq, false, xdq, false, M, K, dev, stream, pro);
    if (e == cudaSuccess)
      e = timed_launch(stream, [&] {
        return launch_dp4a_gemm(xq, xdq, Wq, Wd, y, nullptr, M, N, K, stream, epi);
      });
    return launch_status(e);
  }
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint16_t* A16 = reinterpret_cast<uint16_t*>(w8);
  float* xd = reinterpret_cast<float*>(w8 + align256(static_cast<size_t>(M) * K * 2));
  uint8_t* after_xd = w8 + align256(static_cast<size_t>(M) * K * 2) +
                      align256(static_cast<size_t>(M) * (K / kQK) * 4);
  uint16_t* B16 = with_b16 ? reinterpret_cast<uint16_t*>(after_xd) : const_cast<uint16_t*>(B16_pre);
  float* part = reinterpret_cast<float*>(after_xd + (with_b16 ? align256(static_cast<size_t>(N) * K * 2) : 0));
  cudaError_t e =
      launch_quantize(x, static_cast<int>(xtype), A16, true, xd, false, M, K, dev, stream, pro);
  if (e == cudaSuccess && with_b16) e = launch_codes_to_f16(Wq, B16, N * K, dev, stream);
  if (e == cudaSuccess)
    e = timed_launch(stream, [&] {
      return b8 ? launch_gemm_tc(A16, Wq, true, xd, Wd, y, nullptr, part, splits, M, N, K, dev, stream, epi)
                : launch_gemm_tc(A16, B16, false, xd, Wd, y, nullptr, part, splits, M, N, K, dev, stream, epi);
    });
  return launch_status(e);
}

}  // namespace
}  // namespace q8

using namespace q8;

extern "C" {

q8_status q8_quantize_weights(const float* W, int8_t* Wq, uint16_t* Wd, int64_t N, int64_t K,
                              cudaStream_t stream) {
  q8_status st = check_shape(0, N, K);
  if (st != Q8_OK) return st;
  if (N * K > 0 && (W == nullptr || Wq == nullptr || Wd == nullptr)) return Q8_ERR_NULL;
  if (!aligned16(W) || !aligned16(Wq) || !aligned16(Wd)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != Q8_OK) return st;
  return launch_status(launch_quantize(W, 0, Wq, false, Wd, true, N, K, dev, stream));
}

q8_status q8_quantize_act(const void* x, q8_dtype xtype, int8_t* xq, float* xd, int64_t M,
                          int64_t K, cudaStream_t stream) {
  if (xtype != Q8_F32 && xtype != Q8_BF16) return Q8_ERR_DTYPE;
  q8_status st = check_shape(M, 0, K);
  if (st != Q8_OK) return st;
  if (M * K > 0 && (x == nullptr || xq == nullptr || xd == nullptr)) return Q8_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(xd)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != Q8_OK) return st;
  return launch_status(
      launch_quantize(x, static_cast<int>(xtype), xq, false, xd, false, M, K, dev, stream));
}

q8_status q8_quantize_act_rmsnorm(const void* x, q8_dtype xtype, const float* gamma, float eps,
                                  int8_t* xq, float* xd, float* r, int64_t M, int64_t K,
                                  cudaStream_t stream) {
  if (xtype != Q8_F32 && xtype != Q8_BF16) return Q8_ERR_DTYPE;
  q8_status st = check_shape(M, 0, K);
  if (st != Q8_OK) return st;
  if (!(eps > 0.0f) || !std::isfinite(eps)) return Q8_ERR_VALUE;
  if ((M * K > 0 && (x == nullptr || xq == nullptr || xd == nullptr)) ||
      (K > 0 && gamma == nullptr) || (M > 0 && r == nullptr))
    return Q8_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(xd) || !aligned16(gamma) || !aligned16(r))
    return Q8_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != Q8_OK) return st;
  cudaError_t e = launch_row_rms(x, static_cast<int>(xtype), M, K, eps, r, dev, stream);
  Prologue pro;
  pro.gamma = gamma;
  pro.r = r;
  pro.eps = eps;
  if (e == cudaSuccess)
    e = launch_quantize(x, static_cast<int>(xtype), xq, false, xd, false, M, K, dev, stream, pro);
  return launch_status(e);
}

q8_status q8_linear(const void* x, const int8_t* Wq, const uint16_t* Wd, float* y, int64_t M,
                    int64_t N, int64_t K, cudaStream_t stream) {
  return linear_impl(x, Q8_BF16, Wq, Wd, y, M, N, K, Q8_PATH_AUTO, nullptr, 0, true, stream);
}

q8_status q8_linear_ex(const void* x, q8_dtype xtype, const int8_t* Wq, const uint16_t* Wd,
                       float* y, int64_t M, int64_t N, int64_t K, q8_path path, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  return linear_impl(x, xtype, Wq, Wd, y, M, N, K, path, workspace, workspace_bytes, false, stream);
}

}  // extern "C"

namespace q8 {
namespace {
// The neighbours of q8_linear_fused / q8_linear_prepared, checked.
q8_status fused_neighbours(const float* norm_weight, float norm_eps, q8_epilogue epi,
                           const float* aux, const void* y, q8_dtype ytype, int64_t M, int64_t N,
                           int64_t K, Prologue* pro, Epilogue* e) {
  if (epi != Q8_EPI_NONE && epi != Q8_EPI_ADD && epi != Q8_EPI_SILU_MUL) return Q8_ERR_DTYPE;
  if (ytype != Q8_F32 && ytype != Q8_BF16) return Q8_ERR_DTYPE;
  if (epi != Q8_EPI_NONE && M > 0 && N > 0 && aux == nullptr) return Q8_ERR_NULL;
  if (!aligned16(aux) || !aligned16(norm_weight)) return Q8_ERR_ALIGN;
  if (epi != Q8_EPI_NONE && M > 0 && N > 0 && y != nullptr) {
    // aux is read through the read-only data path while y is written: the two byte ranges
    // must be disjoint (the shape check bounds both below 2^48 bytes)
    const q8_status st = check_shape(M, N, K);
    if (st != Q8_OK) return st;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(aux);
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(y);
    const uintptr_t a1 = a0 + static_cast<uintptr_t>(M * N) * 4u;
    const uintptr_t y1 = y0 + static_cast<uintptr_t>(M * N) * (ytype == Q8_BF16 ? 2u : 4u);
    if (a0 < y1 && y0 < a1) return Q8_ERR_VALUE;
  }
  if (norm_weight != nullptr) {
    if (!(norm_eps > 0.0f) || !std::isfinite(norm_eps)) return Q8_ERR_VALUE;
    pro->gamma = norm_weight;
    pro->eps = norm_eps;
  }
  e->aux = aux;
  e->op = static_cast<int>(epi);
  e->bf16 = ytype == Q8_BF16 ? 1 : 0;
  return Q8_OK;
}
}  // namespace
}  // namespace q8

extern "C" {

q8_status q8_linear_fused(const void* x, q8_dtype xtype, const float* norm_weight,
                          float norm_eps, const int8_t* Wq, const uint16_t* Wd, q8_epilogue epi,
                          const float* aux, void* y, q8_dtype ytype, int64_t M, int64_t N,
                          int64_t K, q8_path path, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  Prologue pro;
  Epilogue e;
  q8_status st = fused_neighbours(norm_weight, norm_eps, epi, aux, y, ytype, M, N, K, &pro, &e);
  if (st != Q8_OK) return st;
  const bool library_ws = workspace == nullptr && workspace_bytes == 0;
  return linear_impl(x, xtype, Wq, Wd, static_cast<float*>(y), M, N, K, path, workspace,
                     workspace_bytes, library_ws, stream, e, pro);
}

q8_status q8_weights_to_f16(const int8_t* Wq, uint16_t* B16, int64_t N, int64_t K,
                            cudaStream_t stream) {
  q8_status st = check_shape(0, N, K);
  if (st != Q8_OK) return st;
  if (N * K > 0 && (Wq == nullptr || B16 == nullptr)) return Q8_ERR_NULL;
  if (!aligned16(Wq) || !aligned16(B16)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != Q8_OK) return st;
  if (N * K == 0) return Q8_OK;
  return launch_status(launch_codes_to_f16(Wq, B16, N * K, dev, stream));
}

q8_status q8_linear_prepared(const void* x, q8_dtype xtype, const float* norm_weight,
                             float norm_eps, const uint16_t* B16, const uint16_t* Wd,
                             q8_epilogue epi, const float* aux, void* y, q8_dtype ytype,
                             int64_t M, int64_t N, int64_t K, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  Prologue pro;
  Epilogue e;
  q8_status st = fused_neighbours(norm_weight, norm_eps, epi, aux, y, ytype, M, N, K, &pro, &e);
  if (st != Q8_OK) return st;
  if (N * K > 0 && B16 == nullptr) return Q8_ERR_NULL;
  const bool library_ws = workspace == nullptr && workspace_bytes == 0;
  // B16 stands in for Wq in the common checks (non-null, aligned); empty shapes return before
  // anything reads it
  return linear_impl(x, xtype, reinterpret_cast<const int8_t*>(B16), Wd, static_cast<float*>(y), M,
                     N, K, Q8_PATH_TENSOR, workspace, workspace_bytes, library_ws, stream, e, pro, B16);
}

size_t q8_linear_prepared_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (check_shape(M, N, K) != Q8_OK) return 0;
  DeviceInfo dev;
  if (current_device(&dev) != Q8_OK) return 0;
  return path_ws_bytes(Q8_PATH_TENSOR, M, N, K, gemm_part_bytes(M, N, K, dev), false);
}

q8_status q8_bsa_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const int32_t* row_ptr, const int32_t* col_idx, int64_t nnz, void* o,
                           q8_dtype otype, int64_t H, int64_t Hkv, int64_t T, int64_t d,
                           cudaStream_t stream) {
  if (otype != Q8_F32 && otype != Q8_BF16) return Q8_ERR_DTYPE;
  if (d != 128 || H < 0 || Hkv <= 0 || T < 0 || T % 64 != 0 || nnz < 0 || H % Hkv != 0 ||
      H > 0x7FFFFFFF || T > 0x7FFFFFFF || static_cast<double>(H) * T * d * 4 > 281474976710656.0 ||
      static_cast<double>(H) * T > 2147483647.0)  // the tiles' row coordinates are 32-bit
    return Q8_ERR_SHAPE;
  if (H * T > 0 && (q == nullptr || k == nullptr || v == nullptr || o == nullptr || row_ptr == nullptr ||
                    (nnz > 0 && col_idx == nullptr)))
    return Q8_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return Q8_ERR_ALIGN;
  // the block lists are read as int32 words on the device
  if ((reinterpret_cast<uintptr_t>(row_ptr) & 3u) != 0 || (reinterpret_cast<uintptr_t>(col_idx) & 3u) != 0)
    return Q8_ERR_ALIGN;
  DeviceInfo dev;
  q8_status st = current_device(&dev);
  if (st != Q8_OK) return st;
  return launch_status(
      launch_bsa(q, k, v, row_ptr, col_idx, nnz, o, static_cast<int>(otype), H, Hkv, T, dev, stream));
}

q8_status q8_kv3_encode(const void* x, q8_dtype xtype, uint32_t* codes, float* scales,
                        int64_t ngroups, cudaStream_t stream) {
  if (xtype != Q8_F32 && xtype != Q8_BF16) return Q8_ERR_DTYPE;
  if (ngroups < 0 || static_cast<double>(ngroups) * 512 > 281474976710656.0) return Q8_ERR_SHAPE;
  if (ngroups > 0 && (x == nullptr || codes == nullptr || scales == nullptr)) return Q8_ERR_NULL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  q8_status st = current_device(&dev);
  if (st != Q8_OK) return st;
  return launch_status(launch_kv3_encode(x, static_cast<int>(xtype), codes, scales, ngroups, dev, stream));
}

q8_status q8_kv3_decode(const uint32_t* codes, const float* scales, void* out, q8_dtype otype,
                        int64_t ngroups, cudaStream_t stream) {
  if (otype != Q8_F32 && otype != Q8_BF16) return Q8_ERR_DTYPE;
  if (ngroups < 0 || static_cast<double>(ngroups) * 512 > 281474976710656.0) return Q8_ERR_SHAPE;
  if (ngroups > 0 && (out == nullptr || codes == nullptr || scales == nullptr)) return Q8_ERR_NULL;
  if (!aligned16(out) || !aligned16(codes) || !aligned16(scales)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  q8_status st = current_device(&dev);
  if (st != Q8_OK) return st;
  return launch_status(launch_kv3_decode(codes, scales, out, static_cast<int>(otype), ngroups, dev, stream));
}

size_t q8_linear_workspace_size(int64_t M, int64_t N, int64_t K, q8_path path) {
  if (check_shape(M, N, K) != Q8_OK) return 0;
  DeviceInfo dev;
  if (current_device(&dev) != Q8_OK) return 0;
  q8_path p;
  if (resolve_path(M, N, K, path, dev, &p) != Q8_OK) return 0;
  return path_ws_bytes(p, M, N, K, gemm_part_bytes(M, N, K, dev), tensor_widens(M, false));
}

q8_status q8_block_sums(const int8_t* xq, const int8_t* Wq, int32_t* isum, int64_t M, int64_t N,
                        int64_t K, q8_path path, cudaStream_t stream) {
  if (path != Q8_PATH_AUTO && path != Q8_PATH_DECODE && path != Q8_PATH_TENSOR &&
      path != Q8_PATH_BATCH && path != Q8_PATH_DP4A)
    return Q8_ERR_DTYPE;
  q8_status st = check_shape(M, N, K);
  if (st != Q8_OK) return st;
  if ((M * K > 0 && xq == nullptr) || (N * K > 0 && Wq == nullptr) || (M * N * K > 0 && isum == nullptr))
    return Q8_ERR_NULL;
  if (!aligned16(xq) || !aligned16(Wq) || !aligned16(isum)) return Q8_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != Q8_OK) return st;
  q8_path p;
  if ((st = resolve_path(M, N, K, path, dev, &p)) != Q8_OK) return st;
  if (M == 0 || N == 0 || K == 0) return Q8_OK;
  if (p == Q8_PATH_DECODE)
    return launch_status(
        launch_decode(nullptr, 0, xq, Wq, nullptr, nullptr, isum, M, N, K, dev, stream));
  if (p == Q8_PATH_DP4A)
    return launch_status(launch_dp4a_gemm(xq, nullptr, Wq, nullptr, nullptr, isum, M, N, K, stream));
  if (p == Q8_PATH_BATCH) {
    void* wsb = nullptr;
    if ((st = library_workspace(dev, stream, batch_ws_bytes(M, K), &wsb)) != Q8_OK) return st;
    return launch_status(
        launch_batch(nullptr, 0, xq, Wq, nullptr, nullptr, isum, M, N, K, wsb, dev, stream));
  }
  const size_t need = align256(static_cast<size_t>(M) * K * 2) + align256(static_cast<size_t>(N) * K * 2);
  void* ws = nullptr;
  if ((st = library_workspace(dev, stream, need, &ws)) != Q8_OK) return st;
  uint16_t* A16 = static_cast<uint16_t*>(ws);
  uint16_t* B16 = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) +
                                              align256(static_cast<size_t>(M) * K * 2));
  cudaError_t e = launch_codes_to_f16(xq, A16, M * K, dev, stream);
  if (e == cudaSuccess) e = launch_codes_to_f16(Wq, B16, N * K, dev, stream);
  if (e == cudaSuccess)
    e = launch_gemm_tc(A16, B16, false, nullptr, nullptr, nullptr, isum, nullptr, 1, M, N, K, dev, stream);
  return launch_status(e);
}

uint32_t q8_device_error(q8_status* status) {
  if (status) *status = Q8_OK;
  DeviceInfo dev;
  q8_status st = current_device(&dev);
  if (st != Q8_OK) {
    if (status) *status = st;
    return 0;
  }
  cudaError_t e = cudaDeviceSynchronize();
  uint32_t word = 0;
  const uint32_t zero = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&word, g_err_word, sizeof word);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_err_word, &zero, sizeof zero);
  if (e != cudaSuccess) {
    cuda_fail(e);
    if (status) *status = Q8_ERR_CUDA;
  }
  return word;
}

const char* q8_status_string(q8_status s) {
  switch (s) {
    case Q8_OK: return "ok";
    case Q8_ERR_NULL: return "a required pointer is NULL";
    case Q8_ERR_SHAPE: return "bad shape (negative size, K not a multiple of 32, too large, or not supported by the chosen path)";
    case Q8_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case Q8_ERR_DTYPE: return "unknown activation type or path";
    case Q8_ERR_NOMEM: return "workspace too small or allocation failed";
    case Q8_ERR_CUDA: return "CUDA runtime error (see q8_last_cuda_error)";
    case Q8_ERR_DEVICE: return "current device is not compute capability 10.3";
    case Q8_ERR_CAPTURE: return "the call would allocate scratch while its stream is captured";
    case Q8_ERR_VALUE: return "a scalar argument is outside its domain";
  }
  return "unknown status";
}

const char* q8_last_cuda_error(void) { return g_last_cuda_error; }

q8_status q8_set_timing_events(cudaEvent_t* starts, cudaEvent_t* stops, int count) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  g_t_start.clear();
  g_t_stop.clear();
  g_t_next = 0;
  if (count <= 0) return Q8_OK;
  if (starts == nullptr || stops == nullptr) return Q8_ERR_NULL;
  g_t_start.assign(starts, starts + count);
  g_t_stop.assign(stops, stops + count);
  return Q8_OK;
}

void q8_release(void) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = -1;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
      if (kv.second.ptr != nullptr) {
        cudaSetDevice(kv.first.first);
        cudaFree(kv.second.ptr);
      }
    }
    g_ws.clear();
    if (cur >= 0) cudaSetDevice(cur);
    // device addresses (the error word) belong to the context they were looked up in
    for (DeviceInfo& d : g_dev) d = DeviceInfo();
  }
  // a later context (e.g. after cudaDeviceReset) starts afresh
  forget_kernel_attributes();
  forget_noalloc_scratch();
  forget_tensor_maps();
}

const char* q8_version(void) { return "0.1.0"; }

}  // extern "C"

namespace q8 {
namespace {
std::mutex g_attr_mu;
std::map<std::pair<const void*, int>, size_t> g_smem_set;
std::map<std::pair<const void*, int>, int> g_regs;
}  // namespace

int device_info(DeviceInfo* out) { return static_cast<int>(current_device(out)); }

cudaError_t ensure_smem(const void* fn, size_t bytes, int device) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  size_t& cur = g_smem_set[{fn, device}];
  if (cur >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) cur = bytes;
  return e;
}

void forget_kernel_attributes() {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  g_smem_set.clear();
  g_regs.clear();
}

cudaError_t kernel_regs(const void* fn, int device, int* regs) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  auto it = g_regs.find({fn, device});
  if (it != g_regs.end()) {
    *regs = it->second;
    return cudaSuccess;
  }
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  g_regs[{fn, device}] = fa.numRegs;
  *regs = fa.numRegs;
  return cudaSuccess;
}

}  // namespace q8
