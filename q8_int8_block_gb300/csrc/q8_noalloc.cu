// q8_noalloc.cu -- q8_linear_noalloc: the tensor-core Q8_0 linear layer with its scratch
// memory in a fixed, statically sized device array, so that the call allocates nothing.
//
// Who needs this: callers that cannot allocate device memory during a call, e.g. a host
// framework that owns every device allocation through its own fixed-size pool, a serving
// loop where cudaMalloc (which synchronizes the device) or an out-of-memory failure in
// the middle of a step is not acceptable.  They pass inputs and outputs as usual; the
// scratch (binary16 activation codes, activation scales, binary16 weight codes) lives in
// the array below, which every GPU that loads this library holds until the process exits.
#include <mutex>

#include "../../include/q8.h"
#include "q8_internal.h"

namespace q8 {
namespace {

// The scratch array.  In host code this name is only a stand-in for the device object:
// its address is obtained per device with cudaGetSymbolAddress and passed to kernels.
static __device__ __align__(256) uint8_t g_noalloc_scratch[Q8_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_na_mu;
void* g_na_ptr[kMaxDev] = {};  // the array's device address, per device (nullptr: not looked up)

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

void forget_noalloc_scratch() {
  std::lock_guard<std::mutex> lock(g_na_mu);
  for (void*& p : g_na_ptr) p = nullptr;
}

}  // namespace q8

using namespace q8;

extern "C" q8_status q8_linear_noalloc(const void* x, q8_dtype xtype, const int8_t* Wq,
                                       const uint16_t* Wd, float* y, int64_t M, int64_t N,
                                       int64_t K, cudaStream_t stream) {
  if (xtype != Q8_F32 && xtype != Q8_BF16) return Q8_ERR_DTYPE;
  const int64_t lim = 0x7FFFFFFF;
  if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim || K % kQK != 0)
    return Q8_ERR_SHAPE;
  if ((M * K > 0 && x == nullptr) || (N * K > 0 && (Wq == nullptr || Wd == nullptr)) ||
      (M * N > 0 && y == nullptr))
    return Q8_ERR_NULL;
  auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis(x) || mis(Wq) || mis(Wd) || mis(y)) return Q8_ERR_ALIGN;
  // scratch layout: A16 [M,K] binary16 codes | xd [M,K/32] f32 | B16 [N,K] binary16 codes
  const double need_d = static_cast<double>(up256(static_cast<size_t>(M) * K * 2)) +
                        static_cast<double>(up256(static_cast<size_t>(M) * (K / kQK) * 4)) +
                        static_cast<double>(up256(static_cast<size_t>(N) * K * 2));
  if (need_d > static_cast<double>(Q8_NOALLOC_SCRATCH_BYTES)) return Q8_ERR_NOMEM;
  if (M == 0 || N == 0) return Q8_OK;

  // the library's checked device info: compute capability, SM count, shared-memory limit,
  // and the device error word that the kernels' bounded waits report into
  DeviceInfo di;
  const int st = device_info(&di);
  if (st != Q8_OK) return static_cast<q8_status>(st);
  if (di.device >= kMaxDev) return Q8_ERR_DEVICE;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (g_na_ptr[di.device] == nullptr) {
      // one-time set-up on this device (it is current): the array's device address
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || ptr == nullptr) return Q8_ERR_CUDA;
      g_na_ptr[di.device] = ptr;
    }
    scratch = g_na_ptr[di.device];
  }
  cudaError_t e;
  if (K == 0) {
    e = cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 4, stream);
    return e == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
  }
  // Every byte of scratch a call reads is written by that call first (codes and scales of
  // all M rows and all N weight rows), so nothing has to be cleared between calls.
  uint8_t* base = static_cast<uint8_t*>(scratch);
  uint16_t* A16 = reinterpret_cast<uint16_t*>(base);
  float* xd = reinterpret_cast<float*>(base + up256(static_cast<size_t>(M) * K * 2));
  uint16_t* B16 = reinterpret_cast<uint16_t*>(base + up256(static_cast<size_t>(M) * K * 2) +
                                              up256(static_cast<size_t>(M) * (K / kQK) * 4));
  e = launch_quantize(x, static_cast<int>(xtype), A16, true, xd, false, M, K, di, stream);
  if (e == cudaSuccess) e = launch_codes_to_f16(Wq, B16, N * K, di, stream);
  if (e == cudaSuccess) e = launch_gemm_tc(A16, B16, false, xd, Wd, y, nullptr, nullptr, 1, M, N, K, di, stream);
  return e == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}
