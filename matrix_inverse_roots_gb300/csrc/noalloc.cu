// spectral_scale_noalloc: the spectral scaling step with its scratch memory
// built into the library instead of supplied by the caller.
//
// Who needs it: code that must not allocate device memory at the time it runs.
// Examples are work recorded into a CUDA graph (allocation calls cannot be
// captured), hooks running inside another framework's memory manager or under a
// fixed device-memory budget, and real-time loops that forbid allocation after
// start-up.  Such callers can still pass the inputs and outputs they own, but
// cannot obtain a scratch buffer.  This entry point gives them the power
// iteration without one.
//
// How: the scratch is one file-scope __device__ array of DASH_NOALLOC_SCRATCH_BYTES
// that every GPU loading the library holds until the process exits.  Host code
// cannot use the array's name as a device pointer (on the host it names a shadow
// object, not device memory), so the device address is looked up once per device
// with cudaGetSymbolAddress and then handed to the kernels like any workspace.
#include <mutex>

#include "dash_internal.h"
#include "dashroot.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DASH_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call made with that device current; nullptr on failure.
void* scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" dash_status spectral_scale_noalloc(const float* A, float ridge, int64_t N, int B,
                                              int mode, int n_vec, int power_iters,
                                              const float* V0, float* lambda_out,
                                              void* stream) {
  size_t need = 0;
  const int prec = (mode == DASH_SCALE_POWER_F16)    ? DASH_FP16
                   : (mode == DASH_SCALE_POWER_BF16) ? DASH_BF16
                                                     : DASH_FP32_3XTF32;
  const dash_status s = dash_workspace_size(DASH_OP_SPECTRAL_SCALE, N, B, prec, n_vec, &need);
  if (s != DASH_OK) return s;
  if (mode == DASH_SCALE_FROBENIUS) need = (static_cast<size_t>(N) * 4 + 255) & ~size_t(255);
  // One pass over all N blocks must fit; larger stacks are refused, not chunked.
  if (need > static_cast<size_t>(DASH_NOALLOC_SCRATCH_BYTES)) return DASH_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = scratch_address();
  if (scratch == nullptr) return DASH_ERR_CUDA;
  return spectral_scale(A, ridge, N, B, mode, n_vec, power_iters, V0, lambda_out, scratch,
                        static_cast<size_t>(DASH_NOALLOC_SCRATCH_BYTES), stream);
}
