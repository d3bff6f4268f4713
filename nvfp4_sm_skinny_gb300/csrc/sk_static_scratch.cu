// sk_gemm_rmsnorm_nvfp4_static: the pooler call (GEMM, pre-expert RMSNorm,
// NVFP4) for callers that cannot allocate device memory, such as the enqueue
// function of an inference-engine plugin that is handed no workspace, or a
// serving loop whose device memory is budgeted once at start-up. The GEMM
// output that the norm reads back lives in a fixed array in the library's
// device image instead of a caller-provided workspace.
//
// The array exists once per device that loads the library and is held until
// the process exits, or until the context that holds it is destroyed (for
// example by cudaDeviceReset); the next call then looks its address up again.
// Every call on a device shares it and it keeps the last call's contents;
// nothing in it has to start at zero, because the GEMM overwrites the part the
// norm reads before the norm reads it. Calls that can overlap on the GPU
// (different streams without ordering between them) race on it and must not be
// issued.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sk.h"
#include "sk_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = SK_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
// The array's device address per device, with the unique ID of the context it
// was looked up in: a device reset (or another context made current) replaces
// the module image that holds the array, so the address is looked up again
// whenever the current context's ID differs.
struct ScratchAddr {
  unsigned long long ctx_id;
  void *addr;
};
ScratchAddr g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique ID of the calling thread's current CUDA context (driver entry points
// cuCtxGetCurrent and cuCtxGetId, CUDA 12.0 and later); false if unavailable.
bool current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" sk_status sk_gemm_rmsnorm_nvfp4_static(const void *x, const void *w, const void *norm_w,
                                                  float eps, float gain_center,
                                                  const float *global_scale, uint8_t *a,
                                                  uint8_t *a_sf, void *z_out, int m, int n, int k,
                                                  int splits, void *stream) {
  char msg[256];
  if (m >= 1 && n >= 1 &&
      static_cast<size_t>(m) * static_cast<size_t>(n) * 2 > kStaticScratchBytes) {
    snprintf(msg, sizeof msg,
             "m=%d, n=%d: the GEMM output (%zu bytes) exceeds the static scratch of %zu bytes "
             "(m * n <= %zu)",
             m, n, static_cast<size_t>(m) * n * 2, kStaticScratchBytes, kStaticScratchBytes / 2);
    return sk::report_error(SK_ERR_INVALID_ARG, msg);
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "no usable CUDA device: %s", cudaGetErrorString(e));
    return sk::report_error(SK_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) return sk::report_error(SK_ERR_CUDA, "device index out of range");
  // The ID of the context the kernels will run in. Before the runtime's first
  // use on this thread no context is current yet: cudaSetDevice makes the
  // device's primary context current (it allocates nothing).
  unsigned long long ctx_id = 0;
  if (!current_context_id(&ctx_id)) {
    e = cudaSetDevice(dev);
    if (e != cudaSuccess || !current_context_id(&ctx_id)) {
      snprintf(msg, sizeof msg, "cannot identify the current CUDA context on device %d: %s", dev,
               cudaGetErrorString(e));
      return sk::report_error(SK_ERR_CUDA, msg);
    }
  }
  void *scratch = nullptr;
  {
    // One-time set-up per device and context, with that device current: the
    // device address of the array (its name in host code is only a host-side
    // handle).
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr &slot = g_scratch[dev];
    if (!slot.addr || slot.ctx_id != ctx_id) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "static scratch address on device %d: %s", dev,
                 cudaGetErrorString(e));
        return sk::report_error(SK_ERR_CUDA, msg);
      }
      slot.ctx_id = ctx_id;
      slot.addr = p;
    }
    scratch = slot.addr;
  }
  return sk_gemm_rmsnorm_nvfp4(x, w, norm_w, eps, gain_center, global_scale, a, a_sf, z_out,
                               scratch, kStaticScratchBytes, m, n, k, splits, stream);
}
