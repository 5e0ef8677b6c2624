// Status strings, device checks and launch accounting for libdora.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace dora {

std::atomic<uint64_t> g_launches{0};

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_known[kMaxDevices] = {};
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
}  // namespace

uint64_t context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<CtxGetCurrentFn>(a);
      get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
  });
  if (!get_current || !get_id) return 0;
  // no context yet (the runtime creates it on first real use): 0, so the
  // caller's set-up runs and records the id that exists after it
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

dora_status current_device(DeviceInfo *info, int *device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DORA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_known[dev]) {
      int major = 0, minor = 0, sms = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DORA_ERR_CUDA;
      g_info[dev].ok_arch = (major == 10 && minor == 3) ? 1 : 0;
      g_info[dev].sms = sms;
      g_known[dev] = true;
    }
    *info = g_info[dev];
  }
  if (device) *device = dev;
  return info->ok_arch ? DORA_OK : DORA_ERR_ARCH;
}

}  // namespace dora

extern "C" const char *dora_status_str(dora_status st) {
  switch (st) {
    case DORA_OK: return "DORA_OK";
    case DORA_ERR_NULL: return "DORA_ERR_NULL: a required pointer is NULL";
    case DORA_ERR_SHAPE: return "DORA_ERR_SHAPE: invalid size";
    case DORA_ERR_ALIGN: return "DORA_ERR_ALIGN: pointer or row stride misaligned";
    case DORA_ERR_DTYPE: return "DORA_ERR_DTYPE: unknown activation dtype";
    case DORA_ERR_WORKSPACE: return "DORA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case DORA_ERR_ARCH: return "DORA_ERR_ARCH: current device is not sm_103";
    case DORA_ERR_CUDA: return "DORA_ERR_CUDA: CUDA call or kernel launch failed";
    case DORA_ERR_DEVICE: return "DORA_ERR_DEVICE: a kernel gave up waiting on an on-chip barrier";
  }
  return "DORA_ERR_UNKNOWN";
}

extern "C" uint64_t dora_kernel_launches(void) {
  return dora::g_launches.load(std::memory_order_relaxed);
}
