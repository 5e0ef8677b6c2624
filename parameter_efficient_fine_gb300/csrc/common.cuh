// Host-side helpers shared by the libdora translation units.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/dora.h"

namespace dora {

// Kernel launches issued by this process through the library.
extern std::atomic<uint64_t> g_launches;

inline void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Per-device facts, read once per device.
struct DeviceInfo {
  int ok_arch;    // 1 when the device is sm_103
  int sms;        // streaming multiprocessors
};

// Returns DORA_OK and fills *info for the current device; DORA_ERR_ARCH when the
// device is not sm_103; DORA_ERR_CUDA when the runtime cannot answer.
dora_status current_device(DeviceInfo *info, int *device);

// Process-unique id of the calling thread's current CUDA context (the driver's
// context id, never reused within a process); 0 when it cannot be read or no
// context is current yet (0 never matches a recorded id).
// Per-device set-up that belongs to a context (symbol addresses, kernel
// attributes) is keyed on it, so a device reset -- which destroys the context
// and reloads the library's module -- makes that set-up run again.
uint64_t context_id();

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The device error word that the library's kernels write when a bounded wait
// gives up (read and cleared by dora_device_error); sets up the tensor-core
// kernels' shared-memory limits on first use of a device.
dora_status error_word(int device, int **errp);

// Device addresses of the failure-test hook (see dora_test_stall_loads): a
// flag that makes the tensor-core producers withhold their loads, and the
// limit of the bounded waits.
dora_status test_hooks(int **stall, unsigned long long **limit_ns);

inline dora_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? DORA_OK : DORA_ERR_CUDA;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace dora
