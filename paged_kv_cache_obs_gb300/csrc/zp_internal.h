// zp_internal.h — host-side helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/zipage.h"

namespace zp {

// Encodes a 3-D bf16 tiled tensor map with 128-byte swizzle.  dims/strides in elements/bytes
// (strides of dims 1 and 2), box in elements.  Returns false if the driver rejects it.
bool encode_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                         uint32_t box2);

// Number of SMs of the current device (cached per device).
int num_sms();

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Runs a set-up step once per device.  Kernel attributes such as the dynamic shared-memory
// limit belong to the device that is current when they are set, so a process that launches on
// several devices must set them on each.  run() calls fn() with the current device's index the
// first time that device is seen (under a lock) and remembers a success; a failure is returned
// and retried on the next call.
class PerDeviceInit {
 public:
  template <class Fn>
  cudaError_t run(Fn&& fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return cudaSuccess;
    e = fn();
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

// NVTX range over the host side of an entry point (a no-op unless a profiler listens), so
// that a timeline shows which call queued which kernels.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace zp
