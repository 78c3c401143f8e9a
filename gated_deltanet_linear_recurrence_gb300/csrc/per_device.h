// per_device.h — host set-up that must happen once on each device.
// Kernel attributes (the opt-in shared-memory size) belong to a device: a
// process that launches on several GPUs sets them on each one it uses.
#pragma once
#include <cuda_runtime.h>

#include <mutex>

namespace gdn {

class PerDeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;
  // Runs f() (returning cudaError_t) on the current device unless it already
  // succeeded there; a failure is returned and retried on the next call.
  template <typename F>
  cudaError_t run(F&& f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return cudaSuccess;
    e = f();
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

}  // namespace gdn
