// Kernel attributes set with cudaFuncSetAttribute belong to the current
// device, so a process that drives several GPUs must set them on each: the
// launchers keep one "done" flag per device.
#pragma once

#include <atomic>

#include <cuda_runtime.h>

namespace mla {

constexpr int kMaxDevices = 64;
using DeviceFlags = std::atomic<bool>[kMaxDevices];

// Runs `set` (returning cudaError_t) once per device; a failure is returned
// and retried on the next call.
template <class F>
cudaError_t once_per_device(DeviceFlags& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace mla
