// kvq_host.h -- host-side helpers shared by the entry points of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace kvq {

// Per-device one-time setup (kernel attributes, symbol addresses) that is
// recorded only once it succeeds: run(dev, f) calls f under a lock until f
// returns true for that device, after which it returns true at once.  A
// failure leaves the device unmarked and clears the CUDA error it left, so
// the next call tries again.  Devices 0 .. 63.
class DeviceOnce {
 public:
  template <typename F>
  bool run(int dev, F&& f) {
    if (dev < 0 || dev >= kMaxDev) return false;
    if (done_[dev].load(std::memory_order_acquire)) return true;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return true;
    if (!f()) {
      cudaGetLastError();
      return false;
    }
    done_[dev].store(true, std::memory_order_release);
    return true;
  }

 private:
  static constexpr int kMaxDev = 64;
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDev]{};
};

// The current device, or -1 (its error cleared) if there is none.
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (cached per device); 0 if no device.
int device_sm_count();

// Launch shape of a kernel whose threads each keep one of the row_units
// chunks of a token row and stride over tokens: a block is the largest
// multiple of row_units that fits 256 threads (or 256 threads, with the grid
// a multiple of the blocks that make up whole rows); the grid fills the SMs
// once (blocks_per_sm blocks of 256 per SM) or covers the tokens, if fewer.
void token_row_shape(int64_t num_tokens, int row_units, int blocks_per_sm, int& grid, int& block);

// Launch with programmatic stream serialization (the kernel must call
// griddepcontrol.wait before reading data written by earlier kernels).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace kvq
