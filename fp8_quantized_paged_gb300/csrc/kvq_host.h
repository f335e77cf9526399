// kvq_host.h -- host-side helpers shared by the entry points of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

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
