// Host-side helpers shared by the libmedusa translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "medusa.h"

namespace medusa {

// Record a message for medusa_last_error() and return `code`.
int fail(int code, const char* fmt, ...);
// Map a CUDA error after a launch to MEDUSA_ERR_CUDA (or MEDUSA_OK).
int check_launch(const char* what);
// Streaming multiprocessors of the current device (cached per device).
int sm_count();
// Validate a medusa_tree_t (host fields and non-null device arrays).
int check_tree(const medusa_tree_t* tree, const char* what);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch through cudaLaunchKernelEx (arguments coerced to the kernel's types).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace medusa
