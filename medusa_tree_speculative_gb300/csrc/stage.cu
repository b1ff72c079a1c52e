// Host <-> device plumbing of a step: the inputs' copy from pinned host
// memory, and the read-out of the device error word.
//
// Copy of a step's inputs from pinned host memory into device memory by a
// kernel.  On a GPU that reads host memory over a coherent chip-to-chip link,
// many CTAs with 16-byte loads in flight move a few megabytes sooner than one
// copy-engine transfer; the host buffer must be page-locked and mapped into
// the device's address space (the runtime is asked for its device address
// first, so the kernel never touches an unmapped page).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyLoads = 8;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads) copy_from_host_kernel(uint4* __restrict__ dst,
                                                                      const uint4* __restrict__ src, int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
  for (int64_t i0 = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; i0 < n16; i0 += stride * kCopyLoads) {
    uint4 v[kCopyLoads];
#pragma unroll
    for (int u = 0; u < kCopyLoads; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n16) v[u] = src[i];
    }
#pragma unroll
    for (int u = 0; u < kCopyLoads; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n16) dst[i] = v[u];
    }
  }
}

// One thread: the error word to its destination, then (clear) back to zero.
__global__ void check_errors_kernel(int32_t* err, int32_t* out, int clear) {
  const int32_t v = *reinterpret_cast<volatile int32_t*>(err);
  *out = v;
  if (clear) *err = 0;
}

// Device address of a pointer that is either device (or managed) memory or
// page-locked host memory mapped into the device's address space.
int device_view(const char* fn, void* p, void** out) {
  cudaPointerAttributes a{};
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MEDUSA_ERR_INVALID, "%s: pointer attributes: %s", fn, cudaGetErrorString(e));
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return MEDUSA_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *out = a.devicePointer;
    return MEDUSA_OK;
  }
  return fail(MEDUSA_ERR_INVALID, "%s: not device memory nor mapped pinned host memory", fn);
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_check_errors(int32_t* err, int32_t* out, int clear, void* stream) {
  const char* fn = "medusa_check_errors";
  if (!err || !out) return fail(MEDUSA_ERR_INVALID, "%s: NULL pointer", fn);
  if ((reinterpret_cast<uintptr_t>(err) | reinterpret_cast<uintptr_t>(out)) % 4)
    return fail(MEDUSA_ERR_INVALID, "%s: pointers must be 4-byte aligned", fn);
  void* err_dev = nullptr;
  void* out_dev = nullptr;
  if (int rc = device_view(fn, err, &err_dev)) return rc;
  if (int rc = device_view(fn, out, &out_dev)) return rc;
  launch_kernel(check_errors_kernel, dim3(1), dim3(1), 0, as_stream(stream), static_cast<int32_t*>(err_dev),
                static_cast<int32_t*>(out_dev), clear);
  return check_launch(fn);
}

extern "C" int medusa_copy_from_host(void* dst, const void* src_host, size_t bytes, void* stream) {
  const char* fn = "medusa_copy_from_host";
  if (bytes == 0) return MEDUSA_OK;
  if (!dst || !src_host) return fail(MEDUSA_ERR_INVALID, "%s: NULL pointer", fn);
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src_host) | bytes) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: pointers and size must be multiples of 16 bytes", fn);
  void* src_dev = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(&src_dev, const_cast<void*>(src_host), 0);
  if (e != cudaSuccess || !src_dev) {
    cudaGetLastError();  // the failed query's error is not left for the next call
    return fail(MEDUSA_ERR_INVALID, "%s: the source is not mapped pinned host memory (%s)", fn,
                cudaGetErrorString(e));
  }
  const int64_t n16 = (int64_t)(bytes / 16);
  const int64_t per_cta = (int64_t)kCopyThreads * kCopyLoads;
  const int grid = (int)std::min<int64_t>((n16 + per_cta - 1) / per_cta, 4 * sm_count());
  launch_kernel(copy_from_host_kernel, dim3(grid), dim3(kCopyThreads), 0, as_stream(stream),
                static_cast<uint4*>(dst), static_cast<const uint4*>(src_dev), n16);
  return check_launch(fn);
}
