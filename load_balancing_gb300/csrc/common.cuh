// Internal helpers shared by the library's translation units (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dbsp.h"

namespace dbsp {

// Records a CUDA error's text for dbsp_last_error_string() and returns DBSP_ERR_CUDA.
int cuda_fail(cudaError_t err, const char* where);

// Checks the current device once (compute capability 10.3 = GB300) and returns
// DBSP_OK, DBSP_ERR_UNSUPPORTED or DBSP_ERR_CUDA. *device receives the ordinal.
int check_device(int* device);

// Device address of the current device's error word (a static __device__ int).
int* error_word(int device);

// SM count of a device (cached).
int sm_count(int device);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch attribute: the kernel may start before the previous grid in the stream has
// finished (programmatic dependent launch); the kernel waits for that grid (griddepcontrol.wait)
// before it touches memory the grid produces or reads.
inline cudaLaunchAttribute overlap_previous_grid() {
  cudaLaunchAttribute a = {};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Device-side error reporting: first error wins.
__device__ __forceinline__ void report(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Launches kernel<<<grid, block, smem, stream>>>(args...) with overlap_previous_grid().
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {overlap_previous_grid()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace dbsp

#define DBSP_LAUNCH_CHECK(where)                                  \
  do {                                                            \
    cudaError_t e_ = cudaGetLastError();                          \
    if (e_ != cudaSuccess) return ::dbsp::cuda_fail(e_, where);   \
  } while (0)
