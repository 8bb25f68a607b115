// Device-side error reporting.  Kernels never trap: a wait that runs out of time, or a launch
// that finds an impossible configuration, records a code here and returns.  The host reads
// and clears the word in fa_sync_status().
//
// The library is built without relocatable device code, so every translation unit that
// launches kernels owns its own status word; FA_DEFINE_STATUS_FETCH gives each one a host
// accessor that fa_sync_status() calls in turn.
#pragma once

#include <cuda_runtime.h>

#include "fa_kernels.h"

namespace fa {

static __device__ unsigned int g_dev_status = 0;
static __device__ int g_dev_where = 0;

__device__ __forceinline__ void report_device_error(unsigned int code, int where) {
  atomicOr(&g_dev_status, code);
  atomicExch(&g_dev_where, where);
}

}  // namespace fa

// Host accessor: copy this TU's status word out (after synchronising ``stream``) and clear it.
#define FA_DEFINE_STATUS_FETCH(NAME)                                                         \
  namespace fa {                                                                             \
  cudaError_t NAME(cudaStream_t stream, unsigned int* code, int* where) {                    \
    cudaError_t e = cudaStreamSynchronize(stream);                                           \
    if (e != cudaSuccess) return e;                                                          \
    e = cudaMemcpyFromSymbol(code, g_dev_status, sizeof(unsigned int));                      \
    if (e != cudaSuccess) return e;                                                          \
    e = cudaMemcpyFromSymbol(where, g_dev_where, sizeof(int));                               \
    if (e != cudaSuccess) return e;                                                          \
    if (*code) {                                                                             \
      const unsigned int zero = 0;                                                           \
      e = cudaMemcpyToSymbol(g_dev_status, &zero, sizeof(unsigned int));                     \
    }                                                                                        \
    return e;                                                                                \
  }                                                                                          \
  }
