// Host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fp8la.h"

namespace fp8la {

// Device status word of the current device (a __device__ variable's
// address, looked up once per device).  nullptr on failure.
unsigned *status_word_ptr();

// Current limit of every bounded wait, in nanoseconds.
uint64_t wait_timeout_ns();

// Number of SMs of the current device (cached per device); <= 0 on failure.
int sm_count();

// True if the current device is a compute-capability 10.x GPU.
bool device_is_sm10x();

// cuTensorMapEncodeTiled, fetched from the driver once (nullptr on failure).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType,
                                   cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline fp8la_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FP8LA_OK : FP8LA_ERR_CUDA;
}

}  // namespace fp8la
