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

// Index of the current device, or -1.
int current_device_index();

// Per-device once-only set-up of a kernel: runs `fn` (returning a
// cudaError_t) the first time it is called for (slot, device) and caches a
// success; later calls return cudaSuccess without touching the runtime, so
// that a call sequence can be captured into a CUDA graph.  `slot` names the
// kernel (a small integer per kernel instantiation).
template <typename F>
cudaError_t once_per_device(int slot, F &&fn);

// Cached cudaOccupancyMaxActiveClusters result for (slot, device), or -1.
int cached_clusters(int slot);
void cache_clusters(int slot, int clusters);

// Diagnostics (bounded-wait tests): the CTA-pair per-tensor GEMM and the
// block-scaled GEMM with their first TMA arrival withheld.
fp8la_status diag_pair_withheld(const uint8_t *A, int64_t lda, const uint8_t *B,
                                int64_t ldb, uint16_t *C, int64_t ldc,
                                int64_t M, int64_t N, int64_t K,
                                const float *scale_a, const float *scale_b,
                                cudaStream_t s);
fp8la_status diag_block32_withheld(const uint8_t *A, int64_t lda,
                                   const uint8_t *B, int64_t ldb, uint16_t *C,
                                   int64_t ldc, int64_t M, int64_t N, int64_t K,
                                   const float *sa, int64_t ld_sa,
                                   const float *sb, int64_t ld_sb,
                                   cudaStream_t s);

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline fp8la_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FP8LA_OK : FP8LA_ERR_CUDA;
}

namespace detail {
constexpr int kSlots = 16;
constexpr int kDevs = 64;
bool setup_done(int slot, int dev);
void mark_setup_done(int slot, int dev);
}  // namespace detail

template <typename F>
cudaError_t once_per_device(int slot, F &&fn) {
  const int dev = current_device_index();
  if (dev < 0 || slot < 0 || slot >= detail::kSlots) return fn();
  if (detail::setup_done(slot, dev)) return cudaSuccess;
  const cudaError_t e = fn();
  if (e == cudaSuccess) detail::mark_setup_done(slot, dev);
  return e;
}

}  // namespace fp8la
