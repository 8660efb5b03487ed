// E4M3 quantisers: per-tensor (amax grid reduction + cast) and 32x32 block.
//
// Method: [P1] "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核", risks
// paragraph (E4M3 spans +-448; per-tensor scaling avoids overflow) and
// optimisation parameter list (scale_max = 448); [P3] "JAX 中使用 Triton 优化
// Blackwell GPU 的 FP8 GEMM 内核", implementation paragraph (32x32 scale
// blocks).  Per tensor (or tile): amax = max|x| (NaN ignored), qscale =
// fp32(448/amax), scale = fp32(amax/448) (amax == 0 or qscale not finite:
// both 1), q = E4M3 round-to-nearest-even saturating of fp32(x * qscale).
//
// The kernels are HBM-bound streams.  The per-tensor path is two launches:
// a 128-bit-load grid reduction whose blocks combine their maxima with one
// atomicMax on the float's bit pattern (non-negative floats order like
// their unsigned bit patterns; max is exact, so the result does not depend
// on the order), then a cast pass that walks the tensor backwards so that
// it starts on the part the reduction left in L2.  Contiguous tensors of at
// most 512K floats take one launch instead: one 16-CTA cluster does both
// passes and combines the CTAs' maxima through distributed shared memory.
// The block quantiser needs one pass: a 32x32 fp32 tile (4 KB) fits one
// warp's registers.  Delayed scaling (the scale from a carried-over amax)
// also needs one pass, which casts and records the new amax together.
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8la {
namespace {

// Grid of the per-tensor passes: two 512-thread blocks per SM.  The
// register cap of the launch bounds (three blocks' worth, <= 40 registers a
// thread) leaves room on every SM for one CTA of the persistent GEMM (320
// threads) beside at least one of the blocks, so that the quantisation of
// the next operands can run on the same SMs while a GEMM is in flight on
// another stream.  Four blocks of 512 threads fill the register file, and
// the GEMM then waits for the whole pass to finish.
constexpr int kThreads = 512;
constexpr int kBlocksPerSm = 2;
constexpr int kMinBlocksBound = 3;
constexpr int kBlock32PerSm = 4;
// Bytes of x's tail that the amax pass asks L2 to keep for the cast pass
// (L2 is 129 MB; the rest of it holds the codes being written and other
// work's data).  96 MB measured 1.5 % faster than 64 MB for an 8192 x 8192
// operand, 112 MB no faster than 96.
constexpr int64_t kL2KeepBytes = int64_t(96) << 20;

// FP8 formats: 0 = E4M3 (max 448), 1 = E5M2 (max 57344).
template <int FMT>
struct Fp8Format;
template <>
struct Fp8Format<0> {
  static constexpr float kMax = 448.0f;
  static constexpr __nv_fp8_interpretation_t kKind = __NV_E4M3;
};
template <>
struct Fp8Format<1> {
  static constexpr float kMax = 57344.0f;
  static constexpr __nv_fp8_interpretation_t kKind = __NV_E5M2;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// fmaxf returns the non-NaN operand, so NaNs drop out of the maximum.
__device__ __forceinline__ float max_abs4(float m, float4 v) {
  return fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))),
               fabsf(v.w));
}

__device__ __forceinline__ void block_max_into(float v, float *out) {
  __shared__ float red[kThreads / 32];
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = (l < static_cast<int>(blockDim.x >> 5)) ? red[l] : 0.0f;
    v = warp_max(v);
    if (l == 0)
      atomicMax(reinterpret_cast<unsigned *>(out), __float_as_uint(v));
  }
}

struct Scales {
  float qscale, scale;
};

template <int FMT = 0>
__device__ __forceinline__ Scales scales_from_amax(float amax) {
  Scales s;
  s.qscale = __fdiv_rn(Fp8Format<FMT>::kMax, amax);
  s.scale = __fdiv_rn(amax, Fp8Format<FMT>::kMax);
  if (amax == 0.0f || !isfinite(s.qscale)) {
    s.qscale = 1.0f;
    s.scale = 1.0f;
  }
  return s;
}

// Two fp32 values -> two FP8 codes (low byte = first value).
template <int FMT = 0>
__device__ __forceinline__ uint32_t cvt2(float a, float b, float qs) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
      make_float2(__fmul_rn(a, qs), __fmul_rn(b, qs)), __NV_SATFINITE,
      Fp8Format<FMT>::kKind));
}

template <int FMT = 0>
__device__ __forceinline__ uint32_t cvt4(float4 v, float qs) {
  return cvt2<FMT>(v.x, v.y, qs) | (cvt2<FMT>(v.z, v.w, qs) << 16);
}

template <int FMT = 0>
__device__ __forceinline__ uint8_t cvt1(float a, float qs) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(
      __fmul_rn(a, qs), __NV_SATFINITE, Fp8Format<FMT>::kKind));
}

__device__ __forceinline__ float4 ld_stream4(const float4 *p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// L2 eviction-priority policies for 128-bit loads.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float4 ld_hint4(const float4 *p, uint64_t policy) {
  float4 v;
  asm volatile(
      "ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p), "l"(policy));
  return v;
}

// ------------------------------------------------------------------- amax
// VEC = 4: x, ldx and cols allow 16-byte loads; VEC = 1: scalar loads.
// A unit is VEC consecutive elements of one row; units are numbered row by
// row, `upr` units per row.
// `keep_from`: units at or past this index are loaded with an evict-last
// L2 policy (the rest evict-first), so that the part of x the cast pass
// reads first -- it walks the tensor backwards -- is still in L2.
template <int VEC>
__global__ void __launch_bounds__(kThreads, kMinBlocksBound)
    amax_kernel(const float *__restrict__ x, int64_t rows, int64_t upr,
                int64_t ldx, bool contiguous, int64_t keep_from,
                float *amax_out) {
  const int64_t n = rows * upr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  float m = 0.0f;
  if (VEC == 4) {
    if (contiguous) {
      const float4 *x4 = reinterpret_cast<const float4 *>(x);
      const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
      for (; i + 3 * stride < n; i += 4 * stride) {
        const uint64_t pol = i + 3 * stride >= keep_from ? keep : drop;
        const float4 a = ld_hint4(x4 + i, pol);
        const float4 b = ld_hint4(x4 + i + stride, pol);
        const float4 c = ld_hint4(x4 + i + 2 * stride, pol);
        const float4 d = ld_hint4(x4 + i + 3 * stride, pol);
        m = max_abs4(max_abs4(m, a), b);
        m = max_abs4(max_abs4(m, c), d);
      }
      for (; i < n; i += stride)
        m = max_abs4(m, ld_hint4(x4 + i, i >= keep_from ? keep : drop));
    } else {
      for (; i < n; i += stride) {
        const int64_t r = i / upr, c = i - r * upr;
        m = max_abs4(m, ld_stream4(reinterpret_cast<const float4 *>(
                            x + r * ldx + c * 4)));
      }
    }
  } else {
    for (; i < n; i += stride) {
      const int64_t r = i / upr, c = i - r * upr;
      m = fmaxf(m, fabsf(x[r * ldx + c]));
    }
  }
  block_max_into(m, amax_out);
}

// ------------------------------------------------------------------- cast
template <int VEC, int FMT>
__global__ void __launch_bounds__(kThreads, kMinBlocksBound)
    cast_kernel(const float *__restrict__ x, int64_t rows, int64_t upr,
                int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                bool contiguous, const float *amax_in, float *scale_out) {
  const Scales s = scales_from_amax<FMT>(*amax_in);
  // A GEMM launched next may start its set-up now; it waits for this
  // kernel to finish before reading the codes or the scale.
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s.scale;
  const float qs = s.qscale;
  const int64_t n = rows * upr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (VEC == 4) {
    if (contiguous) {
      // Walk the tensor from its end: the amax pass has just streamed it
      // front to back, so its tail is still in L2.  Unit u = n - 1 - i.
      const float4 *x4 = reinterpret_cast<const float4 *>(x);
      uint32_t *q4 = reinterpret_cast<uint32_t *>(q);
      const int64_t last = n - 1;
      const uint64_t drop = policy_evict_first();   // last use of x
      for (; i + 3 * stride < n; i += 4 * stride) {
        const float4 a = ld_hint4(x4 + (last - i), drop);
        const float4 b = ld_hint4(x4 + (last - i - stride), drop);
        const float4 c = ld_hint4(x4 + (last - i - 2 * stride), drop);
        const float4 d = ld_hint4(x4 + (last - i - 3 * stride), drop);
        q4[last - i] = cvt4<FMT>(a, qs);
        q4[last - i - stride] = cvt4<FMT>(b, qs);
        q4[last - i - 2 * stride] = cvt4<FMT>(c, qs);
        q4[last - i - 3 * stride] = cvt4<FMT>(d, qs);
      }
      for (; i < n; i += stride)
        q4[last - i] = cvt4<FMT>(ld_hint4(x4 + (last - i), drop), qs);
    } else {
      for (; i < n; i += stride) {
        const int64_t r = i / upr, c = i - r * upr;
        const float4 v = ld_stream4(
            reinterpret_cast<const float4 *>(x + r * ldx + c * 4));
        *reinterpret_cast<uint32_t *>(q + r * ldq + c * 4) = cvt4<FMT>(v, qs);
      }
    }
  } else {
    for (; i < n; i += stride) {
      const int64_t r = i / upr, c = i - r * upr;
      q[r * ldq + c] = cvt1<FMT>(x[r * ldx + c], qs);
    }
  }
}

// ------------------------------------------------ delayed-scaling one pass
// Codes with the scale of a carried-over amax (amax_prev), and this
// tensor's own amax recorded in amax_out for the next call: one read of x
// (4 B) and one write of codes (1 B) per element.  Eight 16-byte loads per
// thread are in flight before their codes are stored (3 % more bandwidth
// than four); the register cap of two blocks per SM still leaves room for
// one CTA of the persistent GEMM beside one block.
template <int VEC, int FMT>
__global__ void __launch_bounds__(kThreads, 2)
    delayed_kernel(const float *__restrict__ x, int64_t rows, int64_t upr,
                   int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                   bool contiguous, const float *amax_prev, float *amax_out,
                   float *scale_out) {
  const Scales s = scales_from_amax<FMT>(*amax_prev);
  // A GEMM launched next may start its set-up now; it waits for this
  // kernel to finish before reading the codes or the scale.
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s.scale;
  const float qs = s.qscale;
  const int64_t n = rows * upr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  float m = 0.0f;
  if (VEC == 4) {
    if (contiguous) {
      const float4 *x4 = reinterpret_cast<const float4 *>(x);
      uint32_t *q4 = reinterpret_cast<uint32_t *>(q);
      const uint64_t drop = policy_evict_first();
      for (; i + 7 * stride < n; i += 8 * stride) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = ld_hint4(x4 + i + j * stride, drop);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = max_abs4(m, v[j]);
#pragma unroll
        for (int j = 0; j < 8; ++j) q4[i + j * stride] = cvt4<FMT>(v[j], qs);
      }
      for (; i < n; i += stride) {
        const float4 v = ld_hint4(x4 + i, drop);
        m = max_abs4(m, v);
        q4[i] = cvt4<FMT>(v, qs);
      }
    } else {
      for (; i < n; i += stride) {
        const int64_t r = i / upr, c = i - r * upr;
        const float4 v = ld_stream4(
            reinterpret_cast<const float4 *>(x + r * ldx + c * 4));
        m = max_abs4(m, v);
        *reinterpret_cast<uint32_t *>(q + r * ldq + c * 4) = cvt4<FMT>(v, qs);
      }
    }
  } else {
    for (; i < n; i += stride) {
      const int64_t r = i / upr, c = i - r * upr;
      const float v = x[r * ldx + c];
      m = fmaxf(m, fabsf(v));
      q[r * ldq + c] = cvt1<FMT>(v, qs);
    }
  }
  block_max_into(m, amax_out);
}

// 32-bit load from the shared memory of a CTA of the cluster (cluster
// address from mapa_shared).
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];"
               : "=f"(v)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

// ------------------------------------------ small tensors: one launch
// For a contiguous tensor of at most kSmallMaxUnits float4 units, where
// launches rather than bytes set the time of the two-pass path, one
// cluster of kSmallCluster CTAs takes both passes in a single launch.  Each
// CTA reduces its share of x to a block maximum in its shared memory; after
// a cluster barrier, warp 0 of every CTA reads the kSmallCluster block maxima
// through distributed shared memory, so every CTA holds the tensor's amax
// without a global atomic (and amax_out needs no clearing); a second cluster
// barrier keeps each CTA's shared memory alive until its peers have read it.
// Each CTA then casts its share; the second read of x hits L2.
constexpr int kSmallCluster = 16;
constexpr int kSmallThreads = 1024;
// Up to 512K floats (2 MB): beyond that the two-pass grid path over all SMs
// is as fast (a 4 MB tensor takes 8.4 µs either way on a GB300) and then
// faster.
constexpr int64_t kSmallMaxUnits = int64_t(1) << 17;

template <int FMT>
__global__ void __launch_bounds__(kSmallThreads, 1)
    quantize_small_kernel(const float4 *__restrict__ x4, int64_t n,
                          uint32_t *__restrict__ q4, float *amax_out,
                          float *scale_out) {
  __shared__ float red[kSmallThreads / 32];
  // A GEMM launched next may start its set-up now; it waits for this
  // kernel to finish before reading the codes or the scale.
  pdl_launch_dependents();
  __shared__ float cta_max;
  const uint32_t rank = cluster_ctarank();
  const int64_t stride = static_cast<int64_t>(kSmallCluster) * kSmallThreads;
  const int64_t first = static_cast<int64_t>(rank) * kSmallThreads + threadIdx.x;
  // Eight 16-byte loads in flight per thread (128 KB per SM).
  float m = 0.0f;
  int64_t i = first;
  for (; i + 7 * stride < n; i += 8 * stride) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = ld_stream4(x4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) m = max_abs4(m, v[u]);
  }
  for (; i < n; i += stride) m = max_abs4(m, ld_stream4(x4 + i));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  m = warp_max(m);
  if (l == 0) red[w] = m;
  __syncthreads();
  if (w == 0) {
    const float v = warp_max(red[l]);
    if (l == 0) cta_max = v;
  }
  cluster_sync_all();            // every CTA's cta_max is visible
  if (w == 0) {
    float v = 0.0f;
    if (l < kSmallCluster)
      v = ld_shared_cluster_f32(
          mapa_shared(smem_addr(&cta_max), static_cast<uint32_t>(l)));
    v = warp_max(v);
    if (l == 0) red[0] = v;
  }
  cluster_sync_all();            // peers done reading; red[0] visible
  const float amax = red[0];
  const Scales s = scales_from_amax<FMT>(amax);
  if (rank == 0 && threadIdx.x == 0) {
    *amax_out = amax;
    *scale_out = s.scale;
  }
  const uint64_t drop = policy_evict_first();   // last use of x
  for (i = first; i + 7 * stride < n; i += 8 * stride) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = ld_hint4(x4 + i + u * stride, drop);
#pragma unroll
    for (int u = 0; u < 8; ++u) q4[i + u * stride] = cvt4<FMT>(v[u], s.qscale);
  }
  for (; i < n; i += stride) q4[i] = cvt4<FMT>(ld_hint4(x4 + i, drop), s.qscale);
}

// --------------------------------------------------------- 32x32 block cast
// One warp per 32x32 tile.  VEC = 4: lane l covers columns 4*(l%8)..+3 of
// rows l/8, l/8+4, ..., l/8+28 with 16-byte loads; VEC = 1: lane l covers
// column l of all 32 rows.  Out-of-range elements are left out of the amax
// and not stored.
template <int VEC>
__global__ void __launch_bounds__(256)
    block32_kernel(const float *__restrict__ x, int64_t rows, int64_t cols,
                   int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                   float *__restrict__ scales, int64_t ld_scales,
                   int64_t tiles_r, int64_t tiles_c) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total =
      static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) +
                   (threadIdx.x >> 5);
       t < tiles_r * tiles_c; t += warps_total) {
    const int64_t tr = t / tiles_c, tc = t - tr * tiles_c;
    const int64_t r0 = tr * 32, c0 = tc * 32;
    if (VEC == 4 && r0 + 32 <= rows && c0 + 32 <= cols) {
      // Interior tile: no bounds checks, rows reached by a constant step.
      const int64_t rstep = 4 * ldx;
      const float *xp = x + (r0 + (lane >> 3)) * ldx + c0 + 4 * (lane & 7);
      float4 v[8];
      float m = 0.0f;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        v[it] = ld_stream4(reinterpret_cast<const float4 *>(xp + it * rstep));
        m = max_abs4(m, v[it]);
      }
      const float amax = warp_max(m);
      const Scales s = scales_from_amax(amax);
      if (lane == 0) scales[tr * ld_scales + tc] = s.scale;
      const int64_t qstep = 4 * ldq;
      uint8_t *qp = q + (r0 + (lane >> 3)) * ldq + c0 + 4 * (lane & 7);
#pragma unroll
      for (int it = 0; it < 8; ++it)
        *reinterpret_cast<uint32_t *>(qp + it * qstep) = cvt4(v[it], s.qscale);
    } else if (VEC == 4) {
      const int64_t col = c0 + 4 * (lane & 7);
      const bool col_ok = col < cols;
      float4 v[8];
      float m = 0.0f;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int64_t row = r0 + (lane >> 3) + 4 * it;
        if (col_ok && row < rows) {
          v[it] = ld_stream4(
              reinterpret_cast<const float4 *>(x + row * ldx + col));
          m = max_abs4(m, v[it]);
        } else {
          v[it] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      const float amax = warp_max(m);
      const Scales s = scales_from_amax(amax);
      if (lane == 0) scales[tr * ld_scales + tc] = s.scale;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int64_t row = r0 + (lane >> 3) + 4 * it;
        if (col_ok && row < rows)
          *reinterpret_cast<uint32_t *>(q + row * ldq + col) =
              cvt4(v[it], s.qscale);
      }
    } else {
      const int64_t col = c0 + lane;
      const bool col_ok = col < cols;
      float v[32];
      float m = 0.0f;
#pragma unroll
      for (int it = 0; it < 32; ++it) {
        const int64_t row = r0 + it;
        v[it] = (col_ok && row < rows) ? x[row * ldx + col] : 0.0f;
        m = fmaxf(m, fabsf(v[it]));
      }
      const float amax = warp_max(m);
      const Scales s = scales_from_amax(amax);
      if (lane == 0) scales[tr * ld_scales + tc] = s.scale;
#pragma unroll
      for (int it = 0; it < 32; ++it) {
        const int64_t row = r0 + it;
        if (col_ok && row < rows) q[row * ldq + col] = cvt1(v[it], s.qscale);
      }
    }
  }
}

// Grid of a grid-stride launch: enough blocks for `units` threads' worth of
// work, at most `per_sm` blocks per SM.
int grid_for(int64_t units, int threads, int per_sm = kBlocksPerSm) {
  const int sms = sm_count();
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * per_sm;
  int64_t g = (units + threads - 1) / threads;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace
}  // namespace fp8la

using namespace fp8la;

namespace fp8la {
namespace {

// Whether this device can run quantize_small_kernel (a cluster of
// kSmallCluster CTAs of kSmallThreads threads, a non-portable cluster
// size); checked once per device, before any stream capture.
template <int FMT>
bool small_path_ready() {
  const int slot = 10 + FMT;
  // The cache holds the cluster count + 1, so that "none" is remembered too.
  const int cached = cached_clusters(slot);
  int c = cached > 0 ? cached - 1 : -1;
  if (c < 0) {
    c = 0;
    if (cudaFuncSetAttribute(quantize_small_kernel<FMT>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kSmallCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(kSmallCluster, 1, 1);
      cfg.blockDim = dim3(kSmallThreads, 1, 1);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&c, quantize_small_kernel<FMT>,
                                         &cfg) != cudaSuccess)
        c = 0;
    }
    cudaGetLastError();   // a refusal here only disables the small path
    cache_clusters(slot, c + 1);
  }
  return c > 0;
}

template <int FMT>
fp8la_status quantize_pertensor_impl(const float *x, int64_t rows,
                                     int64_t cols, int64_t ldx, uint8_t *q,
                                     int64_t ldq, float *amax_out,
                                     float *scale_out, cudaStream_t s) {
  if (!amax_out || !scale_out || rows < 0 || cols < 0)
    return FP8LA_ERR_INVALID_ARG;
  // The cast blocks read amax_out while the first of them writes scale_out.
  if (static_cast<void *>(amax_out) == static_cast<void *>(scale_out))
    return FP8LA_ERR_INVALID_ARG;
  const bool empty = rows == 0 || cols == 0;
  if (!empty && (!x || !q || ldx < cols || ldq < cols))
    return FP8LA_ERR_INVALID_ARG;
  if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40))
    return FP8LA_ERR_UNSUPPORTED;
  if (sm_count() <= 0) return FP8LA_ERR_CUDA;
  if (empty) {
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess)
      return FP8LA_ERR_CUDA;
    cast_kernel<1, FMT><<<1, 32, 0, s>>>(x, 0, 0, 0, q, 0, true, amax_out,
                                         scale_out);
    return launch_status();
  }
  const bool vec4 = cols % 4 == 0 && ldx % 4 == 0 && ldq % 4 == 0 &&
                    aligned16(x) &&
                    (reinterpret_cast<uintptr_t>(q) & 3u) == 0;
  const bool contiguous = ldx == cols && ldq == cols;
  if (vec4 && contiguous && rows * (cols / 4) <= kSmallMaxUnits &&
      small_path_ready<FMT>()) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmallCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(kSmallCluster, 1, 1);
    cfg.blockDim = dim3(kSmallThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, quantize_small_kernel<FMT>,
                           reinterpret_cast<const float4 *>(x),
                           rows * (cols / 4), reinterpret_cast<uint32_t *>(q),
                           amax_out, scale_out) != cudaSuccess)
      return FP8LA_ERR_CUDA;
    return launch_status();
  }
  if (cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  if (vec4) {
    const int64_t upr = cols / 4;
    const int g = grid_for(rows * upr, kThreads);
    // Keep up to kL2KeepBytes of x's tail resident for the cast pass.
    const int64_t units = rows * upr;
    const int64_t keep_units = kL2KeepBytes / 16;
    const int64_t keep_from = units > keep_units ? units - keep_units : 0;
    amax_kernel<4><<<g, kThreads, 0, s>>>(x, rows, upr, ldx, contiguous,
                                          keep_from, amax_out);
    cast_kernel<4, FMT><<<g, kThreads, 0, s>>>(x, rows, upr, ldx, q, ldq,
                                               contiguous, amax_out, scale_out);
  } else {
    const int g = grid_for(rows * cols, kThreads);
    amax_kernel<1><<<g, kThreads, 0, s>>>(x, rows, cols, ldx, contiguous, 0,
                                          amax_out);
    cast_kernel<1, FMT><<<g, kThreads, 0, s>>>(x, rows, cols, ldx, q, ldq,
                                               contiguous, amax_out, scale_out);
  }
  return launch_status();
}

template <int FMT>
fp8la_status quantize_delayed_impl(const float *x, int64_t rows, int64_t cols,
                                   int64_t ldx, uint8_t *q, int64_t ldq,
                                   const float *amax_prev, float *amax_out,
                                   float *scale_out, cudaStream_t s) {
  if (!amax_prev || !amax_out || !scale_out || rows < 0 || cols < 0)
    return FP8LA_ERR_INVALID_ARG;
  // Every block reads amax_prev while others update amax_out and block 0
  // writes scale_out, so the three must be distinct words.
  const void *a = amax_prev, *b = amax_out, *c = scale_out;
  if (a == b || a == c || b == c) return FP8LA_ERR_INVALID_ARG;
  const bool empty = rows == 0 || cols == 0;
  if (!empty && (!x || !q || ldx < cols || ldq < cols))
    return FP8LA_ERR_INVALID_ARG;
  if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40))
    return FP8LA_ERR_UNSUPPORTED;
  if (sm_count() <= 0) return FP8LA_ERR_CUDA;
  if (cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  if (empty) {
    delayed_kernel<1, FMT><<<1, 32, 0, s>>>(x, 0, 0, 0, q, 0, true, amax_prev,
                                            amax_out, scale_out);
    return launch_status();
  }
  const bool vec4 = cols % 4 == 0 && ldx % 4 == 0 && ldq % 4 == 0 &&
                    aligned16(x) &&
                    (reinterpret_cast<uintptr_t>(q) & 3u) == 0;
  const bool contiguous = ldx == cols && ldq == cols;
  if (vec4) {
    const int64_t upr = cols / 4;
    const int g = grid_for(rows * upr, kThreads);
    delayed_kernel<4, FMT><<<g, kThreads, 0, s>>>(
        x, rows, upr, ldx, q, ldq, contiguous, amax_prev, amax_out, scale_out);
  } else {
    const int g = grid_for(rows * cols, kThreads);
    delayed_kernel<1, FMT><<<g, kThreads, 0, s>>>(
        x, rows, cols, ldx, q, ldq, contiguous, amax_prev, amax_out,
        scale_out);
  }
  return launch_status();
}

// ------------------------------------------- grouped per-tensor (MoE rows)
// Rows m_offsets[e] .. m_offsets[e+1]-1 of x form group e (an expert's
// tokens), quantised with their own per-tensor amax and scale.  The offsets
// stay on the device; both passes read them into shared memory, check them
// (m_offsets[0] == 0, non-decreasing, m_offsets[E] <= the row capacity) and
// on failure record kStatusBadDeviceArg and write nothing.  The work is
// split into items of kGroupChunkRows rows of one group; item i belongs to
// the group whose item range [pref[g], pref[g+1]) holds it.
constexpr int kGroupChunkRows = 4;
constexpr int kQuantMaxGroups = 1024;

// The offsets and each group's first item, in dynamic shared memory sized
// for the call's group count (2 (E + 1) words: a few bytes for a handful of
// experts, so that the quantiser's blocks still fit beside a GEMM's).
struct GroupTable {
  int32_t *offs;   // [E + 1]
  int32_t *pref;   // [E + 1]
  int *bad;
};

__device__ __forceinline__ GroupTable group_table(int E) {
  extern __shared__ int32_t gt_words[];
  __shared__ int gt_bad;
  return GroupTable{gt_words, gt_words + E + 1, &gt_bad};
}

// Fills `t` from m_offsets (all threads of the block take part); returns
// false for offsets that fail the check.
__device__ bool load_group_table(const GroupTable &t, const int32_t *m_offsets,
                                 int E, int64_t rows_cap) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) t.offs[e] = m_offsets[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    int bad = t.offs[0] != 0 || t.offs[E] > rows_cap;
    int32_t acc = 0;
    for (int e = 0; e < E; ++e) {
      const int32_t n = t.offs[e + 1] - t.offs[e];
      if (n < 0) bad = 1;
      t.pref[e] = acc;
      acc += n > 0 ? (n + kGroupChunkRows - 1) / kGroupChunkRows : 0;
    }
    t.pref[E] = acc;
    *t.bad = bad;
  }
  __syncthreads();
  return !*t.bad;
}

// The group of work item i (pref[g] <= i < pref[g+1]; empty groups have
// an empty range).
__device__ __forceinline__ int group_of_item(const GroupTable &t, int E,
                                             int32_t i) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.pref[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int VEC>
__global__ void __launch_bounds__(kThreads, kMinBlocksBound)
    amax_grouped_kernel(const float *__restrict__ x, int64_t ldx,
                        int64_t cols, const int32_t *m_offsets, int E,
                        int64_t rows_cap, float *amax_out, unsigned *status) {
  const GroupTable t = group_table(E);
  if (!load_group_table(t, m_offsets, E, rows_cap)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadDeviceArg);
    return;
  }
  const int64_t units = VEC == 4 ? cols / 4 : cols;
  for (int32_t i = blockIdx.x; i < t.pref[E]; i += gridDim.x) {
    const int g = group_of_item(t, E, i);
    const int64_t r0 = t.offs[g] + static_cast<int64_t>(i - t.pref[g]) * kGroupChunkRows;
    const int64_t r1 = min(r0 + kGroupChunkRows, static_cast<int64_t>(t.offs[g + 1]));
    const int nr = static_cast<int>(r1 - r0);
    float m = 0.0f;
    // A thread takes a column of the item's rows: up to kGroupChunkRows
    // independent loads in flight.
    for (int64_t c = threadIdx.x; c < units; c += blockDim.x) {
      if (VEC == 4) {
        const float4 *col = reinterpret_cast<const float4 *>(x + r0 * ldx) + c;
        const int64_t ld4 = ldx / 4;
        if (nr == kGroupChunkRows) {
          // a whole item: all its loads in flight before the first use
          float4 v[kGroupChunkRows];
#pragma unroll
          for (int k = 0; k < kGroupChunkRows; ++k) v[k] = ld_stream4(col + k * ld4);
#pragma unroll
          for (int k = 0; k < kGroupChunkRows; ++k) m = max_abs4(m, v[k]);
        } else {
          for (int k = 0; k < nr; ++k) m = max_abs4(m, ld_stream4(col + k * ld4));
        }
      } else {
        const float *col = x + r0 * ldx + c;
        float v[kGroupChunkRows];
#pragma unroll
        for (int k = 0; k < kGroupChunkRows; ++k) v[k] = k < nr ? col[k * ldx] : 0.0f;
#pragma unroll
        for (int k = 0; k < kGroupChunkRows; ++k) m = fmaxf(m, fabsf(v[k]));
      }
    }
    block_max_into(m, amax_out + g);
    __syncthreads();   // block_max_into's shared buffer is reused next item
  }
}

template <int VEC, int FMT>
__global__ void __launch_bounds__(kThreads, kMinBlocksBound)
    cast_grouped_kernel(const float *__restrict__ x, int64_t ldx, int64_t cols,
                        uint8_t *__restrict__ q, int64_t ldq,
                        const int32_t *m_offsets, int E, int64_t rows_cap,
                        const float *amax_in, float *scale_out,
                        unsigned *status) {
  const GroupTable t = group_table(E);
  if (!load_group_table(t, m_offsets, E, rows_cap)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadDeviceArg);
    return;
  }
  // Every group's scale, empty groups included, from block 0.
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      scale_out[e] = scales_from_amax<FMT>(amax_in[e]).scale;
  const int64_t units = VEC == 4 ? cols / 4 : cols;
  for (int32_t i = blockIdx.x; i < t.pref[E]; i += gridDim.x) {
    const int g = group_of_item(t, E, i);
    const int64_t r0 = t.offs[g] + static_cast<int64_t>(i - t.pref[g]) * kGroupChunkRows;
    const int64_t r1 = min(r0 + kGroupChunkRows, static_cast<int64_t>(t.offs[g + 1]));
    const float qs = scales_from_amax<FMT>(amax_in[g]).qscale;
    const int nr = static_cast<int>(r1 - r0);
    for (int64_t c = threadIdx.x; c < units; c += blockDim.x) {
      if (VEC == 4) {
        const float4 *col = reinterpret_cast<const float4 *>(x + r0 * ldx) + c;
        uint32_t *qcol = reinterpret_cast<uint32_t *>(q + r0 * ldq) + c;
        const int64_t ld4 = ldx / 4, ldq4 = ldq / 4;
        if (nr == kGroupChunkRows) {
          // a whole item: all its loads in flight before the first store
          float4 v[kGroupChunkRows];
#pragma unroll
          for (int k = 0; k < kGroupChunkRows; ++k) v[k] = ld_stream4(col + k * ld4);
#pragma unroll
          for (int k = 0; k < kGroupChunkRows; ++k) qcol[k * ldq4] = cvt4<FMT>(v[k], qs);
        } else {
          for (int k = 0; k < nr; ++k)
            qcol[k * ldq4] = cvt4<FMT>(ld_stream4(col + k * ld4), qs);
        }
      } else {
        const float *col = x + r0 * ldx + c;
        uint8_t *qcol = q + r0 * ldq + c;
        float v[kGroupChunkRows];
#pragma unroll
        for (int k = 0; k < kGroupChunkRows; ++k)
          if (k < nr) v[k] = col[k * ldx];
#pragma unroll
        for (int k = 0; k < kGroupChunkRows; ++k)
          if (k < nr) qcol[k * ldq] = cvt1<FMT>(v[k], qs);
      }
    }
  }
}

fp8la_status quantize_grouped_impl(const float *x, int32_t E,
                                   const int32_t *m_offsets, int64_t rows_cap,
                                   int64_t cols, int64_t ldx, uint8_t *q,
                                   int64_t ldq, float *amax_out,
                                   float *scale_out, cudaStream_t s) {
  if (E < 0 || E > kQuantMaxGroups || rows_cap < 0 || cols < 0)
    return FP8LA_ERR_INVALID_ARG;
  if (E == 0) return FP8LA_OK;
  if (!m_offsets || !amax_out || !scale_out) return FP8LA_ERR_INVALID_ARG;
  // The cast blocks read amax_out while block 0 writes scale_out.
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(amax_out);
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(scale_out);
  const uintptr_t bytes = static_cast<uintptr_t>(E) * sizeof(float);
  if (a0 < s0 + bytes && s0 < a0 + bytes) return FP8LA_ERR_INVALID_ARG;
  if (rows_cap > 0 && cols > 0 && (!x || !q || ldx < cols || ldq < cols))
    return FP8LA_ERR_INVALID_ARG;
  if (rows_cap >= (int64_t(1) << 31) || cols > (int64_t(1) << 40))
    return FP8LA_ERR_UNSUPPORTED;
  if (sm_count() <= 0) return FP8LA_ERR_CUDA;
  unsigned *status = status_word_ptr();
  if (!status) return FP8LA_ERR_CUDA;
  if (cudaMemsetAsync(amax_out, 0, bytes, s) != cudaSuccess) return FP8LA_ERR_CUDA;
  const bool vec4 = cols % 4 == 0 && ldx % 4 == 0 && ldq % 4 == 0 &&
                    aligned16(x) && (reinterpret_cast<uintptr_t>(q) & 3u) == 0;
  // Items: at most rows_cap / kGroupChunkRows + E of them.
  const int64_t items = (rows_cap + kGroupChunkRows - 1) / kGroupChunkRows + E;
  const int g = grid_for(items * kThreads, kThreads);
  const int64_t c = cols > 0 ? cols : 0;
  const size_t table = 2 * (static_cast<size_t>(E) + 1) * sizeof(int32_t);
  if (vec4) {
    amax_grouped_kernel<4><<<g, kThreads, table, s>>>(x, ldx, c, m_offsets, E,
                                                      rows_cap, amax_out, status);
    cast_grouped_kernel<4, 0><<<g, kThreads, table, s>>>(
        x, ldx, c, q, ldq, m_offsets, E, rows_cap, amax_out, scale_out, status);
  } else {
    amax_grouped_kernel<1><<<g, kThreads, table, s>>>(x, ldx, c, m_offsets, E,
                                                      rows_cap, amax_out, status);
    cast_grouped_kernel<1, 0><<<g, kThreads, table, s>>>(
        x, ldx, c, q, ldq, m_offsets, E, rows_cap, amax_out, scale_out, status);
  }
  return launch_status();
}

}  // namespace
}  // namespace fp8la

extern "C" fp8la_status fp8_quantize_pertensor(const float *x, int64_t rows,

                                               int64_t cols, int64_t ldx,
                                               uint8_t *q, int64_t ldq,
                                               float *amax_out,
                                               float *scale_out,
                                               fp8la_stream_t stream) {
  return quantize_pertensor_impl<0>(x, rows, cols, ldx, q, ldq, amax_out,
                                    scale_out,
                                    reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8la_status fp8_quantize_pertensor_ex(
    const float *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
    int64_t ldq, float *amax_out, float *scale_out, int32_t format,
    fp8la_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (format == FP8LA_FORMAT_E4M3)
    return quantize_pertensor_impl<0>(x, rows, cols, ldx, q, ldq, amax_out,
                                      scale_out, s);
  if (format == FP8LA_FORMAT_E5M2)
    return quantize_pertensor_impl<1>(x, rows, cols, ldx, q, ldq, amax_out,
                                      scale_out, s);
  return FP8LA_ERR_INVALID_ARG;
}

extern "C" fp8la_status fp8_quantize_blockwise_32x32(
    const float *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
    int64_t ldq, float *scales, int64_t ld_scales, fp8la_stream_t stream) {
  if (rows < 0 || cols < 0) return FP8LA_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8LA_OK;
  const int64_t tiles_r = (rows + 31) / 32, tiles_c = (cols + 31) / 32;
  if (!x || !q || !scales || ldx < cols || ldq < cols || ld_scales < tiles_c)
    return FP8LA_ERR_INVALID_ARG;
  if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40))
    return FP8LA_ERR_UNSUPPORTED;
  if (sm_count() <= 0) return FP8LA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool vec4 = cols % 4 == 0 && ldx % 4 == 0 && ldq % 4 == 0 &&
                    aligned16(x) &&
                    (reinterpret_cast<uintptr_t>(q) & 3u) == 0;
  // 256-thread blocks of 64 registers: four per SM fill the register file.
  const int g = grid_for(tiles_r * tiles_c * 32, 256, kBlock32PerSm);
  if (vec4)
    block32_kernel<4><<<g, 256, 0, s>>>(x, rows, cols, ldx, q, ldq, scales,
                                        ld_scales, tiles_r, tiles_c);
  else
    block32_kernel<1><<<g, 256, 0, s>>>(x, rows, cols, ldx, q, ldq, scales,
                                        ld_scales, tiles_r, tiles_c);
  return launch_status();
}

extern "C" fp8la_status fp8_quantize_pertensor_delayed(
    const float *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
    int64_t ldq, const float *amax_prev, float *amax_out, float *scale_out,
    int32_t format, fp8la_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (format == FP8LA_FORMAT_E4M3)
    return quantize_delayed_impl<0>(x, rows, cols, ldx, q, ldq, amax_prev,
                                    amax_out, scale_out, s);
  if (format == FP8LA_FORMAT_E5M2)
    return quantize_delayed_impl<1>(x, rows, cols, ldx, q, ldq, amax_prev,
                                    amax_out, scale_out, s);
  return FP8LA_ERR_INVALID_ARG;
}

extern "C" fp8la_status fp8_quantize_pertensor_grouped(
    const float *x, int32_t num_groups, const int32_t *m_offsets,
    int64_t rows_capacity, int64_t cols, int64_t ldx, uint8_t *q, int64_t ldq,
    float *amax_out, float *scale_out, fp8la_stream_t stream) {
  return quantize_grouped_impl(x, num_groups, m_offsets, rows_capacity, cols,
                               ldx, q, ldq, amax_out, scale_out,
                               reinterpret_cast<cudaStream_t>(stream));
}
