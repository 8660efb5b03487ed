// 32x32 block-scaled E4M3 GEMM: tcgen05 partial sums per 32-wide K block,
// promoted into FP32 register accumulators on the CUDA cores.
//
// Method: [P3] "JAX 中使用 Triton 优化 Blackwell GPU 的 FP8 GEMM 内核",
// implementation paragraph (one scale per 32x32 block, "microscaling") and
// warp-specialisation paragraph (one warp loads by TMA, one issues the FP8
// MMA, a third promotes on the CUDA cores); output rule of [P1]
// "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (FP32 accumulator,
// BF16 output).
//
//   C[m][n] = bf16( sum_kb sa[m/32][kb] * sb[n/32][kb] * S_kb[m][n] )
//
// The tile scales are arbitrary fp32 values, so they cannot be folded into
// the tensor-core instruction; each 32-wide K block's product S_kb is formed
// by one tcgen05.mma (M=128, N=64, K=32) into a fresh TMEM buffer and then
// weighted and added on the CUDA cores.
//
// Design (one CTA per SM, persistent, 18 warps).  The promotion costs one
// FP32 FMA per output per 32-wide K block, against 32 tensor-core FMAs: on
// 128 FP32 lanes per SM versus 8192 tensor FMAs per clock this caps the
// kernel near half the dense FP8 peak.  What holds it below that is the
// latency of each handoff between the MMA warp and the promotion warps, so
// the CTA's 128 x 128 tile is split into two 128 x 64 halves, each with its
// own TMEM partial set and its own promotion group, which hides one group's
// waits behind the other's FMAs; all synchronisation is at the granularity
// of 128-wide K stages:
//   * warp 16: producer (lane 0).  Per 128-wide K stage (7-stage ring) it
//     issues four TMA loads on one barrier: a 128 x 128 A tile, a 128 x 128
//     B tile (both halves' columns), and the stage's scale boxes sa[4 row
//     tiles][4 K blocks] and sb[4 column tiles][4 K blocks].  The two
//     halves share the stage's A tile.  Nothing on the producer waits for
//     global memory, so it runs up to seven stages ahead.
//   * warp 17: MMA issuer (lane 0).  Per stage and half g, four MMAs (M=128,
//     N=64, K=32, one per 32-wide K block; B = rows 64g.. of the stage's B
//     tile) into the four 64-column TMEM partial buffers of set g; one
//     commit hands the whole set to group g.  Half 0 is issued before half
//     1, so the two groups run about half a stage apart.
//   * warps 8g .. 8g+7: promotion group g.  Warp w reads TMEM lanes
//     32(w%4).. (C rows) and columns 32((w%8)/4)..+31 of each partial of its
//     set, exactly one 32 x 32 scale tile, so its scale is one number per K
//     block: sa * sb from two 16-byte shared-memory vectors per stage.  Each
//     thread keeps its row's 32 FP32 accumulators in registers (as 16 packed
//     pairs) and adds (sa*sb) * partial with packed FMAs (fma.rn.f32x2), one
//     K block per asm statement.  After the last stage of a tile it rounds
//     to BF16 and stores 64 bytes.
//   * A stage is recycled once all sixteen promotion warps have read its
//     scales (empty count 16): each group reads them only after its set for
//     the stage is committed, which implies that its MMAs, readers of the
//     stage's operand tiles, have completed.  The scale reads are
//     generic-proxy loads and the slot's next fill is an async-proxy (TMA)
//     write, so each warp issues fence.proxy.async before it arrives;
//     without it the next fill's scale boxes were seen to land under the
//     reads at tile changes.  A partial-buffer set is reused once its eight
//     warps hold its data in registers (pempty count 8).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8la {
namespace {

constexpr int BM = 128;
constexpr int BN = 64;           // columns of one group's half tile
constexpr int BNS = 2 * BN;      // columns of a CTA tile (two halves)
constexpr int BK = 128;          // K per stage (bytes = E4M3 values)
constexpr int KB = 32;           // scale block along K, = K per MMA
constexpr int KPS = BK / KB;     // K blocks per stage (4)
constexpr int STAGES = 7;
constexpr int NSETS = 2;         // TMEM partial-buffer sets, KPS buffers each
constexpr int kGroups = 2;       // promotion groups: group g uses set g
constexpr int kGroupWarps = 8;   // promotion warps per group
constexpr int kPromoWarps = kGroups * kGroupWarps;
constexpr int kProducerWarp = kPromoWarps;
constexpr int kMmaWarp = kPromoWarps + 1;
constexpr int kThreads = 32 * (kPromoWarps + 2);
constexpr int GROUP_M = 16;
constexpr int kTmemCols = NSETS * KPS * BN;  // 512

struct BsArgs {
  uint16_t *C;
  int64_t ldc;
  int32_t M, N, K;
  const float *sa;
  int64_t ld_sa;
  const float *sb;
  int64_t ld_sb;
  unsigned *status;
  uint64_t timeout_ns;
  int32_t c_vec16;
  int32_t withhold_first;  // diagnostic: skip the first stage's TMA arrival
};

struct Lay {
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BNS * BK;
  static constexpr int kSaBytes = 4 * KPS * 4;
  static constexpr int kSbBytes = 4 * KPS * 4;
  static constexpr int kStageBytes = kABytes + kBBytes + kSaBytes + kSbBytes;
  static constexpr int kA = 0;
  static constexpr int kB = kA + STAGES * kABytes;
  // Per stage: the A-scale box [4 row tiles][4 K blocks] (64 B) at +0 and
  // the B-scale box [4 column tiles][4 K blocks] (64 B) at +128.  Every TMA
  // destination in shared memory starts on a 128-byte boundary.
  static constexpr int kSbOffset = 128;
  static constexpr int kScaleSlot = 256;
  static constexpr int kScale = kB + STAGES * kBBytes;
  static constexpr int kBar = kScale + STAGES * kScaleSlot;
  static constexpr int kNumBars = 2 * STAGES + 2 * NSETS + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16;
  static constexpr int kAlloc = kEnd + 1024;
};

// TMA writes to shared memory must start on 128-byte boundaries (the
// swizzled operand tiles additionally on their 1024-byte swizzle atoms).
static_assert(Lay::kA % 1024 == 0 && Lay::kABytes % 1024 == 0, "A tiles");
static_assert(Lay::kB % 1024 == 0 && Lay::kBBytes % 1024 == 0, "B tiles");
static_assert(Lay::kScale % 128 == 0 && Lay::kScaleSlot % 128 == 0 &&
                  Lay::kSbOffset % 128 == 0 &&
                  Lay::kSbOffset >= Lay::kSaBytes &&
                  Lay::kSbOffset + Lay::kSbBytes <= Lay::kScaleSlot,
              "scale boxes");
static_assert(Lay::kBar % 8 == 0, "mbarriers");
static_assert(Lay::kAlloc <= 227 * 1024, "shared memory");

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n,
                                            int &mb, int &nb) {
  const int per_group = GROUP_M * tiles_n;
  const int g = t / per_group;
  const int first_m = g * GROUP_M;
  const int gm = min(tiles_m - first_m, GROUP_M);
  const int r = t - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

// Promotion of one K block's partial (32 columns, one lane row): loads it
// from TMEM, waits, and adds s * partial into the 32 FP32 accumulators held
// as 16 packed pairs, with packed FMAs.  One asm statement.
__device__ __forceinline__ void promote_one(uint64_t (&acc)[16], uint32_t taddr,
                                            float s) {
  asm volatile(
      "{\n\t"
      ".reg .b32 p<32>;\n\t"
      ".reg .b64 q<16>, sc;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {p0, p1, p2, p3, p4, p5, p6, p7, p8, p9, p10, p11, p12, p13, p14, p15, p16, p17, p18, p19, p20, p21, p22, p23, p24, p25, p26, p27, p28, p29, p30, p31}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 sc, {%17, %17};\n\t"
      "mov.b64 q0, {p0, p1};\n\t"
      "mov.b64 q1, {p2, p3};\n\t"
      "mov.b64 q2, {p4, p5};\n\t"
      "mov.b64 q3, {p6, p7};\n\t"
      "mov.b64 q4, {p8, p9};\n\t"
      "mov.b64 q5, {p10, p11};\n\t"
      "mov.b64 q6, {p12, p13};\n\t"
      "mov.b64 q7, {p14, p15};\n\t"
      "mov.b64 q8, {p16, p17};\n\t"
      "mov.b64 q9, {p18, p19};\n\t"
      "mov.b64 q10, {p20, p21};\n\t"
      "mov.b64 q11, {p22, p23};\n\t"
      "mov.b64 q12, {p24, p25};\n\t"
      "mov.b64 q13, {p26, p27};\n\t"
      "mov.b64 q14, {p28, p29};\n\t"
      "mov.b64 q15, {p30, p31};\n\t"
      "fma.rn.f32x2 %0, sc, q0, %0;\n\t"
      "fma.rn.f32x2 %1, sc, q1, %1;\n\t"
      "fma.rn.f32x2 %2, sc, q2, %2;\n\t"
      "fma.rn.f32x2 %3, sc, q3, %3;\n\t"
      "fma.rn.f32x2 %4, sc, q4, %4;\n\t"
      "fma.rn.f32x2 %5, sc, q5, %5;\n\t"
      "fma.rn.f32x2 %6, sc, q6, %6;\n\t"
      "fma.rn.f32x2 %7, sc, q7, %7;\n\t"
      "fma.rn.f32x2 %8, sc, q8, %8;\n\t"
      "fma.rn.f32x2 %9, sc, q9, %9;\n\t"
      "fma.rn.f32x2 %10, sc, q10, %10;\n\t"
      "fma.rn.f32x2 %11, sc, q11, %11;\n\t"
      "fma.rn.f32x2 %12, sc, q12, %12;\n\t"
      "fma.rn.f32x2 %13, sc, q13, %13;\n\t"
      "fma.rn.f32x2 %14, sc, q14, %14;\n\t"
      "fma.rn.f32x2 %15, sc, q15, %15;\n\t"
      "}"
      : "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]), "+l"(acc[7]), "+l"(acc[8]), "+l"(acc[9]), "+l"(acc[10]), "+l"(acc[11]), "+l"(acc[12]), "+l"(acc[13]), "+l"(acc[14]), "+l"(acc[15])
      : "r"(taddr), "f"(s)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_e4m3_block32_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSa,
                             const __grid_constant__ CUtensorMap tmSb,
                             const BsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = base + Lay::kBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto pfull_bar = [&](int p) { return bar0 + 8u * (2 * STAGES + p); };
  auto pempty_bar = [&](int p) { return bar0 + 8u * (2 * STAGES + NSETS + p); };
  const uint32_t final_bar = bar0 + 8u * (2 * STAGES + 2 * NSETS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + Lay::kMisc);
  volatile int *abort_flag =
      reinterpret_cast<volatile int *>(sbase + Lay::kMisc + 4);

  const int tiles_m = (a.M + BM - 1) / BM;
  const int tiles_n = (a.N + BNS - 1) / BNS;    // tiles of 128 columns
  const int total_tiles = tiles_m * tiles_n;
  const int nks = (a.K + BK - 1) / BK;          // stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kPromoWarps);     // both groups read it
    }
    for (int p = 0; p < NSETS; ++p) {
      mbar_init(pfull_bar(p), 1);
      mbar_init(pempty_bar(p), kGroupWarps);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSa);
    tma_prefetch_desc(&tmSb);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t s = 0, ph = 0, issued = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, tiles_m, tiles_n, mb, nb);
      const int m0 = mb * BM, n0 = nb * BNS;
      for (int ks = 0; ks < nks; ++ks) {
        const bool ready = mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns,
                                     a.status, abort_flag);
        if (!__all_sync(0xffffffffu, ready)) {
          ok = false;
          break;
        }
        // Operand tiles and the stage's scale boxes, all on one barrier.
        // TMA zero-fills scale entries past the grid's edge.
        if (lane == 0 && !(a.withhold_first && issued == 0)) {
          const uint32_t fb = full_bar(s);
          const uint32_t sslot = base + Lay::kScale + s * Lay::kScaleSlot;
          mbar_arrive_expect_tx(fb, Lay::kStageBytes);
          tma_load_2d(base + Lay::kA + s * Lay::kABytes, &tmA, fb, ks * BK, m0);
          tma_load_2d(base + Lay::kB + s * Lay::kBBytes, &tmB, fb, ks * BK, n0);
          tma_load_2d(sslot, &tmSa, fb, ks * KPS, m0 / 32);
          tma_load_2d(sslot + Lay::kSbOffset, &tmSb, fb, ks * KPS, n0 / 32);
        }
        ++issued;
        if (++s == STAGES) { s = 0; ph ^= 1u; }
      }
    }
    // Wait for the copies this warp armed before the CTA may exit.
    if (lane == 0) {
      for (uint32_t st = 0; st < STAGES; ++st) {
        if (issued <= st) break;
        const uint32_t arms = (issued - 1 - st) / STAGES + 1;
        if (a.withhold_first && st == 0 && arms == 1) continue;  // never armed
        mbar_wait_drain(full_bar(st), (arms - 1) & 1u, a.timeout_ns, a.status);
      }
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
      uint32_t s = 0, ph = 0, use = 0;  // stage ring; uses of each set
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        for (int ks = 0; ok && ks < nks; ++ks, ++use) {
          if (!mbar_wait(full_bar(s), ph, a.timeout_ns, a.status,
                         abort_flag)) {
            ok = false;
            break;
          }
          const uint64_t adesc =
              smem_desc_k128_sw128(base + Lay::kA + s * Lay::kABytes);
          for (int g = 0; g < kGroups; ++g) {
            if (!mbar_wait(pempty_bar(g), (use & 1u) ^ 1u, a.timeout_ns,
                           a.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // Group g's half of the B tile: rows 64 g .. 64 g + 63.
            const uint64_t bdesc = smem_desc_k128_sw128(
                base + Lay::kB + s * Lay::kBBytes + g * BN * BK);
#pragma unroll
            for (int k = 0; k < KPS; ++k)
              umma_f8f6f4(tmem_base + (g * KPS + k) * BN, adesc + 2u * k,
                          bdesc + 2u * k, idesc, 0u);
            // The stage's shared memory is released by both groups after
            // their sets' commits, which imply the stage's MMAs are done.
            umma_commit(pfull_bar(g));
          }
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      umma_commit(final_bar);
      mbar_wait_drain(final_bar, 0, a.timeout_ns, a.status);
    }
  } else {
    // ----------------------------------------------------------- promotion
    const int grp = warp / kGroupWarps;          // which half of the tile
    const int gw = warp % kGroupWarps;
    const int q = warp & 3;          // TMEM lane quarter = 32-row tile
    const int c = gw >> 2;           // 32-column slice within the half
    const uint32_t col0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          32 * c + grp * KPS * BN;
    uint32_t s = 0, ph = 0, use = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, tiles_m, tiles_n, mb, nb);
      uint64_t acc[16];   // packed FP32 pairs: columns 2j, 2j+1
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0;
      for (int ks = 0; ok && ks < nks; ++ks, ++use) {
        // Scale products of this stage (acquired through the stage's full
        // barrier), then let the stage go as far as this warp is concerned.
        const bool sready = mbar_wait(full_bar(s), ph, a.timeout_ns,
                                      a.status, abort_flag);
        const bool pready = sready &&
                            mbar_wait(pfull_bar(grp), use & 1u, a.timeout_ns,
                                      a.status, abort_flag);
        if (!__all_sync(0xffffffffu, sready && pready)) {
          ok = false;
          break;
        }
        const float4 va = *reinterpret_cast<const float4 *>(
            sbase + Lay::kScale + s * Lay::kScaleSlot + q * KPS * 4);
        const float4 vb = *reinterpret_cast<const float4 *>(
            sbase + Lay::kScale + s * Lay::kScaleSlot + Lay::kSbOffset +
            (2 * grp + c) * KPS * 4);
        const float4 sc = make_float4(__fmul_rn(va.x, vb.x), __fmul_rn(va.y, vb.y),
                                      __fmul_rn(va.z, vb.z), __fmul_rn(va.w, vb.w));
        // Order these generic reads before the TMA writes of the slot's next
        // fill, which the arrival below lets the producer issue.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
        if (++s == STAGES) { s = 0; ph ^= 1u; }
        tc_fence_after();
        promote_one(acc, col0, sc.x);
        promote_one(acc, col0 + BN, sc.y);
        promote_one(acc, col0 + 2 * BN, sc.z);
        promote_one(acc, col0 + 3 * BN, sc.w);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pempty_bar(grp));
      }
      if (!ok) break;
      // Epilogue: round to BF16 and store this thread's 32 columns.
      const int row = mb * BM + q * 32 + lane;
      const int n = nb * BNS + grp * BN + 32 * c;
      if (row < a.M && n < a.N) {
        uint16_t *crow = a.C + static_cast<int64_t>(row) * a.ldc;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(
              __uint_as_float(static_cast<uint32_t>(acc[j])),
              __uint_as_float(static_cast<uint32_t>(acc[j] >> 32)));
          w[j] = *reinterpret_cast<const uint32_t *>(&b2);
        }
        if (a.c_vec16 && n + 32 <= a.N) {
          uint4 *dst = reinterpret_cast<uint4 *>(crow + n);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2],
                                w[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < a.N)
              crow[n + j] = static_cast<uint16_t>(
                  (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

__global__ void zero_c_kernel_bs(uint16_t *C, int64_t ldc, int64_t M,
                                 int64_t N) {
  const int64_t n = M * N;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    C[r * ldc + c] = 0;
  }
}

bool encode_2d_f32(CUtensorMap *m, const void *ptr, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                   uint32_t box_outer) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d_bs(CUtensorMap *m, const void *ptr, uint64_t inner,
                  uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                  uint32_t box_outer) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fp8la

using namespace fp8la;

namespace fp8la {
namespace {

fp8la_status blockscaled_impl(const uint8_t *A, int64_t lda, const uint8_t *B,
                              int64_t ldb, uint16_t *C, int64_t ldc, int64_t M,
                              int64_t N, int64_t K, const float *sa,
                              int64_t ld_sa, const float *sb, int64_t ld_sb,
                              cudaStream_t s, int withhold) {
  if (M < 0 || N < 0 || K < 0) return FP8LA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FP8LA_OK;
  if (!C || ldc < N) return FP8LA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 1u) != 0) return FP8LA_ERR_ALIGNMENT;
  if (K == 0) {
    if (!device_is_sm10x()) return FP8LA_ERR_UNSUPPORTED;
    const int sms = sm_count();
    zero_c_kernel_bs<<<sms > 0 ? sms * 4 : 1, 256, 0, s>>>(C, ldc, M, N);
    return launch_status();
  }
  const int64_t nkb = (K + 31) / 32;
  if (!A || !B || !sa || !sb || lda < K || ldb < K || ld_sa < nkb ||
      ld_sb < nkb)
    return FP8LA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0 ||
      !aligned16(sa) || !aligned16(sb) || ld_sa % 4 != 0 || ld_sb % 4 != 0)
    return FP8LA_ERR_ALIGNMENT;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31) || lda >= (int64_t(1) << 39) ||
      ldb >= (int64_t(1) << 39) || ld_sa >= (int64_t(1) << 31) ||
      ld_sb >= (int64_t(1) << 31))
    return FP8LA_ERR_UNSUPPORTED;
  if (!device_is_sm10x()) return FP8LA_ERR_UNSUPPORTED;
  CUtensorMap tmA, tmB, tmSa, tmSb;
  if (!encode_2d_bs(&tmA, A, K, M, lda, BK, BM) ||
      !encode_2d_bs(&tmB, B, K, N, ldb, BK, BNS) ||
      !encode_2d_f32(&tmSa, sa, nkb, (M + 31) / 32, ld_sa * 4, KPS, BM / 32) ||
      !encode_2d_f32(&tmSb, sb, nkb, (N + 31) / 32, ld_sb * 4, KPS, BNS / 32))
    return FP8LA_ERR_CUDA;
  unsigned *status = status_word_ptr();
  if (!status) return FP8LA_ERR_CUDA;
  BsArgs args{};
  args.C = C;
  args.ldc = ldc;
  args.M = static_cast<int32_t>(M);
  args.N = static_cast<int32_t>(N);
  args.K = static_cast<int32_t>(K);
  args.sa = sa;
  args.ld_sa = ld_sa;
  args.sb = sb;
  args.ld_sb = ld_sb;
  args.status = status;
  args.timeout_ns = wait_timeout_ns();
  args.c_vec16 = aligned16(C) && ldc % 8 == 0;
  args.withhold_first = withhold;
  if (once_per_device(4, [] {
        return cudaFuncSetAttribute(gemm_e4m3_block32_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Lay::kAlloc);
      }) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return FP8LA_ERR_CUDA;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BNS - 1) / BNS);
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  gemm_e4m3_block32_kernel<<<grid, kThreads, Lay::kAlloc, s>>>(tmA, tmB, tmSa,
                                                               tmSb, args);
  return launch_status();
}

}  // namespace

fp8la_status diag_block32_withheld(const uint8_t *A, int64_t lda,
                                   const uint8_t *B, int64_t ldb, uint16_t *C,
                                   int64_t ldc, int64_t M, int64_t N, int64_t K,
                                   const float *sa, int64_t ld_sa,
                                   const float *sb, int64_t ld_sb,
                                   cudaStream_t s) {
  if (M <= 0 || N <= 0 || K <= 0) return FP8LA_ERR_INVALID_ARG;
  return blockscaled_impl(A, lda, B, ldb, C, ldc, M, N, K, sa, ld_sa, sb,
                          ld_sb, s, 1);
}

}  // namespace fp8la

extern "C" fp8la_status fp8_gemm_blockscaled_32x32(
    const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb, uint16_t *C,
    int64_t ldc, int64_t M, int64_t N, int64_t K, const float *sa,
    int64_t ld_sa, const float *sb, int64_t ld_sb, fp8la_stream_t stream) {
  return blockscaled_impl(A, lda, B, ldb, C, ldc, M, N, K, sa, ld_sa, sb,
                          ld_sb, reinterpret_cast<cudaStream_t>(stream), 0);
}
