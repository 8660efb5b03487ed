// Per-tensor-scaled and grouped (MoE) E4M3 GEMMs on tcgen05 tensor cores.
//
// Method: [P1] "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核", kernel-code
// paragraph (C tile = sum over K blocks of A tile x B tile, FP32
// accumulator), scale paragraph (acc * scale_a * scale_b) and parameter
// list (E4M3 in, FP32 accumulate, BF16 out); [P3] "JAX 中使用 Triton 优化
// Blackwell GPU 的 FP8 GEMM 内核", TMA paragraph, warp-specialisation
// paragraph (one warp loads by TMA, one issues the MMA) and MoE paragraph
// (grouped GEMM over experts).
//
// Two kernels live here.  The default for large problems is the CTA-pair
// kernel further down (tcgen05 cta_group::2, 256 x 256 tiles per pair of
// SMs; its own comment describes it).  The single-CTA kernel described next
// serves small problems (128 x 128 tiles) and an explicit variant choice.
//
// Single-CTA design (sm_103a, one CTA per SM, persistent):
//   * warp 4 (one lane): TMA producer.  For every 128-wide K block it loads
//     a 128 x 128 A tile and a BN x 128 B tile (both K-major, 128-byte
//     swizzle) into one stage of a STAGES-deep shared-memory ring, arming
//     the stage's `full` mbarrier with the byte count.
//   * warp 5 (one lane): MMA issuer.  Four tcgen05.mma kind::f8f6f4
//     (M=128, N=BN, K=32 each) per stage into an FP32 accumulator in tensor
//     memory; tcgen05.commit frees the stage (`empty`) and, after the last
//     K block, hands the accumulator to the epilogue (`tmem_full`).
//     Tensor memory holds two accumulators (2 x BN of 512 columns) so the
//     epilogue of tile i overlaps the MMAs of tile i+1.
//   * warps 0-3: epilogue.  Warp w owns TMEM lanes (= C rows) 32w..32w+31;
//     each thread loads its row's accumulator 32 columns at a time
//     (tcgen05.ld), multiplies by scale_a and then by scale_b, rounds to
//     BF16 and writes 16-byte vectors; then releases the accumulator
//     (`tmem_empty`).
//   * Tiles are visited in a grouped order (GROUP_M row blocks per group)
//     so that concurrently running CTAs share A and B tiles through L2.
//   * Ragged M, N, K: TMA fills out-of-range operand elements with zeros;
//     the epilogue stores only in-range elements.
//   * Grouped GEMM: A is the concatenation of all groups' rows; B is a 3-D
//     tensor [E][N][K].  The tile space is the concatenation of every
//     group's own tile grid; each CTA derives it from m_offsets on the
//     device.  Rows of a tile past its group's end are computed (they hold
//     the next group's rows, or TMA zeros) and not stored.
#include <cuda_bf16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace fp8la {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;                  // bytes = E4M3 values per K block
constexpr int UMMA_K = 32;               // K per tcgen05.mma for 8-bit inputs
constexpr int kThreads = 192;            // 6 warps
constexpr int kMaxGroups = 1024;
constexpr int GROUP_M = 16;

struct GemmArgs {
  uint16_t *C;
  int64_t ldc;
  int32_t M, N, K;
  const float *scale_a;  // per-tensor: [1]; grouped: [E]
  const float *scale_b;
  const int32_t *m_offsets;  // grouped only
  int32_t num_groups;        // grouped only
  unsigned *status;
  uint64_t timeout_ns;
  int32_t withhold_first;  // diagnostic: skip the first TMA arrival (CTA-pair
                           // kernel: the second CTA's first loads)
  int32_t c_vec16;         // C rows allow 16-byte stores (C 16-byte aligned, ldc % 8 == 0)
  int32_t c_tma;           // CTA-pair kernel: C written through its tensor map
  uint32_t fmt_bits;       // operand-format bits of the MMA instruction descriptor
  int32_t split_tail;      // CTA-pair kernel: last tiles computed as two 128-column halves
};

template <int BN, int STAGES>
struct Smem {
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
  // Layout (offsets from a 1024-byte-aligned base).
  static constexpr int kA = 0;
  static constexpr int kB = kA + STAGES * kABytes;
  static constexpr int kBar = kB + STAGES * kBBytes;
  static constexpr int kNumBars = 2 * STAGES + 4 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kPrefix = kMisc + 16;  // int32 [kMaxGroups + 1]
  static constexpr int kEnd = kPrefix + (kMaxGroups + 1) * 4;
  static constexpr int kAlloc = kEnd + 1024;  // slack for aligning the base
};

// TMA destinations: operand tiles start on their 1024-byte swizzle atoms.
static_assert(Smem<256, 4>::kB % 1024 == 0 && Smem<256, 4>::kBBytes % 1024 == 0,
              "B tiles");
static_assert(Smem<256, 4>::kAlloc <= 227 * 1024, "shared memory");
static_assert(Smem<128, 6>::kB % 1024 == 0 && Smem<128, 6>::kBBytes % 1024 == 0,
              "B tiles");
static_assert(Smem<128, 6>::kAlloc <= 227 * 1024, "shared memory");

// Tile t of a tiles_m x tiles_n grid in grouped order.
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

struct TileInfo {
  int32_t row0;     // first C row of the tile
  int32_t row_end;  // rows >= row_end are not stored
  int32_t n0;
  int32_t group;
  int32_t tn;       // CTA-pair grouped tail tile computed transposed: its
                    // MMA width (a multiple of 32, <= 256); 0 otherwise
};

template <bool GROUPED, int TBM>
__device__ __forceinline__ TileInfo tile_info(int t, const GemmArgs &a,
                                              int tiles_n, const int32_t *pref,
                                              const int32_t *offs_smem,
                                              int BN) {
  TileInfo ti;
  ti.tn = 0;
  if (!GROUPED) {
    const int tiles_m = (a.M + TBM - 1) / TBM;
    int mb, nb;
    tile_coords(t, tiles_m, tiles_n, mb, nb);
    ti.row0 = mb * TBM;
    ti.row_end = a.M;
    ti.n0 = nb * BN;
    ti.group = 0;
  } else {
    // pref[e] = number of tiles of groups 0..e-1; find e with
    // pref[e] <= t < pref[e+1] (binary search over num_groups + 1 entries).
    int lo = 0, hi = a.num_groups;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pref[mid] <= t) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int m_lo = offs_smem[e], m_hi = offs_smem[e + 1];
    const int tiles_m = (m_hi - m_lo + TBM - 1) / TBM;
    int mb, nb;
    tile_coords(t - pref[e], tiles_m, tiles_n, mb, nb);
    ti.row0 = m_lo + mb * TBM;
    ti.row_end = min(m_hi, a.M);   // m_offsets are checked at set-up as well
    ti.n0 = nb * BN;
    ti.group = e;
    // A group's last row tile, when partial, is computed transposed by the
    // CTA-pair kernel (C_tail^T = B_e A_tail^T: MMA M = 256 over C columns,
    // N = the tail's rows rounded up to 32) instead of as a 256-row tile
    // whose rows past the group are padding.
    const int rows = ti.row_end - ti.row0;
    if (TBM == 256 && rows < TBM) ti.tn = (rows + 31) & ~31;
  }
  return ti;
}

// Grouped set-up, one warp: copy m_offsets to shared memory and build
// pref[e] = number of tiles of groups 0..e-1 (TBM-row tiles, tiles_n column
// tiles each).  Offsets that do not start at 0, decrease, or end past
// m_capacity (a.M) leave pref[num_groups] = 0, so the CTA computes and
// stores nothing, and the first CTA records kStatusBadDeviceArg.
template <int TBM>
__device__ __forceinline__ void load_group_offsets(const GemmArgs &a,
                                                   int tiles_n,
                                                   int32_t *offs_smem,
                                                   int32_t *pref, int lane) {
  for (int e = lane; e <= a.num_groups; e += 32) offs_smem[e] = a.m_offsets[e];
  __syncwarp();
  if (lane == 0) {
    bool ok = offs_smem[0] == 0 && offs_smem[a.num_groups] <= a.M;
    int acc = 0;
    for (int e = 0; e < a.num_groups; ++e) {
      pref[e] = acc;
      const int me = offs_smem[e + 1] - offs_smem[e];
      ok = ok && me >= 0;
      acc += (me > 0 ? (me + TBM - 1) / TBM : 0) * tiles_n;
    }
    if (!ok) {
      acc = 0;
      if (blockIdx.x == 0) atomicOr(a.status, kStatusBadDeviceArg);
    }
    pref[a.num_groups] = acc;
  }
}

// acc * scale_a * scale_b, evaluated left to right as the scale paragraph
// writes it: (acc * scale_a) * scale_b.  The two scales are never multiplied
// together, so a product of scales outside the FP32 range (two tiny scales,
// or two huge ones) does not flush or overflow an output that is itself in
// range, and a zero accumulator stays zero.  scale = {scale_a, scale_b}.
__device__ __forceinline__ float apply_scales(uint32_t acc, float2 scale) {
  return __fmul_rn(__fmul_rn(__uint_as_float(acc), scale.x), scale.y);
}

// Epilogue of one accumulator row: 32 FP32 columns of TMEM -> x scales ->
// BF16 (round to nearest even) -> C[row][n .. n+31], clipped at N.  Every
// lane of the warp must call it (tcgen05.ld is warp-collective).
__device__ __forceinline__ void store_chunk32(uint32_t taddr, bool row_ok,
                                              uint16_t *crow, int n, int N,
                                              float2 scale, bool vec16) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  if (!row_ok || n >= N) return;
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const __nv_bfloat162 h =
        __floats2bfloat162_rn(apply_scales(v[2 * j], scale),
                              apply_scales(v[2 * j + 1], scale));
    w[j] = *reinterpret_cast<const uint32_t *>(&h);
  }
  if (vec16 && n + 32 <= N) {
    uint4 *dst = reinterpret_cast<uint4 *>(crow + n);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  } else {
    // Fully unrolled so that w[] stays in registers.
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n + j < N)
        crow[n + j] = static_cast<uint16_t>((j & 1) ? (w[j >> 1] >> 16)
                                                    : (w[j >> 1] & 0xFFFFu));
  }
}

// Epilogue of a transposed tile: this lane's TMEM row is C column n, its 32
// TMEM columns from taddr are C rows m0 .. m0+31; rows at or past m_end and
// columns at or past N are not stored.  Across the warp each store writes 32
// consecutive BF16 of one C row.  Every lane of the warp must call it.
__device__ __forceinline__ void store_chunk32_t(uint32_t taddr, uint16_t *C,
                                                int64_t ldc, int m0, int m_end,
                                                int n, int N, float2 scale) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  if (n >= N) return;
  uint16_t *cp = C + static_cast<int64_t>(m0) * ldc + n;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (m0 + j < m_end) {
      const __nv_bfloat16 h =
          __float2bfloat16_rn(apply_scales(v[j], scale));
      cp[static_cast<int64_t>(j) * ldc] = *reinterpret_cast<const uint16_t *>(&h);
    }
}

// As store_chunk32, for a whole 32 x 32 block through a TMA store: the warp
// (lane = row) writes the block into the 2 KB shared buffer `stage` in the
// 64-byte swizzled layout of the C tensor map (16-byte chunk q of row r at
// r * 64 + 16 * (q ^ ((r >> 1) & 3)), which spreads each quarter-warp's
// stores over all 32 banks), and lane 0 stores the box at (column n, row
// row0).  Only blocks that lie inside C (and inside their group) come here;
// edge blocks go through store_chunk32.  Lane 0 first waits until its
// previous store has read the buffer.
__device__ __forceinline__ void store_chunk32_tma(uint32_t taddr,
                                                  uint32_t stage, int lane,
                                                  const CUtensorMap *tmC,
                                                  int n, int row0,
                                                  float2 scale) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const __nv_bfloat162 h =
        __floats2bfloat162_rn(apply_scales(v[2 * j], scale),
                              apply_scales(v[2 * j + 1], scale));
    w[j] = *reinterpret_cast<const uint32_t *>(&h);
  }
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  const uint32_t rowbase = stage + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
  for (uint32_t q = 0; q < 4; ++q)
    st_shared_v4(rowbase + 16u * (q ^ sw), w[4 * q], w[4 * q + 1],
                 w[4 * q + 2], w[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmC, stage, n, row0);
    bulk_commit_group();
  }
}

template <int BN, int STAGES, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_e4m3_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs a) {
  using L = Smem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The grouped set-up reads m_offsets, so it waits for the previous
  // kernel in the stream first (a no-op unless launched with programmatic
  // stream serialization).
  if (GROUPED) pdl_wait();

  const uint32_t bar0 = base + L::kBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t final_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + L::kMisc + 4);
  int32_t *pref = reinterpret_cast<int32_t *>(sbase + L::kPrefix);
  __shared__ int32_t offs_smem[GROUPED ? kMaxGroups + 1 : 1];

  const int tiles_n = (a.N + BN - 1) / BN;
  const int nkb = (a.K + BK - 1) / BK;

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), BM);  // every epilogue thread arrives
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  int total_tiles;
  if (GROUPED && warp == 0)
    load_group_offsets<BM>(a, tiles_n, offs_smem, pref, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The set-up above reads no input memory, so it may overlap the previous
  // kernel in the stream; operands and scales are read only after this.
  if (!GROUPED) pdl_wait();
  const uint32_t tmem_base = *tmem_slot;
  total_tiles = GROUPED ? pref[a.num_groups]
                        : ((a.M + BM - 1) / BM) * tiles_n;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t s = 0, ph = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        const TileInfo ti =
            tile_info<GROUPED, BM>(t, a, tiles_n, pref, offs_smem, BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns, a.status,
                         abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + L::kA + s * L::kABytes;
          const uint32_t sb = base + L::kB + s * L::kBBytes;
          if (!(a.withhold_first && issued == 0)) {
            mbar_arrive_expect_tx(full_bar(s), L::kStageBytes);
            tma_load_2d(sa, &tmA, full_bar(s), kb * BK, ti.row0);
            if (GROUPED)
              tma_load_3d(sb, &tmB, full_bar(s), kb * BK, ti.n0, ti.group);
            else
              tma_load_2d(sb, &tmB, full_bar(s), kb * BK, ti.n0);
          }
          ++issued;
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      // Drain: wait for the last load issued into each stage, so that no
      // copy is still writing shared memory when the CTA exits.
      for (uint32_t st = 0; st < STAGES; ++st) {
        if (issued <= st) break;
        const uint32_t arms = (issued - 1 - st) / STAGES + 1;
        if (a.withhold_first && st == 0 && arms == 1) continue;
        mbar_wait_drain(full_bar(st), (arms - 1) & 1u, a.timeout_ns, a.status);
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_e4m3_f32(BM, BN) | a.fmt_bits;
      uint32_t s = 0, ph = 0;
      uint32_t local = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles;
           t += gridDim.x, ++local) {
        const uint32_t buf = local & 1u, use = local >> 1;
        if (!mbar_wait(tempty_bar(buf), (use & 1u) ^ 1u, a.timeout_ns,
                       a.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(s), ph, a.timeout_ns, a.status,
                         abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc =
              smem_desc_k128_sw128(base + L::kA + s * L::kABytes);
          const uint64_t bdesc =
              smem_desc_k128_sw128(base + L::kB + s * L::kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            // +32 bytes along K inside the 128-byte swizzled row = +2 in
            // the descriptor's (address >> 4) field.
            umma_f8f6f4(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc,
                        (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(empty_bar(s));
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull_bar(buf));
      }
      // Make sure every MMA issued has finished before tensor memory is
      // released at exit.
      umma_commit(final_bar);
      mbar_wait_drain(final_bar, 0, a.timeout_ns, a.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    uint32_t local = 0;
    float2 scale = make_float2(1.0f, 1.0f);
    int cur_group = -1;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++local) {
      const TileInfo ti =
          tile_info<GROUPED, BM>(t, a, tiles_n, pref, offs_smem, BN);
      if (ti.group != cur_group) {
        scale = make_float2(a.scale_a[ti.group], a.scale_b[ti.group]);
        cur_group = ti.group;
      }
      const uint32_t buf = local & 1u, use = local >> 1;
      // The whole warp must agree before the warp-collective tcgen05.ld.
      const bool ready = mbar_wait(tfull_bar(buf), use & 1u, a.timeout_ns,
                                   a.status, abort_flag);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      const int row = ti.row0 + warp * 32 + lane;
      const bool row_ok = row < ti.row_end && row < ti.row0 + BM;
      uint16_t *crow = a.C + static_cast<int64_t>(row) * a.ldc;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + buf * BN;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32)
        store_chunk32(taddr + c, row_ok, crow, ti.n0 + c, a.N, scale,
                      a.c_vec16 != 0);
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
    }
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

// --------------------------------------------------------------------------
// CTA-pair variant (tcgen05 cta_group::2).  A cluster of two CTAs on two SMs
// computes a 256 x 256 tile: CTA r loads A rows row0 + 128r .. +127 and B
// rows (= C columns) n0 + 128r .. +127 into its own shared memory (32 KB per
// 128-wide K stage, 6 stages), and one thread of the leader CTA (rank 0)
// issues M=256, N=256, K=32 MMAs that read both CTAs' shared memory and
// accumulate into both CTAs' tensor memory (CTA r holds rows 128r.. of the
// tile, all 256 columns).  Per SM this halves the B bytes moved per MMA
// FLOP compared with the single-CTA 128 x 256 tile.  When the last wave of
// tiles would fill at most half the clusters, those tiles are computed as
// two 256 x 128 halves (N = 128 MMAs, 64 B rows per CTA), so the tail takes
// half a tile's time.  Both CTAs' TMA loads
// complete on the leader's `full` barrier; the leader's commits are
// multicast to both CTAs' `empty` / `tmem_full` barriers; both CTAs'
// epilogue warps release an accumulator on the leader's `tmem_empty`.
// The epilogue writes each whole 32 x 32 BF16 block of C through a 2 KB
// shared-memory staging buffer per warp and one TMA store (store_chunk32_tma);
// blocks on the edge of C, or of a group in the grouped GEMM, are stored
// row by row (store_chunk32).
constexpr int P_BM = 256;   // tile rows per CTA pair
constexpr int P_BN = 256;   // tile columns per CTA pair
constexpr int P_STAGES = 6;
// Warps 0-3 and 6-9 are epilogue warps (two per TMEM lane quarter, each
// storing half of the tile's columns); warp 4 loads, warp 5 issues MMAs.
constexpr int P_THREADS = 320;
constexpr int P_EPI_WARPS = 8;

struct PairSmem {
  static constexpr int kABytes = 128 * BK;   // this CTA's half of A
  static constexpr int kBBytes = 128 * BK;   // this CTA's half of B
  static constexpr int kTmemCols = 2 * P_BN;
  static constexpr int kA = 0;
  static constexpr int kB = kA + P_STAGES * kABytes;
  static constexpr int kBar = kB + P_STAGES * kBBytes;
  static constexpr int kNumBars = 2 * P_STAGES + 4 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kPrefix = kMisc + 16;
  static constexpr int kEnd = kPrefix + (kMaxGroups + 1) * 4;
  // One 2 KB staging buffer (32 rows x 32 BF16) per epilogue warp for the
  // TMA-store epilogue, 1024-byte aligned for the 64-byte swizzle.
  static constexpr int kCStage = (kEnd + 1023) / 1024 * 1024;
  static constexpr int kCStageBytes = 32 * 32 * 2;
  static constexpr int kAlloc = kCStage + P_EPI_WARPS * kCStageBytes + 1024;
};

static_assert(PairSmem::kCStage % 1024 == 0 &&
                  PairSmem::kCStageBytes % 1024 == 0,
              "C staging buffers");
static_assert(PairSmem::kB % 1024 == 0 && PairSmem::kABytes % 1024 == 0 &&
                  PairSmem::kBBytes % 1024 == 0 && PairSmem::kBar % 8 == 0,
              "pair layout");
static_assert(PairSmem::kAlloc <= 227 * 1024, "shared memory");

// QUAD (per-tensor GEMM only): clusters of four CTAs, two CTA pairs that
// compute horizontally adjacent 256 x 256 tiles (one 256 x 512 cluster tile)
// and so need the same rows of A.  Each CTA loads 64 of the 128 A rows its
// pair position needs and multicasts them to itself and to the CTA at the
// same position in the other pair, which loads the other 64: every A byte
// leaves L2 once per cluster instead of once per pair.  A stage is refilled
// only after both pairs' MMAs have finished with it (each pair's commit
// arrives on the stage's empty barrier in all four CTAs).
template <bool GROUPED, bool QUAD = false>
__global__ void __launch_bounds__(P_THREADS, 1)
    gemm_e4m3_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmB64,
                          const __grid_constant__ CUtensorMap tmC,
                          const __grid_constant__ CUtensorMap tmA64,
                          const GemmArgs a) {
  static_assert(!(GROUPED && QUAD), "clusters of four: per-tensor GEMM only");
  using L = PairSmem;
  constexpr int STAGES = P_STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The grouped set-up reads m_offsets, so it waits for the previous
  // kernel in the stream first (a no-op unless launched with programmatic
  // stream serialization).
  if (GROUPED) pdl_wait();
  const uint32_t rank = cluster_ctarank();
  const uint32_t pair = QUAD ? rank >> 1 : 0;      // which CTA pair
  const uint32_t prank = rank & 1u;                // position in the pair
  const uint32_t lrank = rank & ~1u;               // this pair's leader
  const bool leader = prank == 0;

  const uint32_t bar0 = base + L::kBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t final_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + L::kMisc);
  volatile int *abort_flag =
      reinterpret_cast<volatile int *>(sbase + L::kMisc + 4);
  int32_t *pref = reinterpret_cast<int32_t *>(sbase + L::kPrefix);
  __shared__ int32_t offs_smem[GROUPED ? kMaxGroups + 1 : 1];

  // Column tiles of the work items: 256 per pair, 512 per cluster of four.
  constexpr int kCBN = QUAD ? 2 * P_BN : P_BN;
  const int tiles_n = (a.N + kCBN - 1) / kCBN;
  const int nkb = (a.K + BK - 1) / BK;
  const int cluster_id = QUAD ? blockIdx.x >> 2 : blockIdx.x >> 1;
  const int num_clusters = QUAD ? gridDim.x >> 2 : gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), QUAD ? 2 : 1);   // one commit per pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * P_EPI_WARPS);  // epilogue warps of both CTAs
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(QUAD ? &tmA64 : &tmA);
    tma_prefetch_desc(&tmB);
    if (a.split_tail > 0) tma_prefetch_desc(&tmB64);
  }
  if (warp == 5) {
    tmem_alloc_pair(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish_pair();
  }
  if (GROUPED && warp == 0)
    load_group_offsets<P_BM>(a, tiles_n, offs_smem, pref, lane);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // peer barriers initialised before any remote use
  tc_fence_after();
  // The set-up above reads no input memory, so it may overlap the previous
  // kernel in the stream; operands and scales are read only after this.
  if (!GROUPED) pdl_wait();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = GROUPED ? pref[a.num_groups]
                                  : ((a.M + P_BM - 1) / P_BM) * tiles_n;
  // Work items: the first total_tiles - split tiles whole, the last `split`
  // tiles as two 256 x 128 halves each (so that a last, partly filled wave
  // of tiles takes half as long).
  const int split = GROUPED ? 0 : a.split_tail;
  const int n_whole = total_tiles - split;
  const int n_items = n_whole + 2 * split;
  // Item i -> its tile and half (-1 = whole tile).
  auto item = [&](int i, int &half) {
    int t = i;
    half = -1;
    if (i >= n_whole) {
      t = n_whole + ((i - n_whole) >> 1);
      half = (i - n_whole) & 1;
    }
    TileInfo ti = tile_info<GROUPED, P_BM>(t, a, tiles_n, pref, offs_smem, kCBN);
    // A cluster of four splits its 512 columns between the pairs: 256 each
    // for a whole tile, 128 each for a half (half h covers 256 h .. +255).
    if (QUAD)
      ti.n0 += half < 0 ? 256 * static_cast<int>(pair)
                        : 256 * half + 128 * static_cast<int>(pair);
    else if (half >= 0)
      ti.n0 += 128 * half;
    return ti;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t s = 0, ph = 0, issued = 0;
      bool ok = true;
      for (int i = cluster_id; ok && i < n_items; i += num_clusters) {
        int half;
        const TileInfo ti = item(i, half);
        // A whole tile takes 128 B rows per CTA, a half tile 64.  A
        // transposed tail tile puts this CTA's 128 rows of B_e in the A
        // slot (the MMA's M operand) and the tail rows of A, tn / 2 per CTA
        // (a 128-row box, of which the MMA reads the first tn / 2 <= 128),
        // in the B slot.
        const int brows = half < 0 ? 128 : 64;
        const int arow = ti.row0 + (ti.tn ? ti.tn / 2 : 128) * static_cast<int>(prank);
        const int brow = ti.n0 + brows * static_cast<int>(prank);
        const uint32_t bytes = 2u * (L::kABytes + brows * BK);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, a.timeout_ns, a.status,
                         abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t lf = mapa_shared(full_bar(s), lrank);
          if (leader) mbar_arrive_expect_tx(full_bar(s), bytes);
          // (Diagnostic only: the second CTA leaves out its first loads, so
          // the leader's first stage never fills.)
          if (!(a.withhold_first && !leader && issued == 0)) {
            const uint32_t aslot = base + (ti.tn ? L::kB + s * L::kBBytes
                                                 : L::kA + s * L::kABytes);
            const uint32_t bslot = base + (ti.tn ? L::kA + s * L::kABytes
                                                 : L::kB + s * L::kBBytes);
            if (QUAD)
              // This CTA's 64-row half of its A rows, to itself and to the
              // CTA at the same position in the other pair.
              tma_load_2d_pair_mc(aslot + 8192u * pair, &tmA64, lf, kb * BK,
                                  arow + 64 * static_cast<int>(pair),
                                  static_cast<uint16_t>((1u << rank) |
                                                        (1u << (rank ^ 2u))));
            else
              tma_load_2d_pair(aslot, &tmA, lf, kb * BK, arow);
            if (GROUPED)
              tma_load_3d_pair(bslot, &tmB, lf, kb * BK, brow, ti.group);
            else
              tma_load_2d_pair(base + L::kB + s * L::kBBytes,
                               half < 0 ? &tmB : &tmB64, lf, kb * BK, brow);
          }
          ++issued;
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      // The leader's full barriers count both CTAs' copies: drain them.
      if (leader) {
        for (uint32_t st = 0; st < STAGES; ++st) {
          if (issued <= st) break;
          const uint32_t arms = (issued - 1 - st) / STAGES + 1;
          mbar_wait_drain(full_bar(st), (arms - 1) & 1u, a.timeout_ns,
                          a.status);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------- MMA (leader CTA only)
    // The whole warp runs the loop and waits; one elected lane issues each
    // MMA and commit, so the warp never branches around them.
    if (leader) {
      const uint32_t idesc_whole = idesc_e4m3_f32(P_BM, P_BN) | a.fmt_bits;
      const uint32_t idesc_half = idesc_e4m3_f32(P_BM, P_BN / 2) | a.fmt_bits;
      uint32_t s = 0, ph = 0, local = 0;
      bool ok = true;
      for (int i = cluster_id; ok && i < n_items; i += num_clusters, ++local) {
        uint32_t idesc = i < n_whole ? idesc_whole : idesc_half;
        if (GROUPED) {
          int half;
          const TileInfo ti = item(i, half);
          if (ti.tn) idesc = idesc_e4m3_f32(P_BM, ti.tn) | a.fmt_bits;
        }
        const uint32_t buf = local & 1u, use = local >> 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(tempty_bar(buf), (use & 1u) ^ 1u,
                                  a.timeout_ns, a.status, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * P_BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(full_bar(s), ph, a.timeout_ns, a.status,
                                    abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc =
              smem_desc_k128_sw128(base + L::kA + s * L::kABytes);
          const uint64_t bdesc =
              smem_desc_k128_sw128(base + L::kB + s * L::kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_f8f6f4_pair_warp(d_tmem, adesc + 2u * k, bdesc + 2u * k,
                                  idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair_warp(empty_bar(s), QUAD ? 0xF : 0x3);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair_warp(tfull_bar(buf),
                              static_cast<uint16_t>(0x3u << (2u * pair)));
      }
      umma_commit_pair_warp(final_bar, static_cast<uint16_t>(1u << rank));
      mbar_wait_drain(final_bar, 0, a.timeout_ns, a.status);
    }
  } else {
    // ----------------------------------------------- epilogue (both CTAs)
    uint32_t local = 0;
    float2 scale = make_float2(1.0f, 1.0f);
    int cur_group = -1;
    const uint32_t leader_tempty0 = mapa_shared(tempty_bar(0), lrank);
    const uint32_t leader_tempty1 = mapa_shared(tempty_bar(1), lrank);
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter..
    const int col_half = warp >= 6 ? 1 : 0;       // which half of the columns
    const uint32_t cstage = base + L::kCStage +
                            static_cast<uint32_t>(warp < 4 ? warp : warp - 2) *
                                L::kCStageBytes;
    for (int i = cluster_id; i < n_items; i += num_clusters, ++local) {
      int half;
      const TileInfo ti = item(i, half);
      const int width = (half < 0 ? P_BN : P_BN / 2) / 2;   // this warp's share
      const int col0 = col_half * width;
      if (ti.group != cur_group) {
        scale = make_float2(a.scale_a[ti.group], a.scale_b[ti.group]);
        cur_group = ti.group;
      }
      const uint32_t buf = local & 1u, use = local >> 1;
      const bool ready = mbar_wait(tfull_bar(buf), use & 1u, a.timeout_ns,
                                   a.status, abort_flag);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      if (GROUPED && ti.tn) {
        // Transposed tail tile: TMEM lane = C column, TMEM column = C row;
        // the two warps of a lane quarter take alternate 32-row chunks.
        const int n = ti.n0 + 128 * static_cast<int>(prank) + quarter * 32 + lane;
        const uint32_t tbase = tmem_base +
                               (static_cast<uint32_t>(quarter * 32) << 16) +
                               buf * P_BN;
#pragma unroll 1
        for (int c = 32 * col_half; c < ti.tn; c += 64)
          store_chunk32_t(tbase + c, a.C, a.ldc, ti.row0 + c, ti.row_end, n, a.N,
                          scale);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(tempty_bar(buf));
          else
            mbar_arrive_cluster(buf ? leader_tempty1 : leader_tempty0);
        }
        continue;
      }
      const int row_chunk0 =
          ti.row0 + 128 * static_cast<int>(prank) + quarter * 32;
      const int row = row_chunk0 + lane;
      const bool row_ok = row < ti.row_end;
      uint16_t *crow = a.C + static_cast<int64_t>(row) * a.ldc;
      const uint32_t taddr = tmem_base +
                             (static_cast<uint32_t>(quarter * 32) << 16) +
                             buf * P_BN + col0;
      // Whole 32 x 32 blocks inside C (and inside the group) go out by TMA;
      // blocks on an edge are stored row by row.
      const bool rows_whole = a.c_tma != 0 && row_chunk0 + 32 <= ti.row_end;
      if (rows_whole) {
#pragma unroll 1
        for (int c = 0; c < width; c += 32) {
          const int n = ti.n0 + col0 + c;
          if (n + 32 <= a.N)
            store_chunk32_tma(taddr + c, cstage, lane, &tmC, n, row_chunk0,
                              scale);
          else
            store_chunk32(taddr + c, true, crow, n, a.N, scale,
                          a.c_vec16 != 0);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < width; c += 32)
          store_chunk32(taddr + c, row_ok, crow, ti.n0 + col0 + c, a.N, scale,
                        a.c_vec16 != 0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(tempty_bar(buf));
        else
          mbar_arrive_cluster(buf ? leader_tempty1 : leader_tempty0);
      }
    }
    // C stores in flight finish before the CTA (and its shared memory) ends.
    if (lane == 0) bulk_wait_all();
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::kTmemCols);
  }
}

__global__ void zero_c_kernel(uint16_t *C, int64_t ldc, int64_t M, int64_t N) {
  const int64_t n = M * N;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    C[r * ldc + c] = 0;
  }
}

// Grouped variant of the K = 0 case: zero the rows each group owns, after
// the same check of m_offsets as the GEMM kernels make (on failure nothing
// is written and kStatusBadDeviceArg is recorded).
__global__ void zero_c_grouped_kernel(uint16_t *C, int64_t ldc,
                                      const int32_t *m_offsets, int32_t E,
                                      int64_t N, int64_t m_capacity,
                                      unsigned *status) {
  __shared__ int bad;
  if (threadIdx.x == 0)
    bad = m_offsets[0] != 0 || m_offsets[E] > m_capacity;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (m_offsets[e + 1] < m_offsets[e]) bad = 1;
  __syncthreads();
  if (bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadDeviceArg);
    return;
  }
  const int64_t rows = m_offsets[E];
  const int64_t n = rows * N;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    C[r * ldc + c] = 0;
  }
}

constexpr int kBN = 256;
constexpr int kStages = 4;
// 128 x 128 tiles for problems with few 256 x 256 tiles: more CTAs share the
// work (1024^3: 64 CTAs instead of 16 pairs).
constexpr int kSmallBN = 128;
constexpr int kSmallStages = 6;

bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
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

bool encode_3d(CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1,
               uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0,
               uint32_t b1) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TBN, int TSTAGES, bool GROUPED>
fp8la_status launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB,
                         const GemmArgs &args, int64_t max_tiles,
                         cudaStream_t s) {
  using L = Smem<TBN, TSTAGES>;
  auto kern = gemm_e4m3_kernel<TBN, TSTAGES, GROUPED>;
  const int slot = TBN == kSmallBN ? 5 : (GROUPED ? 1 : 0);
  if (once_per_device(slot, [&] {
        return cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
      }) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return FP8LA_ERR_CUDA;
  int64_t grid = max_tiles < sms ? max_tiles : sms;
  if (grid < 1) grid = 1;
  // Plain GEMMs start while the previous kernel in the stream finishes (the
  // kernel waits for it before reading operands; see pdl_wait).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = GROUPED ? 0 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, args) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  return launch_status();
}

// C as a BF16 tensor of `rows` x N with row stride ldc, stored in 32 x 32
// boxes with the 64-byte swizzle (the layout store_chunk32_tma writes).
bool encode_c(CUtensorMap *m, const uint16_t *C, int64_t ldc, int64_t rows,
              int64_t N) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<uint16_t *>(C), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch the CTA-pair kernel on clusters of two CTAs (QUAD: four, two
// pairs), as many clusters as can be resident at once (at most one per work
// tile: a pair tile, or for QUAD a 256 x 512 cluster tile).
template <bool GROUPED, bool QUAD = false>
fp8la_status launch_gemm_pair(const CUtensorMap &tmA, const CUtensorMap &tmB,
                              const CUtensorMap &tmB64, const CUtensorMap &tmC,
                              const CUtensorMap &tmA64, GemmArgs args,
                              int64_t max_tiles, cudaStream_t s) {
  using L = PairSmem;
  auto kern = gemm_e4m3_pair_kernel<GROUPED, QUAD>;
  constexpr int kCluster = QUAD ? 4 : 2;
  const int slot = QUAD ? 6 : (GROUPED ? 3 : 2);
  if (once_per_device(slot, [&] {
        return cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
      }) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(P_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(kCluster, 1, 1);
  int clusters = cached_clusters(slot);
  if (clusters < 1) {
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess ||
        clusters < 1)
      return FP8LA_ERR_CUDA;
    cache_clusters(slot, clusters);
  }
  // Split the tiles of a last, at most half-filled wave into halves (for
  // the per-tensor GEMM, where max_tiles is the exact tile count).
  args.split_tail = 0;
  if (!GROUPED) {
    const int64_t rem = max_tiles % clusters;
    if (rem > 0 && 2 * rem <= clusters) args.split_tail = static_cast<int32_t>(rem);
  }
  const int64_t items = max_tiles + args.split_tail;
  int64_t n = items < clusters ? items : clusters;
  if (n < 1) n = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(kCluster * n), 1, 1);
  // Plain GEMMs start while the previous kernel in the stream finishes (the
  // kernel waits for it before reading operands; see pdl_wait).
  cudaLaunchAttribute attrs[2] = {attr[0], {}};
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = GROUPED ? 1 : 2;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmB64, tmC, tmA64, args) !=
      cudaSuccess)
    return FP8LA_ERR_CUDA;
  return launch_status();
}

// Kernel choice: 0 = by shape, 1 = single-CTA kernel (128 x 256 tiles),
// 2 = CTA-pair kernel, 3 = single-CTA kernel with 128 x 128 tiles, 4 = two
// CTA pairs per cluster sharing A by multicast.
std::atomic<int> g_variant{0};

fp8la_status check_operands(const uint8_t *A, int64_t lda, const uint8_t *B,
                            int64_t ldb, const uint16_t *C, int64_t ldc,
                            int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return FP8LA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FP8LA_OK;
  if (!C || ldc < N) return FP8LA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 1u) != 0) return FP8LA_ERR_ALIGNMENT;
  if (K == 0) return FP8LA_OK;
  if (!A || !B || lda < K || ldb < K) return FP8LA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0)
    return FP8LA_ERR_ALIGNMENT;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31) || lda >= (int64_t(1) << 39) ||
      ldb >= (int64_t(1) << 39))
    return FP8LA_ERR_UNSUPPORTED;
  return FP8LA_OK;
}

fp8la_status gemm_pertensor_impl(const uint8_t *A, int64_t lda,
                                 const uint8_t *B, int64_t ldb, uint16_t *C,
                                 int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 const float *scale_a, const float *scale_b,
                                 cudaStream_t s, int withhold,
                                 uint32_t fmt_bits = 0) {
  fp8la_status st = check_operands(A, lda, B, ldb, C, ldc, M, N, K);
  if (st != FP8LA_OK) return st;
  if (M == 0 || N == 0) return FP8LA_OK;
  if (K > 0 && (!scale_a || !scale_b)) return FP8LA_ERR_INVALID_ARG;
  if (!device_is_sm10x()) return FP8LA_ERR_UNSUPPORTED;
  if (K == 0) {
    const int sms = sm_count();
    zero_c_kernel<<<sms > 0 ? sms * 4 : 1, 256, 0, s>>>(C, ldc, M, N);
    return launch_status();
  }
  // The CTA-pair kernel (256 x 256 tiles) unless the problem has too few
  // rows to fill a pair tile, or so few pair tiles that they would leave
  // three quarters of the SMs idle (then 128 x 128 single-CTA tiles), or the
  // caller asked otherwise.  The diagnostic path uses the single-CTA 128 x 256
  // kernel (withhold == 1) or the CTA-pair kernel (withhold == 2).
  const int v = g_variant.load();
  const int sms = sm_count();
  const int64_t pair_tiles = ((M + P_BM - 1) / P_BM) * ((N + P_BN - 1) / P_BN);
  const bool small = !withhold &&
                     (v == 3 || (v == 0 && sms > 0 && pair_tiles * 4 < sms));
  const bool quad = !withhold && !small && v == 4;
  const bool pair = withhold == 2 || quad ||
                    (!withhold && !small && (v == 2 || (v == 0 && M > BM)));
  CUtensorMap tmA, tmB, tmB64, tmA64{};
  if (!encode_2d(&tmA, A, K, M, lda, BK, BM) ||
      !encode_2d(&tmB, B, K, N, ldb, BK, pair || small ? 128 : kBN) ||
      (pair && !encode_2d(&tmB64, B, K, N, ldb, BK, 64)) ||
      (quad && !encode_2d(&tmA64, A, K, M, lda, BK, 64)))
    return FP8LA_ERR_CUDA;
  unsigned *status = status_word_ptr();
  if (!status) return FP8LA_ERR_CUDA;
  GemmArgs args{};
  args.C = C;
  args.ldc = ldc;
  args.M = static_cast<int32_t>(M);
  args.N = static_cast<int32_t>(N);
  args.K = static_cast<int32_t>(K);
  args.scale_a = scale_a;
  args.scale_b = scale_b;
  args.status = status;
  args.timeout_ns = wait_timeout_ns();
  args.withhold_first = withhold;
  args.c_vec16 = aligned16(C) && ldc % 8 == 0;
  args.fmt_bits = fmt_bits;
  if (pair) {
    CUtensorMap tmC{};
    if (args.c_vec16) {
      if (!encode_c(&tmC, C, ldc, M, N)) return FP8LA_ERR_CUDA;
      args.c_tma = 1;
    }
    if (quad) {
      const int64_t ctiles = ((M + P_BM - 1) / P_BM) * ((N + 2 * P_BN - 1) / (2 * P_BN));
      return launch_gemm_pair<false, true>(tmA, tmB, tmB64, tmC, tmA64, args,
                                           ctiles, s);
    }
    const int64_t tiles = ((M + P_BM - 1) / P_BM) * ((N + P_BN - 1) / P_BN);
    return launch_gemm_pair<false>(tmA, tmB, tmB64, tmC, tmA64, args, tiles, s);
  }
  if (small) {
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + kSmallBN - 1) / kSmallBN);
    return launch_gemm<kSmallBN, kSmallStages, false>(tmA, tmB, args, tiles, s);
  }
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + kBN - 1) / kBN);
  return launch_gemm<kBN, kStages, false>(tmA, tmB, args, tiles, s);
}

}  // namespace
}  // namespace fp8la

using namespace fp8la;

extern "C" fp8la_status fp8_gemm(const uint8_t *A, int64_t lda,
                                 const uint8_t *B, int64_t ldb, uint16_t *C,
                                 int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 const float *scale_a, const float *scale_b,
                                 fp8la_stream_t stream) {
  return gemm_pertensor_impl(A, lda, B, ldb, C, ldc, M, N, K, scale_a,
                             scale_b, reinterpret_cast<cudaStream_t>(stream),
                             0);
}

extern "C" fp8la_status fp8_gemm_ex(const uint8_t *A, int64_t lda,
                                    const uint8_t *B, int64_t ldb, uint16_t *C,
                                    int64_t ldc, int64_t M, int64_t N,
                                    int64_t K, const float *scale_a,
                                    const float *scale_b, int32_t a_format,
                                    int32_t b_format, fp8la_stream_t stream) {
  const auto ok = [](int32_t f) {
    return f == FP8LA_FORMAT_E4M3 || f == FP8LA_FORMAT_E5M2;
  };
  if (!ok(a_format) || !ok(b_format)) return FP8LA_ERR_INVALID_ARG;
  // kind::f8f6f4 format codes: E4M3 = 0, E5M2 = 1 (A at bits 7-9, B at 10-12).
  const uint32_t bits = (static_cast<uint32_t>(a_format) << 7) |
                        (static_cast<uint32_t>(b_format) << 10);
  return gemm_pertensor_impl(A, lda, B, ldb, C, ldc, M, N, K, scale_a,
                             scale_b, reinterpret_cast<cudaStream_t>(stream),
                             0, bits);
}

extern "C" fp8la_status fp8la_diag_gemm_withheld_arrival(
    const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb, uint16_t *C,
    int64_t ldc, const float *scale_a, const float *scale_b,
    fp8la_stream_t stream) {
  return gemm_pertensor_impl(A, lda, B, ldb, C, ldc, BM, kBN, BK, scale_a,
                             scale_b, reinterpret_cast<cudaStream_t>(stream),
                             1);
}

namespace fp8la {
// The CTA-pair kernel with the second CTA's first loads withheld (the
// diagnostic entry point for the block-scaled kernel lives beside it).
fp8la_status diag_pair_withheld(const uint8_t *A, int64_t lda, const uint8_t *B,
                                int64_t ldb, uint16_t *C, int64_t ldc,
                                int64_t M, int64_t N, int64_t K,
                                const float *scale_a, const float *scale_b,
                                cudaStream_t s) {
  if (M <= BM || K <= 0) return FP8LA_ERR_INVALID_ARG;
  return gemm_pertensor_impl(A, lda, B, ldb, C, ldc, M, N, K, scale_a, scale_b,
                             s, 2);
}
}  // namespace fp8la

extern "C" fp8la_status fp8_grouped_gemm(
    int32_t num_groups, const int32_t *m_offsets, int64_t m_capacity,
    const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
    int64_t b_group_stride, uint16_t *C, int64_t ldc, int64_t N, int64_t K,
    const float *scale_a, const float *scale_b, fp8la_stream_t stream) {
  if (num_groups < 1 || num_groups > kMaxGroups || !m_offsets ||
      m_capacity < 0)
    return FP8LA_ERR_INVALID_ARG;
  fp8la_status st = check_operands(A, lda, B, ldb, C, ldc, m_capacity, N, K);
  if (st != FP8LA_OK) return st;
  if (m_capacity == 0 || N == 0) return FP8LA_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!device_is_sm10x()) return FP8LA_ERR_UNSUPPORTED;
  if (K == 0) {
    const int sms = sm_count();
    unsigned *status = status_word_ptr();
    if (!status) return FP8LA_ERR_CUDA;
    zero_c_grouped_kernel<<<sms > 0 ? sms * 4 : 1, 256, 0, s>>>(
        C, ldc, m_offsets, num_groups, N, m_capacity, status);
    return launch_status();
  }
  if (!scale_a || !scale_b) return FP8LA_ERR_INVALID_ARG;
  if (b_group_stride % 16 != 0 || b_group_stride < N * ldb)
    return b_group_stride % 16 != 0 ? FP8LA_ERR_ALIGNMENT
                                    : FP8LA_ERR_INVALID_ARG;
  // CTA pairs when groups average at least one pair tile of rows.
  const int v = g_variant.load() >= 3 ? 0 : g_variant.load();
  const bool pair = v == 2 || (v == 0 && m_capacity >= int64_t(P_BM) * num_groups);
  CUtensorMap tmA, tmB;
  if (!encode_2d(&tmA, A, K, m_capacity, lda, BK, BM) ||
      !encode_3d(&tmB, B, K, N, num_groups, ldb, b_group_stride, BK,
                 pair ? 128 : kBN))
    return FP8LA_ERR_CUDA;
  unsigned *status = status_word_ptr();
  if (!status) return FP8LA_ERR_CUDA;
  GemmArgs args{};
  args.C = C;
  args.ldc = ldc;
  args.M = static_cast<int32_t>(m_capacity);
  args.N = static_cast<int32_t>(N);
  args.K = static_cast<int32_t>(K);
  args.scale_a = scale_a;
  args.scale_b = scale_b;
  args.m_offsets = m_offsets;
  args.num_groups = num_groups;
  args.c_vec16 = aligned16(C) && ldc % 8 == 0;
  args.status = status;
  args.timeout_ns = wait_timeout_ns();
  // Upper bound on the tile count without reading m_offsets: each group
  // adds at most one partial row block.
  if (pair) {
    CUtensorMap tmC{};
    if (args.c_vec16) {
      if (!encode_c(&tmC, C, ldc, m_capacity, N)) return FP8LA_ERR_CUDA;
      args.c_tma = 1;
    }
    const int64_t tiles = ((m_capacity + P_BM - 1) / P_BM + num_groups) *
                          ((N + P_BN - 1) / P_BN);
    return launch_gemm_pair<true>(tmA, tmB, tmB, tmC, tmA, args, tiles, s);
  }
  const int64_t tiles =
      ((m_capacity + BM - 1) / BM + num_groups) * ((N + kBN - 1) / kBN);
  return launch_gemm<kBN, kStages, true>(tmA, tmB, args, tiles, s);
}

extern "C" fp8la_status fp8la_set_gemm_variant(int32_t variant) {
  if (variant < 0 || variant > 4) return FP8LA_ERR_INVALID_ARG;
  g_variant.store(variant);
  return FP8LA_OK;
}
