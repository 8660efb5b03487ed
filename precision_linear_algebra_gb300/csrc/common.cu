// Library-wide state: the device status word, the wait limit, device
// queries, the tensor-map encoder, status strings and the version.
#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fp8la {

// One status word per device (each device holds its own copy of this
// module variable).  Kernels OR error bits into it.
__device__ unsigned g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
int g_cc_major[kMaxDevices] = {};
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return -1;
  return dev;
}

bool fill_device_info(int dev) {
  if (g_sm_count[dev] > 0) return true;
  int sms = 0, major = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
          cudaSuccess)
    return false;
  g_sm_count[dev] = sms;
  g_cc_major[dev] = major;
  return true;
}
}  // namespace

unsigned *status_word_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned *>(p);
  }
  return g_status_ptr[dev];
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

int current_device_index() { return current_device(); }

namespace {
std::atomic<bool> g_setup[detail::kSlots][detail::kDevs];
std::atomic<int> g_clusters[detail::kSlots][detail::kDevs];
}  // namespace

namespace detail {
bool setup_done(int slot, int dev) { return g_setup[slot][dev].load(); }
void mark_setup_done(int slot, int dev) { g_setup[slot][dev].store(true); }
}  // namespace detail

int cached_clusters(int slot) {
  const int dev = current_device();
  if (dev < 0 || slot < 0 || slot >= detail::kSlots) return -1;
  const int v = g_clusters[slot][dev].load();
  return v > 0 ? v : -1;
}

void cache_clusters(int slot, int clusters) {
  const int dev = current_device();
  if (dev < 0 || slot < 0 || slot >= detail::kSlots) return;
  g_clusters[slot][dev].store(clusters);
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  return fill_device_info(dev) ? g_sm_count[dev] : -1;
}

bool device_is_sm10x() {
  const int dev = current_device();
  if (dev < 0) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  return fill_device_info(dev) && g_cc_major[dev] == 10;
}

EncodeTiledFn encode_tiled_fn() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

}  // namespace fp8la

extern "C" {

fp8la_status fp8_get_device_status(fp8la_stream_t stream) {
  unsigned *p = fp8la::status_word_ptr();
  if (!p) return FP8LA_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FP8LA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FP8LA_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return FP8LA_ERR_CUDA;
  }
  if (v & fp8la::kStatusTimeout) return FP8LA_ERR_DEVICE_TIMEOUT;
  if (v & fp8la::kStatusBadDeviceArg) return FP8LA_ERR_DEVICE_ARG;
  return FP8LA_OK;
}

fp8la_status fp8la_set_wait_timeout_ns(int64_t timeout_ns) {
  if (timeout_ns < 1000) return FP8LA_ERR_INVALID_ARG;
  fp8la::g_timeout_ns.store(static_cast<uint64_t>(timeout_ns));
  return FP8LA_OK;
}

const char *fp8la_status_string(fp8la_status s) {
  switch (s) {
    case FP8LA_OK: return "FP8LA_OK";
    case FP8LA_ERR_INVALID_ARG: return "FP8LA_ERR_INVALID_ARG";
    case FP8LA_ERR_ALIGNMENT: return "FP8LA_ERR_ALIGNMENT";
    case FP8LA_ERR_UNSUPPORTED: return "FP8LA_ERR_UNSUPPORTED";
    case FP8LA_ERR_CUDA: return "FP8LA_ERR_CUDA";
    case FP8LA_ERR_DEVICE_TIMEOUT: return "FP8LA_ERR_DEVICE_TIMEOUT";
    case FP8LA_ERR_DEVICE_ARG: return "FP8LA_ERR_DEVICE_ARG";
    default: return "FP8LA_ERR_UNKNOWN";
  }
}

int fp8la_version(void) { return 101; }

fp8la_status fp8la_diag_withheld_arrival(
    int32_t kernel, const uint8_t *A, int64_t lda, const uint8_t *B,
    int64_t ldb, uint16_t *C, int64_t ldc, int64_t M, int64_t N, int64_t K,
    const float *scale_a, int64_t ld_sa, const float *scale_b, int64_t ld_sb,
    fp8la_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kernel == FP8LA_DIAG_KERNEL_PAIR)
    return fp8la::diag_pair_withheld(A, lda, B, ldb, C, ldc, M, N, K, scale_a,
                                     scale_b, s);
  if (kernel == FP8LA_DIAG_KERNEL_BLOCK32)
    return fp8la::diag_block32_withheld(A, lda, B, ldb, C, ldc, M, N, K,
                                        scale_a, ld_sa, scale_b, ld_sb, s);
  return FP8LA_ERR_INVALID_ARG;
}

}  // extern "C"
