// 32x32 block-scaled E4M3 GEMM (tcgen05 partials + CUDA-core promotion).
#include "internal.h"

extern "C" fp8la_status fp8_gemm_blockscaled_32x32(
    const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb, uint16_t *C,
    int64_t ldc, int64_t M, int64_t N, int64_t K, const float *sa,
    int64_t ld_sa, const float *sb, int64_t ld_sb, fp8la_stream_t stream) {
  (void)A; (void)lda; (void)B; (void)ldb; (void)C; (void)ldc; (void)M;
  (void)N; (void)K; (void)sa; (void)ld_sa; (void)sb; (void)ld_sb;
  (void)stream;
  return FP8LA_ERR_UNSUPPORTED;
}
