// gemm_simt.cu -- instantiations and host launchers of the fp32 SIMT GEMM.
#include "internal.h"
#include "simt_gemm.cuh"

namespace lce {

namespace {

template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_sg(const float* A, const float* B, int64_t lda, int64_t ldb, int64_t M, int64_t N, int64_t K,
                      const typename Epi::Params& ep, int kid, cudaStream_t s, int splits = 1) {
  auto kern = simt_gemm_kernel<A_MN, B_MN, Epi>;
  {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), SG_SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  if (M == 0 || N == 0) return cudaSuccess;
  const int64_t gx = (N + SG_BN - 1) / SG_BN, gy = (M + SG_BM - 1) / SG_BM;
  if (gy > 65535 || gx > 2147483647LL) return cudaErrorInvalidValue;
  prof_before(kid, s, 2.0 * M * N * static_cast<double>(K));
  kern<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(splits)), SG_THREADS,
         SG_SMEM_BYTES, s>>>(A, B, lda, ldb, M, N, K, ep);
  cudaError_t e = cudaGetLastError();
  prof_after(kid, s);
  return e;
}

}  // namespace

cudaError_t launch_simt_logits(const float* A, const float* B, int64_t lda, int64_t ldb, int64_t M, int64_t N,
                               int64_t K, const EpiLse::Params& ep, cudaStream_t s) {
  return launch_sg<false, false, EpiLse>(A, B, lda, ldb, M, N, K, ep, K_GEMM_LOGITS_SIMT, s);
}

cudaError_t launch_simt_store(int op, const float* A, const float* B, int64_t lda, int64_t ldb, int64_t M,
                              int64_t N, int64_t K, const EpiStore::Params& ep, cudaStream_t s) {
  switch (op) {
    case TC_DX: {
      // few output tiles and a long K (= C): split K over z so every SM has
      // work; the splits add into the zeroed fp32 output (mode 4)
      const int64_t tiles = ((M + SG_BM - 1) / SG_BM) * ((N + SG_BN - 1) / SG_BN);
      if (ep.mode == 0 && ep.out_dt == LCE_F32 && ep.row_scale == nullptr && tiles < 2 * num_sms() && K >= 1024) {
        int64_t splits = (2 * num_sms() + tiles - 1) / tiles;
        if (splits > 16) splits = 16;
        if (splits > K / 256) splits = K / 256;
        if (splits > 1) {
          EpiStore::Params e2 = ep;
          e2.mode = 4;
          cudaError_t e = cudaMemsetAsync(ep.out, 0, static_cast<size_t>(M) * ep.ldo * sizeof(float), s);
          if (e != cudaSuccess) return e;
          return launch_sg<false, true, EpiStore>(A, B, lda, ldb, M, N, K, e2, K_GEMM_DX_SIMT, s,
                                                   static_cast<int>(splits));
        }
      }
      return launch_sg<false, true, EpiStore>(A, B, lda, ldb, M, N, K, ep, K_GEMM_DX_SIMT, s);
    }
    case TC_DW:
      return launch_sg<true, true, EpiStore>(A, B, lda, ldb, M, N, K, ep, K_GEMM_DW_SIMT, s);
    case TC_TEST_KK:
      return launch_sg<false, false, EpiStore>(A, B, lda, ldb, M, N, K, ep, K_GEMM_TEST, s);
    case TC_TEST_KM:
      return launch_sg<false, true, EpiStore>(A, B, lda, ldb, M, N, K, ep, K_GEMM_TEST, s);
    case TC_TEST_MK:
      return launch_sg<true, false, EpiStore>(A, B, lda, ldb, M, N, K, ep, K_GEMM_TEST, s);
    case TC_TEST_MM:
      return launch_sg<true, true, EpiStore>(A, B, lda, ldb, M, N, K, ep, K_GEMM_TEST, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace lce
