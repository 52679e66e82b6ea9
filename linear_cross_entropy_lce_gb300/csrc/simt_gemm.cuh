// simt_gemm.cuh -- fp32 GEMM on the CUDA cores (exact fp32 FMA products).
//
// out[m, n] = sum_k A(m, k) B(n, k); A(m, k) = A[m*lda + k] (K-major) or
// A[k*lda + m] (M-major), B(n, k) = B[n*ldb + k] or B[k*ldb + n]. Used for
// fp32 inputs, where tensor-core TF32 products would miss a 1e-5 relative
// loss tolerance. 128x128 tiles, 256 threads with 8x8 outputs each; after
// the K loop the tile is staged in shared memory and two threads per row
// run the row epilogue over 64 columns each.
#pragma once

#include "common.cuh"

namespace lce {

constexpr int SG_BM = 128;
constexpr int SG_BN = 128;
constexpr int SG_BK = 16;
constexpr int SG_THREADS = 256;
constexpr int SG_SEG = 64;  // epilogue segment width (columns per thread)
constexpr int SG_CT_LD = SG_BN + 1;
constexpr int SG_SMEM_BYTES = SG_BM * SG_CT_LD * 4;  // >= the two K-loop tiles

template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(SG_THREADS)
    simt_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B, int64_t lda, int64_t ldb,
                     int64_t M, int64_t N, int64_t K, const typename Epi::Params ep) {
  extern __shared__ float sm[];
  float* As = sm;                           // [SG_BK][SG_BM + 4]
  float* Bs = sm + SG_BK * (SG_BM + 4);     // [SG_BK][SG_BN + 4]
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * SG_BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * SG_BN;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  for (int64_t k0 = 0; k0 < K; k0 += SG_BK) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + i * SG_THREADS;
      int mm, kk;
      if (A_MN) {
        kk = idx / SG_BM;
        mm = idx % SG_BM;
      } else {
        mm = idx / SG_BK;
        kk = idx % SG_BK;
      }
      const int64_t gm = m0 + mm, gk = k0 + kk;
      float a = 0.0f;
      if (gm < M && gk < K) a = A_MN ? A[gk * lda + gm] : A[gm * lda + gk];
      As[kk * (SG_BM + 4) + mm] = a;
      int nn;
      if (B_MN) {
        kk = idx / SG_BN;
        nn = idx % SG_BN;
      } else {
        nn = idx / SG_BK;
        kk = idx % SG_BK;
      }
      const int64_t gn = n0 + nn, gk2 = k0 + kk;
      float b = 0.0f;
      if (gn < N && gk2 < K) b = B_MN ? B[gk2 * ldb + gn] : B[gn * ldb + gk2];
      Bs[kk * (SG_BN + 4) + nn] = b;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk * (SG_BM + 4) + ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk * (SG_BM + 4) + 64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk * (SG_BN + 4) + tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk * (SG_BN + 4) + 64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  // stage the tile, then the row epilogue
  float* Ct = sm;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = (j < 4) ? tx * 4 + j : 64 + tx * 4 + (j - 4);
      Ct[r * SG_CT_LD + c] = acc[i][j];
    }
  }
  __syncthreads();
  const int r = tid >> 1, half = tid & 1;
  const int64_t col0 = n0 + half * SG_SEG;
  EpiIO io{nullptr, nullptr, 0, static_cast<int>(threadIdx.x & 31), 0};
  Epi::template run<SG_SEG / 32>(
      ep, m0 + r, col0, col0 / SG_SEG,
      [&](int c, float (&v)[32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = Ct[r * SG_CT_LD + half * SG_SEG + c * 32 + i];
      },
      io);
}

}  // namespace lce
