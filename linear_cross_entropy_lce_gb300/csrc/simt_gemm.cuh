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
constexpr int SG_SMEM_BYTES = SG_BM * SG_CT_LD * 4;  // >= the 2 x 2 double-buffered K tiles

template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(SG_THREADS)
    simt_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B, int64_t lda, int64_t ldb,
                     int64_t M, int64_t N, int64_t K, const typename Epi::Params ep) {
  extern __shared__ float sm[];
  // two K-tile buffers: [buf][SG_BK][SG_BM + 4] for A, then the same for B
  constexpr int A_TILE = SG_BK * (SG_BM + 4);
  constexpr int B_TILE = SG_BK * (SG_BN + 4);
  float* As = sm;
  float* Bs = sm + 2 * A_TILE;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * SG_BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * SG_BN;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  // split K: blockIdx.z takes the K range [k_begin, k_end)
  const int64_t kchunk = (K + gridDim.z - 1) / gridDim.z;
  const int64_t k_begin = static_cast<int64_t>(blockIdx.z) * kchunk;
  const int64_t k_end = (k_begin + kchunk < K) ? k_begin + kchunk : K;

  // Each thread moves 8 elements of A and 8 of B per K tile; the next tile
  // is fetched into registers while the current one is multiplied.
  float ra[8], rb[8];
  auto fetch = [&](int64_t k0) {
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
      ra[i] = (gm < M && gk < k_end) ? (A_MN ? A[gk * lda + gm] : A[gm * lda + gk]) : 0.0f;
      int nn;
      if (B_MN) {
        kk = idx / SG_BN;
        nn = idx % SG_BN;
      } else {
        nn = idx / SG_BK;
        kk = idx % SG_BK;
      }
      const int64_t gn = n0 + nn, gk2 = k0 + kk;
      rb[i] = (gn < N && gk2 < k_end) ? (B_MN ? B[gk2 * ldb + gn] : B[gn * ldb + gk2]) : 0.0f;
    }
  };
  auto stash = [&](int buf) {
    float* as = As + buf * A_TILE;
    float* bs = Bs + buf * B_TILE;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + i * SG_THREADS;
      const int amm = A_MN ? idx % SG_BM : idx / SG_BK;
      const int akk = A_MN ? idx / SG_BM : idx % SG_BK;
      as[akk * (SG_BM + 4) + amm] = ra[i];
      const int bnn = B_MN ? idx % SG_BN : idx / SG_BK;
      const int bkk = B_MN ? idx / SG_BN : idx % SG_BK;
      bs[bkk * (SG_BN + 4) + bnn] = rb[i];
    }
  };
  int buf = 0;
  if (k_begin < k_end) {
    fetch(k_begin);
    stash(0);
  }
  __syncthreads();
  for (int64_t k0 = k_begin; k0 < k_end; k0 += SG_BK) {
    const bool more = k0 + SG_BK < k_end;
    if (more) fetch(k0 + SG_BK);
    const float* as = As + buf * A_TILE;
    const float* bs = Bs + buf * B_TILE;
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&as[kk * (SG_BM + 4) + ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&as[kk * (SG_BM + 4) + 64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&bs[kk * (SG_BN + 4) + tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&bs[kk * (SG_BN + 4) + 64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) stash(buf ^ 1);  // the other buffer was last read before the previous barrier
    __syncthreads();
    buf ^= 1;
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
  EpiIO io{nullptr, nullptr, 0, static_cast<int>(threadIdx.x & 31), 0, nullptr};
  Epi::template run<SG_SEG / 32, SG_SEG / 32>(
      ep, m0 + r, col0, col0 / SG_SEG,
      [&](int, float (&v)[SG_SEG]) {
#pragma unroll
        for (int i = 0; i < SG_SEG; ++i) v[i] = Ct[r * SG_CT_LD + half * SG_SEG + i];
      },
      io);
}

}  // namespace lce
