// gemm_tf32.cu -- fp32 inputs on the tensor cores: the TF32 hi / lo split
// and the host launchers of the 3xTF32 CTA-pair GEMM.
#include <cstdlib>

#include "internal.h"
#include "tc2x3_gemm.cuh"

namespace lce {

namespace {

// hi = x rounded to TF32; lo = (x - hi) rounded to TF32. x - hi is exact in
// fp32 (hi keeps the leading 11 significant bits of x). A non-finite hi
// (x infinite or NaN, or a finite x that rounds past the largest float)
// keeps x itself and lo = 0, so infinities and NaNs reach the product once.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = round_tf32(x);
  if (isfinite(hi)) {
    lo = round_tf32(x - hi);
  } else {
    hi = x;
    lo = 0.0f;
  }
}

// One 32 x 32 tile of src per iteration, 256 threads (8 rows of 32 lanes,
// 4 rows each); the transposed outputs go through shared memory so both the
// reads and the writes are coalesced.
__global__ void __launch_bounds__(256) split_tf32_kernel(const SplitArgs a) {
  __shared__ float th[32][33];
  __shared__ float tl[32][33];
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;
  const int64_t tiles_c = (a.cols + 31) / 32;
  const int64_t ntiles = ((a.rows + 31) / 32) * tiles_c;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * 32;
    const int64_t c0 = (t % tiles_c) * 32;
    const int64_t c = c0 + tx;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t r = r0 + ty + 8 * k;
      float hi = 0.0f, lo = 0.0f;
      if (r < a.rows && c < a.cols) {
        split_tf32(a.src[r * a.lds + c], hi, lo);
        if (a.hi != nullptr) {
          a.hi[r * a.ldo + c] = hi;
          a.lo[r * a.ldo + c] = lo;
        }
      }
      th[ty + 8 * k][tx] = hi;
      tl[ty + 8 * k][tx] = lo;
    }
    if (a.hiT != nullptr) {
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t cc = c0 + ty + 8 * k;  // row of the transposed outputs
        const int64_t rr = r0 + tx;
        if (cc < a.cols && rr < a.rows) {
          a.hiT[cc * a.ldt + rr] = th[tx][ty + 8 * k];
          a.loT[cc * a.ldt + rr] = tl[tx][ty + 8 * k];
        }
      }
    }
    __syncthreads();
  }
}

template <class Epi>
cudaError_t launch_tx(const TxOperands& o, int M, int N, int K, int m_inner, int splits, int* status,
                      const typename Epi::Params& ep, int kid, cudaStream_t s) {
  auto kern = tc2x3_gemm_kernel<Epi>;
  static bool attr_set = false;  // one device per process is assumed for the attribute cache
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TX_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  TxArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.num_m_blocks = (M + 255) / 256;
  g.num_n_blocks = (N + 255) / 256;
  g.mn_tiles = g.num_m_blocks * g.num_n_blocks;
  const int nkb = (K + TX_BK - 1) / TX_BK;
  if (splits < 1) splits = 1;
  if (splits > nkb) splits = nkb;
  g.kb_per_split = (nkb + splits - 1) / splits;
  splits = (nkb + g.kb_per_split - 1) / g.kb_per_split;  // no empty work item
  g.num_tiles = g.mn_tiles * splits;
  g.m_inner = m_inner;
  g.status = status;
  if (g.mn_tiles == 0 || nkb == 0) return cudaSuccess;
  const int max_pairs = num_sms() / 2;
  const int pairs = g.num_tiles < max_pairs ? g.num_tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(TX_THREADS);
  cfg.dynamicSmemBytes = TX_SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(kid, s, 2.0 * M * N * static_cast<double>(K));
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, o.ah, o.al, o.bh, o.bl, g, ep);
  prof_after(kid, s);
  return e;
}

}  // namespace

bool f32_tensor_default() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LCE_F32_SIMT");
    v = (e != nullptr && e[0] == '1') ? 0 : 1;
  }
  return v == 1;
}

cudaError_t launch_split_tf32(const SplitArgs& a, cudaStream_t s) {
  if (a.rows == 0 || a.cols == 0) return cudaSuccess;
  const int64_t ntiles = ((a.rows + 31) / 32) * ((a.cols + 31) / 32);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  const int grid = static_cast<int>(ntiles < cap ? ntiles : cap);
  const double outs = (a.hi != nullptr ? 2.0 : 0.0) + (a.hiT != nullptr ? 2.0 : 0.0);
  prof_before(K_SPLIT_TF32, s, 4.0 * (1.0 + outs) * a.rows * static_cast<double>(a.cols));
  split_tf32_kernel<<<grid, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  prof_after(K_SPLIT_TF32, s);
  return e;
}

cudaError_t launch_tx_logits(const TxOperands& o, int M, int N, int K, int* status, const EpiLse::Params& ep,
                             cudaStream_t s) {
  return launch_tx<EpiLse>(o, M, N, K, 1, 1, status, ep, K_GEMM_LOGITS_TX, s);
}

cudaError_t launch_tx_store(int op, const TxOperands& o, int M, int N, int K, int* status,
                            const EpiStore::Params& ep, cudaStream_t s, int test_splits) {
  if (op == TC_DX) {
    // few output tiles and a long K (= C): split K so that every SM pair has
    // work; the splits add into the zeroed fp32 output (mode 4)
    const int64_t tiles = static_cast<int64_t>((M + 255) / 256) * ((N + 255) / 256);
    const int pairs = num_sms() / 2;
    if (ep.mode == 0 && ep.out_dt == LCE_F32 && ep.row_scale == nullptr && ep.scalar_scale == nullptr &&
        tiles < pairs && K >= 1024) {
      int64_t splits = (pairs + tiles - 1) / tiles;
      if (splits > 16) splits = 16;
      if (splits > K / 512) splits = K / 512;
      if (splits > 1) {
        EpiStore::Params e2 = ep;
        e2.mode = 4;
        cudaError_t e = cudaMemsetAsync(ep.out, 0, static_cast<size_t>(M) * ep.ldo * sizeof(float), s);
        if (e != cudaSuccess) return e;
        return launch_tx<EpiStore>(o, M, N, K, 0, static_cast<int>(splits), status, e2, K_GEMM_DX_TX, s);
      }
    }
    return launch_tx<EpiStore>(o, M, N, K, 0, 1, status, ep, K_GEMM_DX_TX, s);
  }
  if (op == TC_DW) return launch_tx<EpiStore>(o, M, N, K, 0, 1, status, ep, K_GEMM_DW_TX, s);
  if (op == TC_TEST_KK) {
    if (test_splits > 1) {
      EpiStore::Params e2 = ep;
      e2.mode = 4;
      cudaError_t e = cudaMemsetAsync(ep.out, 0, static_cast<size_t>(M) * ep.ldo * sizeof(float), s);
      if (e != cudaSuccess) return e;
      return launch_tx<EpiStore>(o, M, N, K, 0, test_splits, status, e2, K_GEMM_TEST, s);
    }
    return launch_tx<EpiStore>(o, M, N, K, 0, 1, status, ep, K_GEMM_TEST, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lce
