// gemm_tf32.cu -- fp32 inputs on the tensor cores: the TF32 hi / lo split
// and the host launchers of the 3xTF32 CTA-pair GEMM.
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "tc2x3_gemm.cuh"

namespace lce {

static_assert(TX_MN_ROWS == TX_BK, "an MN-major box holds one K block");

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

// One 64 x 64 tile per iteration, 256 threads, over the tiles of a and then
// of b (b.rows == 0: none); reads and writes move float4s (16 threads per
// 64-float row segment) when the matrix's pitches and base pointers allow it
// (vec_a, vec_b), scalar code covers ragged tile edges.
//
// GRAD (a only): a.src is the chunk buffer holding P~ of the fp32 path, and
// the value split is G itself, formed on the way in: G[r, j] = P~[r, j] *
// scale of (j's segment, r), or gt[r] at the row's target column (the same G
// as the stand-alone G formation); with g.db_acc the tile's column sums of G
// are added to it (one atomic per column per tile). G is never written in
// fp32: its hi part goes over P~ in place (a.hi == a.src) and its lo part to
// its buffer, so the G formation and the split read the buffer once.
constexpr int SP_T = 64;
__host__ __device__ inline int64_t split_tiles(const SplitArgs& m) {
  return ((m.rows + SP_T - 1) / SP_T) * ((m.cols + SP_T - 1) / SP_T);
}
template <bool GRAD>
__global__ void __launch_bounds__(256) split_tf32_kernel(const SplitArgs a, const SplitArgs b, const GradArgs g,
                                                         int vec_a, int vec_b) {
  __shared__ float cs[GRAD ? 16 : 1][SP_T];
  const int t = threadIdx.x;
  const int64_t na = split_tiles(a);
  const int64_t ntiles = na + split_tiles(b);
  const int cq = (t & 15) * 4;  // column of this thread's float4 within the tile
  const int rq = t >> 4;        // first row (of 16) within the tile
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const bool in_a = tile < na;
    const float* src = in_a ? a.src : b.src;
    float* hi = in_a ? a.hi : b.hi;
    float* lo = in_a ? a.lo : b.lo;
    const int64_t rows = in_a ? a.rows : b.rows, cols = in_a ? a.cols : b.cols;
    const int64_t lds = in_a ? a.lds : b.lds, ldo = in_a ? a.ldo : b.ldo;
    const int64_t lt = in_a ? tile : tile - na;
    const int64_t tiles_c = (cols + SP_T - 1) / SP_T;
    const int64_t r0 = (lt / tiles_c) * SP_T;
    const int64_t c0 = (lt % tiles_c) * SP_T;
    const bool full_c = (in_a ? vec_a : vec_b) && c0 + cq + 4 <= cols;
    const int seg = GRAD ? static_cast<int>((c0 + cq) / g.segw) : 0;  // the float4 lies in one segment
    float colsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t r = r0 + rq + 16 * k;
      if (r >= rows) continue;
      float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (full_c) {
        const float4 v = *reinterpret_cast<const float4*>(src + r * lds + c0 + cq);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c0 + cq + e < cols) x[e] = src[r * lds + c0 + cq + e];
      }
      if (GRAD) {
        const float sc = g.scale[seg * g.sld + r].x;
        const int64_t tc = g.tcol[r];
        const float gtv = g.gt[r];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[e] = (c0 + cq + e == tc) ? gtv : x[e] * sc;
          colsum[e] += x[e];
        }
      }
      float h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_tf32(x[e], h[e], l[e]);
      if (full_c) {
        *reinterpret_cast<float4*>(hi + r * ldo + c0 + cq) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(lo + r * ldo + c0 + cq) = make_float4(l[0], l[1], l[2], l[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (c0 + cq + e < cols) {
            hi[r * ldo + c0 + cq + e] = h[e];
            lo[r * ldo + c0 + cq + e] = l[e];
          }
        }
      }
    }
    if (GRAD && g.db_acc != nullptr) {
#pragma unroll
      for (int e = 0; e < 4; ++e) cs[rq][cq + e] = colsum[e];
      __syncthreads();
      if (t < SP_T) {
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 16; ++q) sum += cs[q][t];
        if (c0 + t < g.C) atomicAdd(g.db_acc + c0 + t, sum);
      }
      __syncthreads();
    }
  }
}

template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_tx(const TxOperands& o, int M, int N, int K, int m_inner, int splits, int* status,
                      const typename Epi::Params& ep, int kid, cudaStream_t s) {
  auto kern = tc2x3_gemm_kernel<A_MN, B_MN, Epi>;
  {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), TX_SMEM_BYTES);
    if (e != cudaSuccess) return e;
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
  g.single = g.kb_per_split <= TX_KB_CHUNK ? 1 : 0;
  g.num_tiles = g.mn_tiles * splits;
  g.m_inner = m_inner ? m_group_for(g.num_m_blocks, 256, K, 8) : 0;  // hi + lo fp32 parts of A
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

// The kernel for the operands' layouts.
cudaError_t launch_tx_store_any(const TxOperands& o, int M, int N, int K, int splits, int* status,
                                const EpiStore::Params& ep, int kid, cudaStream_t s) {
  if (o.a_mn) {
    return o.b_mn ? launch_tx<true, true, EpiStore>(o, M, N, K, 0, splits, status, ep, kid, s)
                  : launch_tx<true, false, EpiStore>(o, M, N, K, 0, splits, status, ep, kid, s);
  }
  return o.b_mn ? launch_tx<false, true, EpiStore>(o, M, N, K, 0, splits, status, ep, kid, s)
                : launch_tx<false, false, EpiStore>(o, M, N, K, 0, splits, status, ep, kid, s);
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

namespace {
template <bool GRAD>
cudaError_t launch_split(const SplitArgs& a, const SplitArgs& b, const GradArgs& g, int kid, cudaStream_t s) {
  const int64_t ntiles = split_tiles(a) + split_tiles(b);
  if (ntiles == 0) return cudaSuccess;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  auto vec = [&](const SplitArgs& m) {
    return (m.lds % 4 == 0) && (m.ldo % 4 == 0) && al16(m.src) && al16(m.hi) && al16(m.lo) ? 1 : 0;
  };
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  const int grid = static_cast<int>(ntiles < cap ? ntiles : cap);
  // algorithmic bytes: each source read once, its hi and lo parts written
  prof_before(kid, s, 12.0 * (a.rows * static_cast<double>(a.cols) + b.rows * static_cast<double>(b.cols)));
  split_tf32_kernel<GRAD><<<grid, 256, 0, s>>>(a, b, g, vec(a), vec(b));
  cudaError_t e = cudaGetLastError();
  prof_after(kid, s);
  return e;
}
}  // namespace

cudaError_t launch_split_tf32(const SplitArgs& a, cudaStream_t s, const SplitArgs* b) {
  SplitArgs none;
  memset(&none, 0, sizeof(none));
  if (a.rows > 0 && a.cols > 0 && (a.hi == nullptr || a.lo == nullptr)) return cudaErrorInvalidValue;
  if (b != nullptr && b->rows > 0 && b->cols > 0 && (b->hi == nullptr || b->lo == nullptr))
    return cudaErrorInvalidValue;
  GradArgs ng;
  memset(&ng, 0, sizeof(ng));
  return launch_split<false>(a, b != nullptr && b->cols > 0 ? *b : none, ng, K_SPLIT_TF32, s);
}

cudaError_t launch_grad_split_tf32(const GradArgs& g, const SplitArgs& a, cudaStream_t s) {
  if (g.segw % SP_T != 0) return cudaErrorInvalidValue;  // a tile's float4 must lie in one segment
  if (a.hi == nullptr || a.lo == nullptr) return cudaErrorInvalidValue;
  SplitArgs none;
  memset(&none, 0, sizeof(none));
  return launch_split<true>(a, none, g, K_GRAD_SPLIT_TF32, s);
}

cudaError_t launch_tx_logits(const TxOperands& o, int M, int N, int K, int* status, const EpiLse::Params& ep,
                             cudaStream_t s) {
  if (o.a_mn || o.b_mn) return cudaErrorInvalidValue;
  return launch_tx<false, false, EpiLse>(o, M, N, K, 1, 1, status, ep, K_GEMM_LOGITS_TX, s);
}

cudaError_t launch_tx_store(int op, const TxOperands& o, int M, int N, int K, int* status,
                            const EpiStore::Params& ep, cudaStream_t s, int test_splits) {
  if (op == TC_DX) {
    // few output tiles and a long K (= C): split K so that every SM pair has
    // work; the splits add into the zeroed fp32 output (mode 4)
    const int64_t tiles = static_cast<int64_t>((M + 255) / 256) * ((N + 255) / 256);
    const int64_t pairs = num_sms() / 2;
    if (ep.mode == 0 && ep.out_dt == LCE_F32 && ep.row_scale == nullptr && ep.scalar_scale == nullptr &&
        tiles < pairs && K >= 1024) {
      // cost of a split count: K blocks on the busiest pair (waves x K
      // blocks per work item); take the fewest splits (fewest output
      // atomics) within 10 % of the best, at most 16, >= 16 K blocks each
      const int64_t nkb = (K + TX_BK - 1) / TX_BK;
      auto cost = [&](int64_t sp) { return ((tiles * sp + pairs - 1) / pairs) * ((nkb + sp - 1) / sp); };
      int64_t best = nkb;
      for (int64_t sp = 2; sp <= 16 && nkb / sp >= 16; ++sp) best = cost(sp) < best ? cost(sp) : best;
      int64_t splits = 1;
      while (cost(splits) * 10 > best * 11) ++splits;
      if (splits > 1) {
        EpiStore::Params e2 = ep;
        e2.mode = 4;
        cudaError_t e = cudaMemsetAsync(ep.out, 0, static_cast<size_t>(M) * ep.ldo * sizeof(float), s);
        if (e != cudaSuccess) return e;
        return launch_tx_store_any(o, M, N, K, static_cast<int>(splits), status, e2, K_GEMM_DX_TX, s);
      }
    }
    return launch_tx_store_any(o, M, N, K, 1, status, ep, K_GEMM_DX_TX, s);
  }
  if (op == TC_DW) return launch_tx_store_any(o, M, N, K, 1, status, ep, K_GEMM_DW_TX, s);
  if (op == TC_TEST_KK) {
    if (test_splits > 1) {
      EpiStore::Params e2 = ep;
      e2.mode = 4;
      cudaError_t e = cudaMemsetAsync(ep.out, 0, static_cast<size_t>(M) * ep.ldo * sizeof(float), s);
      if (e != cudaSuccess) return e;
      return launch_tx_store_any(o, M, N, K, test_splits, status, e2, K_GEMM_TEST, s);
    }
    return launch_tx_store_any(o, M, N, K, 1, status, ep, K_GEMM_TEST, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lce
