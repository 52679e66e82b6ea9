// gemm_tc.cu -- instantiations and host launchers of the tcgen05 GEMM.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "tc_gemm.cuh"
#include "tc2_gemm.cuh"

namespace lce {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tile order of a launch (the m_group argument of the launchers): 0 walks
// the column blocks of one row block before the next row block; k > 0
// walks groups of k row blocks, down the rows of a group before the next
// column block; kGroupForL2 sizes the groups so that their rows of A fit in
// L2 (the logits: the tiles in flight share one W panel).
constexpr int kGroupForL2 = -1;
// dX and dW on CTA pairs: groups of 8 row blocks shape a wave of 76 tiles
// about 8 row blocks by 9.5 column blocks, so each operand panel in L2
// serves more of the tiles in flight. On the bf16 LLM head (one box, ncu)
// dX read 5.9 instead of 7.9 GB per launch and dW 4.4 instead of 4.7 GB
// than with whole rows of tiles in turn, and ran 3 % and 1 % faster.
constexpr int kDxDwGroup = 8;

inline int tile_group(int m_group, int num_m_blocks, int tile_m, int K) {
  return m_group == kGroupForL2 ? m_group_for(num_m_blocks, tile_m, K, 2) : m_group;
}

template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int N, int K, int m_group,
                      int* status, const typename Epi::Params& ep, int kid, cudaStream_t s) {
  auto kern = tc_gemm_kernel<A_MN, B_MN, Epi>;
  {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), TC_SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  TcGemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.num_m_blocks = (M + TC_BM - 1) / TC_BM;
  g.num_n_blocks = (N + TC_BN - 1) / TC_BN;
  g.num_tiles = g.num_m_blocks * g.num_n_blocks;
  g.m_inner = tile_group(m_group, g.num_m_blocks, TC_BM, K);
  g.status = status;
  g.use_tma_out = 0;
  g.sched = nullptr;
  if (g.num_tiles == 0) return cudaSuccess;
  const int grid = g.num_tiles < num_sms() ? g.num_tiles : num_sms();
  prof_before(kid, s, 2.0 * M * N * static_cast<double>(K));
  kern<<<grid, TC_THREADS, TC_SMEM_BYTES, s>>>(tmA, tmB, g, ep);
  cudaError_t e = cudaGetLastError();
  prof_after(kid, s);
  return e;
}

template <bool A_MN, bool B_MN, class Epi, bool F16 = false>
cudaError_t launch_tc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap* tmOut, int M, int N,
                       int K, int m_group, int* status, const typename Epi::Params& ep, int kid, cudaStream_t s,
                       const SideGrad* side = nullptr, int* sched = nullptr) {
  auto kern = tc2_gemm_kernel<A_MN, B_MN, Epi, F16>;
  {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), TC2_SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  TcGemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.num_m_blocks = (M + TC2_TILE_M - 1) / TC2_TILE_M;
  g.num_n_blocks = (N + TC2_TILE_N - 1) / TC2_TILE_N;
  g.num_tiles = g.num_m_blocks * g.num_n_blocks;
  g.m_inner = tile_group(m_group, g.num_m_blocks, TC2_TILE_M, K);
  g.status = status;
  g.use_tma_out = tmOut != nullptr ? 1 : 0;
  g.sched = sched;
  if (g.num_tiles == 0) return cudaSuccess;
  const int max_pairs = num_sms() / 2;
  const int pairs = g.num_tiles < max_pairs ? g.num_tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(TC2_THREADS);
  cfg.dynamicSmemBytes = TC2_SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(kid, s, 2.0 * M * N * static_cast<double>(K));
  SideGrad sd;
  if (side != nullptr) {
    sd = *side;
  } else {
    memset(&sd, 0, sizeof(sd));
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmOut != nullptr ? *tmOut : tmA, g, ep, sd);
  prof_after(kid, s);
  return e;
}

}  // namespace

bool tc_pair_default() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LCE_TC_PAIR");
    v = (e != nullptr && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

static CUtensorMapDataType map_dtype(int dt) {
  return dt == LCE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

bool encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t ld,
                      uint32_t box_rows, int dt) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, map_dtype(dt), 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t ld, bool mn_major) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {32, mn_major ? TX_MN_ROWS : 128u};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = mn_major ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_bf16_store(CUtensorMap* map, void* base, uint64_t inner, uint64_t rows, uint64_t ld, int dt) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, map_dtype(dt), 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// logits: A = X [M rows, K] K-major, B = W [N rows, K] K-major; consecutive
// tiles walk down the rows so the CTAs in flight share one W panel.
cudaError_t launch_tc_logits(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap* tmOut, int M, int N,
                             int K, int* status, const EpiLse::Params& ep, bool pair, cudaStream_t s,
                             const SideGrad* side, bool f16, int* sched) {
  if (f16)
    return launch_tc2<false, false, EpiLse, true>(tmX, tmW, tmOut, M, N, K, kGroupForL2, status, ep, K_GEMM_LOGITS_TC,
                                                  s, side, sched);
  if (pair)
    return launch_tc2<false, false, EpiLse>(tmX, tmW, tmOut, M, N, K, kGroupForL2, status, ep, K_GEMM_LOGITS_TC, s,
                                            side, sched);
  return launch_tc<false, false, EpiLse>(tmX, tmW, M, N, K, kGroupForL2, status, ep, K_GEMM_LOGITS_TC, s);
}

// recomputed logits of one class chunk with the gradient epilogue: the
// same operands and tile order as the logits GEMM
cudaError_t launch_tc_grad(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap* tmOut, int M, int N,
                           int K, int* status, const EpiGrad::Params& ep, bool pair, cudaStream_t s, bool f16,
                           int* sched) {
  if (f16)
    return launch_tc2<false, false, EpiGrad, true>(tmX, tmW, tmOut, M, N, K, kGroupForL2, status, ep,
                                                   K_GEMM_RECOMPUTE_TC, s, nullptr, sched);
  if (pair)
    return launch_tc2<false, false, EpiGrad>(tmX, tmW, tmOut, M, N, K, kGroupForL2, status, ep, K_GEMM_RECOMPUTE_TC, s,
                                             nullptr, sched);
  return launch_tc<false, false, EpiGrad>(tmX, tmW, M, N, K, kGroupForL2, status, ep, K_GEMM_RECOMPUTE_TC, s);
}

cudaError_t launch_tc_store(int op, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap* tmOut, int M,
                            int N, int K, int* status, const EpiStore::Params& ep, bool pair, cudaStream_t s,
                            bool f16, const SideGrad* side, int* sched) {
  if (side != nullptr && !(op == TC_DX && (pair || f16))) return cudaErrorInvalidValue;
  if (f16) {  // fp16 operands: CTA-pair kernel only
    switch (op) {
      case TC_DX:
        return launch_tc2<false, true, EpiStore, true>(tmA, tmB, tmOut, M, N, K, kDxDwGroup, status, ep, K_GEMM_DX_TC,
                                                       s, side, sched);
      case TC_DW:
        return launch_tc2<true, true, EpiStore, true>(tmA, tmB, tmOut, M, N, K, kDxDwGroup, status, ep, K_GEMM_DW_TC, s,
                                                      nullptr, sched);
      default:
        return cudaErrorInvalidValue;
    }
  }
  if (pair) {
    switch (op) {
      case TC_DX:
        return launch_tc2<false, true, EpiStore>(tmA, tmB, tmOut, M, N, K, kDxDwGroup, status, ep, K_GEMM_DX_TC, s,
                                                 side, sched);
      case TC_DW:
        return launch_tc2<true, true, EpiStore>(tmA, tmB, tmOut, M, N, K, kDxDwGroup, status, ep, K_GEMM_DW_TC, s,
                                                nullptr, sched);
      case TC_TEST_KK:
        return launch_tc2<false, false, EpiStore>(tmA, tmB, tmOut, M, N, K, 0, status, ep, K_GEMM_TEST, s);
      case TC_TEST_KM:
        return launch_tc2<false, true, EpiStore>(tmA, tmB, tmOut, M, N, K, 0, status, ep, K_GEMM_TEST, s);
      case TC_TEST_MK:
        return launch_tc2<true, false, EpiStore>(tmA, tmB, tmOut, M, N, K, 0, status, ep, K_GEMM_TEST, s);
      case TC_TEST_MM:
        return launch_tc2<true, true, EpiStore>(tmA, tmB, tmOut, M, N, K, 0, status, ep, K_GEMM_TEST, s);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (op) {
    case TC_DX:  // A = G [rows, C] K-major, B = W [C, D] N-major
      return launch_tc<false, true, EpiStore>(tmA, tmB, M, N, K, 0, status, ep, K_GEMM_DX_TC, s);
    case TC_DW:  // A = G^T from G [rows, C] (M-major), B = X [rows, D] N-major
      return launch_tc<true, true, EpiStore>(tmA, tmB, M, N, K, 0, status, ep, K_GEMM_DW_TC, s);
    case TC_TEST_KK:
      return launch_tc<false, false, EpiStore>(tmA, tmB, M, N, K, 0, status, ep, K_GEMM_TEST, s);
    case TC_TEST_KM:
      return launch_tc<false, true, EpiStore>(tmA, tmB, M, N, K, 0, status, ep, K_GEMM_TEST, s);
    case TC_TEST_MK:
      return launch_tc<true, false, EpiStore>(tmA, tmB, M, N, K, 0, status, ep, K_GEMM_TEST, s);
    case TC_TEST_MM:
      return launch_tc<true, true, EpiStore>(tmA, tmB, M, N, K, 0, status, ep, K_GEMM_TEST, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace lce
