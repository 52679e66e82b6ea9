// tc_gemm.cuh -- persistent bf16 GEMM on the sm_103a tensor cores.
//
// out[m, n] = sum_k A(m, k) B(n, k) with bf16 operands and fp32
// accumulation, for the three products of the fused loss: the logits
// z = X W^T (A = X, B = W, both K-major), dX = G W (A = G K-major, B = W
// N-major) and dW = G^T X (A = G M-major, B = X N-major).
//
// One CTA per SM, 8 warps, warp-specialised:
//   warp 0      TMA producer: 128x64 A and 256x64 B tiles (128-byte
//               swizzle) into a 4-stage shared-memory ring
//   warp 1      MMA issuer: 4 x tcgen05.mma (M=128, N=256, K=16) per stage
//               into an fp32 accumulator in tensor memory
//   warp 2      allocates / frees the 512 tensor-memory columns
//   warps 4-7   epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//               32*(w%4)..+31, i.e. one output row per thread) and the
//               per-row epilogue functor
// Two 256-column accumulators alternate between tiles, so the epilogue of
// one tile overlaps the main loop of the next. Every mbarrier wait is
// bounded (see mbar_wait); a wait that gives up sets LCE_ERR_TIMEOUT.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace lce {

constexpr int TC_BK = 64;
constexpr int TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_SMEM_BYTES = TC_STAGES * TC_STAGE_BYTES + 1024 + 256;
constexpr int TC_THREADS = 256;
constexpr int TC_TMEM_COLS = 512;

// Row blocks per group for the grouped M-inner walk: the A rows of a group
// (block_rows x K x a_bytes each) within about 40 MB of L2.
inline int m_group_for(int num_m_blocks, int block_rows, int K, int a_bytes) {
  const double per_block = static_cast<double>(block_rows) * K * a_bytes;
  int gm = static_cast<int>((40.0 * 1024 * 1024) / per_block);
  if (gm < 1) gm = 1;
  return gm < num_m_blocks ? gm : num_m_blocks;
}

struct TcGemmArgs {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles;
  // 0: consecutive tiles walk along N. k >= 1: they walk down M in groups of
  // k row blocks (all N blocks of one group before the next group), so the
  // CTAs in flight share a B panel and the group's A rows stay in L2.
  int m_inner;
  int* status;  // device status word or NULL
  int use_tma_out;  // CTA-pair kernel: epilogue stores bf16 results through the output tensor map
  // CTA-pair kernel: NULL for the static schedule (pair p takes tiles p,
  // p + pairs, ...), or a zeroed device counter from which the pairs claim
  // tiles in order, one at a time (see tc2_gemm.cuh)
  int* sched;
};

__device__ __forceinline__ void tc_tile_coords(const TcGemmArgs& g, int tile, int& mb, int& nb) {
  if (g.m_inner) {
    const int per_group = g.m_inner * g.num_n_blocks;
    const int grp = tile / per_group;
    const int m_first = grp * g.m_inner;
    const int rows_in = g.m_inner < g.num_m_blocks - m_first ? g.m_inner : g.num_m_blocks - m_first;
    const int r = tile - grp * per_group;
    mb = m_first + r % rows_in;
    nb = r / rows_in;
  } else {
    nb = tile % g.num_n_blocks;
    mb = tile / g.num_n_blocks;
  }
}

template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcGemmArgs g, const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TC_STAGES * TC_STAGE_BYTES);
  uint64_t* empty = full + TC_STAGES;
  uint64_t* tfull = empty + TC_STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nkb = (g.K + TC_BK - 1) / TC_BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tc_tile_coords(g, tile, mb, nb);
        const int m0 = mb * TC_BM, n0 = nb * TC_BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * TC_STAGE_BYTES;
          uint8_t* sB = sA + TC_A_BYTES;
          mbar_arrive_expect_tx(&full[stage], TC_STAGE_BYTES);
          const int k0 = kb * TC_BK;
          if (!A_MN) {
            tma_load_2d(sA, &tmA, &full[stage], k0, m0);
          } else {
            tma_load_2d(sA, &tmA, &full[stage], m0, k0);
            tma_load_2d(sA + 8192, &tmA, &full[stage], m0 + 64, k0);
          }
          if (!B_MN) {
            tma_load_2d(sB, &tmB, &full[stage], k0, n0);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) tma_load_2d(sB + 8192 * i, &tmB, &full[stage], n0 + 64 * i, k0);
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == TC_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every issued copy must land before the CTA can exit.
      for (int s = 0; s < TC_STAGES; ++s)
        if (issued_mask & (1u << s)) mbar_wait_drain(&full[s], (issued_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t kIdesc = idesc_16_f32(TC_BM, TC_BN, A_MN, B_MN, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < g.num_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_par ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TC_BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * TC_STAGE_BYTES);
          const uint32_t b_base = a_base + TC_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            // K-major, 128B swizzle: a K step of 16 bf16 is 32 bytes inside
            // the swizzle atom; SBO = 1024 (8 rows of 128 B).
            // MN-major, 128B swizzle: a K step of 16 is 16 rows of 128 B;
            // LBO = 8192 (next 64-wide MN block), SBO = 1024 (next 8 K rows).
            const uint64_t adesc = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024)
                                        : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                        : sdesc_sw128(b_base + kk * 32, 16, 1024);
            tc_mma_bf16(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == TC_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(&tfull[acc]);
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue
    const int q = warp & 3;
    int it = 0;
    for (int tile = blockIdx.x; tile < g.num_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_par, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int mb, nb;
      tc_tile_coords(g, tile, mb, nb);
      const int64_t row = static_cast<int64_t>(mb) * TC_BM + q * 32 + lane;
      const int64_t col0 = static_cast<int64_t>(nb) * TC_BN;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TC_BN;
      EpiIO io{nullptr, nullptr, 0, lane, 0, nullptr};
      Epi::template run<TC_BN / 32, 4>(
          ep, row, col0, nb, [&](int g, float (&v)[128]) { tmem_ld128(taddr + g * 128, v); }, io);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, TC_TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag && g.status != nullptr) atomicOr(g.status, kStatusTimeout);
}

}  // namespace lce
