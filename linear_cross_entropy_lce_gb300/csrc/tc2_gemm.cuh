// tc2_gemm.cuh -- persistent bf16 GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same contraction and epilogues as tc_gemm.cuh, but each cluster of two
// CTAs (on two SMs) owns a 256 x 256 output tile:
//   * CTA r of the pair loads rows [128r, 128r+128) of the A tile and rows
//     [128r, 128r+128) of the 256-row B tile into its own shared memory; the
//     even CTA issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16), which
//     reads both CTAs' halves and leaves rows 128r.. of the accumulator in
//     CTA r's tensor memory. Each SM thus streams 32 KB per 64-wide K step
//     instead of 48 KB for the same flops, and the 192 KB of shared memory
//     hold 6 stages instead of 4.
//   * both CTAs' TMA loads complete on the even CTA's "full" barrier
//     (cta_group::2 form of the tensor load); the MMA completion is
//     multicast to the "empty" / "accumulator full" barriers of both CTAs;
//     both CTAs' epilogue warps release an accumulator on the even CTA's
//     "accumulator empty" barrier (8 arrivals).
// Warps: 0 TMA producer, 1 MMA issuer (even CTA), 2 tensor-memory
// allocation, 2-3 an optional side job (the per-row merge and G formation
// of another row slab, see SideGrad), 4-7 epilogue (128-column tensor-memory
// loads, stores through TMA where an output map is given). Every wait is
// bounded as in tc_gemm.cuh. Tiles are taken in a static round-robin order,
// or, with a schedule counter, claimed one at a time by the even CTA's
// producer (TC2_SLOTS), so that the tiles in flight on all pairs stay
// consecutive in the tile order however the pairs' speeds differ.
#pragma once

#include "common.cuh"
#include "combine_unit.cuh"
#include "grad_unit.cuh"
#include "ptx.cuh"

namespace lce {

// G formation in idle warps: work chunks of side_rb_group 64-row blocks of
// one column segment. With a bias gradient, 8 blocks share one flush of the
// column sums; without one, single blocks keep the CTAs working at the same
// time on neighbouring segments of the same 64 rows (better DRAM locality).
__host__ __device__ inline int64_t side_rb_group(const GradArgs& a) { return a.db_acc != nullptr ? 8 : 1; }
__host__ __device__ inline int64_t side_chunks(const GradArgs& a) {
  const int64_t rows_per_chunk = 64 * side_rb_group(a);
  return ((a.rows + rows_per_chunk - 1) / rows_per_chunk) * a.nseg;
}

constexpr int TC2_BK = 64;
constexpr int TC2_STAGES = 6;
constexpr int TC2_A_BYTES = 128 * TC2_BK * 2;  // this CTA's 128 rows of A
constexpr int TC2_B_BYTES = 128 * TC2_BK * 2;  // this CTA's 128 rows of the 256-row B tile
constexpr int TC2_STAGE_BYTES = TC2_A_BYTES + TC2_B_BYTES;
constexpr int TC2_STAGING_BYTES = 4 * 2 * 2048;  // epilogue: 2 x 2 KB per epilogue warp
constexpr int TC2_SIDE_BYTES = 2 * 256 * 4;       // warps 2-3: column-sum scratch of the G formation
constexpr int TC2_BIAS_BYTES = 4 * 256 * 4;       // epilogue: one segment of bias per epilogue warp
constexpr int TC2_SMEM_BYTES =
    TC2_STAGES * TC2_STAGE_BYTES + TC2_STAGING_BYTES + TC2_SIDE_BYTES + TC2_BIAS_BYTES + 1024 + 512;
constexpr int TC2_THREADS = 256;
constexpr int TC2_TMEM_COLS = 512;
constexpr int TC2_TILE_M = 256;  // rows per pair tile (128 per CTA)
constexpr int TC2_TILE_N = 256;
// Dynamic schedule: the even CTA's producer claims tiles from a counter and
// passes each tile index through a ring of slots in both CTAs' shared
// memory. Every role of the pair reads every slot in order: the MMA warp,
// the 4 epilogue warps of each CTA and the odd CTA's producer release a slot
// on the even CTA's "slot empty" barrier.
constexpr int TC2_SLOTS = 8;
constexpr int TC2_SLOT_READERS = 10;

// The tile of iteration `it` of the dynamic schedule: wait until the even
// CTA has filled the slot, read it, release it. -1 when a wait gave up.
__device__ __forceinline__ int take_slot(uint64_t* sfull, uint64_t* sempty, volatile int* stile, int it,
                                         volatile int* abort_flag) {
  const int s = it % TC2_SLOTS;
  const uint32_t ph = static_cast<uint32_t>(it / TC2_SLOTS) & 1u;
  if (!mbar_wait_cluster(&sfull[s], ph, abort_flag)) return -1;
  const int t = stile[s];
  mbar_arrive_cluster(mapa_u32(&sempty[s], 0));
  return t;
}

// The side job of warps 2-3 (64 threads, named barrier 1): an optional
// merge phase, then the G formation of side.a (see SideGrad).
template <bool F16>
__device__ __forceinline__ void run_side_job(const SideGrad& side, float* side_red, volatile int* unit_slot,
                                          volatile int* abort_flag) {
  const int tid = threadIdx.x - 64;
  auto bar = [] { asm volatile("bar.sync 1, 64;" ::: "memory"); };
  bool go = true;
  if (side.comb) {
    // merge phase: claimed 32-row blocks, then wait until every block
    // (merged by any CTA) is done before forming G from the scales
    const int64_t nblk = (side.ca.rows + 31) / 32;
    while (true) {
      if (tid == 0) *unit_slot = atomicAdd(side.cclaim, 1);
      bar();
      const int64_t u = *unit_slot;
      bar();
      if (u >= nblk) break;
      combine_rows32<64>(side.ca, u * 32, tid, side_red, bar);
      __threadfence();
      bar();
      if (tid == 0) atomicAdd(side.cdone, 1);
    }
    if (tid == 0) {
      int ok = 1;
      const long long t0 = clock64();
      while (ld_acquire_gpu(side.cdone) < nblk) {
        if (*abort_flag || clock64() - t0 > kWaitLimitCycles) {
          *abort_flag = 1;
          ok = 0;
          break;
        }
      }
      // with the barrier below, the other threads' plain loads of the
      // merged rows see what the merging CTAs wrote before counting
      __threadfence();
      *unit_slot = ok;
    }
    bar();
    go = *unit_slot != 0;
    bar();
  }
  // Work chunks ordered row-group-major (chunk c -> row group c / nseg,
  // segment c % nseg): the column sums are flushed once per chunk and the
  // CTAs working at the same time read neighbouring segments of the same
  // rows.
  const int64_t nrb = (side.a.rows + 63) / 64;
  const int64_t nchunks = side_chunks(side.a);
  const int64_t kRbGroup = side_rb_group(side.a);
  auto run_chunk = [&](int64_t c) {
    using U16 = GradUnit<__half, 256, 64, 64, 16>;
    using UB = GradUnit<__nv_bfloat16, 256, 64, 64, 16>;
    const int seg = static_cast<int>(c % side.a.nseg);
    const int64_t rb0 = (c / side.a.nseg) * kRbGroup;
    float colsum[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) colsum[i] = 0.0f;
    for (int64_t rb = rb0; rb < rb0 + kRbGroup && rb < nrb; ++rb) {
      if (F16)
        U16::form(side.a, seg, rb * 64, tid, colsum);
      else
        UB::form(side.a, seg, rb * 64, tid, colsum);
    }
    if (F16)
      U16::flush(side.a, seg, tid, colsum, side_red, bar);
    else
      UB::flush(side.a, seg, tid, colsum, side_red, bar);
  };
  if (!go) {
    // a merge wait gave up: the launch reports a timeout
  } else if (side.claim == nullptr) {
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) run_chunk(c);
  } else {
    // claimed chunks: progress does not depend on which CTAs are resident
    while (true) {
      if (tid == 0) *unit_slot = atomicAdd(side.claim, 1);
      bar();
      const int64_t c = *unit_slot;
      bar();  // every thread has read the slot before it is rewritten
      if (c >= nchunks) break;
      run_chunk(c);
      fence_proxy_async_all();  // G stores visible to the TMA loads of other CTAs
      __threadfence();
      bar();
      if (tid == 0) atomicAdd(side.done, 1);
    }
  }
}

// Bounded wait of a producer until the side job's G formation is complete
// (all chunks counted), then the proxy fence that lets its TMA loads see
// the G stores. False (abort flag set) when the wait gives up.
__device__ __forceinline__ bool wait_side_done(const SideGrad& side, volatile int* abort_flag) {
  const int target = static_cast<int>(side_chunks(side.a));
  const long long t0 = clock64();
  while (ld_acquire_gpu(side.done) < target) {
    if (*abort_flag || clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
  fence_proxy_async_all();
  return true;
}

template <bool A_MN, bool B_MN, class Epi, bool F16>
__global__ void __launch_bounds__(TC2_THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmOut, const TcGemmArgs g,
                    const typename Epi::Params ep, const SideGrad side) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + TC2_STAGES * TC2_STAGE_BYTES;
  float* side_red = reinterpret_cast<float*>(staging + TC2_STAGING_BYTES);
  float* bias_s = side_red + TC2_SIDE_BYTES / 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + TC2_STAGING_BYTES + TC2_SIDE_BYTES + TC2_BIAS_BYTES);
  uint64_t* empty = full + TC2_STAGES;
  uint64_t* tfull = empty + TC2_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;              // [TC2_SLOTS] dynamic schedule: slot filled
  uint64_t* sempty = sfull + TC2_SLOTS;      // [TC2_SLOTS] slot read by every role (even CTA's are used)
  volatile int* stile = reinterpret_cast<volatile int*>(sempty + TC2_SLOTS);  // [TC2_SLOTS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sempty + TC2_SLOTS) + TC2_SLOTS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* unit_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);  // side job: claimed unit

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = the CTA that issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(nclusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC2_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    for (int q = 0; q < TC2_SLOTS; ++q) {
      mbar_init(&sfull[q], 1);
      mbar_init(&sempty[q], TC2_SLOT_READERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, TC2_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nkb = (g.K + TC2_BK - 1) / TC2_BK;
  const bool dyn = g.sched != nullptr;
  // tile of iteration `it` for the roles that read slots (or the static order)
  auto tile_of = [&](int it) -> int {
    if (!dyn) return pair + it * npairs;
    return take_slot(sfull, sempty, stile, it, abort_flag);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      // rows of A formed by the side job of this launch: wait for all its units once
      bool dep_wait = side.enabled && side.claim != nullptr;
      for (int it = 0; ok; ++it) {
        int tile;
        if (dyn && rank == 0) {
          // claim the next tile and hand it to both CTAs' roles
          const int s = it % TC2_SLOTS;
          const uint32_t ph = static_cast<uint32_t>(it / TC2_SLOTS) & 1u;
          if (!mbar_wait_cluster(&sempty[s], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tile = atomicAdd(g.sched, 1);
          if (tile > g.num_tiles) tile = g.num_tiles;  // the end, for every reader
          stile[s] = tile;
          st_cluster_u32(mapa_u32(const_cast<int*>(&stile[s]), 1), static_cast<uint32_t>(tile));
          mbar_arrive_cluster(mapa_u32(&sfull[s], 0));
          mbar_arrive_cluster(mapa_u32(&sfull[s], 1));
        } else {
          tile = tile_of(it);
          if (tile < 0) {
            ok = false;
            break;
          }
        }
        if (tile >= g.num_tiles) break;
        int mb, nb;
        tc_tile_coords(g, tile, mb, nb);
        const int m0 = mb * TC2_TILE_M + static_cast<int>(rank) * 128;
        const int n0 = nb * TC2_TILE_N + static_cast<int>(rank) * 128;
        if (dep_wait && m0 + 128 > side.dep_row0 && m0 < side.dep_row0 + side.a.rows) {
          if (!wait_side_done(side, abort_flag)) {
            ok = false;
            break;
          }
          dep_wait = false;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * TC2_STAGE_BYTES;
          uint8_t* sB = sA + TC2_A_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * TC2_STAGE_BYTES);
          const uint32_t bar = mapa_u32(&full[stage], 0);
          const int k0 = kb * TC2_BK;
          if (!A_MN) {
            tma_load_2d_pair(sA, &tmA, bar, k0, m0);
          } else {
            tma_load_2d_pair(sA, &tmA, bar, m0, k0);
            tma_load_2d_pair(sA + 8192, &tmA, bar, m0 + 64, k0);
          }
          if (!B_MN) {
            tma_load_2d_pair(sB, &tmB, bar, k0, n0);
          } else {
            tma_load_2d_pair(sB, &tmB, bar, n0, k0);
            tma_load_2d_pair(sB + 8192, &tmB, bar, n0 + 64, k0);
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == TC2_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: a stage's copies have landed once the MMAs that read it are
      // done, which arrives on this CTA's empty barrier.
      for (int s = 0; s < TC2_STAGES; ++s)
        if (issued_mask & (1u << s)) mbar_wait_cluster_drain(&empty[s], (issued_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA only)
      constexpr uint32_t kIdesc = idesc_16_f32(TC2_TILE_M, TC2_TILE_N, A_MN, B_MN, F16);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int tile = tile_of(it);
        if (tile < 0 || tile >= g.num_tiles) break;
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!mbar_wait_cluster(&tempty[acc], acc_par ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TC2_TILE_N;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * TC2_STAGE_BYTES);
          const uint32_t b_base = a_base + TC2_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC2_BK / 16; ++kk) {
            const uint64_t adesc = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024)
                                        : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                        : sdesc_sw128(b_base + kk * 32, 16, 1024);
            tc_mma_bf16_pair(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == TC2_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit_pair_mc(&tfull[acc], 0x3);
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------- side job: merge and G formation of another row slab
    if (side.enabled) run_side_job<F16>(side, side_red, unit_slot, abort_flag);
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs): this CTA's 128 rows of the tile
    const int q = warp & 3;
    EpiIO io{g.use_tma_out ? &tmOut : nullptr, staging + q * 4096, 0, lane, 0, bias_s + q * 256};
    for (int it = 0;; ++it) {
      int tile = 0;
      if (lane == 0) tile = tile_of(it);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0 || tile >= g.num_tiles) break;
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_cluster(&tfull[acc], acc_par, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int mb, nb;
      tc_tile_coords(g, tile, mb, nb);
      const int64_t row = static_cast<int64_t>(mb) * TC2_TILE_M + rank * 128 + q * 32 + lane;
      const int64_t col0 = static_cast<int64_t>(nb) * TC2_TILE_N;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TC2_TILE_N;
      io.row_base = static_cast<int64_t>(mb) * TC2_TILE_M + rank * 128 + q * 32;
      Epi::template run<TC2_TILE_N / 32, 4>(
          ep, row, col0, nb, [&](int g, float (&v)[128]) { tmem_ld128(taddr + g * 128, v); }, io);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_u32(&tempty[acc], 0));
    }
    if (lane == 0) bulk_wait_all();  // every TMA store of this warp has landed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA frees or leaves while its peer may still use it
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem_base, TC2_TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag && g.status != nullptr) atomicOr(g.status, kStatusTimeout);
}

}  // namespace lce
