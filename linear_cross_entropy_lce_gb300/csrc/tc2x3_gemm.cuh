// tc2x3_gemm.cuh -- fp32 GEMM on the tensor cores by three TF32 products.
//
// out[m, n] = sum_k A(m, k) B(n, k) for fp32 A and B given as hi / lo pairs
// (hi = x rounded to TF32, lo = x - hi, exact in fp32): the accumulator
// receives Ahi*Bhi + Ahi*Blo + Alo*Bhi in fp32 (the dropped Alo*Blo is
// below 2^-21 of |A||B|), so products carry about fp32 accuracy while the
// multiply runs at the TF32 tensor rate (Ootomo & Yokota, 2022).
//
// Each operand is K-major (stored [rows, K]: the logits' X and W, dX's G) or
// MN-major (stored [K, rows]: dX's W, dW's G and X); kind::tf32 takes both,
// as the 16-bit kinds do, so no operand is ever transposed in memory.
//
// The loads and MMAs follow tc2_gemm.cuh (CTA pairs, cta_group::2, 256 x 256
// tiles, bounded waits): per stage each CTA loads 128 rows x 32 fp32 of Ahi,
// Alo, Bhi, Blo (64 KB), 3 stages. A K-major part is one 128-row box of 128
// bytes of K per row, 128-byte swizzle; an MN-major part is four boxes of
// 32 K rows x 32 fp32 (128 bytes) of MN, 4 KB apart, in the 128-byte
// swizzle with 32-byte atoms that tcgen05 takes 32-bit MN-major operands in.
//
// Accumulation. The tensor cores add each MMA's products into the fp32
// accumulator with an error that does not average out over a long K (on
// GB300 it grew about linearly with the number of MMAs: 2e-6 of the largest
// entry at K = 256, 5e-5 at K = 8192 with three products per K step). So
// the MMAs accumulate only TX_KB_CHUNK K blocks (512 values of K) at a time
// into a partial P in tensor memory (columns 0-255); the epilogue warps fold
// each partial into a running sum R (columns 256-511) with ordinary fp32
// adds (tcgen05.ld P and R, add, tcgen05.st R) and release P to the next
// chunk; the tile's epilogue then reads R. The error stays that of a
// 512-long chain whatever K is (about 4e-6 of the largest entry).
//
// When every work item's K range fits in one chunk (g.single), no partial
// ever needs folding: the two halves of tensor memory are then two
// accumulators used in turn, the epilogue reads each directly, and the MMAs
// of the next item run while the epilogue drains the previous one.
//
// The K range may be split over k_splits work items per output tile, whose
// epilogues then add into a zeroed fp32 output (EpiStore mode 4).
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "tc_gemm.cuh"

namespace lce {

struct TxArgs {
  int M, N, K;
  int num_m_blocks, num_n_blocks;  // 256-row / 256-column tiles
  int mn_tiles;                    // num_m_blocks * num_n_blocks
  int num_tiles;                   // mn_tiles * k_splits
  int kb_per_split;                // 32-wide K blocks per work item
  int m_inner;                     // as TcGemmArgs::m_inner (0, or row blocks per group)
  int single;                      // every work item has at most TX_KB_CHUNK K blocks
  int* status;
};

__device__ __forceinline__ void tx_tile(const TxArgs& g, int tile, int& mb, int& nb, int& kb0, int& kb1) {
  const int mn = tile % g.mn_tiles;
  const int ks = tile / g.mn_tiles;
  if (g.m_inner) {
    const int per_group = g.m_inner * g.num_n_blocks;
    const int grp = mn / per_group;
    const int m_first = grp * g.m_inner;
    const int rows_in = g.m_inner < g.num_m_blocks - m_first ? g.m_inner : g.num_m_blocks - m_first;
    const int r = mn - grp * per_group;
    mb = m_first + r % rows_in;
    nb = r / rows_in;
  } else {
    nb = mn % g.num_n_blocks;
    mb = mn / g.num_n_blocks;
  }
  const int nkb = (g.K + 31) / 32;
  kb0 = ks * g.kb_per_split;
  kb1 = kb0 + g.kb_per_split < nkb ? kb0 + g.kb_per_split : nkb;
}

constexpr int TX_BK = 32;  // fp32 elements per 128-byte row
constexpr int TX_STAGES = 3;
constexpr int TX_OP_BYTES = 128 * TX_BK * 4;  // 16 KB: 128 rows of one operand part
constexpr int TX_STAGE_BYTES = 4 * TX_OP_BYTES;
constexpr int TX_SMEM_BYTES = TX_STAGES * TX_STAGE_BYTES + 1024 + 512;
constexpr int TX_THREADS = 256;
constexpr int TX_KB_CHUNK = 16;  // K blocks of 32 accumulated in tensor memory before a fold
constexpr int TX_MN_BOX_BYTES = TX_BK * 32 * 4;  // MN-major box: 32 K rows x 32 fp32

// kind::tf32 instruction descriptor with the operands' major-ness: bit 15
// (A) / bit 16 (B) set = MN-major.
__host__ __device__ constexpr uint32_t idesc_tf32_major(int M, int N, bool a_mn, bool b_mn) {
  return idesc_tf32_f32(M, N) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16);
}

// Shared-memory descriptor of K step kk (8 fp32 of K) of one 128-row part.
// K-major: rows of 128 bytes of K, 8-row groups 1024 bytes apart, K step
// 32 bytes into the swizzled row. MN-major: rows of 128 bytes of MN (one K
// value each, consecutive), the four 32-wide MN boxes TX_MN_BOX_BYTES apart
// (leading offset), 4-row K groups (the 32-byte-atom swizzle's period)
// 512 bytes apart; a K step of 8 rows is 1024 bytes.
template <bool MN>
__device__ __forceinline__ uint64_t tx_sdesc(uint32_t part, int kk) {
  return MN ? sdesc_sw128_atom32(part + kk * 1024, TX_MN_BOX_BYTES, 512) : sdesc_sw128(part + kk * 32, 16, 1024);
}

template <bool MN>
__device__ __forceinline__ void tx_load_part(uint8_t* dst, const CUtensorMap* map, uint32_t bar, int k0, int r0) {
  if (!MN) {
    tma_load_2d_pair(dst, map, bar, k0, r0);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d_pair(dst + j * TX_MN_BOX_BYTES, map, bar, r0 + 32 * j, k0);
  }
}

template <bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(TX_THREADS, 1)
    tc2x3_gemm_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                      const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                      const TxArgs g, const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TX_STAGES * TX_STAGE_BYTES);
  uint64_t* empty = full + TX_STAGES;
  // [2]: partial P complete (MMA -> fold), or with g.single accumulator b complete
  uint64_t* pfull = empty + TX_STAGES;
  // [2]: P folded into R (fold -> MMA), or accumulator b drained; 8 arrivals
  uint64_t* pempty = pfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(nclusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < TX_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmAh);
    tma_prefetch_desc(&tmAl);
    tma_prefetch_desc(&tmBh);
    tma_prefetch_desc(&tmBl);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      for (int tile = pair; tile < g.num_tiles && ok; tile += npairs) {
        int mb, nb, kb0, kb1;
        tx_tile(g, tile, mb, nb, kb0, kb1);
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int n0 = nb * 256 + static_cast<int>(rank) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * TX_STAGE_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * TX_STAGE_BYTES);
          const uint32_t bar = mapa_u32(&full[stage], 0);
          const int k0 = kb * TX_BK;
          tx_load_part<A_MN>(st, &tmAh, bar, k0, m0);
          tx_load_part<A_MN>(st + TX_OP_BYTES, &tmAl, bar, k0, m0);
          tx_load_part<B_MN>(st + 2 * TX_OP_BYTES, &tmBh, bar, k0, n0);
          tx_load_part<B_MN>(st + 3 * TX_OP_BYTES, &tmBl, bar, k0, n0);
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == TX_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < TX_STAGES; ++s)
        if (issued_mask & (1u << s)) mbar_wait_cluster_drain(&empty[s], (issued_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA only): 3 TF32 products per K
      // step into the partial P, one chunk of TX_KB_CHUNK K blocks at a time
      constexpr uint32_t kIdesc = idesc_tf32_major(256, 256, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t q = 0;  // chunks issued so far (pfull / pempty phase)
      const bool single = g.single != 0;
      bool ok = true;
      for (int tile = pair; tile < g.num_tiles && ok; tile += npairs) {
        int mb, nb, kb0, kb1;
        tx_tile(g, tile, mb, nb, kb0, kb1);
        for (int c0 = kb0; c0 < kb1 && ok; c0 += TX_KB_CHUNK, ++q) {
          const int c1 = c0 + TX_KB_CHUNK < kb1 ? c0 + TX_KB_CHUNK : kb1;
          // accumulator of this chunk: P (columns 0-255), or with single
          // work items the two halves in turn
          const uint32_t buf = single ? (q & 1u) : 0u;
          const uint32_t par = single ? ((q >> 1) & 1u) : (q & 1u);
          if (!mbar_wait_cluster(&pempty[buf], par ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = c0; kb < c1; ++kb) {
            if (!mbar_wait_cluster(&full[stage], phase, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t base = smem_u32(smem + stage * TX_STAGE_BYTES);
#pragma unroll
            for (int kk = 0; kk < TX_BK / 8; ++kk) {
              const uint64_t ah = tx_sdesc<A_MN>(base, kk);
              const uint64_t al = tx_sdesc<A_MN>(base + TX_OP_BYTES, kk);
              const uint64_t bh = tx_sdesc<B_MN>(base + 2 * TX_OP_BYTES, kk);
              const uint64_t bl = tx_sdesc<B_MN>(base + 3 * TX_OP_BYTES, kk);
              const uint32_t acc = (kb == c0 && kk == 0) ? 0u : 1u;
              const uint32_t d = tmem_base + buf * 256;
              tc_mma_tf32_pair(d, ah, bh, kIdesc, acc);
              tc_mma_tf32_pair(d, ah, bl, kIdesc, 1u);
              tc_mma_tf32_pair(d, al, bh, kIdesc, 1u);
            }
            tc_commit_pair_mc(&empty[stage], 0x3);
            if (++stage == TX_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc_commit_pair_mc(&pfull[buf], 0x3);
        }
      }
    }
  } else if (warp >= 4) {
    // ---------------- fold + epilogue (both CTAs): this CTA's 128 rows
    const int qw = warp & 3;
    const uint32_t tP = tmem_base + (static_cast<uint32_t>(qw * 32) << 16);
    const uint32_t tR = tP + 256;
    EpiIO io{nullptr, nullptr, 0, lane, 0, nullptr};
    uint32_t q = 0;
    bool ok = true;
    for (int tile = pair; tile < g.num_tiles && ok; tile += npairs) {
      int mb, nb, kb0, kb1;
      tx_tile(g, tile, mb, nb, kb0, kb1);
      const int64_t row = static_cast<int64_t>(mb) * 256 + rank * 128 + qw * 32 + lane;
      const int64_t col0 = static_cast<int64_t>(nb) * 256;
      if (g.single) {
        // one chunk: the epilogue reads the accumulator itself, then frees it
        const uint32_t buf = q & 1u;
        int okw = 1;
        if (lane == 0) okw = mbar_wait_cluster(&pfull[buf], (q >> 1) & 1u, abort_flag) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        tc_fence_after();
        const uint32_t tA = tP + buf * 256;
        Epi::template run<8, 4>(
            ep, row, col0, nb, [&](int g, float (&v)[128]) { tmem_ld128(tA + g * 128, v); }, io);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_u32(&pempty[buf], 0));
        ++q;
        continue;
      }
      for (int c0 = kb0; c0 < kb1; c0 += TX_KB_CHUNK, ++q) {
        int okw = 1;
        if (lane == 0) okw = mbar_wait_cluster(&pfull[0], q & 1u, abort_flag) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool first = c0 == kb0;
#pragma unroll 1
        for (int c = 0; c < 256; c += 64) {
          // 64 columns of P and of R per wait; the first chunk of a tile
          // copies P (R's old contents are the previous tile's)
          float p[64], r[64];
          tmem_ld64x2(tP + c, tR + c, p, r);
          float (&p0)[32] = *reinterpret_cast<float(*)[32]>(&p[0]);
          float (&p1)[32] = *reinterpret_cast<float(*)[32]>(&p[32]);
          if (!first) {
#pragma unroll
            for (int i = 0; i < 64; ++i) p[i] += r[i];
          }
          tmem_st32(tR + c, p0);
          tmem_st32(tR + c + 32, p1);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_u32(&pempty[0], 0));
      }
      if (!ok) break;
      Epi::template run<8, 4>(
          ep, row, col0, nb, [&](int g, float (&v)[128]) { tmem_ld128(tR + g * 128, v); }, io);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem_base, 512);
  if (threadIdx.x == 0 && *abort_flag && g.status != nullptr) atomicOr(g.status, kStatusTimeout);
}

}  // namespace lce
