// grad_unit.cuh -- forming the gradient tile G from the stored P~, for one
// (column segment, block of RB rows) unit, with NT cooperating threads.
//
// G[r, j] = P~[r, j] * scale[seg(j), r], replaced by gt[r] at the target
// column, written in place over P~ (linear_cross_entropy.py: logits scaled
// by w / denominator, then the one-hot correction). With db_acc the column
// sums of G are accumulated per thread (`form`) and added to db_acc by
// `flush` (one fp32 atomic per column); a caller that forms several row
// blocks of the same segment in a row flushes once for all of them. When G
// is stored without the row weights (wrow given) each row's contribution to
// the column sums is multiplied by wrow[r]. Used by the stand-alone kernel
// (256 threads, one unit per CTA) and by the otherwise idle warps 2-3 of the
// CTA-pair GEMM (64 threads), which convert one row slab while another GEMM
// runs.
#pragma once

#include "internal.h"

namespace lce {

// NRMAX: rows per thread loaded before any store (bytes in flight); the
// 64-thread idle-warp form takes 16 so that few threads keep enough loads
// in flight.
template <class T, int SEGW, int NT, int RB, int NRMAX = 8>
struct GradUnit {
  static constexpr int VE = 16 / static_cast<int>(sizeof(T));
  static constexpr int TPR = SEGW / VE;  // threads per row
  static constexpr int RPP = NT / TPR;   // rows per pass of all threads
  static constexpr int NR = (RB / RPP) < NRMAX ? (RB / RPP) : NRMAX;
  static constexpr int PASSES = RB / (RPP * NR);
  static_assert(NT % TPR == 0 && RB % (RPP * NR) == 0, "unit shape");

  // G for rows [r_begin, r_begin + RB) of segment seg; this thread's
  // weighted column sums are added into colsum (its VE columns).
  __device__ static __forceinline__ void form(const GradArgs& a, int seg, int64_t r_begin, int tid,
                                              float (&colsum)[VE]) {
    const int64_t r_end = (r_begin + RB < a.rows) ? r_begin + RB : a.rows;
    const int lt = tid % TPR;
    const int rsub = tid / TPR;
    const int64_t col = static_cast<int64_t>(seg) * SEGW + lt * VE;
#pragma unroll 1
    for (int pass = 0; pass < PASSES; ++pass) {
      const int64_t rp = r_begin + pass * RPP * NR + rsub;
      uint4 raw[NR];
      float sc[NR];
      int tc[NR];
      float wr[NR];
      float gtv[NR];
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        const int64_t r = rp + k * RPP;
        if (r < r_end) {
          raw[k] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.L) + r * a.ld + col);
          sc[k] = a.scale[seg * a.sld + r].x;
          tc[k] = a.tcol[r];
          wr[k] = a.wrow != nullptr ? a.wrow[r] : 1.0f;
          gtv[k] = a.gt[r];
        }
      }
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        const int64_t r = rp + k * RPP;
        if (r >= r_end) continue;
        T* e = reinterpret_cast<T*>(&raw[k]);
#pragma unroll
        for (int i = 0; i < VE; ++i) {
          float gv = to_f32(e[i]) * sc[k];
          if (col + i == tc[k]) gv = gtv[k];
          e[i] = from_f32<T>(gv);
          colsum[i] += wr[k] * to_f32(e[i]);
        }
        *reinterpret_cast<uint4*>(static_cast<T*>(a.L) + r * a.ld + col) = raw[k];
      }
    }
  }

  // Adds the NT threads' column sums of segment seg into db_acc and clears
  // colsum. red: RPP * SEGW floats of shared memory; bar(): a barrier over
  // the NT threads. No-op without db_acc.
  template <class Bar>
  __device__ static __forceinline__ void flush(const GradArgs& a, int seg, int tid, float (&colsum)[VE], float* red,
                                               Bar&& bar) {
    if (a.db_acc == nullptr) return;
    const int lt = tid % TPR;
    const int rsub = tid / TPR;
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      red[rsub * SEGW + lt * VE + i] = colsum[i];
      colsum[i] = 0.0f;
    }
    bar();
    for (int c = tid; c < SEGW; c += NT) {
      float acc = 0.0f;
#pragma unroll 4
      for (int q = 0; q < RPP; ++q) acc += red[q * SEGW + c];
      const int64_t gc = static_cast<int64_t>(seg) * SEGW + c;
      if (gc < a.C) atomicAdd(&a.db_acc[gc], acc);
    }
    bar();  // red is reused by the next flush
  }
};

// One unit, formed and flushed (the stand-alone kernel's form).
template <class T, int SEGW, int NT, int RB, int NRMAX = 8, class Bar>
__device__ __forceinline__ void grad_unit(const GradArgs& a, int seg, int64_t r_begin, int tid, float* red,
                                          Bar&& bar) {
  using U = GradUnit<T, SEGW, NT, RB, NRMAX>;
  float colsum[U::VE];
#pragma unroll
  for (int i = 0; i < U::VE; ++i) colsum[i] = 0.0f;
  U::form(a, seg, r_begin, tid, colsum);
  U::flush(a, seg, tid, colsum, red, bar);
}

}  // namespace lce
