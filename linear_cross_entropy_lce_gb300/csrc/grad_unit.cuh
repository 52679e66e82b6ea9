// grad_unit.cuh -- forming the gradient tile G from the stored P~, for one
// (column segment, block of RB rows) unit, with NT cooperating threads.
//
// G[r, j] = P~[r, j] * scale[seg(j), r], replaced by gt[r] at the target
// column, written in place over P~ (linear_cross_entropy.py: logits scaled
// by w / denominator, then the one-hot correction). With db_acc the column
// sums of G over the unit's rows are added to db_acc (one fp32 atomic per
// column per unit); when G is stored without the row weights (wrow given)
// each row's contribution is multiplied by wrow[r]. Used by the stand-alone kernel (256 threads) and by the
// otherwise idle warps 2-3 of the CTA-pair GEMM (64 threads), which convert
// one row slab while the next slab's logits are being computed.
#pragma once

#include "internal.h"

namespace lce {

// NRMAX: rows per thread loaded before any store (bytes in flight); the
// 64-thread idle-warp form takes 16 so that few threads keep enough loads
// in flight.
template <class T, int SEGW, int NT, int RB, int NRMAX = 8, class Bar>
__device__ __forceinline__ void grad_unit(const GradArgs& a, int seg, int64_t r_begin, int tid, float* red,
                                          Bar&& bar) {
  constexpr int VE = 16 / static_cast<int>(sizeof(T));
  constexpr int TPR = SEGW / VE;          // threads per row
  constexpr int RPP = NT / TPR;           // rows per pass of all threads
  constexpr int NR = (RB / RPP) < NRMAX ? (RB / RPP) : NRMAX;
  constexpr int PASSES = RB / (RPP * NR);
  static_assert(NT % TPR == 0 && RB % (RPP * NR) == 0, "unit shape");
  const int64_t r_end = (r_begin + RB < a.rows) ? r_begin + RB : a.rows;
  const int lt = tid % TPR;
  const int rsub = tid / TPR;
  const int64_t col = static_cast<int64_t>(seg) * SEGW + lt * VE;
  float colsum[VE];
#pragma unroll
  for (int i = 0; i < VE; ++i) colsum[i] = 0.0f;
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
  if (a.db_acc == nullptr) return;
#pragma unroll
  for (int i = 0; i < VE; ++i) red[rsub * SEGW + lt * VE + i] = colsum[i];
  bar();
  for (int c = tid; c < SEGW; c += NT) {
    float acc = 0.0f;
#pragma unroll 4
    for (int q = 0; q < RPP; ++q) acc += red[q * SEGW + c];
    const int64_t gc = static_cast<int64_t>(seg) * SEGW + c;
    if (gc < a.C) atomicAdd(&a.db_acc[gc], acc);
  }
  bar();  // red is reused by the next unit
}

}  // namespace lce
