// combine_unit.cuh -- merge of a row's per-segment (max, sum-exp) pairs into
// its log-sum-exp, loss and gradient scales, for a block of 32 rows.
//
// lse = M + log sum_s s_s exp(m_s - M), loss_n = lse - z_t (0 on ignored
// rows). For the backward each pair of a stored segment becomes the scale
// w_n exp(m_s - lse) that maps the stored P~ to G (and the row's lse and
// weight are kept for classes recomputed later), and G at the target column is
// w_n (softmax_t - 1) from the fp32 target logit (expm1 keeps it accurate
// when softmax_t ~ 1). Used by the stand-alone merge kernel and by the
// otherwise idle warps of the next GEMM (64 threads).
#pragma once

#include "internal.h"

namespace lce {

__device__ __forceinline__ void merge_pair(float& M, float& S, float m2, float s2) {
  if (m2 == -INFINITY) return;  // an empty pair (also covers M == m2 == -inf)
  if (m2 > M) {
    S = (M == -INFINITY ? 0.0f : S * expf(M - m2)) + s2;
    M = m2;
  } else {
    S += s2 * expf(m2 - M);
  }
}

// Rows [r0, r0 + 32) of a.partial (chunk-local). NT threads (a multiple of
// 32): thread t takes row r0 + t % 32 and the segments t / 32, t / 32 + SL,
// ... (SL = NT / 32), 8 loads in flight at a time; warps of the same row set
// meet in shared memory. A warp's 32 threads read one segment of 32
// consecutive rows: one coalesced 256-byte row of the [segment][row] array.
// sm: 2 * NT + 64 floats. bar(): a barrier over the NT threads.
template <int NT, class Bar>
__device__ __forceinline__ void combine_rows32(const CombineArgs& a, int64_t r0, int t, float* sm, Bar&& bar) {
  constexpr int SL = NT / 32;
  float* sM = sm;
  float* sS = sm + NT;
  float* sLse = sm + 2 * NT;
  float* sW = sLse + 32;
  const int rl = t & 31;
  const int sl = t >> 5;
  const int64_t r = r0 + rl;
  const bool in = r < a.rows;
  float M = -INFINITY, S = 0.0f;
  if (in) {
    for (int s0 = sl; s0 < a.nseg; s0 += 8 * SL) {
      float2 p[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int s = s0 + k * SL;
        p[k] = s < a.nseg ? a.partial[s * a.ld + r] : make_float2(-INFINITY, 0.0f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) merge_pair(M, S, p[k].x, p[k].y);
    }
  }
  sM[sl * 32 + rl] = M;
  sS[sl * 32 + rl] = S;
  bar();
  if (sl == 0 && in) {
#pragma unroll 1
    for (int k = 1; k < SL; ++k) merge_pair(M, S, sM[k * 32 + rl], sS[k * 32 + rl]);
    const float lse = M + logf(S);
    const int64_t g = a.row0 + r;
    const int64_t tg = a.target[g];
    const bool valid = target_valid(tg, a.ignore_index, a.C);
    const float zt = valid ? a.zt[r] : 0.0f;
    a.loss_rows[g] = valid ? class_w(a.rw, tg, true) * (lse - zt) : 0.0f;
    if (a.lse_out != nullptr) a.lse_out[g] = lse;
    if (a.backward) {
      const float w = row_weight(a.rw, a.hdr, g, tg, valid);
      // with wrow the stored G leaves w_n out: unit weight on valid rows, 0 on the others
      const float ws = a.wrow != nullptr ? (valid ? 1.0f : 0.0f) : w;
      a.tcol[r] = valid ? static_cast<int>(tg) : -1;
      a.gt[r] = valid ? ws * expm1f(zt - lse) : 0.0f;
      if (a.wrow != nullptr) a.wrow[r] = w;
      if (a.lse_rows != nullptr) a.lse_rows[r] = lse;
      if (a.w_rows != nullptr) a.w_rows[r] = ws;
      sLse[rl] = lse;
      sW[rl] = ws;
    }
  }
  if (a.backward) {
    bar();
    if (in) {
      const float lse = sLse[rl];
      const float ws = sW[rl];
      for (int s0 = sl; s0 < a.nseg_store; s0 += 8 * SL) {
        float m[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int s = s0 + k * SL;
          m[k] = s < a.nseg_store ? a.partial[s * a.ld + r].x : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int s = s0 + k * SL;
          if (s < a.nseg_store) a.partial[s * a.ld + r].x = ws * expf(m[k] - lse);
        }
      }
    }
  }
  bar();  // sm is reused by the next call
}

}  // namespace lce
