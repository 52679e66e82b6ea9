// common.cuh -- types shared by the kernels and the host side of liblce.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/lce.h"

namespace lce {

// Output tile of the tcgen05 GEMM (rows x columns); TC_BN is also the
// segment width of the per-row (max, sum-exp) partials on the bf16 path.
constexpr int TC_BM = 128;
constexpr int TC_BN = 256;

// Bits of the device status word (workspace header).
constexpr int kStatusTargetRange = 1;
constexpr int kStatusTimeout = 2;

// Workspace header, at offset 0 of every workspace.
struct WsHeader {
  int status;       // kStatus* bits, OR-ed by kernels
  int n_valid;      // rows whose target is a class index (not ignored, in range)
  double weight_sum;  // sum of class weights over valid rows (class-weighted calls)
  // the mean's denominator d: n_valid, or weight_sum with class weights, or
  // the caller's given value; written once by the last block of the prep
  // kernel, read by everything after it
  double denom;
  int prep_done;    // prep blocks finished
  int pad[57];
};
static_assert(sizeof(WsHeader) <= 256, "header must fit 256 bytes");

// Per-row weight parameters: w_n = valid ? c_n * base * (vec ? g[n] : g0) : 0,
// with c_n = class_weight[target_n] (1 without class weights) and base = 1
// (sum, none) or 1 / d (mean; d = hdr->denom: n_valid, or the sum of c_n over
// valid rows with class weights, or a denominator the caller gives; NaN for
// every row when d == 0).
struct RowWeight {
  const float* grad_out;      // device scalar (sum/mean) or [N] (none); may be NULL
  const float* class_weight;  // [C] or NULL
  int reduction;
  int grad_is_vector;
};

// Element load / store helpers.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
template <class T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) {
  return __float2half_rn(x);
}

// Class weight of a row: class_weight[t] on valid rows (1 without class
// weights), 0 on ignored rows.
__device__ __forceinline__ float class_w(const RowWeight& rw, int64_t t, bool valid) {
  if (!valid) return 0.0f;
  return rw.class_weight != nullptr ? rw.class_weight[t] : 1.0f;
}

__device__ __forceinline__ float row_weight(const RowWeight& rw, const WsHeader* hdr, int64_t n, int64_t t,
                                            bool valid) {
  const bool mean = rw.reduction == LCE_RED_MEAN;
  const bool empty = hdr->denom == 0.0;
  if (!valid) {
    // an ignored row still sees NaN under mean when the divisor is 0
    return (mean && empty) ? __int_as_float(0x7fc00000) : 0.0f;
  }
  float g = 1.0f;
  if (rw.grad_out != nullptr) g = rw.grad_is_vector ? rw.grad_out[n] : rw.grad_out[0];
  const float c = rw.class_weight != nullptr ? rw.class_weight[t] : 1.0f;
  if (mean) {
    if (empty) return __int_as_float(0x7fc00000);
    const float d = static_cast<float>(hdr->denom);
    return c * (1.0f / d) * g;
  }
  return c * g;
}

// A row's target is valid iff it is not ignore_index; a target outside
// [0, C) that is not ignore_index is an error (status bit) and the row is
// treated as ignored.
__device__ __forceinline__ bool target_valid(int64_t t, int64_t ignore_index, int64_t C) {
  return t != ignore_index && t >= 0 && t < C;
}

}  // namespace lce
