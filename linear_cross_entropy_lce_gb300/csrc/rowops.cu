// rowops.cu -- the per-row and elementwise steps around the GEMMs:
// valid-target count, merge of the per-segment (max, sum-exp) pairs into
// the row log-sum-exp and loss, formation of the gradient tile G, and the
// final loss / bias-gradient reductions.
#include "combine_unit.cuh"
#include "grad_unit.cuh"
#include "internal.h"

namespace lce {

namespace {

// n_valid = #rows whose target is a class index; a target that is neither
// ignore_index nor in [0, C) sets the target-range status bit
// (linear_cross_entropy.py: the _mask / corrected_target / neg_weight_target
// d = sum of unmasked weights). The last block to finish sets the mean's
// denominator: the caller's given value, else the class-weight sum or
// n_valid. out_denom (optional) receives it as fp32.
__global__ void prep_kernel(const int64_t* __restrict__ target, int64_t N, int64_t C, int64_t ign,
                            const float* __restrict__ cw, const float* __restrict__ given_denom, WsHeader* hdr,
                            float* out_denom) {
  __shared__ int s_cnt[32];
  __shared__ int s_bad[32];
  __shared__ double s_ws[32];
  int cnt = 0, bad = 0;
  double ws = 0.0;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < N;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = target[i];
    if (t != ign) {
      if (t >= 0 && t < C) {
        ++cnt;
        if (cw != nullptr) ws += cw[t];
      } else {
        bad = 1;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    ws += __shfl_xor_sync(0xffffffffu, ws, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_cnt[warp] = cnt;
    s_bad[warp] = bad;
    s_ws[warp] = ws;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    cnt = lane < nw ? s_cnt[lane] : 0;
    bad = lane < nw ? s_bad[lane] : 0;
    ws = lane < nw ? s_ws[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
      ws += __shfl_xor_sync(0xffffffffu, ws, o);
    }
    if (lane == 0) {
      if (cnt) atomicAdd(&hdr->n_valid, cnt);
      if (bad) atomicOr(&hdr->status, kStatusTargetRange);
      if (cw != nullptr && ws != 0.0) atomicAdd(&hdr->weight_sum, ws);
      __threadfence();  // this block's sums are visible before it counts itself done
      if (atomicAdd(&hdr->prep_done, 1) == static_cast<int>(gridDim.x) - 1) {
        __threadfence();
        double d;
        if (given_denom != nullptr)
          d = static_cast<double>(*given_denom);
        else if (cw != nullptr)
          d = atomicAdd(&hdr->weight_sum, 0.0);
        else
          d = static_cast<double>(atomicAdd(&hdr->n_valid, 0));
        hdr->denom = d;
        if (out_denom != nullptr) *out_denom = static_cast<float>(d);
      }
    }
  }
}

// Stand-alone per-row merge: 32 rows x COMBINE_SL segment lanes per block.
constexpr int COMBINE_SL = 32;

__global__ void __launch_bounds__(32 * COMBINE_SL) combine_kernel(const CombineArgs a) {
  __shared__ float sm[2 * 32 * COMBINE_SL + 64];
  combine_rows32<32 * COMBINE_SL>(a, static_cast<int64_t>(blockIdx.x) * 32, threadIdx.x, sm,
                                  [] { __syncthreads(); });
}

// Stand-alone G formation: one (segment, 64-row block) unit per CTA.
template <class T, int SEGW>
__global__ void __launch_bounds__(256) grad_logits_kernel(const GradArgs a) {
  __shared__ float red[256 / (SEGW / (16 / sizeof(T)))][SEGW];
  grad_unit<T, SEGW, 256, 64>(a, blockIdx.x, static_cast<int64_t>(blockIdx.y) * 64, threadIdx.x, &red[0][0],
                              [] { __syncthreads(); });
}

// max |w| over the rows, NaN if any w is NaN (single block).
__global__ void wmax_kernel(const float* __restrict__ w, int64_t rows, float* out) {
  __shared__ float s_m[32];
  __shared__ int s_nan[32];
  float m = 0.0f;
  int nan = 0;
  for (int64_t i = threadIdx.x; i < rows; i += blockDim.x) {
    const float x = w[i];
    nan |= isnan(x) ? 1 : 0;
    m = fmaxf(m, fabsf(x));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    nan |= __shfl_xor_sync(0xffffffffu, nan, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_m[warp] = m;
    s_nan[warp] = nan;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    m = lane < nw ? s_m[lane] : 0.0f;
    nan = lane < nw ? s_nan[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      nan |= __shfl_xor_sync(0xffffffffu, nan, o);
    }
    if (lane == 0) out[0] = nan ? __int_as_float(0x7fc00000) : m;
  }
}

// Xs[r, :] = (w_r / wbar) X[r, :], fp16, 8 elements per thread (D % 8 == 0).
__global__ void scale_rows_kernel(const __half* __restrict__ X, const float* __restrict__ w,
                                  const float* __restrict__ wbar, __half* __restrict__ Xs, int64_t rows, int64_t D) {
  const int64_t nvec = rows * (D / 8);
  const float wb = wbar[0];
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = v / (D / 8);
    const float f = wb > 0.0f ? w[r] / wb : (isnan(wb) ? wb : 0.0f);
    uint4 raw = reinterpret_cast<const uint4*>(X)[v];
    __half2* h = reinterpret_cast<__half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __half22float2(h[i]);
      h[i] = __floats2half2_rn(x.x * f, x.y * f);
    }
    reinterpret_cast<uint4*>(Xs)[v] = raw;
  }
}

// Deterministic single-block sum of the per-row losses in fp64; mean
// divides by n_valid (NaN when it is 0).
__global__ void loss_finalize_kernel(const float* __restrict__ loss_rows, int64_t N, int reduction,
                                     const WsHeader* hdr, int weighted, float* loss_out) {
  __shared__ double s[32];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) acc += loss_rows[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s[warp] = acc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    acc = lane < nw ? s[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if (reduction == LCE_RED_SUM) {
        loss_out[0] = static_cast<float>(acc);
      } else {
        // mean: over the valid rows, their class weights, or the given denominator
        const double d = hdr->denom;
        loss_out[0] = d == 0.0 ? __int_as_float(0x7fc00000) : static_cast<float>(acc / d);
      }
    }
  }
}

template <class T>
__global__ void db_finalize_kernel(const float* __restrict__ db_acc, T* db, int64_t C) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < C;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    db[i] = from_f32<T>(db_acc[i]);
}

}  // namespace

cudaError_t launch_prep(const int64_t* target, int64_t N, int64_t C, int64_t ignore_index, const float* cw,
                        const float* given_denom, WsHeader* hdr, cudaStream_t s, float* out_denom) {
  int64_t blocks = (N + 1023) / 1024;
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  if (blocks < 1) blocks = 1;  // no rows: one block still sets the denominator
  prof_before(K_PREP, s, 8.0 * N);
  prep_kernel<<<static_cast<unsigned>(blocks), 1024, 0, s>>>(target, N, C, ignore_index, cw, given_denom, hdr,
                                                              out_denom);
  cudaError_t e = cudaGetLastError();
  prof_after(K_PREP, s);
  return e;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const int64_t blocks = (a.rows + 31) / 32;  // 32 rows per block
  prof_before(K_LSE_COMBINE, s, 8.0 * a.rows * a.nseg * (a.backward ? 2 : 1));
  combine_kernel<<<static_cast<unsigned>(blocks), 32 * COMBINE_SL, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  prof_after(K_LSE_COMBINE, s);
  return e;
}

cudaError_t launch_grad_logits(const GradArgs& a, int dt, cudaStream_t s) {
  const bool bf16 = dt != LCE_F32;
  if (a.rows == 0) return cudaSuccess;
  const int64_t gy = (a.rows + 63) / 64;
  if (gy > 65535) return cudaErrorInvalidValue;
  if (bf16 ? a.segw != 256 : (a.segw != 64 && a.segw != 256)) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(a.nseg), static_cast<unsigned>(gy));
  prof_before(K_GRAD_LOGITS, s, 2.0 * (bf16 ? 2 : 4) * a.rows * static_cast<double>(a.ld));  // 16-bit or fp32
  if (dt == LCE_F16)
    grad_logits_kernel<__half, 256><<<grid, 256, 0, s>>>(a);
  else if (dt == LCE_BF16)
    grad_logits_kernel<__nv_bfloat16, 256><<<grid, 256, 0, s>>>(a);
  else if (a.segw == 256)  // fp32 on the tensor cores: 256-column segments
    grad_logits_kernel<float, 256><<<grid, 256, 0, s>>>(a);
  else
    grad_logits_kernel<float, 64><<<grid, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  prof_after(K_GRAD_LOGITS, s);
  return e;
}

cudaError_t launch_row_scale(const void* X, const float* wrow, float* wbar, void* Xs, int64_t rows, int64_t D,
                             cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  prof_before(K_ROW_SCALE, s, 4.0 * rows * static_cast<double>(D) + 4.0 * rows);
  wmax_kernel<<<1, 1024, 0, s>>>(wrow, rows, wbar);
  int64_t blocks = (rows * (D / 8) + 255) / 256;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  scale_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const __half*>(X), wrow, wbar,
                                                                 static_cast<__half*>(Xs), rows, D);
  cudaError_t e = cudaGetLastError();
  prof_after(K_ROW_SCALE, s);
  return e;
}

cudaError_t launch_loss_finalize(const float* loss_rows, int64_t N, int reduction, const WsHeader* hdr,
                                 bool weighted, float* loss_out, cudaStream_t s) {
  prof_before(K_LOSS_FINALIZE, s, 4.0 * N);
  loss_finalize_kernel<<<1, 1024, 0, s>>>(loss_rows, N, reduction, hdr, weighted ? 1 : 0, loss_out);
  cudaError_t e = cudaGetLastError();
  prof_after(K_LOSS_FINALIZE, s);
  return e;
}

cudaError_t launch_db_finalize(const float* db_acc, void* db, int64_t C, int dt, cudaStream_t s) {
  int64_t blocks = (C + 255) / 256;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  prof_before(K_DB_FINALIZE, s, (dt == LCE_F32 ? 8.0 : 6.0) * C);
  if (dt == LCE_BF16)
    db_finalize_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        db_acc, static_cast<__nv_bfloat16*>(db), C);
  else if (dt == LCE_F16)
    db_finalize_kernel<__half><<<static_cast<unsigned>(blocks), 256, 0, s>>>(db_acc, static_cast<__half*>(db), C);
  else
    db_finalize_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, s>>>(db_acc, static_cast<float*>(db), C);
  cudaError_t e = cudaGetLastError();
  prof_after(K_DB_FINALIZE, s);
  return e;
}

// Per-row weights and target columns of a backward given the row lse.
__global__ void backward_rows_kernel(const BackwardRowsArgs a) {
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < a.rows;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = a.row0 + r;
    const int64_t t = a.target[g];
    const bool valid = target_valid(t, a.ignore_index, a.C);
    const float w = row_weight(a.rw, a.hdr, g, t, valid);
    a.tcol[r] = valid ? static_cast<int>(t) : -1;
    a.w_rows[r] = a.wrow != nullptr ? (valid ? 1.0f : 0.0f) : w;
    if (a.wrow != nullptr) a.wrow[r] = w;
  }
}

cudaError_t launch_backward_rows(const BackwardRowsArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  int64_t blocks = (a.rows + 255) / 256;
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  prof_before(K_BACKWARD_ROWS, s, 24.0 * a.rows);
  backward_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  prof_after(K_BACKWARD_ROWS, s);
  return e;
}

// Gradients times a device scalar g, in place, for the backward of the
// scalar-reduction ops (linear_cross_entropy.py precomputes the gradients in
// the forward and multiplies them by grad_output in the backward). Every
// block reads g first and returns at once when g == 1, so a caller needs no
// host-side test of g (no synchronisation) to skip the pass.
template <class T>
__device__ __forceinline__ void scale_span(T* p, int64_t n, float g, int64_t tid, int64_t nthreads) {
  if (p == nullptr || n <= 0) return;
  constexpr int VE = 16 / static_cast<int>(sizeof(T));
  const bool vec = (reinterpret_cast<uintptr_t>(p) & 15) == 0;
  const int64_t nv = vec ? n / VE : 0;
  for (int64_t i = tid; i < nv; i += nthreads) {
    uint4 raw = reinterpret_cast<const uint4*>(p)[i];
    T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
    for (int k = 0; k < VE; ++k) e[k] = from_f32<T>(to_f32(e[k]) * g);
    reinterpret_cast<uint4*>(p)[i] = raw;
  }
  for (int64_t i = nv * VE + tid; i < n; i += nthreads) p[i] = from_f32<T>(to_f32(p[i]) * g);
}

template <class T>
__global__ void __launch_bounds__(256) scale_grads_kernel(T* a, int64_t na, T* b, int64_t nb, T* c, int64_t nc,
                                                          const float* __restrict__ g) {
  const float gv = *g;
  if (gv == 1.0f) return;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  scale_span(a, na, gv, tid, nthreads);
  scale_span(b, nb, gv, tid, nthreads);
  scale_span(c, nc, gv, tid, nthreads);
}

cudaError_t launch_scale_grads(void* a, int64_t na, void* b, int64_t nb, void* c, int64_t nc, int dt,
                               const float* g, cudaStream_t s) {
  const int64_t total = na + nb + nc;
  if (total == 0) return cudaSuccess;
  const int esz = dt == LCE_F32 ? 4 : 2;
  int64_t blocks = (total / (16 / esz) + 255) / 256;
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  if (blocks < 1) blocks = 1;
  prof_before(K_SCALE_GRADS, s, 2.0 * esz * total);
  const unsigned nbk = static_cast<unsigned>(blocks);
  if (dt == LCE_BF16)
    scale_grads_kernel<__nv_bfloat16><<<nbk, 256, 0, s>>>(static_cast<__nv_bfloat16*>(a), na,
                                                          static_cast<__nv_bfloat16*>(b), nb,
                                                          static_cast<__nv_bfloat16*>(c), nc, g);
  else if (dt == LCE_F16)
    scale_grads_kernel<__half><<<nbk, 256, 0, s>>>(static_cast<__half*>(a), na, static_cast<__half*>(b), nb,
                                                   static_cast<__half*>(c), nc, g);
  else
    scale_grads_kernel<float><<<nbk, 256, 0, s>>>(static_cast<float*>(a), na, static_cast<float*>(b), nb,
                                                  static_cast<float*>(c), nc, g);
  cudaError_t e = cudaGetLastError();
  prof_after(K_SCALE_GRADS, s);
  return e;
}

}  // namespace lce
