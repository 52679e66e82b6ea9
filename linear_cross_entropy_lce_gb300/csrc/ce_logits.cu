// ce_logits.cu -- cross entropy on given logits, gradient written in place.
//
// Liger-Kernel issue #343 ("cross entropy kernel: inplace modification of
// input") describes one kernel that produces the loss and overwrites the
// logits with dLoss/dlogits during the forward. Here the whole row is read
// from HBM once and written once:
//
//  * resident kernel: a thread-block cluster of CS CTAs (CS = 1..16) owns a
//    row; each CTA holds a 16384-element slice in registers (512 threads x
//    32 elements, 16-byte vector loads), replaces each x_i by
//    e_i = exp(x_i - m_thread) (one exponential per element), reduces its
//    slice to (max, sum-exp), exchanges the pairs through distributed
//    shared memory, and writes g * w_n * (softmax - onehot) back from
//    registers as e_i * g * w_n * exp(m_thread - lse). Clusters walk the
//    rows persistently, each CTA prefetching its slice of the next row into
//    L2 with the copy engine. Needs V <= 16 * 16384 and 16-byte aligned rows.
//  * streaming kernel (any V, any alignment; used when V > 262144, rows are
//    not 16-byte aligned, or no cluster fits): one CTA per row, online
//    (max, sum-exp) in a first pass, gradient in a second pass that reads
//    the row again (largely from L2).
#include <cfloat>

#include "internal.h"

namespace lce {

namespace {

constexpr int CE_THREADS = 512;
constexpr int CE_EPT = 32;
constexpr int64_t CE_SLICE = static_cast<int64_t>(CE_THREADS) * CE_EPT;  // 16384

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Warp-wide merge of per-lane (max, sum of exp(x - max)) pairs: the warp's
// max first, then one rescale per lane and a sum. Every lane gets the pair.
__device__ __forceinline__ void warp_merge_ms(float& m, float& s) {
  const float wm = warp_max(m);
  s = warp_sum(m == -INFINITY ? 0.0f : s * fast_exp2((m - wm) * kLog2e));
  m = wm;
}

// Block-wide reductions over CE_THREADS threads; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* scratch) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = (lane < (int)(blockDim.x >> 5)) ? scratch[lane] : -INFINITY;
  return warp_max(v);
}
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = (lane < (int)(blockDim.x >> 5)) ? scratch[lane] : 0.0f;
  return warp_sum(v);
}

template <class T>
__device__ __forceinline__ void load_vec(const T* p, float* x);
template <>
__device__ __forceinline__ void load_vec<float>(const float* p, float* x) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16>(const __nv_bfloat16* p, float* x) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load_vec<__half>(const __half* p, float* x) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
template <class T>
__device__ __forceinline__ void store_vec(T* p, const float* x);
template <>
__device__ __forceinline__ void store_vec<__half>(__half* p, const float* x) {
  uint4 v;
  __half2* h = reinterpret_cast<__half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = v;
}
template <>
__device__ __forceinline__ void store_vec<float>(float* p, const float* x) {
  *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16>(__nv_bfloat16* p, const float* x) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = v;
}

template <class T>
__global__ void __launch_bounds__(CE_THREADS, 2) ce_resident_kernel(const CeArgs a, int cs) {
  constexpr int VE = 16 / static_cast<int>(sizeof(T));
  constexpr int NV = CE_EPT / VE;
  __shared__ float2 scratch2[32];
  __shared__ float xch[2][2];
  __shared__ float bc[2];
  const uint32_t rank = cluster_ctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = nclusters_x();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t V = a.V;
  const int64_t sbeg = static_cast<int64_t>(rank) * CE_SLICE;
  int iter = 0;
  for (int64_t row = cid; row < a.N; row += ncl, ++iter) {
    T* rowp = static_cast<T*>(a.logits) + row * V;
    float x[CE_EPT];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t col = sbeg + static_cast<int64_t>(tid + k * CE_THREADS) * VE;
      if (col + VE <= V) {
        load_vec<T>(rowp + col, &x[k * VE]);
      } else {
#pragma unroll
        for (int i = 0; i < VE; ++i) x[k * VE + i] = (col + i < V) ? to_f32(rowp[col + i]) : -INFINITY;
      }
    }
    const int64_t t = a.target[row];
    const bool valid = target_valid(t, a.ignore_index, V);
    float zt = 0.0f;
    if (rank == 0 && tid == 0 && valid) zt = to_f32(rowp[t]);  // read before any CTA writes the row
    // One thread starts the copy engine fetching this CTA's slice of its
    // next row into L2, so that those loads find it there; the prefetch
    // holds no registers and no barrier waits for it.
    if (tid == 0 && row + ncl < a.N && sbeg < V) {
      const int64_t n = (V - sbeg < CE_SLICE ? V - sbeg : CE_SLICE) * static_cast<int64_t>(sizeof(T));
      bulk_prefetch_l2(rowp + static_cast<int64_t>(ncl) * V + sbeg, static_cast<uint32_t>(n));
    }
    // Per-thread max cm; x[i] is replaced by e_i = exp(x_i - cm), so that
    // the gradient needs one more exponential per thread, not one per
    // element: softmax_i = e_i * exp(cm - lse). A thread whose values are
    // all -inf (padding past V, or -inf logits) takes no shift: its e_i = 0.
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < CE_EPT; ++i) cm = fmaxf(cm, x[i]);
    const float cm2 = (cm == -INFINITY) ? 0.0f : cm * kLog2e;
    float csum = 0.0f;
#pragma unroll
    for (int i = 0; i < CE_EPT; ++i) {
      x[i] = fast_exp2(fmaf(x[i], kLog2e, -cm2));
      csum += x[i];
    }
    // warp pairs, then warp 0 merges the CTA's pairs for the cluster exchange
    float wm = cm, wsum = csum;
    warp_merge_ms(wm, wsum);
    if (lane == 0) scratch2[warp] = make_float2(wm, wsum);
    __syncthreads();
    if (warp == 0) {
      float2 pr = (lane < CE_THREADS / 32) ? scratch2[lane] : make_float2(-INFINITY, 0.0f);
      warp_merge_ms(pr.x, pr.y);
      if (lane == 0) {
        xch[iter & 1][0] = pr.x;
        xch[iter & 1][1] = pr.y;
      }
    }
    cluster_sync();
    if (warp == 0) {
      float pm = -INFINITY, ps = 0.0f;
      if (lane < cs) {
        pm = dsmem_ld_f32(&xch[iter & 1][0], lane);
        ps = dsmem_ld_f32(&xch[iter & 1][1], lane);
      }
      const float M = warp_max(pm);
      const float S = warp_sum((lane < cs && pm != -INFINITY) ? ps * expf(pm - M) : 0.0f);
      if (lane == 0) {
        bc[0] = M + logf(S);
        bc[1] = row_weight(a.rw, a.hdr, row, t, valid);
      }
    }
    __syncthreads();
    const float lse = bc[0], w = bc[1];
    // w * exp(cm - lse): 0 for all-padding threads (cm = -inf)
    const float ws = w * fast_exp2((cm - lse) * kLog2e);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t col = sbeg + static_cast<int64_t>(tid + k * CE_THREADS) * VE;
      float gv[VE];
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        const float e = x[k * VE + i];
        gv[i] = (valid && col + i == t) ? fmaf(e, ws, -w) : e * ws;
      }
      if (col + VE <= V) {
        store_vec<T>(rowp + col, gv);
      } else {
#pragma unroll
        for (int i = 0; i < VE; ++i)
          if (col + i < V) rowp[col + i] = from_f32<T>(gv[i]);
      }
    }
    if (rank == 0 && tid == 0) a.loss_rows[row] = valid ? class_w(a.rw, t, true) * (lse - zt) : 0.0f;
  }
  cluster_sync();  // no CTA leaves while a peer may still read its xch
}

template <class T>
__global__ void __launch_bounds__(CE_THREADS) ce_stream_kernel(const CeArgs a) {
  __shared__ float scratch[32];
  __shared__ float s_zt;
  const int tid = threadIdx.x;
  const int64_t V = a.V;
  for (int64_t row = blockIdx.x; row < a.N; row += gridDim.x) {
    T* rowp = static_cast<T*>(a.logits) + row * V;
    const int64_t t = a.target[row];
    const bool valid = target_valid(t, a.ignore_index, V);
    if (tid == 0) s_zt = valid ? to_f32(rowp[t]) : 0.0f;
    float m = -INFINITY, s = 0.0f;
    for (int64_t j = tid; j < V; j += CE_THREADS) {
      const float x = to_f32(rowp[j]);
      if (x > m) {
        s = s * fast_exp2((m - x) * kLog2e) + 1.0f;
        m = x;
      } else if (m != -INFINITY) {  // x = m = -inf adds exp(-inf) = 0, not exp(NaN)
        s += fast_exp2((x - m) * kLog2e);
      }
    }
    const float M = block_max(m, scratch);
    const float S = block_sum(m == -INFINITY ? 0.0f : s * fast_exp2((m - M) * kLog2e), scratch);
    const float lse = M + logf(S);
    const float w = row_weight(a.rw, a.hdr, row, t, valid);
    const float zt = s_zt;
    for (int64_t j = tid; j < V; j += CE_THREADS) {
      const float p = fast_exp2((to_f32(rowp[j]) - lse) * kLog2e);
      rowp[j] = from_f32<T>(w * ((valid && j == t) ? p - 1.0f : p));
    }
    if (tid == 0) a.loss_rows[row] = valid ? class_w(a.rw, t, true) * (lse - zt) : 0.0f;
    __syncthreads();  // s_zt is rewritten for the next row
  }
}

template <class T>
cudaError_t launch_ce_t(const CeArgs& a, cudaStream_t s) {
  const size_t esz = sizeof(T);
  const bool aligned = (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) && ((a.V * esz) % 16 == 0);
  // one 16384-element slice per CTA: a cluster of ceil(V / 16384) CTAs,
  // up to 16 (above 8 a non-portable cluster size, allowed per kernel; the
  // occupancy query below falls back to streaming when no cluster fits)
  const int64_t need = (a.V + CE_SLICE - 1) / CE_SLICE;
  int cs = need < 16 ? static_cast<int>(need) : 16;
  if (cs > 8) {
    cudaError_t e = cudaFuncSetAttribute(ce_resident_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      cudaGetLastError();
      cs = 0;  // stream the rows instead
    }
  }
  if (aligned && cs > 0 && static_cast<int64_t>(cs) * CE_SLICE >= a.V) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(CE_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(cs);
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, ce_resident_kernel<T>, &cfg) == cudaSuccess &&
        max_clusters > 0) {
      int64_t ncl = max_clusters;
      if (ncl > a.N) ncl = a.N;
      cfg.gridDim = dim3(static_cast<unsigned>(ncl * cs));
      prof_before(K_CE_RESIDENT, s, 2.0 * sizeof(T) * a.N * static_cast<double>(a.V));
      cudaError_t e = cudaLaunchKernelEx(&cfg, ce_resident_kernel<T>, a, cs);
      prof_after(K_CE_RESIDENT, s);
      return e;
    }
    cudaGetLastError();  // clear a failed occupancy query and stream the rows instead
  }
  int64_t grid = a.N < 4 * num_sms() ? a.N : 4 * num_sms();
  prof_before(K_CE_STREAM, s, 2.0 * sizeof(T) * a.N * static_cast<double>(a.V));
  ce_stream_kernel<T><<<static_cast<unsigned>(grid), CE_THREADS, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  prof_after(K_CE_STREAM, s);
  return e;
}

}  // namespace

cudaError_t launch_ce_logits(const CeArgs& a, int dt, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (dt == LCE_BF16) return launch_ce_t<__nv_bfloat16>(a, s);
  if (dt == LCE_F16) return launch_ce_t<__half>(a, s);
  return launch_ce_t<float>(a, s);
}

}  // namespace lce
