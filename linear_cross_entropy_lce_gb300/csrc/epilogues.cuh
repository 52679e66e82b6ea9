// epilogues.cuh -- per-row epilogues shared by the tcgen05 and the SIMT GEMMs.
//
// Both GEMMs hand each epilogue thread one output row of a tile segment of
// NCHUNK*32 columns starting at col0; load(c, v) fills v with the fp32
// accumulators of columns [col0 + 32c, col0 + 32c + 32) of that row. The
// loads must be called by every lane of a warp in the same order (the
// tcgen05 loads are warp-collective), so row validity only guards stores.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace lce {

// Output path of one epilogue warp. With tmap == NULL every thread stores
// its row directly. Otherwise bf16 results go out per 32-column chunk
// through a TMA store of the warp's 32 x 32 box: the warp stages the chunk
// in a 2 KB buffer (32 rows x 64 B, 64-byte swizzle, so the 16-byte writes
// of the 32 lanes hit distinct banks) and lane 0 issues the store; two
// buffers alternate, and a buffer is rewritten only after the store issued
// from it two chunks earlier has finished reading it. Calls are
// warp-collective; rows and columns outside the tensor are not written.
struct EpiIO {
  const CUtensorMap* tmap;
  uint8_t* stage;    // 2 x 2048 B, 1024-byte aligned
  int64_t row_base;  // first output row of this warp
  int lane;
  int nst;           // stores issued so far (buffer parity)
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void stage_store_bf16(EpiIO& io, const float (&v)[32], int64_t col) {
  uint8_t* buf = io.stage + (io.nst & 1) * 2048;
  if (io.lane == 0) bulk_wait_read_le1();
  __syncwarp();
  const uint32_t row_addr = smem_u32(buf) + io.lane * 64;
  const int sw = (io.lane >> 1) & 3;  // 64-byte swizzle: 16-byte chunk index ^= (row / 2) % 4
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    st_shared_v4(row_addr + ((q ^ sw) << 4), u);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (io.lane == 0) {
    tma_store_2d(io.tmap, buf, static_cast<int32_t>(col), static_cast<int32_t>(io.row_base));
    bulk_commit_group();
  }
  ++io.nst;
}

// ---------------------------------------------------------------------------
// Logits epilogue of the forward GEMM (z = X W^T + b).
//
// For its row and segment the thread computes m = max_j z_j and
// s = sum_j exp(z_j - m) over the segment's columns j < C (padding columns
// are excluded), keeps z at the target column, and, when a buffer is given,
// stores P~_j = exp(z_j - m) in the buffer's type (0 in padding columns).
// The per-(row, segment) pair (m, s) is merged into the row's log-sum-exp
// later; P~ times exp(m - lse) is softmax(z)_j. This replaces the page's
// per-chunk amax / sub_ / exp_ / sum passes over the [chunk, C] logits
// (linear_cross_entropy.py, the chunked loop body) with one pass over each
// tile while it is still on chip.
// ---------------------------------------------------------------------------
struct EpiLse {
  struct Params {
    const void* bias;        // [C] (bf16 or fp32, see bias_bf16) or NULL
    int bias_bf16;
    const int64_t* target;   // chunk-local: target[row]
    int64_t C;
    int rows;                // valid rows in this chunk
    float2* partial;         // [nseg][partial_ld] (m, s)
    int64_t partial_ld;
    float* zt;               // [rows] logit at the target column
    void* ptilde;            // [rows][ld_p] or NULL (forward only)
    int64_t ld_p;
    int ptilde_bf16;
  };

  __device__ static __forceinline__ float bias_at(const Params& p, int64_t col) {
    if (p.bias == nullptr || col >= p.C) return 0.0f;
    return p.bias_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.bias)[col])
                       : static_cast<const float*>(p.bias)[col];
  }

  template <int NCHUNK, class Loader>
  __device__ static __forceinline__ void run(const Params& p, int64_t row, int64_t col0, int64_t seg,
                                             Loader&& load, EpiIO& io) {
    const bool row_ok = row < p.rows;
    const int64_t t = row_ok ? p.target[row] : -1;
    const int tl = (t >= col0 && t < col0 + NCHUNK * 32 && t < p.C) ? static_cast<int>(t - col0) : -1;
    float v[32];
    // pass 1: segment max
    float m = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < NCHUNK; ++c) {
      load(c, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int64_t col = col0 + 32 * c + i;
        const float z = v[i] + bias_at(p, col);
        m = (col < p.C) ? fmaxf(m, z) : m;
      }
    }
    // pass 2: sum of exp(z - m), target logit, optional P~ store
    float s = 0.0f, ztv = 0.0f;
#pragma unroll 1
    for (int c = 0; c < NCHUNK; ++c) {
      load(c, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int64_t col = col0 + 32 * c + i;
        const float z = v[i] + bias_at(p, col);
        const float e = (col < p.C) ? fast_exp2((z - m) * kLog2e) : 0.0f;
        ztv = (32 * c + i == tl) ? z : ztv;
        s += e;
        v[i] = e;
      }
      if (p.ptilde != nullptr && io.tmap != nullptr) {
        stage_store_bf16(io, v, col0 + 32 * c);
      } else if (p.ptilde != nullptr && row_ok) {
        const int64_t off = row * p.ld_p + col0 + 32 * c;
        if (p.ptilde_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.ptilde) + off);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
            u.x = *reinterpret_cast<uint32_t*>(&h0);
            u.y = *reinterpret_cast<uint32_t*>(&h1);
            u.z = *reinterpret_cast<uint32_t*>(&h2);
            u.w = *reinterpret_cast<uint32_t*>(&h3);
            dst[q] = u;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.ptilde) + off);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    }
    if (row_ok && col0 < p.C) {
      p.partial[seg * p.partial_ld + row] = make_float2(m, s);
      if (tl >= 0) p.zt[row] = ztv;
    }
  }
};

// ---------------------------------------------------------------------------
// Store epilogue for the dX = G W and dW = G^T X contractions (and the GEMM
// tests). mode 0: out = acc; 1: acc32 = acc (first chunk of a dW
// accumulated over chunks); 2: acc32 += acc; 3: out = acc32 + acc (last
// chunk); 4: out += acc with fp32 atomics (one split of a split-K GEMM
// into a zeroed fp32 out). out is bf16 or fp32; acc32 is fp32 with the
// same leading dimension as out.
// ---------------------------------------------------------------------------
struct EpiStore {
  struct Params {
    void* out;
    int out_bf16;
    int64_t ldo;
    float* acc32;
    int mode;
    int64_t rows, cols;  // valid output region
    int vec_ok;          // rows of out / acc32 are 16-byte aligned
  };

  __device__ static __forceinline__ void put(const Params& p, int64_t idx, float x) {
    if (p.mode == 4) {  // split-K partial: add into the zeroed fp32 output
      atomicAdd(static_cast<float*>(p.out) + idx, x);
      return;
    }
    if (p.mode == 1) {
      p.acc32[idx] = x;
      return;
    }
    if (p.mode == 2) {
      p.acc32[idx] += x;
      return;
    }
    if (p.mode == 3) x += p.acc32[idx];
    if (p.out_bf16)
      static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(x);
    else
      static_cast<float*>(p.out)[idx] = x;
  }

  template <int NCHUNK, class Loader>
  __device__ static __forceinline__ void run(const Params& p, int64_t row, int64_t col0, int64_t /*seg*/,
                                             Loader&& load, EpiIO& io) {
    const bool row_ok = row < p.rows;
    float v[32];
#pragma unroll 1
    for (int c = 0; c < NCHUNK; ++c) {
      load(c, v);
      if (io.tmap != nullptr) {  // bf16, mode 0 (the host only sets tmap then)
        stage_store_bf16(io, v, col0 + 32 * c);
        continue;
      }
      if (!row_ok) continue;
      const int64_t cb = col0 + 32 * c;
      const int64_t base = row * p.ldo + cb;
      if (p.vec_ok && cb + 32 <= p.cols && p.mode != 4) {
        if (p.mode == 0 && p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + base);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
            u.x = *reinterpret_cast<uint32_t*>(&h0);
            u.y = *reinterpret_cast<uint32_t*>(&h1);
            u.z = *reinterpret_cast<uint32_t*>(&h2);
            u.w = *reinterpret_cast<uint32_t*>(&h3);
            dst[q] = u;
          }
          continue;
        }
        if (p.mode == 0 || p.mode == 1) {
          float* o = (p.mode == 1) ? p.acc32 : static_cast<float*>(p.out);
          float4* dst = reinterpret_cast<float4*>(o + base);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          continue;
        }
        if (p.mode == 2 || (p.mode == 3 && !p.out_bf16)) {
          float4* a = reinterpret_cast<float4*>(p.acc32 + base);
          float4* o = reinterpret_cast<float4*>((p.mode == 2 ? p.acc32 : static_cast<float*>(p.out)) + base);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 x = a[q];
            o[q] = make_float4(x.x + v[4 * q], x.y + v[4 * q + 1], x.z + v[4 * q + 2], x.w + v[4 * q + 3]);
          }
          continue;
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (cb + i < p.cols) put(p, base + i, v[i]);
      }
    }
  }
};

}  // namespace lce
