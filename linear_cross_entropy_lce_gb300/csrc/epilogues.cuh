// epilogues.cuh -- per-row epilogues shared by the tcgen05 and the SIMT GEMMs.
//
// Both GEMMs hand each epilogue thread one output row of a tile segment of
// NCHUNK*32 columns starting at col0, read in groups of GW chunks:
// load(g, v) fills v[GW*32] with the fp32 accumulators of columns
// [col0 + 32 GW g, col0 + 32 GW (g + 1)) of that row. The loads must be
// called by every lane of a warp in the same order (the tcgen05 loads are
// warp-collective), so row validity only guards stores.
// Element types are the lce_dtype_e codes: 0 fp32, 1 bf16, 2 fp16.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace lce {

__device__ __forceinline__ float load_elem(const void* p, int64_t i, int dt) {
  if (dt == LCE_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  if (dt == LCE_F16) return __half2float(static_cast<const __half*>(p)[i]);
  return static_cast<const float*>(p)[i];
}
__device__ __forceinline__ void store_elem(void* p, int64_t i, float x, int dt) {
  if (dt == LCE_BF16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else if (dt == LCE_F16)
    static_cast<__half*>(p)[i] = __float2half_rn(x);
  else
    static_cast<float*>(p)[i] = x;
}
// Two floats as one 32-bit word of two 16-bit values (bf16 or fp16).
__device__ __forceinline__ uint32_t pack2(float a, float b, int dt) {
  if (dt == LCE_F16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// 32 floats -> 64 bytes of 16-bit values at dst (16-byte aligned).
__device__ __forceinline__ void store32_16bit(void* dst, const float (&v)[32], int dt) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack2(v[8 * q + 0], v[8 * q + 1], dt);
    u.y = pack2(v[8 * q + 2], v[8 * q + 3], dt);
    u.z = pack2(v[8 * q + 4], v[8 * q + 5], dt);
    u.w = pack2(v[8 * q + 6], v[8 * q + 7], dt);
    d[q] = u;
  }
}
// 32 floats -> 128 bytes of fp32 at dst (16-byte aligned).
__device__ __forceinline__ void store32_f32(float* dst, const float (&v)[32]) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Output path of one epilogue warp. With tmap == NULL every thread stores
// its row directly. Otherwise 16-bit results go out per 32-column chunk
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
  float* bias_s;     // NULL, or this warp's shared buffer for one segment of bias (NCHUNK * 32 floats)
};

__device__ __forceinline__ void stage_store_16bit(EpiIO& io, const float (&v)[32], int64_t col, int dt) {
  uint8_t* buf = io.stage + (io.nst & 1) * 2048;
  if (io.lane == 0) bulk_wait_read_le1();
  __syncwarp();
  const uint32_t row_addr = smem_u32(buf) + io.lane * 64;
  const int sw = (io.lane >> 1) & 3;  // 64-byte swizzle: 16-byte chunk index ^= (row / 2) % 4
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack2(v[8 * q + 0], v[8 * q + 1], dt);
    u.y = pack2(v[8 * q + 2], v[8 * q + 3], dt);
    u.z = pack2(v[8 * q + 4], v[8 * q + 5], dt);
    u.w = pack2(v[8 * q + 6], v[8 * q + 7], dt);
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
    const void* bias;        // [C] of bias_dt, or NULL
    int bias_dt;
    const int64_t* target;   // chunk-local: target[row]
    int64_t C;
    int rows;                // valid rows in this chunk
    float2* partial;         // [nseg][partial_ld] (m, s)
    int64_t partial_ld;
    float* zt;               // [rows] logit at the target column
    void* ptilde;            // [rows][ld_p] of ptilde_dt, or NULL (forward only)
    int64_t ld_p;
    int ptilde_dt;
    int64_t store_cols;      // P~ is stored for columns < store_cols only (a multiple of the tile width)
  };

  __device__ static __forceinline__ float bias_at(const Params& p, int64_t col) {
    if (p.bias == nullptr || col >= p.C) return 0.0f;
    return load_elem(p.bias, col, p.bias_dt);
  }

  // NCHUNK 32-column chunks, read GW chunks at a time: load(g, v) fills
  // v[GW * 32] with columns [col0 + 32 GW g, col0 + 32 GW (g + 1)).
  template <int NCHUNK, int GW, class Loader>
  __device__ static __forceinline__ void run(const Params& p, int64_t row, int64_t col0, int64_t seg,
                                             Loader&& load, EpiIO& io) {
    static_assert(NCHUNK % GW == 0, "chunk groups");
    constexpr int NG = NCHUNK / GW;
    constexpr int W = GW * 32;
    const bool row_ok = row < p.rows;
    const int64_t t = row_ok ? p.target[row] : -1;
    const int tl = (t >= col0 && t < col0 + NCHUNK * 32 && t < p.C) ? static_cast<int>(t - col0) : -1;
    const bool full = col0 + NCHUNK * 32 <= p.C;  // no padding column in the segment
    // the segment's bias, staged once per tile by the warp in shared memory
    float* bs = (p.bias != nullptr && full) ? io.bias_s : nullptr;
    if (bs != nullptr) {
      __syncwarp();  // the previous tile's reads are done
#pragma unroll
      for (int k = 0; k < NCHUNK; ++k) bs[io.lane + 32 * k] = load_elem(p.bias, col0 + io.lane + 32 * k, p.bias_dt);
      __syncwarp();
    }
    // no per-column tests: no bias, or a full segment with its bias staged
    const bool plain = full && (p.bias == nullptr || bs != nullptr);
    float v[W];
    // pass 1: segment max
    float m = -INFINITY;
#pragma unroll 1
    for (int g = 0; g < NG; ++g) {
      load(g, v);
      if (plain) {
        if (bs != nullptr) {
#pragma unroll
          for (int i = 0; i < W; ++i) v[i] += bs[W * g + i];
        }
#pragma unroll
        for (int i = 0; i < W; ++i) m = fmaxf(m, v[i]);
      } else {
#pragma unroll
        for (int i = 0; i < W; ++i) {
          const int64_t col = col0 + W * g + i;
          const float z = v[i] + bias_at(p, col);
          m = (col < p.C) ? fmaxf(m, z) : m;
        }
      }
    }
    // pass 2: sum of exp(z - m), target logit, optional P~ store (for the
    // first store_cols columns; the others are recomputed later). A segment
    // whose logits are all -inf (a bias of -inf masks classes) is shifted
    // by 0, so that it stores P~ = exp(-inf) = 0 and sums to 0, not NaN.
    if (m == -INFINITY) m = 0.0f;
    float s = 0.0f, ztv = 0.0f;
#pragma unroll 1
    for (int g = 0; g < NG; ++g) {
      load(g, v);
      if (bs != nullptr) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] += bs[W * g + i];
      } else if (!plain) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] += bias_at(p, col0 + W * g + i);
      }
      if (tl >= W * g && tl < W * (g + 1)) {  // at most one group of one segment per row
#pragma unroll
        for (int i = 0; i < W; ++i) ztv = (W * g + i == tl) ? v[i] : ztv;
      }
      if (plain) {
#pragma unroll
        for (int i = 0; i < W; ++i) {
          v[i] = fast_exp2((v[i] - m) * kLog2e);
          s += v[i];
        }
      } else {
#pragma unroll
        for (int i = 0; i < W; ++i) {
          v[i] = (col0 + W * g + i < p.C) ? fast_exp2((v[i] - m) * kLog2e) : 0.0f;
          s += v[i];
        }
      }
      if (p.ptilde == nullptr || col0 >= p.store_cols) continue;
#pragma unroll
      for (int c = 0; c < GW; ++c) {
        float(&vc)[32] = *reinterpret_cast<float(*)[32]>(&v[32 * c]);
        const int64_t cc = col0 + W * g + 32 * c;
        if (io.tmap != nullptr) {
          stage_store_16bit(io, vc, cc, p.ptilde_dt);
        } else if (row_ok) {
          const int64_t off = row * p.ld_p + cc;
          if (p.ptilde_dt == LCE_F32)
            store32_f32(static_cast<float*>(p.ptilde) + off, vc);
          else
            store32_16bit(static_cast<uint16_t*>(p.ptilde) + off, vc, p.ptilde_dt);
        }
      }
    }
    if (row_ok && col0 < p.C) {
      p.partial[seg * p.partial_ld + row] = make_float2(s == 0.0f ? -INFINITY : m, s);
      if (tl >= 0) p.zt[row] = ztv;
    }
  }
};

// Column sums of a warp's 32 rows: on entry x[i] is this lane's (row's)
// value in column i < 32; on return lane L holds the sum over the 32 lanes
// of column L. A transposing butterfly: at each step a lane keeps one half
// of its columns, sends the other half to the lane `s` away and adds what it
// receives, so 31 shuffles cover 32 columns. x is clobbered.
__device__ __forceinline__ float warp_column_sum32(float (&x)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? x[i] : x[i + s];
      const float keep = up ? x[i + s] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return x[0];
}

// ---------------------------------------------------------------------------
// Gradient epilogue of the recomputing GEMM: z = X W_v^T + b_v over one
// chunk v of the classes, for rows whose log-sum-exp is already known.
//
// For its row the thread forms G[r, j] = wg_r (exp(z_j - lse_r) - [j == t_r])
// over the chunk's classes j < cols (the target column from expm1, so that
// softmax_t ~ 1 does not cancel; 0 in padding columns and on rows past the
// chunk) and stores it in the buffer's type, through the output tensor map
// when one is given. With db_acc it also adds the column sums of
// wdb_r * G[r, j] into db_acc (global class col_base + j): each warp's 32
// rows are summed per column with warp_column_sum32, then one lane per
// column adds the sum. This is the second sweep of the page's chunked
// backward (linear_cross_entropy.py: logits recomputed per chunk, scaled by
// the row weight after the max shift, minus the one-hot), done on the tile
// while it is in tensor memory.
// ---------------------------------------------------------------------------
struct EpiGrad {
  struct Params {
    const void* bias;   // [cols] of bias_dt (this chunk's slice), or NULL
    int bias_dt;
    const int* tcol;    // [rows] target class (global index) of a valid row, else -1
    int64_t col_base;   // global class of the chunk's column 0
    int64_t cols;       // classes in the chunk
    int rows;           // rows in the batch chunk
    const float* lse;   // [rows]
    const float* wg;    // [rows] row weight folded into G
    const float* wdb;   // [rows] weight of a row's G in the column sums, or NULL (1)
    float* db_acc;      // [C] fp32, or NULL
    void* g;            // [rows][ld_g] of g_dt: direct stores when no tensor map is given
    int64_t ld_g;
    int g_dt;
  };

  template <int NCHUNK, int GW, class Loader>
  __device__ static __forceinline__ void run(const Params& p, int64_t row, int64_t col0, int64_t /*seg*/,
                                             Loader&& load, EpiIO& io) {
    static_assert(NCHUNK % GW == 0, "chunk groups");
    constexpr int NG = NCHUNK / GW;
    constexpr int W = GW * 32;
    const bool row_ok = row < p.rows;
    const float lse = row_ok ? p.lse[row] : 0.0f;
    const float wg = row_ok ? p.wg[row] : 0.0f;
    const float wdb = (row_ok && p.wdb != nullptr) ? p.wdb[row] : 1.0f;
    const int64_t t = row_ok ? p.tcol[row] : -1;
    const int64_t tloc = t - p.col_base - col0;
    const int tl = (t >= 0 && tloc >= 0 && tloc < NCHUNK * 32) ? static_cast<int>(tloc) : -1;
    const bool full = col0 + NCHUNK * 32 <= p.cols;
    float* bs = (p.bias != nullptr && full) ? io.bias_s : nullptr;
    if (bs != nullptr) {
      __syncwarp();  // the previous tile's reads are done
#pragma unroll
      for (int k = 0; k < NCHUNK; ++k) bs[io.lane + 32 * k] = load_elem(p.bias, col0 + io.lane + 32 * k, p.bias_dt);
      __syncwarp();
    }
    float v[W];
#pragma unroll 1
    for (int g = 0; g < NG; ++g) {
      load(g, v);
      if (bs != nullptr) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] += bs[W * g + i];
      } else if (p.bias != nullptr) {
#pragma unroll
        for (int i = 0; i < W; ++i) {
          const int64_t col = col0 + W * g + i;
          v[i] += col < p.cols ? load_elem(p.bias, col, p.bias_dt) : 0.0f;
        }
      }
      // the target column: wg (softmax_t - 1) from expm1, once per row
      const bool t_here = tl >= W * g && tl < W * (g + 1);
      float xt = 0.0f;
      if (t_here) {
#pragma unroll
        for (int i = 0; i < W; ++i) xt = (W * g + i == tl) ? v[i] : xt;
      }
      const float et = t_here ? wg * expm1f(xt - lse) : 0.0f;
      if (full && row_ok) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = wg * fast_exp2((v[i] - lse) * kLog2e);
      } else {
#pragma unroll
        for (int i = 0; i < W; ++i) {
          const float e = wg * fast_exp2((v[i] - lse) * kLog2e);
          v[i] = (row_ok && col0 + W * g + i < p.cols) ? e : 0.0f;
        }
      }
      if (t_here) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = (W * g + i == tl) ? et : v[i];
      }
#pragma unroll
      for (int c = 0; c < GW; ++c) {
        float(&vc)[32] = *reinterpret_cast<float(*)[32]>(&v[32 * c]);
        const int64_t cc = col0 + W * g + 32 * c;
        if (io.tmap != nullptr) {
          stage_store_16bit(io, vc, cc, p.g_dt);
        } else if (row_ok) {
          const int64_t off = row * p.ld_g + cc;
          if (p.g_dt == LCE_F32)
            store32_f32(static_cast<float*>(p.g) + off, vc);
          else
            store32_16bit(static_cast<uint16_t*>(p.g) + off, vc, p.g_dt);
        }
        if (p.db_acc != nullptr && cc < p.cols) {
          // column sums of the fp32 values (before the 16-bit rounding of the store)
          if (p.wdb != nullptr) {
#pragma unroll
            for (int i = 0; i < 32; ++i) vc[i] *= wdb;
          }
          const float sum = warp_column_sum32(vc, io.lane);
          if (cc + io.lane < p.cols) atomicAdd(p.db_acc + p.col_base + cc + io.lane, sum);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Store epilogue for the dX = G W and dW = G^T X contractions (and the GEMM
// tests). mode 0: out = acc; 1: acc32 = acc (first part of a gradient
// accumulated over batch chunks (dW) or class chunks (dX)); 2: acc32 += acc;
// 3: out = acc32 + acc (last part; like mode 0 it may store through the
// output tensor map); 4: out += acc with fp32 atomics (one split of a split-K GEMM
// into a zeroed fp32 out). out is fp32, bf16 or fp16 (out_dt); acc32 is
// fp32 with the same leading dimension as out. Before any of this the
// accumulator may be scaled per row (row_scale[row]) and by one device
// scalar (scalar_scale[0]): the fp16 backward stores G without the row
// weights, so dX takes them per row and dW as one scalar.
// ---------------------------------------------------------------------------
struct EpiStore {
  struct Params {
    void* out;
    int out_dt;
    int64_t ldo;
    float* acc32;
    int mode;
    int64_t rows, cols;         // valid output region
    int vec_ok;                 // rows of out / acc32 are 16-byte aligned
    const float* row_scale;     // [rows] or NULL
    const float* scalar_scale;  // device scalar or NULL
  };

  // mode: p.mode, except that mode 3 arrives here as 0 (its accumulator is
  // already added)
  __device__ static __forceinline__ void put(const Params& p, int mode, int64_t idx, float x) {
    if (mode == 4) {  // split-K partial: add into the zeroed fp32 output
      atomicAdd(static_cast<float*>(p.out) + idx, x);
      return;
    }
    if (mode == 1) {
      p.acc32[idx] = x;
      return;
    }
    if (mode == 2) {
      p.acc32[idx] += x;
      return;
    }
    store_elem(p.out, idx, x, p.out_dt);
  }

  template <int NCHUNK, int GW, class Loader>
  __device__ static __forceinline__ void run(const Params& p, int64_t row, int64_t col0, int64_t /*seg*/,
                                             Loader&& load, EpiIO& io) {
    static_assert(NCHUNK % GW == 0, "chunk groups");
    constexpr int W = GW * 32;
    const bool row_ok = row < p.rows;
    float scale = 1.0f;
    if (p.row_scale != nullptr) scale = row_ok ? p.row_scale[row] : 0.0f;
    if (p.scalar_scale != nullptr) scale *= p.scalar_scale[0];
    const bool scaled = p.row_scale != nullptr || p.scalar_scale != nullptr;
    float vg[W];
#pragma unroll 1
    for (int g = 0; g < NCHUNK / GW; ++g) {
      load(g, vg);
      if (scaled) {
#pragma unroll
        for (int i = 0; i < W; ++i) vg[i] *= scale;
      }
#pragma unroll
      for (int c = 0; c < GW; ++c) {
        float(&v)[32] = *reinterpret_cast<float(*)[32]>(&vg[32 * c]);
        const int64_t cb = col0 + W * g + 32 * c;
        const int64_t base = row * p.ldo + cb;
        const bool vec = p.vec_ok && cb + 32 <= p.cols;
        if (p.mode == 3 && row_ok) {  // last part of an accumulation: add the fp32 sum so far
          if (vec) {
            const float4* a = reinterpret_cast<const float4*>(p.acc32 + base);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 x = a[q];
              v[4 * q] += x.x;
              v[4 * q + 1] += x.y;
              v[4 * q + 2] += x.z;
              v[4 * q + 3] += x.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i < p.cols) v[i] += p.acc32[base + i];
          }
        }
        const int mode = p.mode == 3 ? 0 : p.mode;
        if (io.tmap != nullptr) {  // 16-bit, mode 0 or 3 (the host only sets tmap then)
          stage_store_16bit(io, v, cb, p.out_dt);
          continue;
        }
        if (!row_ok) continue;
        if (vec && mode == 4) {  // split-K partial: 8 vector reductions
          float* o = static_cast<float*>(p.out) + base;
#pragma unroll
          for (int q = 0; q < 8; ++q) red_add_v4(o + 4 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          continue;
        }
        if (vec) {
          if (mode == 0 && p.out_dt != LCE_F32) {
            store32_16bit(static_cast<uint16_t*>(p.out) + base, v, p.out_dt);
            continue;
          }
          if (mode == 0 || mode == 1) {
            store32_f32((mode == 1 ? p.acc32 : static_cast<float*>(p.out)) + base, v);
            continue;
          }
          if (mode == 2) {
            float4* a = reinterpret_cast<float4*>(p.acc32 + base);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 x = a[q];
              a[q] = make_float4(x.x + v[4 * q], x.y + v[4 * q + 1], x.z + v[4 * q + 2], x.w + v[4 * q + 3]);
            }
            continue;
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (cb + i < p.cols) put(p, mode, base + i, v[i]);
        }
      }
    }
  }
};

}  // namespace lce
