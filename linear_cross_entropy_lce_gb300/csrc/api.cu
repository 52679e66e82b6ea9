// api.cu -- the C ABI of liblce.so: argument checks, workspace plan, and the
// launch sequence of the fused linear + cross-entropy loss.
//
// Launch sequence of lce_forward_backward for one call (all on `stream`):
//   prep            valid-target count n_valid, target-range check, the
//                   mean's denominator
//   per batch chunk of Bc rows (all rows unless the gradient buffer cannot
//   hold D classes of them):
//     logits GEMM   z = X_c W^T (+ b) with the per-segment (max, sum-exp)
//                   epilogue; stores P~ = exp(z - m_seg) in the gradient
//                   buffer for the classes [0, Cs) it holds
//     combine       row lse, loss_n, scales w_n exp(m_seg - lse) of the
//                   stored classes, G at target, the row's lse and weight
//     grad          P~ -> G in place for the stored classes (+ bias-gradient
//                   column sums)
//     dX GEMM       dX_c (+)= G W over the stored classes
//     dW GEMM       dW[0:Cs] (+)= G^T X_c
//     per recomputed chunk of up to Cb classes [c0, c0 + cw):
//       recompute   z again for those classes, G formed in the epilogue
//                   (EpiGrad) into the buffer, bias-gradient column sums
//       dX GEMM     dX_c += G W[c0 : c0 + cw] (fp32 accumulator, the last
//                   part stored in grad_dtype)
//       dW GEMM     dW[c0 : c0 + cw] (+)= G^T X_c
//   loss finalize, bias-gradient finalize
// lce_backward (given lse) skips the logits sweep and the merge: every class
// is a recomputed chunk. On the bf16 / fp16 CTA-pair path with >= 1024
// chunk rows the logits GEMM runs over up to 4 row slabs of growing size,
// and combine + grad of slab k run in the idle warps of the GEMM that
// follows it (slab k+1's logits GEMM, or the dX GEMM for the last slab,
// whose producer waits for those rows), so no combine or grad kernel is
// launched. fp32 inputs add the TF32 hi / lo splits of W and X_c before the
// GEMMs that read them, and form G together with its split (3xTF32 engine).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/lce.h"
#include "../../include/lce_testing.h"
#include "internal.h"

namespace lce {

// ------------------------------------------------------------ device facts
namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
int g_cc_ok[kMaxDevices] = {0};  // 0 unknown, 1 ok, -1 not sm_103

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}
}  // namespace

int num_sms() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 148;
  if (g_sms[d] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 148;
  }
  return g_sms[d];
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& kd : done)
    if (kd.first == kernel && kd.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}

static int check_device() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return LCE_ERR_CUDA;
  if (g_cc_ok[d] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
      return LCE_ERR_CUDA;
    g_cc_ok[d] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_cc_ok[d] == 1 ? LCE_OK : LCE_ERR_DEVICE;
}

// ------------------------------------------------------------ profiler
namespace {
struct ProfRec {
  int id;
  cudaEvent_t a, b;
  double work;
};
std::vector<ProfRec> g_recs;
bool g_prof = false;
std::atomic<int64_t> g_launches{0};
const char* kNames[K_NUM_IDS] = {
    "prep",          "gemm_logits_tc", "gemm_dx_tc",  "gemm_dw_tc",      "gemm_logits_simt",
    "gemm_dx_simt",  "gemm_dw_simt",   "lse_combine", "grad_logits",     "loss_finalize",
    "db_finalize",   "ce_resident",    "ce_stream",   "gemm_test",       "row_scale",
    "gemm_logits_3xtf32", "gemm_dx_3xtf32", "gemm_dw_3xtf32", "split_tf32", "scale_grads",
    "gemm_recompute_tc", "backward_rows", "grad_split_tf32"};
}  // namespace

const char* kernel_id_name(int id) { return (id >= 0 && id < K_NUM_IDS) ? kNames[id] : "?"; }

void prof_before(int id, cudaStream_t s, double work) {
  g_launches.fetch_add(1);
  if (!g_prof) return;
  ProfRec r{id, nullptr, nullptr, work};
  cudaEventCreate(&r.a);
  cudaEventCreate(&r.b);
  cudaEventRecord(r.a, s);
  g_recs.push_back(r);
}
void prof_after(int id, cudaStream_t s) {
  if (!g_prof || g_recs.empty() || g_recs.back().id != id) return;
  cudaEventRecord(g_recs.back().b, s);
}

// ------------------------------------------------------------ workspace plan
namespace {

constexpr size_t kAlign = 256;
// Budget of the default plan for the backward's gradient buffer ([rows,
// classes] of the input type): 1 GiB. The forward-only plan applies it to
// its (max, sum-exp) pairs.
constexpr int64_t kDefaultBufferBytes = int64_t(1) << 30;

inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int esize(int dt) { return dt == LCE_F32 ? 4 : 2; }
// Counters per batch chunk, zeroed at the start of every call. Work counters
// of the idle-warp side jobs: (claimed, done) for the merge of slabs 0..3 at
// [2k, 2k + 1], for the last slab's G formation in the dX GEMM at [8, 9].
// Tile-schedule counters of the CTA-pair GEMMs (one per launch): logits slab
// k at kSched + k, dX and dW of the stored classes at kSched + 4 and + 5,
// and for recomputed chunk v the recompute, dX and dW at kSched + 6 + 3v,
// + 7 + 3v and + 8 + 3v.
constexpr int kSideCounters = 16;
constexpr int kSched = kSideCounters;
inline int64_t counters_per_chunk(int64_t nvc) { return kSched + 6 + 3 * nvc; }

struct Plan {
  bool tc;          // tensor-core (bf16 / fp16) path
  bool tf32;        // fp32 inputs on the tensor cores (3xTF32)
  bool backward;    // a gradient call
  bool given_lse;   // gradients from a given row lse (tensor-core path): no forward sweep
  int segw;         // columns per (max, sum-exp) segment
  int nseg;
  int64_t C_pad;    // classes padded to the tile width
  int64_t Bc;       // rows per batch chunk
  int64_t nchunks;
  // Classes of the backward. The gradient buffer has Cb columns. The forward
  // sweep stores P~ for classes [0, Cs) in it; classes [Cs, C) are
  // recomputed afterwards in nvc chunks of up to Cb classes, each formed
  // into the same buffer (tensor-core path only). Without recomputation
  // Cs = Cb = C_pad and nvc = 0; with a given lse, Cs = 0.
  int64_t Cb, Cs, nvc;
  bool dw_acc;      // fp32 dW accumulator in the workspace (bf16 / fp16 dW over several batch chunks)
  bool dx_acc;      // fp32 dX accumulator (16-bit dX over several class chunks)
  size_t off_cnt, off_loss, off_zt, off_tcol, off_gt, off_partial, off_L, off_dw, off_db, total;
  // fp16 backward: per-row weights [Bc], their max |w| (one float), and the
  // rows of X scaled by w / max|w| for dW ([Bc, D] fp16)
  size_t off_wrow, off_wbar, off_xs;
  // recomputed classes: the rows' lse and G weight [Bc], the fp32 dX
  // accumulator [Bc, D]
  size_t off_lse, off_wv, off_dx;
  // 3xTF32: TF32 hi / lo parts of W [C, ldD] and of the chunk's X [Bc, ldD]
  // (each read K-major by the logits, MN-major by dX / dW), and the lo part
  // of G [Bc, C_pad] (its hi part replaces G in the chunk buffer)
  int64_t ldD;
  size_t off_wh, off_wl, off_xh, off_xl, off_gl;
};

inline bool is_backward_op(int op) { return op == LCE_OP_FORWARD_BACKWARD || op == LCE_OP_BACKWARD; }

// Fewest classes a recomputed chunk of the tensor-core path takes: D
// rounded up to the tile width (so the fp32 dX accumulator's traffic per
// chunk, 8 bytes per row and feature, stays below the chunk's own G
// traffic), at least one tile, at most all classes.
int64_t min_class_chunk(int64_t D, int64_t C_pad) {
  const int64_t c = std::max<int64_t>(256, ceil_div(D, 256) * 256);
  return std::min(c, C_pad);
}

// The plan for batch chunks of Bc rows and a gradient buffer of Cb columns
// (rounded down to the tile width and clamped to [256, C_pad] on the
// tensor-core backward; C_pad elsewhere).
void make_plan(int op, int64_t N, int64_t D, int64_t C, int dtype, int grad_dtype, bool want_dx, bool want_dw,
               bool want_db, int64_t Bc, int64_t Cb, Plan* p) {
  const bool backward = is_backward_op(op);
  p->backward = backward;
  p->tc = dtype != LCE_F32;
  p->tf32 = dtype == LCE_F32 && f32_tensor_default();
  // fp32 inputs have no recomputing GEMM: a given lse is not used there and
  // the call runs its own forward sweep
  p->given_lse = op == LCE_OP_BACKWARD && p->tc;
  p->segw = (p->tc || p->tf32) ? 256 : 64;
  p->nseg = static_cast<int>(ceil_div(C, p->segw));
  p->C_pad = (p->tc || p->tf32) ? ceil_div(C, 256) * 256 : ceil_div(C, 128) * 128;
  if (N == 0) Bc = 0;
  p->Bc = Bc;
  p->nchunks = Bc > 0 ? ceil_div(N, Bc) : 0;
  const bool vocab = backward && p->tc;
  if (vocab) {
    Cb = Cb / 256 * 256;
    Cb = std::max<int64_t>(256, std::min(Cb, p->C_pad));
  } else {
    Cb = p->C_pad;
  }
  p->Cb = Cb;
  p->Cs = p->given_lse ? 0 : Cb;
  p->nvc = (vocab && C > p->Cs) ? ceil_div(C - p->Cs, Cb) : 0;
  const int64_t dx_parts = (p->Cs > 0 ? 1 : 0) + p->nvc;
  p->dw_acc = backward && want_dw && p->nchunks > 1 && grad_dtype != LCE_F32;
  p->dx_acc = backward && want_dx && dx_parts > 1 && grad_dtype != LCE_F32;
  const bool recompute = p->nvc > 0;
  const bool sweep = !p->given_lse;  // forward sweep with (max, sum-exp) pairs
  size_t off = align_up(sizeof(WsHeader));
  p->off_cnt = off;  // zeroed with the header at the start of every call
  off = align_up(off + static_cast<size_t>(p->nchunks) * counters_per_chunk(p->nvc) * sizeof(int));
  p->off_loss = off;
  if (sweep) off = align_up(off + static_cast<size_t>(N) * 4);
  p->off_zt = off;
  off = align_up(off + static_cast<size_t>(Bc) * 4);
  p->off_tcol = off;
  off = align_up(off + static_cast<size_t>(Bc) * 4);
  p->off_gt = off;
  off = align_up(off + static_cast<size_t>(Bc) * 4);
  p->off_partial = off;
  if (sweep) off = align_up(off + static_cast<size_t>(p->nseg) * static_cast<size_t>(Bc) * 8);
  p->off_L = off;
  if (backward) off = align_up(off + static_cast<size_t>(Bc) * static_cast<size_t>(Cb) * esize(dtype));
  p->off_dw = off;
  if (p->dw_acc) off = align_up(off + static_cast<size_t>(C) * static_cast<size_t>(D) * 4);
  p->off_db = off;
  if (backward && want_db) off = align_up(off + static_cast<size_t>(C) * 4);
  const bool f16bw = backward && dtype == LCE_F16;
  p->off_wrow = off;
  if (f16bw) off = align_up(off + static_cast<size_t>(Bc) * 4);
  p->off_wbar = off;
  if (f16bw) off = align_up(off + 4);
  p->off_xs = off;
  if (f16bw && want_dw) off = align_up(off + static_cast<size_t>(Bc) * static_cast<size_t>(D) * 2);
  p->off_lse = off;
  if (recompute) off = align_up(off + static_cast<size_t>(Bc) * 4);
  p->off_wv = off;
  if (recompute) off = align_up(off + static_cast<size_t>(Bc) * 4);
  p->off_dx = off;
  if (p->dx_acc) off = align_up(off + static_cast<size_t>(Bc) * static_cast<size_t>(D) * 4);
  p->ldD = ceil_div(D, 4) * 4;
  const bool tx = p->tf32;
  const bool tx_g = tx && backward && (want_dx || want_dw);
  auto take = [&off](bool on, size_t bytes) {
    const size_t at = off;
    if (on) off = align_up(off + bytes);
    return at;
  };
  const size_t w_bytes = static_cast<size_t>(C) * p->ldD * 4;
  const size_t x_bytes = static_cast<size_t>(Bc) * p->ldD * 4;
  const size_t gl_bytes = static_cast<size_t>(Bc) * p->C_pad * 4;
  p->off_wh = take(tx, w_bytes);
  p->off_wl = take(tx, w_bytes);
  p->off_xh = take(tx, x_bytes);
  p->off_xl = take(tx, x_bytes);
  p->off_gl = take(tx_g, gl_bytes);
  p->total = off;
}

// Rows per batch chunk and buffer columns of the plan whose gradient buffer
// fits `budget` bytes: on the tensor-core backward all rows and as many
// classes as fit (every class if they all do; at least min_class_chunk,
// else fewer rows); elsewhere all rows if their per-row regions fit, else
// the largest 128 * 2^k rows that do.
void budget_dims(int op, int64_t N, int64_t D, int64_t C, int dtype, int64_t budget, int64_t* Bc, int64_t* Cb) {
  const bool tf32 = dtype == LCE_F32 && f32_tensor_default();
  const bool tc = dtype != LCE_F32;
  const bool bw = is_backward_op(op);
  const int64_t C_pad = (tc || tf32) ? ceil_div(C, 256) * 256 : ceil_div(C, 128) * 128;
  *Cb = C_pad;
  if (N == 0) {
    *Bc = 0;
    return;
  }
  if (bw && tc) {
    const int64_t esz = esize(dtype);
    const int64_t cmin = min_class_chunk(D, C_pad);
    if (N * C_pad * esz <= budget) {
      *Bc = N;
    } else if (N * cmin * esz <= budget) {
      *Bc = N;
      *Cb = std::min(C_pad, budget / (N * esz) / 256 * 256);
    } else {
      int64_t bc = std::max<int64_t>(256, budget / (cmin * esz) / 256 * 256);
      *Bc = std::min(bc, N);
      *Cb = std::max(cmin, std::min(C_pad, budget / (*Bc * esz) / 256 * 256));
    }
    return;
  }
  int64_t per_row = (bw ? C_pad * esize(dtype) : 0) + ceil_div(C, 64) * 8;
  if (tf32) per_row += 8 * D + (bw ? 4 * C_pad : 0);  // TF32 parts of X, lo part of G
  if (N * per_row <= budget) {
    *Bc = N;
    return;
  }
  int64_t bc = 128;
  while (bc * 2 * per_row <= budget && bc * 2 < N) bc *= 2;
  *Bc = bc;
}

// The fastest plan that fits ws_bytes: all rows and all classes; else all
// rows and the widest class chunk (>= min_class_chunk) that fits; else the
// same for the largest batch chunk of 128 * 2^k rows that fits.
bool choose_plan(int op, int64_t N, int64_t D, int64_t C, int dtype, int grad_dtype, bool want_dx, bool want_dw,
                 bool want_db, size_t ws_bytes, Plan* p) {
  auto fits = [&](int64_t bc, int64_t cb) {
    make_plan(op, N, D, C, dtype, grad_dtype, want_dx, want_dw, want_db, bc, cb, p);
    return p->total <= ws_bytes;
  };
  if (N == 0) return fits(0, 0);
  std::vector<int64_t> cands;
  cands.push_back(N);
  int64_t bc = 128;
  while (bc * 2 < N) bc *= 2;
  for (; bc >= 128; bc /= 2)
    if (bc < N) cands.push_back(bc);
  make_plan(op, N, D, C, dtype, grad_dtype, want_dx, want_dw, want_db, N, 0, p);
  const bool vocab = p->backward && p->tc;
  const int64_t C_pad = p->C_pad;
  const int64_t cmin = min_class_chunk(D, C_pad);
  for (int64_t rows : cands) {
    if (fits(rows, C_pad)) return true;
    if (!vocab || cmin >= C_pad || !fits(rows, cmin)) continue;
    int64_t lo = cmin / 256, hi = C_pad / 256;  // fits(lo * 256), !fits(hi * 256)
    while (hi - lo > 1) {
      const int64_t mid = (lo + hi) / 2;
      if (fits(rows, mid * 256))
        lo = mid;
      else
        hi = mid;
    }
    return fits(rows, lo * 256);
  }
  return false;
}

// Row slabs of a chunk of `rows` rows: slab k is [off[k], off[k+1]),
// k < the returned count (1 when not slabbed). Slab k's G formation runs
// beside slab k+1's logits GEMM, so the slabs grow, about 4 : 7 : 9 : 12 of
// the rows: each side job forms no more rows than the GEMM beside it
// computes, and the largest, last slab goes to the long dX GEMM. The
// boundaries are the cumulative shares rounded down to the 256-row tile
// height, so every slab but the last is within 256 rows of its share and
// the last one never gets less. Where four slabs would not come out
// non-decreasing (fewer than 2048 rows), three slabs of shares 7 : 9 : 12
// are tried, then two of 9 : 12, then one. Sizes are non-decreasing for
// every row count and strictly growing from 8192 rows on.
int row_slabs(int64_t rows, bool slabbed, int64_t off[5]) {
  for (int k = 0; k < 5; ++k) off[k] = rows;
  off[0] = 0;
  if (!slabbed) return 1;
  if (rows <= 0) return 0;
  static const int64_t kShares[3][4] = {{4, 7, 9, 12}, {7, 9, 12, 0}, {9, 12, 0, 0}};
  for (int n = 4; n >= 2; --n) {
    const int64_t* sh = kShares[4 - n];
    int64_t total = 0;
    for (int k = 0; k < n; ++k) total += sh[k];
    int64_t cand[5];
    cand[0] = 0;
    int64_t cum = 0;
    for (int k = 0; k + 1 < n; ++k) {
      cum += sh[k];
      cand[k + 1] = rows * cum / total / 256 * 256;
    }
    cand[n] = rows;
    bool ok = true;
    for (int k = 0; k < n && ok; ++k) {
      const int64_t sz = cand[k + 1] - cand[k];
      ok = sz > 0 && (k == 0 || sz >= cand[k] - cand[k - 1]);
    }
    if (!ok) continue;
    for (int k = 0; k <= n; ++k) off[k] = cand[k];
    return n;
  }
  return 1;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? LCE_OK : LCE_ERR_CUDA; }

int check_common(int64_t N, int64_t D, int64_t C, int dtype, int acc_dtype, int reduction) {
  if (dtype != LCE_F32 && dtype != LCE_BF16 && dtype != LCE_F16) return LCE_ERR_DTYPE;
  if (acc_dtype != LCE_F32) return LCE_ERR_DTYPE;
  if (reduction != LCE_RED_NONE && reduction != LCE_RED_SUM && reduction != LCE_RED_MEAN) return LCE_ERR_REDUCTION;
  if (N < 0 || D < 1 || C < 1) return LCE_ERR_SHAPE;
  if (N > (int64_t(1) << 40) || D > (int64_t(1) << 30) || C > (int64_t(1) << 30)) return LCE_ERR_SHAPE;
  return LCE_OK;
}

#define LCE_TRY(expr)                        \
  do {                                       \
    cudaError_t _e = (expr);                 \
    if (_e != cudaSuccess) return LCE_ERR_CUDA; \
  } while (0)

// The shared body of lce_forward, lce_forward_backward and lce_backward
// (op: LCE_OP_FORWARD, LCE_OP_FORWARD_BACKWARD or LCE_OP_BACKWARD; lse_in
// is the given row lse of LCE_OP_BACKWARD).
int run_lce(int op, const void* X, const void* W, const void* b, const int64_t* target, const float* class_weight,
            const float* denominator, int64_t N, int64_t D, int64_t C, int dtype, int acc_dtype, int reduction,
            int64_t ignore_index,
            const float* lse_in, const float* grad_out, float* loss_out, float* lse_out, void* dX, void* dW,
            void* db, int grad_dtype, void* workspace, size_t ws_bytes, void* stream) {
  const bool backward = is_backward_op(op);
  const bool given = op == LCE_OP_BACKWARD;
  int st = check_common(N, D, C, dtype, acc_dtype, reduction);
  if (st != LCE_OK) return st;
  if (backward && grad_dtype != LCE_F32 && grad_dtype != LCE_BF16 && grad_dtype != LCE_F16) return LCE_ERR_DTYPE;
  if (N > 0 && (X == nullptr || W == nullptr || target == nullptr)) return LCE_ERR_NULL;
  if (!given && N > 0 && loss_out == nullptr) return LCE_ERR_NULL;
  if (!given && reduction != LCE_RED_NONE && loss_out == nullptr) return LCE_ERR_NULL;
  if (given && N > 0 && lse_in == nullptr) return LCE_ERR_NULL;
  if (backward && reduction == LCE_RED_NONE && N > 0 && grad_out == nullptr) return LCE_ERR_GRAD_OUT;
  if (workspace == nullptr) return LCE_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LCE_ERR_ALIGN;
  const bool want_dx = backward && dX != nullptr;
  const bool want_dw = backward && dW != nullptr;
  const bool want_db = backward && db != nullptr && b != nullptr;
  if (dtype != LCE_F32) {
    if (D % 8 != 0) return LCE_ERR_ALIGN;
    if (N > 0 && (!aligned16(X) || !aligned16(W))) return LCE_ERR_ALIGN;
    if ((want_dx && !aligned16(dX)) || (want_dw && !aligned16(dW))) return LCE_ERR_ALIGN;
  }
  Plan p;
  if (!choose_plan(op, N, D, C, dtype, grad_dtype, want_dx, want_dw, want_db, ws_bytes, &p)) return LCE_ERR_WORKSPACE;
  if (p.Bc > 2147483647LL) return LCE_ERR_SHAPE;
  st = check_device();
  if (st != LCE_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* loss_rows = reinterpret_cast<float*>(ws + p.off_loss);
  float* zt = reinterpret_cast<float*>(ws + p.off_zt);
  int* tcol = reinterpret_cast<int*>(ws + p.off_tcol);
  float* gt = reinterpret_cast<float*>(ws + p.off_gt);
  float2* partial = reinterpret_cast<float2*>(ws + p.off_partial);
  void* Lbuf = ws + p.off_L;
  float* dw_acc = reinterpret_cast<float*>(ws + p.off_dw);
  float* db_acc = reinterpret_cast<float*>(ws + p.off_db);
  float* lse_ws = reinterpret_cast<float*>(ws + p.off_lse);
  float* wv_ws = reinterpret_cast<float*>(ws + p.off_wv);
  float* dx_acc = reinterpret_cast<float*>(ws + p.off_dx);
  const bool f16 = dtype == LCE_F16;
  float* wrow = f16 && backward ? reinterpret_cast<float*>(ws + p.off_wrow) : nullptr;
  float* wbar = reinterpret_cast<float*>(ws + p.off_wbar);
  void* Xs = ws + p.off_xs;
  const int gsz = esize(grad_dtype);
  const int isz = esize(dtype);
  const bool sweep = !p.given_lse;  // forward sweep (a given lse is only used on the tensor-core path)
  const bool recompute = p.nvc > 0;
  // classes whose G comes from the forward sweep's stored P~
  const int64_t Cs_eff = std::min(p.Cs, C);
  const int nseg_store = static_cast<int>(std::min<int64_t>(p.nseg, ceil_div(Cs_eff, p.segw)));

  const int64_t cstride = counters_per_chunk(p.nvc);
  LCE_TRY(cudaMemsetAsync(hdr, 0, p.off_cnt + static_cast<size_t>(p.nchunks) * cstride * sizeof(int), s));
  int* counters = reinterpret_cast<int*>(ws + p.off_cnt);
  if (N == 0) {
    if (!given && reduction != LCE_RED_NONE) {
      LCE_TRY(launch_prep(target, 0, C, ignore_index, class_weight, denominator, hdr, s));
      LCE_TRY(launch_loss_finalize(loss_rows, 0, reduction, hdr, class_weight != nullptr, loss_out, s));
    }
    if (want_dw) LCE_TRY(cudaMemsetAsync(dW, 0, static_cast<size_t>(C) * D * gsz, s));
    if (want_db) LCE_TRY(cudaMemsetAsync(db, 0, static_cast<size_t>(C) * gsz, s));
    return LCE_OK;
  }
  LCE_TRY(launch_prep(target, N, C, ignore_index, class_weight, denominator, hdr, s));
  if (want_db) LCE_TRY(cudaMemsetAsync(db_acc, 0, static_cast<size_t>(C) * 4, s));
  // per-row losses: the caller's vector for 'none', else the workspace (a
  // given-lse call on the fp32 path runs a forward sweep whose losses are
  // not returned)
  float* rows_out = (reduction == LCE_RED_NONE && !given) ? loss_out : loss_rows;

  RowWeight rw;
  rw.grad_out = grad_out;
  rw.class_weight = class_weight;
  rw.reduction = reduction;
  rw.grad_is_vector = reduction == LCE_RED_NONE ? 1 : 0;

  CUtensorMap tmW_k, tmW_n;
  const bool pair = tc_pair_default() || f16;  // fp16 runs on the CTA-pair kernel only
  if (p.tc) {
    if (!encode_tmap_bf16(&tmW_k, W, D, C, D, pair ? 128 : TC_BN, dtype)) return LCE_ERR_CUDA;
    if (want_dx && !encode_tmap_bf16(&tmW_n, W, D, C, D, 64, dtype)) return LCE_ERR_CUDA;
  }
  // 3xTF32: TF32 hi / lo parts of W, X and G in their own row-major layouts;
  // the logits read X and W K-major, dX reads G K-major and W MN-major (K =
  // classes), dW reads G and X MN-major (K = rows), so nothing is transposed
  auto wsf = [ws](size_t off) { return reinterpret_cast<float*>(ws + off); };
  TxOperands tx_lg{}, tx_dx{}, tx_dw{};
  tx_dx.b_mn = 1;
  tx_dw.a_mn = 1;
  tx_dw.b_mn = 1;
  SplitArgs split_w{};  // W's split, launched with the first chunk's X split
  if (p.tf32) {
    split_w.src = static_cast<const float*>(W);
    split_w.rows = C;
    split_w.cols = D;
    split_w.lds = D;
    split_w.hi = wsf(p.off_wh);
    split_w.lo = wsf(p.off_wl);
    split_w.ldo = p.ldD;
    bool ok = encode_tmap_f32(&tx_lg.bh, split_w.hi, D, C, p.ldD, false) &&
              encode_tmap_f32(&tx_lg.bl, split_w.lo, D, C, p.ldD, false);
    if (want_dx)
      ok = ok && encode_tmap_f32(&tx_dx.bh, split_w.hi, D, C, p.ldD, true) &&
           encode_tmap_f32(&tx_dx.bl, split_w.lo, D, C, p.ldD, true);
    if (!ok) return LCE_ERR_CUDA;
  }

  for (int64_t ci = 0; ci < p.nchunks; ++ci) {
    const int64_t row0 = ci * p.Bc;
    const int64_t rows = std::min(p.Bc, N - row0);
    if (p.tf32) {  // TF32 parts of the chunk's rows of X (and of W with the first chunk)
      SplitArgs sa;
      sa.src = static_cast<const float*>(X) + row0 * D;
      sa.rows = rows;
      sa.cols = D;
      sa.lds = D;
      sa.hi = wsf(p.off_xh);
      sa.lo = wsf(p.off_xl);
      sa.ldo = p.ldD;
      LCE_TRY(launch_split_tf32(sa, s, ci == 0 ? &split_w : nullptr));
    }
    const bool slabbed = sweep && p.tc && pair && backward && rows >= 1024;
    GradArgs ga_last, ga_tx;
    CombineArgs ca_last;  // the last slab's merge, deferred into the dX GEMM's idle warps
    bool have_last = false;
    int64_t last_row0 = 0, last_si = 0;
    int* cnt = counters + ci * cstride;
    int* sched = cnt + kSched;  // tile-schedule counters of this chunk's pair GEMMs
    const float* lse_rows = nullptr;  // the chunk's row lse for recomputed classes
    if (sweep) {
      // ---- logits, row lse / loss, and G of the stored classes, over row
      // slabs of the chunk. On the CTA-pair path with a backward (>= 1024
      // rows), the chunk is cut into up to 4 slabs; the idle warps of slab
      // k's logits GEMM merge the rows of slab k-1 and form its G, and those
      // of the dX GEMM do the same for the last slab.
      int64_t slab_off[5];
      const int64_t nslab = row_slabs(rows, slabbed, slab_off);
      GradArgs ga_prev;
      CombineArgs ca_prev;
      bool have_prev = false;
      for (int64_t si = 0; si < nslab; ++si) {
        const int64_t so = slab_off[si];           // slab offset within the chunk
        const int64_t sr = slab_off[si + 1] - so;  // rows in the slab
        EpiLse::Params el;
        el.bias = b;
        el.bias_dt = dtype;
        el.target = target + row0 + so;
        el.C = C;
        el.rows = static_cast<int>(sr);
        el.partial = partial + so;
        el.partial_ld = p.Bc;
        el.zt = zt + so;
        el.ptilde =
            backward ? static_cast<uint8_t*>(Lbuf) + static_cast<size_t>(so) * p.Cb * isz : nullptr;
        el.ld_p = p.Cb;
        el.ptilde_dt = dtype;
        el.store_cols = p.Cs;
        if (p.tc) {
          const void* Xc = static_cast<const uint16_t*>(X) + (row0 + so) * D;
          CUtensorMap tmX_k, tmL;
          if (!encode_tmap_bf16(&tmX_k, Xc, D, sr, D, TC_BM, dtype)) return LCE_ERR_CUDA;
          const bool tma_out = pair && backward;
          if (tma_out && !encode_tmap_bf16_store(&tmL, el.ptilde, p.Cs, sr, p.Cb, dtype)) return LCE_ERR_CUDA;
          SideGrad side;
          side.a = ga_prev;
          side.enabled = have_prev ? 1 : 0;
          side.claim = nullptr;
          side.done = nullptr;
          side.dep_row0 = 0;
          side.ca = ca_prev;  // merge of slab si - 1, then its G formation
          side.comb = have_prev ? 1 : 0;
          side.cclaim = cnt + 2 * (si - 1);
          side.cdone = cnt + 2 * (si - 1) + 1;
          LCE_TRY(launch_tc_logits(tmX_k, tmW_k, tma_out ? &tmL : nullptr, static_cast<int>(sr), static_cast<int>(C),
                                   static_cast<int>(D), &hdr->status, el, pair, s, have_prev ? &side : nullptr, f16,
                                   sched + si));
        } else if (p.tf32) {
          const float* xh = wsf(p.off_xh) + so * p.ldD;
          const float* xl = wsf(p.off_xl) + so * p.ldD;
          if (!encode_tmap_f32(&tx_lg.ah, xh, D, sr, p.ldD, false) ||
              !encode_tmap_f32(&tx_lg.al, xl, D, sr, p.ldD, false))
            return LCE_ERR_CUDA;
          LCE_TRY(launch_tx_logits(tx_lg, static_cast<int>(sr), static_cast<int>(C), static_cast<int>(D),
                                   &hdr->status, el, s));
        } else {
          const float* Xc = static_cast<const float*>(X) + (row0 + so) * D;
          LCE_TRY(launch_simt_logits(Xc, static_cast<const float*>(W), D, D, sr, C, D, el, s));
        }
        CombineArgs ca;
        ca.partial = partial + so;
        ca.ld = p.Bc;
        ca.nseg = p.nseg;
        ca.rows = sr;
        ca.row0 = row0 + so;
        ca.zt = zt + so;
        ca.tcol = tcol + so;
        ca.gt = gt + so;
        ca.target = target;
        ca.ignore_index = ignore_index;
        ca.C = C;
        ca.rw = rw;
        ca.hdr = hdr;
        ca.loss_rows = rows_out;
        ca.lse_out = lse_out;
        ca.backward = backward ? 1 : 0;
        ca.wrow = wrow != nullptr ? wrow + so : nullptr;
        ca.nseg_store = nseg_store;
        ca.lse_rows = recompute ? lse_ws + so : nullptr;
        ca.w_rows = recompute ? wv_ws + so : nullptr;
        // on the slabbed path the merge runs in the next GEMM's idle warps
        const bool defer = slabbed && (si + 1 < nslab || want_dx);
        if (!defer) LCE_TRY(launch_combine(ca, s));
        if (!backward) continue;
        GradArgs ga;
        ga.L = el.ptilde;
        ga.ld = p.Cb;
        ga.rows = sr;
        ga.C = Cs_eff;
        ga.segw = p.segw;
        ga.nseg = nseg_store;
        ga.scale = partial + so;
        ga.sld = p.Bc;
        ga.tcol = tcol + so;
        ga.gt = gt + so;
        ga.db_acc = want_db ? db_acc : nullptr;
        ga.wrow = wrow != nullptr ? wrow + so : nullptr;
        if (slabbed && si + 1 < nslab) {
          ga_prev = ga;  // merged and formed by the next slab's GEMM
          ca_prev = ca;
          have_prev = true;
        } else if (slabbed && want_dx) {
          ga_last = ga;  // merged and formed by the dX GEMM's idle warps before it reads these rows
          ca_last = ca;
          have_last = true;
          last_row0 = so;
          last_si = si;
        } else if (p.tf32 && (want_dx || want_dw)) {
          ga_tx = ga;  // formed together with its TF32 split below
        } else {
          if (nseg_store > 0) LCE_TRY(launch_grad_logits(ga, dtype, s));
          have_prev = false;
        }
      }
      lse_rows = lse_ws;
    } else {
      // ---- given lse: the rows' weights and target columns
      BackwardRowsArgs br;
      br.target = target;
      br.row0 = row0;
      br.rows = rows;
      br.C = C;
      br.ignore_index = ignore_index;
      br.rw = rw;
      br.hdr = hdr;
      br.tcol = tcol;
      br.w_rows = wv_ws;
      br.wrow = wrow;
      LCE_TRY(launch_backward_rows(br, s));
      lse_rows = lse_in + row0;
    }
    if (!backward) continue;
    if (p.tf32 && (want_dx || want_dw)) {  // G formed from P~ and split: hi over P~ itself, lo beside it
      SplitArgs sa;
      sa.src = static_cast<const float*>(Lbuf);
      sa.rows = rows;
      sa.cols = C;
      sa.lds = p.C_pad;
      sa.hi = static_cast<float*>(Lbuf);
      sa.lo = wsf(p.off_gl);
      sa.ldo = p.C_pad;
      LCE_TRY(launch_grad_split_tf32(ga_tx, sa, s));
    }
    // dX is the sum over the class parts (the stored classes, then each
    // recomputed chunk); with several parts a 16-bit dX is summed in fp32
    const int64_t nparts = (Cs_eff > 0 ? 1 : 0) + p.nvc;
    auto dx_params = [&](int64_t part) {
      EpiStore::Params es;
      es.out = static_cast<uint8_t*>(dX) + static_cast<size_t>(row0) * D * gsz;
      es.out_dt = grad_dtype;
      es.ldo = D;
      es.rows = rows;
      es.cols = D;
      es.vec_ok = aligned16(dX) && ((D * gsz) % 16 == 0);
      es.row_scale = wrow;  // fp16: G without the row weights
      es.scalar_scale = nullptr;
      if (nparts == 1) {
        es.mode = 0;
        es.acc32 = nullptr;
      } else if (grad_dtype == LCE_F32) {
        es.mode = part == 0 ? 0 : 2;
        es.acc32 = static_cast<float*>(es.out);
      } else {
        es.mode = part == 0 ? 1 : (part == nparts - 1 ? 3 : 2);
        es.acc32 = dx_acc;
      }
      return es;
    };
    // dW rows [c0, c0 + cw): accumulated over the batch chunks
    auto dw_params = [&](int64_t c0, int64_t cw) {
      EpiStore::Params es;
      es.out = static_cast<uint8_t*>(dW) + static_cast<size_t>(c0) * D * gsz;
      es.out_dt = grad_dtype;
      es.ldo = D;
      es.rows = cw;
      es.cols = D;
      es.vec_ok = aligned16(dW) && ((D * gsz) % 16 == 0);
      es.row_scale = nullptr;
      es.scalar_scale = f16 ? wbar : nullptr;  // fp16: dW = max|w| * G^T (X * w / max|w|)
      if (p.nchunks == 1) {
        es.mode = 0;
        es.acc32 = nullptr;
      } else if (grad_dtype == LCE_F32) {
        es.mode = ci == 0 ? 0 : 2;
        es.acc32 = static_cast<float*>(es.out);
      } else {
        es.mode = ci == 0 ? 1 : (ci == p.nchunks - 1 ? 3 : 2);
        es.acc32 = dw_acc + static_cast<size_t>(c0) * D;
      }
      return es;
    };
    const void* Xc = p.tc ? static_cast<const void*>(static_cast<const uint16_t*>(X) + row0 * D) : nullptr;
    const void* Xdw = Xc;  // the B operand of dW (fp16: X scaled per row)
    bool xs_done = false;
    auto prepare_dw = [&]() -> cudaError_t {
      if (!f16 || xs_done) return cudaSuccess;
      xs_done = true;
      Xdw = Xs;
      return launch_row_scale(Xc, wrow, wbar, Xs, rows, D, s);
    };
    int64_t part = 0;
    if (Cs_eff > 0) {
      // ---- dX = G W over the stored classes
      if (want_dx) {
        EpiStore::Params es = dx_params(part);
        if (p.tc) {
          CUtensorMap tmG_k, tmdX;
          if (!encode_tmap_bf16(&tmG_k, Lbuf, Cs_eff, rows, p.Cb, TC_BM, dtype)) return LCE_ERR_CUDA;
          const bool tma_out = pair && (es.mode == 0 || es.mode == 3) && es.out_dt != LCE_F32 && es.vec_ok;
          if (tma_out && !encode_tmap_bf16_store(&tmdX, es.out, D, rows, D, grad_dtype)) return LCE_ERR_CUDA;
          SideGrad side;
          if (have_last) {
            side.a = ga_last;
            side.enabled = 1;
            side.claim = cnt + 8;
            side.done = cnt + 9;
            side.dep_row0 = last_row0;
            side.ca = ca_last;
            side.comb = 1;
            side.cclaim = cnt + 2 * last_si;
            side.cdone = cnt + 2 * last_si + 1;
          }
          LCE_TRY(launch_tc_store(TC_DX, tmG_k, tmW_n, tma_out ? &tmdX : nullptr, static_cast<int>(rows),
                                  static_cast<int>(D), static_cast<int>(Cs_eff), &hdr->status, es, pair, s, f16,
                                  have_last ? &side : nullptr, sched + 4));
        } else if (p.tf32) {
          if (!encode_tmap_f32(&tx_dx.ah, Lbuf, C, rows, p.C_pad, false) ||
              !encode_tmap_f32(&tx_dx.al, wsf(p.off_gl), C, rows, p.C_pad, false))
            return LCE_ERR_CUDA;
          LCE_TRY(launch_tx_store(TC_DX, tx_dx, static_cast<int>(rows), static_cast<int>(D), static_cast<int>(C),
                                  &hdr->status, es, s));
        } else {
          LCE_TRY(launch_simt_store(TC_DX, static_cast<const float*>(Lbuf), static_cast<const float*>(W), p.C_pad,
                                    D, rows, D, C, es, s));
        }
      }
      // ---- dW (+)= G^T X_c over the stored classes
      if (want_dw) {
        EpiStore::Params es = dw_params(0, Cs_eff);
        if (p.tc) {
          LCE_TRY(prepare_dw());
          CUtensorMap tmG_m, tmX_n, tmdW;
          if (!encode_tmap_bf16(&tmG_m, Lbuf, Cs_eff, rows, p.Cb, 64, dtype)) return LCE_ERR_CUDA;
          if (!encode_tmap_bf16(&tmX_n, Xdw, D, rows, D, 64, dtype)) return LCE_ERR_CUDA;
          const bool tma_out = pair && (es.mode == 0 || es.mode == 3) && es.out_dt != LCE_F32 && es.vec_ok;
          if (tma_out && !encode_tmap_bf16_store(&tmdW, es.out, D, Cs_eff, D, grad_dtype)) return LCE_ERR_CUDA;
          LCE_TRY(launch_tc_store(TC_DW, tmG_m, tmX_n, tma_out ? &tmdW : nullptr, static_cast<int>(Cs_eff),
                                  static_cast<int>(D), static_cast<int>(rows), &hdr->status, es, pair, s, f16,
                                  nullptr, sched + 5));
        } else if (p.tf32) {
          bool ok = encode_tmap_f32(&tx_dw.ah, Lbuf, C, rows, p.C_pad, true) &&
                    encode_tmap_f32(&tx_dw.al, wsf(p.off_gl), C, rows, p.C_pad, true) &&
                    encode_tmap_f32(&tx_dw.bh, wsf(p.off_xh), D, rows, p.ldD, true) &&
                    encode_tmap_f32(&tx_dw.bl, wsf(p.off_xl), D, rows, p.ldD, true);
          if (!ok) return LCE_ERR_CUDA;
          LCE_TRY(launch_tx_store(TC_DW, tx_dw, static_cast<int>(C), static_cast<int>(D), static_cast<int>(rows),
                                  &hdr->status, es, s));
        } else {
          const float* Xf = static_cast<const float*>(X) + row0 * D;
          LCE_TRY(launch_simt_store(TC_DW, static_cast<const float*>(Lbuf), Xf, p.C_pad, D, C, D, rows, es, s));
        }
      }
      ++part;
    }
    // ---- the recomputed classes, one chunk of up to Cb classes at a time:
    // logits again with the gradient epilogue (G into the buffer), then the
    // chunk's share of dX and its rows of dW
    if (recompute) {
      CUtensorMap tmXc_k;
      if (!encode_tmap_bf16(&tmXc_k, Xc, D, rows, D, TC_BM, dtype)) return LCE_ERR_CUDA;
      for (int64_t v = 0; v < p.nvc; ++v, ++part) {
        const int64_t c0 = p.Cs + v * p.Cb;
        const int64_t cw = std::min(p.Cb, C - c0);
        const void* Wv = static_cast<const uint16_t*>(W) + c0 * D;
        CUtensorMap tmWv_k, tmGv;
        if (!encode_tmap_bf16(&tmWv_k, Wv, D, cw, D, pair ? 128 : TC_BN, dtype)) return LCE_ERR_CUDA;
        if (pair && !encode_tmap_bf16_store(&tmGv, Lbuf, cw, rows, p.Cb, dtype)) return LCE_ERR_CUDA;
        EpiGrad::Params eg;
        eg.bias = b != nullptr ? static_cast<const void*>(static_cast<const uint16_t*>(b) + c0) : nullptr;
        eg.bias_dt = dtype;
        eg.tcol = tcol;
        eg.col_base = c0;
        eg.cols = cw;
        eg.rows = static_cast<int>(rows);
        eg.lse = lse_rows;
        eg.wg = wv_ws;
        eg.wdb = wrow;
        eg.db_acc = want_db ? db_acc : nullptr;
        eg.g = Lbuf;
        eg.ld_g = p.Cb;
        eg.g_dt = dtype;
        LCE_TRY(launch_tc_grad(tmXc_k, tmWv_k, pair ? &tmGv : nullptr, static_cast<int>(rows), static_cast<int>(cw),
                               static_cast<int>(D), &hdr->status, eg, pair, s, f16, sched + 6 + 3 * v));
        if (want_dx) {
          EpiStore::Params es = dx_params(part);
          CUtensorMap tmG_k, tmWv_n, tmdX;
          if (!encode_tmap_bf16(&tmG_k, Lbuf, cw, rows, p.Cb, TC_BM, dtype)) return LCE_ERR_CUDA;
          if (!encode_tmap_bf16(&tmWv_n, Wv, D, cw, D, 64, dtype)) return LCE_ERR_CUDA;
          const bool tma_out = pair && (es.mode == 0 || es.mode == 3) && es.out_dt != LCE_F32 && es.vec_ok;
          if (tma_out && !encode_tmap_bf16_store(&tmdX, es.out, D, rows, D, grad_dtype)) return LCE_ERR_CUDA;
          LCE_TRY(launch_tc_store(TC_DX, tmG_k, tmWv_n, tma_out ? &tmdX : nullptr, static_cast<int>(rows),
                                  static_cast<int>(D), static_cast<int>(cw), &hdr->status, es, pair, s, f16, nullptr,
                                  sched + 7 + 3 * v));
        }
        if (want_dw) {
          EpiStore::Params es = dw_params(c0, cw);
          LCE_TRY(prepare_dw());
          CUtensorMap tmG_m, tmX_n, tmdW;
          if (!encode_tmap_bf16(&tmG_m, Lbuf, cw, rows, p.Cb, 64, dtype)) return LCE_ERR_CUDA;
          if (!encode_tmap_bf16(&tmX_n, Xdw, D, rows, D, 64, dtype)) return LCE_ERR_CUDA;
          const bool tma_out = pair && (es.mode == 0 || es.mode == 3) && es.out_dt != LCE_F32 && es.vec_ok;
          if (tma_out && !encode_tmap_bf16_store(&tmdW, es.out, D, cw, D, grad_dtype)) return LCE_ERR_CUDA;
          LCE_TRY(launch_tc_store(TC_DW, tmG_m, tmX_n, tma_out ? &tmdW : nullptr, static_cast<int>(cw),
                                  static_cast<int>(D), static_cast<int>(rows), &hdr->status, es, pair, s, f16,
                                  nullptr, sched + 8 + 3 * v));
        }
      }
    }
  }
  if (!given && reduction != LCE_RED_NONE)
    LCE_TRY(launch_loss_finalize(loss_rows, N, reduction, hdr, class_weight != nullptr, loss_out, s));
  if (want_db) LCE_TRY(launch_db_finalize(db_acc, db, C, grad_dtype, s));
  return LCE_OK;
}

}  // namespace
}  // namespace lce

using namespace lce;

extern "C" {

size_t lce_workspace_size(int op, int64_t N, int64_t D, int64_t C, int dtype, int reduction, int grad_dtype,
                          int64_t chunk_rows) {
  if (op == LCE_OP_CE_FROM_LOGITS) {
    if (N < 0 || C < 1) return 0;
    return align_up(sizeof(WsHeader)) + align_up(static_cast<size_t>(N) * 4);
  }
  if (op != LCE_OP_FORWARD && op != LCE_OP_FORWARD_BACKWARD && op != LCE_OP_BACKWARD) return 0;
  if (check_common(N, D, C, dtype, LCE_F32, reduction) != LCE_OK) return 0;
  if (is_backward_op(op) && grad_dtype != LCE_F32 && grad_dtype != LCE_BF16 && grad_dtype != LCE_F16) return 0;
  if (chunk_rows < 0) return 0;
  int64_t bc, cb;
  if (chunk_rows == 0) {
    budget_dims(op, N, D, C, dtype, kDefaultBufferBytes, &bc, &cb);
  } else {
    // batch chunks of the given rows (the calls use N or a power of two
    // times 128 rows), every class in one buffer
    if (chunk_rows >= N) {
      bc = N;
    } else {
      bc = 128;
      while (bc * 2 <= chunk_rows) bc *= 2;
      if (bc >= N) bc = N;
    }
    cb = int64_t(1) << 40;  // clamped to every class
  }
  Plan p;
  make_plan(op, N, D, C, dtype, grad_dtype, true, true, true, bc, cb, &p);
  return p.total;
}

int64_t lce_aspect_ratio_chunk_rows(int64_t N, int64_t D, int64_t C, int64_t divisor) {
  if (N < 1 || D < 1 || C < 1 || divisor < 1) return 0;
  // next_pow2(ceil(N / ceil(C / D))), divided by the divisor, at least 1
  const int64_t per = ceil_div(N, ceil_div(C, D));
  int64_t p2 = 1;
  while (p2 < per) p2 <<= 1;
  const int64_t rows = p2 / divisor;
  return rows < 1 ? 1 : rows;
}

size_t lce_workspace_size_for_buffer(int op, int64_t N, int64_t D, int64_t C, int dtype, int reduction,
                                     int grad_dtype, size_t buffer_bytes) {
  if (op != LCE_OP_FORWARD && op != LCE_OP_FORWARD_BACKWARD && op != LCE_OP_BACKWARD) return 0;
  if (check_common(N, D, C, dtype, LCE_F32, reduction) != LCE_OK) return 0;
  if (is_backward_op(op) && grad_dtype != LCE_F32 && grad_dtype != LCE_BF16 && grad_dtype != LCE_F16) return 0;
  const int64_t budget = buffer_bytes == 0 ? kDefaultBufferBytes
                                           : static_cast<int64_t>(std::min<size_t>(buffer_bytes, size_t(1) << 62));
  int64_t bc, cb;
  budget_dims(op, N, D, C, dtype, budget, &bc, &cb);
  Plan p;
  make_plan(op, N, D, C, dtype, grad_dtype, true, true, true, bc, cb, &p);
  return p.total;
}

int lce_forward(const void* X, const void* W, const void* b, const int64_t* target, int64_t N, int64_t D, int64_t C,
                int dtype, int acc_dtype, int reduction, int64_t ignore_index, float* loss_out, float* lse_out,
                void* workspace, size_t ws_bytes, void* stream) {
  return run_lce(LCE_OP_FORWARD, X, W, b, target, nullptr, nullptr, N, D, C, dtype, acc_dtype, reduction,
                 ignore_index, nullptr, nullptr, loss_out, lse_out, nullptr, nullptr, nullptr, LCE_F32, workspace, ws_bytes,
                 stream);
}

int lce_forward_ex(const void* X, const void* W, const void* b, const int64_t* target, const float* class_weight,
                   const float* denominator, int64_t N, int64_t D, int64_t C, int dtype, int acc_dtype, int reduction,
                   int64_t ignore_index, float* loss_out, float* lse_out, void* workspace, size_t ws_bytes,
                   void* stream) {
  return run_lce(LCE_OP_FORWARD, X, W, b, target, class_weight, denominator, N, D, C, dtype, acc_dtype, reduction,
                 ignore_index, nullptr, nullptr, loss_out, lse_out, nullptr, nullptr, nullptr, LCE_F32, workspace, ws_bytes,
                 stream);
}

int lce_forward_backward(const void* X, const void* W, const void* b, const int64_t* target, int64_t N, int64_t D,
                         int64_t C, int dtype, int acc_dtype, int reduction, int64_t ignore_index,
                         const float* grad_out, float* loss_out, void* dX, void* dW, void* db, int grad_dtype,
                         void* workspace, size_t ws_bytes, void* stream) {
  return run_lce(LCE_OP_FORWARD_BACKWARD, X, W, b, target, nullptr, nullptr, N, D, C, dtype, acc_dtype, reduction,
                 ignore_index, nullptr, grad_out, loss_out, nullptr, dX, dW, db, grad_dtype, workspace, ws_bytes,
                 stream);
}

int lce_forward_backward_ex(const void* X, const void* W, const void* b, const int64_t* target,
                            const float* class_weight, const float* denominator, int64_t N, int64_t D, int64_t C,
                            int dtype, int acc_dtype, int reduction, int64_t ignore_index, const float* grad_out,
                            float* loss_out, void* dX, void* dW, void* db, int grad_dtype, void* workspace,
                            size_t ws_bytes, void* stream) {
  return run_lce(LCE_OP_FORWARD_BACKWARD, X, W, b, target, class_weight, denominator, N, D, C, dtype, acc_dtype,
                 reduction, ignore_index, nullptr, grad_out, loss_out, nullptr, dX, dW, db, grad_dtype, workspace, ws_bytes,
                 stream);
}

int lce_backward(const void* X, const void* W, const void* b, const int64_t* target, const float* lse, int64_t N,
                 int64_t D, int64_t C, int dtype, int acc_dtype, int reduction, int64_t ignore_index,
                 const float* grad_out, void* dX, void* dW, void* db, int grad_dtype, void* workspace,
                 size_t ws_bytes, void* stream) {
  return run_lce(LCE_OP_BACKWARD, X, W, b, target, nullptr, nullptr, N, D, C, dtype, acc_dtype, reduction,
                 ignore_index, lse,
                 grad_out, nullptr, nullptr, dX, dW, db, grad_dtype, workspace, ws_bytes, stream);
}

int lce_backward_ex(const void* X, const void* W, const void* b, const int64_t* target, const float* class_weight,
                    const float* denominator, const float* lse, int64_t N, int64_t D, int64_t C, int dtype,
                    int acc_dtype, int reduction, int64_t ignore_index, const float* grad_out, void* dX, void* dW,
                    void* db, int grad_dtype, void* workspace, size_t ws_bytes, void* stream) {
  return run_lce(LCE_OP_BACKWARD, X, W, b, target, class_weight, denominator, N, D, C, dtype, acc_dtype, reduction,
                 ignore_index, lse, grad_out, nullptr, nullptr, dX, dW, db, grad_dtype, workspace, ws_bytes, stream);
}

int lce_cross_entropy_from_logits(void* logits_inout, const int64_t* target, int64_t N, int64_t V, int dtype,
                                  int reduction, int64_t ignore_index, const float* grad_out, float* loss_out,
                                  void* workspace, size_t ws_bytes, void* stream) {
  return lce_cross_entropy_from_logits_ex(logits_inout, target, nullptr, nullptr, N, V, dtype, reduction,
                                          ignore_index, grad_out, loss_out, workspace, ws_bytes, stream);
}

int lce_cross_entropy_from_logits_ex(void* logits_inout, const int64_t* target, const float* class_weight,
                                     const float* denominator, int64_t N, int64_t V, int dtype, int reduction,
                                     int64_t ignore_index, const float* grad_out, float* loss_out, void* workspace,
                                     size_t ws_bytes, void* stream) {
  if (dtype != LCE_F32 && dtype != LCE_BF16 && dtype != LCE_F16) return LCE_ERR_DTYPE;
  if (reduction != LCE_RED_NONE && reduction != LCE_RED_SUM && reduction != LCE_RED_MEAN) return LCE_ERR_REDUCTION;
  if (N < 0 || V < 1 || N > (int64_t(1) << 40) || V > (int64_t(1) << 40)) return LCE_ERR_SHAPE;
  if (N > 0 && (logits_inout == nullptr || target == nullptr || loss_out == nullptr)) return LCE_ERR_NULL;
  if (reduction != LCE_RED_NONE && loss_out == nullptr) return LCE_ERR_NULL;
  if (reduction == LCE_RED_NONE && N > 0 && grad_out == nullptr) return LCE_ERR_GRAD_OUT;
  if (workspace == nullptr) return LCE_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LCE_ERR_ALIGN;
  if (ws_bytes < lce_workspace_size(LCE_OP_CE_FROM_LOGITS, N, 1, V, dtype, reduction, dtype, 0))
    return LCE_ERR_WORKSPACE;
  int st = check_device();
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* loss_rows = reinterpret_cast<float*>(ws + align_up(sizeof(WsHeader)));
  LCE_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
  LCE_TRY(launch_prep(target, N, V, ignore_index, class_weight, denominator, hdr, s));
  if (N > 0) {
    CeArgs a;
    a.logits = logits_inout;
    a.N = N;
    a.V = V;
    a.target = target;
    a.ignore_index = ignore_index;
    a.rw.grad_out = grad_out;
    a.rw.class_weight = class_weight;
    a.rw.reduction = reduction;
    a.rw.grad_is_vector = reduction == LCE_RED_NONE ? 1 : 0;
    a.hdr = hdr;
    a.loss_rows = reduction == LCE_RED_NONE ? loss_out : loss_rows;
    a.status = &hdr->status;
    LCE_TRY(launch_ce_logits(a, dtype, s));
  }
  if (reduction != LCE_RED_NONE)
    LCE_TRY(launch_loss_finalize(loss_rows, N, reduction, hdr, class_weight != nullptr, loss_out, s));
  return LCE_OK;
}

int lce_scale_gradients(void* dX, int64_t n_dx, void* dW, int64_t n_dw, void* db, int64_t n_db, int grad_dtype,
                        const float* grad_out, void* stream) {
  if (grad_dtype != LCE_F32 && grad_dtype != LCE_BF16 && grad_dtype != LCE_F16) return LCE_ERR_DTYPE;
  if (grad_out == nullptr) return LCE_ERR_NULL;
  if (n_dx < 0 || n_dw < 0 || n_db < 0) return LCE_ERR_SHAPE;
  if ((n_dx > 0 && dX == nullptr) || (n_dw > 0 && dW == nullptr) || (n_db > 0 && db == nullptr)) return LCE_ERR_NULL;
  const int st = check_device();
  if (st != LCE_OK) return st;
  return from_cuda(launch_scale_grads(dX, dX ? n_dx : 0, dW, dW ? n_dw : 0, db, db ? n_db : 0, grad_dtype, grad_out,
                                      static_cast<cudaStream_t>(stream)));
}

int lce_mean_denominator(const int64_t* target, const float* class_weight, int64_t N, int64_t C,
                         int64_t ignore_index, float* denominator_out, void* workspace, size_t ws_bytes,
                         void* stream) {
  if (denominator_out == nullptr || workspace == nullptr) return LCE_ERR_NULL;
  if (N > 0 && target == nullptr) return LCE_ERR_NULL;
  if (N < 0 || C < 1 || N > (int64_t(1) << 40) || C > (int64_t(1) << 40)) return LCE_ERR_SHAPE;
  if (ws_bytes < sizeof(WsHeader)) return LCE_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LCE_ERR_ALIGN;
  const int st = check_device();
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  LCE_TRY(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
  LCE_TRY(launch_prep(target, N, C, ignore_index, class_weight, nullptr, hdr, s, denominator_out));
  return LCE_OK;
}

const char* lce_status_string(int status) {
  switch (status) {
    case LCE_OK: return "ok";
    case LCE_ERR_NULL: return "a required pointer is NULL";
    case LCE_ERR_SHAPE: return "invalid problem size";
    case LCE_ERR_DTYPE: return "unsupported dtype (inputs and gradients fp32, bf16 or fp16; accumulation fp32)";
    case LCE_ERR_REDUCTION: return "reduction must be none, sum or mean";
    case LCE_ERR_GRAD_OUT: return "reduction none needs a per-row upstream gradient";
    case LCE_ERR_WORKSPACE: return "workspace missing or too small";
    case LCE_ERR_CUDA: return "CUDA runtime error or kernel launch failure";
    case LCE_ERR_TARGET_RANGE: return "a target is neither ignore_index nor a class index";
    case LCE_ERR_ALIGN:
      return "bf16 / fp16 inputs need D % 8 == 0 and 16-byte aligned X, W, dX, dW; every workspace 16-byte aligned";
    case LCE_ERR_TIMEOUT: return "a device pipeline wait timed out";
    case LCE_ERR_DEVICE: return "device is not compute capability 10.3 (GB300)";
    default: return "unknown status";
  }
}

int lce_read_device_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return LCE_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LCE_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LCE_ERR_CUDA;
  if (v & kStatusTimeout) return LCE_ERR_TIMEOUT;
  if (v & kStatusTargetRange) return LCE_ERR_TARGET_RANGE;
  return LCE_OK;
}

int64_t lce_launch_count(void) { return g_launches.load(); }

int lce_profile_enable(int on) {
  g_prof = on != 0;
  return LCE_OK;
}

int lce_profile_reset(void) {
  for (auto& r : g_recs) {
    if (r.a) cudaEventDestroy(r.a);
    if (r.b) cudaEventDestroy(r.b);
  }
  g_recs.clear();
  return LCE_OK;
}

int lce_profile_query(int kernel_id, int64_t* launches, double* total_ms, double* total_work) {
  if (launches == nullptr || total_ms == nullptr) return LCE_ERR_NULL;
  int64_t n = 0;
  double tot = 0.0, work = 0.0;
  for (auto& r : g_recs) {
    if (r.id != kernel_id || r.b == nullptr) continue;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return LCE_ERR_CUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return LCE_ERR_CUDA;
    ++n;
    tot += ms;
    work += r.work;
  }
  *launches = n;
  *total_ms = tot;
  if (total_work != nullptr) *total_work = work;
  return LCE_OK;
}

const char* lce_kernel_name(int kernel_id) { return kernel_id_name(kernel_id); }
int lce_num_kernel_ids(void) { return K_NUM_IDS; }

int lce_test_gemm_bf16(const void* A, const void* B, float* out, int64_t M, int64_t N, int64_t K, int a_mn_major,
                       int b_mn_major, int cta_pair, int* dev_status, void* stream) {
  if (A == nullptr || B == nullptr || out == nullptr) return LCE_ERR_NULL;
  if (M < 1 || N < 1 || K < 1 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return LCE_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return LCE_ERR_ALIGN;
  if ((a_mn_major ? M : K) % 8 != 0 || (b_mn_major ? N : K) % 8 != 0) return LCE_ERR_ALIGN;
  int st = check_device();
  if (st != LCE_OK) return st;
  CUtensorMap ta, tb;
  bool ok = a_mn_major ? encode_tmap_bf16(&ta, A, M, K, M, 64) : encode_tmap_bf16(&ta, A, K, M, K, TC_BM);
  ok = ok && (b_mn_major ? encode_tmap_bf16(&tb, B, N, K, N, 64)
                         : encode_tmap_bf16(&tb, B, K, N, K, cta_pair ? 128 : TC_BN));
  if (!ok) return LCE_ERR_CUDA;
  EpiStore::Params es;
  es.out = out;
  es.out_dt = LCE_F32;
  es.row_scale = nullptr;
  es.scalar_scale = nullptr;
  es.ldo = N;
  es.acc32 = nullptr;
  es.mode = 0;
  es.rows = M;
  es.cols = N;
  es.vec_ok = (N % 4) == 0;
  const int op = a_mn_major ? (b_mn_major ? TC_TEST_MM : TC_TEST_MK) : (b_mn_major ? TC_TEST_KM : TC_TEST_KK);
  return from_cuda(launch_tc_store(op, ta, tb, nullptr, static_cast<int>(M), static_cast<int>(N),
                                   static_cast<int>(K), dev_status, es, cta_pair != 0,
                                   static_cast<cudaStream_t>(stream)));
}

int lce_test_gemm_bf16_unmet_dependency(const void* A, const void* B, float* out, int64_t M, int64_t N, int64_t K,
                                        int* counters, int* dev_status, void* stream) {
  if (A == nullptr || B == nullptr || out == nullptr || counters == nullptr || dev_status == nullptr)
    return LCE_ERR_NULL;
  if (M < 1 || N < 1 || K < 1 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return LCE_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return LCE_ERR_ALIGN;
  if (K % 8 != 0 || N % 8 != 0) return LCE_ERR_ALIGN;
  int st = check_device();
  if (st != LCE_OK) return st;
  CUtensorMap ta, tb;
  if (!encode_tmap_bf16(&ta, A, K, M, K, TC_BM) || !encode_tmap_bf16(&tb, B, N, K, N, 64)) return LCE_ERR_CUDA;
  EpiStore::Params es;
  es.out = out;
  es.out_dt = LCE_F32;
  es.row_scale = nullptr;
  es.scalar_scale = nullptr;
  es.ldo = N;
  es.acc32 = nullptr;
  es.mode = 0;
  es.rows = M;
  es.cols = N;
  es.vec_ok = (N % 4) == 0;
  SideGrad side;
  memset(&side, 0, sizeof(side));
  side.enabled = 1;
  side.a.rows = M;  // the dependency covers every A row
  side.a.nseg = 1;
  side.claim = counters;
  side.done = counters + 1;
  side.dep_row0 = 0;
  return from_cuda(launch_tc_store(TC_DX, ta, tb, nullptr, static_cast<int>(M), static_cast<int>(N),
                                   static_cast<int>(K), dev_status, es, true, static_cast<cudaStream_t>(stream),
                                   false, &side));
}

int lce_test_gemm_tf32x3(const float* A, const float* B, float* out, int64_t M, int64_t N, int64_t K,
                         int a_mn_major, int b_mn_major, int k_splits, void* workspace, size_t ws_bytes,
                         int* dev_status, void* stream) {
  if (A == nullptr || B == nullptr || out == nullptr || workspace == nullptr) return LCE_ERR_NULL;
  if (M < 1 || N < 1 || K < 1 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return LCE_ERR_SHAPE;
  if (!aligned16(workspace)) return LCE_ERR_ALIGN;
  // each operand split into hi / lo parts in its own layout: [rows, K] when
  // K-major, [K, rows] when MN-major, the contiguous dimension padded to 4
  const bool mn[2] = {a_mn_major != 0, b_mn_major != 0};
  const int64_t rows[2] = {M, N};
  int64_t pr[2], pc[2], ld[2];
  size_t bytes[2];
  for (int op = 0; op < 2; ++op) {
    pr[op] = mn[op] ? K : rows[op];
    pc[op] = mn[op] ? rows[op] : K;
    ld[op] = ceil_div(pc[op], 4) * 4;
    bytes[op] = align_up(static_cast<size_t>(pr[op]) * ld[op] * 4);
  }
  if (ws_bytes < 2 * bytes[0] + 2 * bytes[1]) return LCE_ERR_WORKSPACE;
  int st = check_device();
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* parts[4] = {reinterpret_cast<float*>(ws), reinterpret_cast<float*>(ws + bytes[0]),
                     reinterpret_cast<float*>(ws + 2 * bytes[0]),
                     reinterpret_cast<float*>(ws + 2 * bytes[0] + bytes[1])};
  SplitArgs sa[2];
  for (int op = 0; op < 2; ++op) {
    sa[op].src = op == 0 ? A : B;
    sa[op].rows = pr[op];
    sa[op].cols = pc[op];
    sa[op].lds = pc[op];
    sa[op].hi = parts[2 * op];
    sa[op].lo = parts[2 * op + 1];
    sa[op].ldo = ld[op];
  }
  if (launch_split_tf32(sa[0], s, &sa[1]) != cudaSuccess) return LCE_ERR_CUDA;
  TxOperands o{};
  o.a_mn = mn[0] ? 1 : 0;
  o.b_mn = mn[1] ? 1 : 0;
  bool ok = encode_tmap_f32(&o.ah, parts[0], pc[0], pr[0], ld[0], mn[0]) &&
            encode_tmap_f32(&o.al, parts[1], pc[0], pr[0], ld[0], mn[0]) &&
            encode_tmap_f32(&o.bh, parts[2], pc[1], pr[1], ld[1], mn[1]) &&
            encode_tmap_f32(&o.bl, parts[3], pc[1], pr[1], ld[1], mn[1]);
  if (!ok) return LCE_ERR_CUDA;
  EpiStore::Params es;
  es.out = out;
  es.out_dt = LCE_F32;
  es.row_scale = nullptr;
  es.scalar_scale = nullptr;
  es.ldo = N;
  es.acc32 = nullptr;
  es.mode = 0;
  es.rows = M;
  es.cols = N;
  es.vec_ok = aligned16(out) && (N % 4) == 0;
  return from_cuda(launch_tx_store(TC_TEST_KK, o, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                   dev_status, es, s, k_splits));
}

int lce_test_gemm_f32(const float* A, const float* B, float* out, int64_t M, int64_t N, int64_t K, int a_mn_major,
                      int b_mn_major, void* stream) {
  if (A == nullptr || B == nullptr || out == nullptr) return LCE_ERR_NULL;
  if (M < 1 || N < 1 || K < 1) return LCE_ERR_SHAPE;
  int st = check_device();
  if (st != LCE_OK) return st;
  EpiStore::Params es;
  es.out = out;
  es.out_dt = LCE_F32;
  es.row_scale = nullptr;
  es.scalar_scale = nullptr;
  es.ldo = N;
  es.acc32 = nullptr;
  es.mode = 0;
  es.rows = M;
  es.cols = N;
  es.vec_ok = aligned16(out) && (N % 4) == 0;
  const int op = a_mn_major ? (b_mn_major ? TC_TEST_MM : TC_TEST_MK) : (b_mn_major ? TC_TEST_KM : TC_TEST_KK);
  return from_cuda(launch_simt_store(op, A, B, a_mn_major ? M : K, b_mn_major ? N : K, M, N, K, es,
                                     static_cast<cudaStream_t>(stream)));
}

int lce_test_row_slabs(int64_t rows, int64_t* slab_off) {
  if (slab_off == nullptr) return -1;
  if (rows < 0) return -1;
  return row_slabs(rows, true, slab_off);
}

int lce_test_plan(int op, int64_t N, int64_t D, int64_t C, int dtype, int grad_dtype, int want_dx, int want_dw,
                  int want_db, size_t ws_bytes, int64_t* out, int n_out) {
  if (out == nullptr || n_out < LCE_TEST_PLAN_FIELDS) return -1;
  if (op != LCE_OP_FORWARD && op != LCE_OP_FORWARD_BACKWARD && op != LCE_OP_BACKWARD) return -1;
  if (check_common(N, D, C, dtype, LCE_F32, LCE_RED_MEAN) != LCE_OK) return -1;
  Plan p;
  if (!choose_plan(op, N, D, C, dtype, grad_dtype, want_dx != 0, want_dw != 0, want_db != 0, ws_bytes, &p))
    return 0;
  const int64_t v[LCE_TEST_PLAN_FIELDS] = {
      p.Bc, p.nchunks, static_cast<int64_t>(p.total), p.C_pad, p.nseg,
      static_cast<int64_t>(p.off_cnt), static_cast<int64_t>(p.off_loss), static_cast<int64_t>(p.off_zt),
      static_cast<int64_t>(p.off_tcol), static_cast<int64_t>(p.off_gt), static_cast<int64_t>(p.off_partial),
      static_cast<int64_t>(p.off_L), static_cast<int64_t>(p.off_dw), static_cast<int64_t>(p.off_db),
      static_cast<int64_t>(p.off_wrow), static_cast<int64_t>(p.off_wbar), static_cast<int64_t>(p.off_xs),
      static_cast<int64_t>(p.off_lse), static_cast<int64_t>(p.off_wv), static_cast<int64_t>(p.off_dx),
      static_cast<int64_t>(p.off_wh), static_cast<int64_t>(p.off_wl), static_cast<int64_t>(p.off_xh),
      static_cast<int64_t>(p.off_xl), static_cast<int64_t>(p.off_gl),
      p.Cb, p.Cs, p.nvc};
  for (int i = 0; i < LCE_TEST_PLAN_FIELDS; ++i) out[i] = v[i];
  return LCE_TEST_PLAN_FIELDS;
}

}  // extern "C"
