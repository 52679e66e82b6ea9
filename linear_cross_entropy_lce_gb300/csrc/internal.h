// internal.h -- host-side launchers shared between the translation units of
// liblce.so. Every launcher enqueues on `stream` and returns cudaSuccess or
// the launch error.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "common.cuh"
#include "epilogues.cuh"

namespace lce {

// Kernel ids for the launch accounting / profiler.
enum KernelId {
  K_PREP = 0,
  K_GEMM_LOGITS_TC,
  K_GEMM_DX_TC,
  K_GEMM_DW_TC,
  K_GEMM_LOGITS_SIMT,
  K_GEMM_DX_SIMT,
  K_GEMM_DW_SIMT,
  K_LSE_COMBINE,
  K_GRAD_LOGITS,
  K_LOSS_FINALIZE,
  K_DB_FINALIZE,
  K_CE_RESIDENT,
  K_CE_STREAM,
  K_GEMM_TEST,
  K_ROW_SCALE,
  K_GEMM_LOGITS_TX,
  K_GEMM_DX_TX,
  K_GEMM_DW_TX,
  K_SPLIT_TF32,
  K_SCALE_GRADS,
  K_GEMM_RECOMPUTE_TC,
  K_BACKWARD_ROWS,
  K_GRAD_SPLIT_TF32,
  K_NUM_IDS
};
const char* kernel_id_name(int id);

// Launch accounting: called around every launch. work = the launch's
// algorithmic flop (GEMM kernels) or bytes (every other kernel).
void prof_before(int id, cudaStream_t s, double work = 0.0);
void prof_after(int id, cudaStream_t s);

int num_sms();

// Sets the kernel's maximum dynamic shared memory on the current device the
// first time the kernel is launched there (a per-device, per-kernel cache,
// so one process may use the library on several GPUs).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

struct SideGrad;

// ---- tcgen05 GEMM (gemm_tc.cu)
enum TcOp { TC_LOGITS = 0, TC_DX = 1, TC_DW = 2, TC_TEST_KK = 3, TC_TEST_KM = 4, TC_TEST_MK = 5, TC_TEST_MM = 6 };
// Encodes a 2-D bf16 tensor map over a row-major matrix with `rows` rows of
// `inner` elements, row pitch `ld` elements, box {64, box_rows}, 128B swizzle.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t ld,
                      uint32_t box_rows, int dt = LCE_BF16);
// pair: run the CTA-pair kernel (256 x 256 tiles, cta_group::2); its B
// operand maps use boxes of 128 rows (K-major) instead of 256.
// tmOut (pair kernel only; NULL = direct stores): bf16 output tensor map
// with 32 x 32 boxes and 64-byte swizzle (encode_tmap_bf16_store) through
// which the epilogue writes P~ (logits) or the mode-0 bf16 result (store).
// f16: fp16 operands (CTA-pair kernel); otherwise bf16.
// sched (pair kernel; NULL = static tile order): a zeroed device counter
// from which the CTA pairs claim tiles in order (one counter per launch).
cudaError_t launch_tc_logits(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap* tmOut, int M, int N,
                             int K, int* status, const EpiLse::Params& ep, bool pair, cudaStream_t s,
                             const SideGrad* side = nullptr, bool f16 = false, int* sched = nullptr);
// The logits GEMM of one class chunk again, with the gradient epilogue
// (EpiGrad): tmW covers the chunk's rows of W; tmOut (pair kernel; NULL =
// direct stores) is the store map of the chunk's G buffer.
cudaError_t launch_tc_grad(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap* tmOut, int M, int N,
                           int K, int* status, const EpiGrad::Params& ep, bool pair, cudaStream_t s, bool f16,
                           int* sched = nullptr);
// side (TC_DX on the pair kernel only): G formation run in the GEMM's idle
// warps, in the dynamic form of SideGrad.
cudaError_t launch_tc_store(int op, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap* tmOut, int M,
                            int N, int K, int* status, const EpiStore::Params& ep, bool pair, cudaStream_t s,
                            bool f16 = false, const SideGrad* side = nullptr, int* sched = nullptr);
bool encode_tmap_bf16_store(CUtensorMap* map, void* base, uint64_t inner, uint64_t rows, uint64_t ld,
                            int dt = LCE_BF16);
// Whether the fused path uses the CTA-pair GEMM (default yes; LCE_TC_PAIR=0 selects the one-CTA kernel).
bool tc_pair_default();

// ---- fp32 GEMM on the tensor cores by three TF32 products (gemm_tf32.cu)
constexpr uint32_t TX_MN_ROWS = 32;  // box rows of an MN-major operand map: one K block
// Encodes a 2-D fp32 tensor map over a row-major matrix (rows x inner, row
// pitch ld elements, ld * 4 a multiple of 16 bytes) for a 3xTF32 operand:
// K-major (inner = K) box {32, 128} with the 128-byte swizzle, or MN-major
// (inner = M or N) box {32, TX_MN_ROWS} with the 128-byte swizzle of
// 32-byte atoms.
bool encode_tmap_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t ld, bool mn_major);
// Operands as hi / lo pairs of tensor maps; a_mn / b_mn = 1: that operand
// is MN-major (A stored [K, M], B [K, N]; maps with 32-row boxes), else
// K-major (A [M, K], B [N, K]; 128-row boxes). The logits take both K-major
// (launch_tx_logits, EpiLse); launch_tx_store (EpiStore) takes any layout:
// op TC_DX (A K-major G, B MN-major W), TC_DW (both MN-major) or
// TC_TEST_KK. TC_DX with an fp32 mode-0 output and few tiles splits K over
// work items that add into the output after zeroing it; TC_TEST_KK does the
// same with test_splits work items per tile when test_splits > 1 (fp32
// mode-0 output).
struct TxOperands {
  CUtensorMap ah, al, bh, bl;
  int a_mn, b_mn;
};
cudaError_t launch_tx_logits(const TxOperands& o, int M, int N, int K, int* status, const EpiLse::Params& ep,
                             cudaStream_t s);
cudaError_t launch_tx_store(int op, const TxOperands& o, int M, int N, int K, int* status,
                            const EpiStore::Params& ep, cudaStream_t s, int test_splits = 0);
// Splits an fp32 matrix src [rows, cols] (pitch lds) into TF32 hi / lo parts:
// hi[r, c] = x rounded to TF32, lo[r, c] = (x - hi) rounded to TF32, written
// in the layout of src (pitch ldo; hi may be src itself with ldo == lds).
struct SplitArgs {
  const float* src;
  int64_t rows, cols, lds;
  float* hi;
  float* lo;
  int64_t ldo;
};
// b (optional): a second matrix split in the same launch.
cudaError_t launch_split_tf32(const SplitArgs& a, cudaStream_t s, const SplitArgs* b = nullptr);
struct GradArgs;
// The G formation of the fp32 tensor-core path fused with G's split: forms
// G from P~ in a.src (= g.L) exactly as launch_grad_logits would (bias
// gradient included) and writes only its TF32 parts (a.hi may be a.src).
cudaError_t launch_grad_split_tf32(const GradArgs& g, const SplitArgs& a, cudaStream_t s);
// Whether fp32 inputs take the 3xTF32 tensor-core path (default) or the
// SIMT fp32 GEMM (LCE_F32_SIMT=1).
bool f32_tensor_default();

// ---- SIMT fp32 GEMM (gemm_simt.cu); op as TcOp (LOGITS: A K-major, B
// K-major; DX: A K-major, B N-major; DW: A M-major, B N-major).
cudaError_t launch_simt_logits(const float* A, const float* B, int64_t lda, int64_t ldb, int64_t M, int64_t N,
                               int64_t K, const EpiLse::Params& ep, cudaStream_t s);
cudaError_t launch_simt_store(int op, const float* A, const float* B, int64_t lda, int64_t ldb, int64_t M,
                              int64_t N, int64_t K, const EpiStore::Params& ep, cudaStream_t s);

// ---- row kernels (rowops.cu)
// Valid-target count, class-weight sum, target-range check and the mean's
// denominator (given_denom: NULL or a device fp32 scalar that replaces it);
// out_denom (optional, device fp32) receives the denominator. The header
// must be zeroed before.
cudaError_t launch_prep(const int64_t* target, int64_t N, int64_t C, int64_t ignore_index, const float* cw,
                        const float* given_denom, WsHeader* hdr, cudaStream_t s, float* out_denom = nullptr);
struct CombineArgs {
  float2* partial;  // [nseg][ld]; overwritten: .x = w_n exp(m - lse) when backward
  int64_t ld;
  int nseg;
  int64_t rows;
  int64_t row0;              // global index of chunk row 0
  const float* zt;           // [rows]
  int* tcol;                 // [rows] out: target column or -1
  float* gt;                 // [rows] out: G at the target column
  const int64_t* target;     // global
  int64_t ignore_index;
  int64_t C;
  RowWeight rw;
  const WsHeader* hdr;
  float* loss_rows;          // global [N]
  float* lse_out;            // global [N] or NULL
  int backward;
  // fp16 backward: scales and G at the target leave out w_n, which goes to
  // wrow[r] instead (NULL otherwise)
  float* wrow;
  // backward: scales are written for segments < nseg_store only (the
  // classes whose P~ the forward stored)
  int nseg_store;
  // backward with classes recomputed later (NULL otherwise): the row's lse
  // and the weight folded into G (w_n, or 1 / 0 with wrow), [rows]
  float* lse_rows;
  float* w_rows;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);
// Per-row inputs of a backward whose row lse is given (no forward sweep):
// tcol[r] = target (global class) of a valid row, else -1; w_rows[r] = the
// weight folded into G (w_n, or with wrow: 1 on valid rows, 0 otherwise,
// and wrow[r] = w_n), for chunk rows r < rows of global row row0 + r.
struct BackwardRowsArgs {
  const int64_t* target;  // global
  int64_t row0, rows, C, ignore_index;
  RowWeight rw;
  const WsHeader* hdr;
  int* tcol;
  float* w_rows;
  float* wrow;  // NULL unless fp16
};
cudaError_t launch_backward_rows(const BackwardRowsArgs& a, cudaStream_t s);
struct GradArgs {
  void* L;  // [rows][ld] P~ in, G out
  int64_t ld;
  int64_t rows;
  int64_t C;
  int segw;
  int nseg;
  const float2* scale;  // [nseg][sld] (.x)
  int64_t sld;
  const int* tcol;
  const float* gt;
  float* db_acc;       // [C] or NULL
  const float* wrow;   // [rows] row weights when G is stored without them (fp16), else NULL
};
cudaError_t launch_grad_logits(const GradArgs& a, int dt, cudaStream_t s);
// G formation for a row slab (bf16, 256-column segments) done by the idle
// warps of the CTA-pair logits GEMM of the next slab.
struct SideGrad {
  GradArgs a;
  int enabled;
  // Dynamic form (the dX GEMM): units are claimed from *claim and counted in
  // *done once their G is stored; the GEMM's producer loads A rows
  // [dep_row0, dep_row0 + a.rows) only after *done reaches the unit count.
  // claim == NULL: units are taken by block index, with no dependency.
  int* claim;
  int* done;
  int64_t dep_row0;
  // Optional merge phase first (comb != 0): the rows of `ca` in blocks of
  // 32, claimed from *cclaim and counted in *cdone; the G formation starts
  // once *cdone reaches the block count (the merging threads fence before
  // counting; the waiting thread fences after its acquiring wait).
  CombineArgs ca;
  int comb;
  int* cclaim;
  int* cdone;
};
// fp16 backward: wbar = max_r |w_r| over the chunk rows (NaN if any w_r is
// NaN), then Xs[r, :] = (w_r / wbar) X[r, :] in fp16 (0 when wbar is 0).
cudaError_t launch_row_scale(const void* X, const float* wrow, float* wbar, void* Xs, int64_t rows, int64_t D,
                             cudaStream_t s);
cudaError_t launch_loss_finalize(const float* loss_rows, int64_t N, int reduction, const WsHeader* hdr,
                                 bool weighted, float* loss_out, cudaStream_t s);
cudaError_t launch_db_finalize(const float* db_acc, void* db, int64_t C, int dt, cudaStream_t s);
// a[:na], b[:nb], c[:nc] (type dt; NULL spans skipped) *= *g in place,
// nothing touched when *g == 1 (decided on the device).
cudaError_t launch_scale_grads(void* a, int64_t na, void* b, int64_t nb, void* c, int64_t nc, int dt,
                               const float* g, cudaStream_t s);

// ---- cross entropy on given logits (ce_logits.cu)
struct CeArgs {
  void* logits;
  int64_t N, V;
  const int64_t* target;
  int64_t ignore_index;
  RowWeight rw;
  const WsHeader* hdr;
  float* loss_rows;  // [N]
  int* status;
};
cudaError_t launch_ce_logits(const CeArgs& a, int dt, cudaStream_t s);

}  // namespace lce
