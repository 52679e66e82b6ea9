/*
 * lce_testing.h -- building-block entry points of liblce.so for tests.
 *
 * These expose the two GEMM engines that the fused loss is built from, so a
 * test can check a contraction on its own. They are not part of the loss
 * computation's interface. The source pages define the contractions used
 * (PyTorch commit ddfa80bd "Fix NJT linear_backward() memory usage":
 * dX = G W and dW = G^T X; linear_cross_entropy.py: logits = X W^T); the
 * operand layouts below are the three that those products need.
 *
 * out[m, n] = sum_k A(m, k) B(n, k), fp32 [M, N] row-major, written.
 *   A(m, k) = A[m * K + k] when a_mn_major == 0 (A stored [M, K]),
 *             A[k * M + m] when a_mn_major == 1 (A stored [K, M]).
 *   B(n, k) = B[n * K + k] when b_mn_major == 0 (B stored [N, K]),
 *             B[k * N + n] when b_mn_major == 1 (B stored [K, N]).
 * All pointers are device pointers; stream is a cudaStream_t. dev_status
 * is NULL or a device int that receives LCE status bits (2 = a pipeline
 * wait timed out); it is OR-ed, not cleared.
 *
 * lce_test_gemm_bf16: bf16 A, B on the tcgen05 tensor cores (TMA-fed,
 *   fp32 accumulation in tensor memory). cta_pair = 0: one CTA per 128x256
 *   tile; 1: a pair of CTAs on two SMs per 256x256 tile (cta_group::2).
 *   Needs the contiguous dimension of each operand to be a multiple of 8 and
 *   16-byte aligned pointers.
 * lce_test_gemm_f32: fp32 A, B with fp32 FMA on the CUDA cores; any shape.
 * lce_test_gemm_tf32x3: fp32 A, B on the tensor cores as three TF32
 *   products (hi*hi + hi*lo + lo*hi, hi = x rounded to TF32, lo = the
 *   rounded remainder; Ootomo & Yokota 2022), accumulated in fp32. Each
 *   operand is first split into hi / lo copies in its own layout in
 *   `workspace` (device, 16-byte aligned); an operand stored [R, S] takes
 *   two copies of R * ceil(S / 4) * 4 floats, each rounded up to 256 bytes
 *   (2 * (M + N) * ceil(K / 4) * 16 + 1024 bytes always suffice when M, N
 *   and K are multiples of 4); the tensor cores read them K-major or
 *   MN-major as stored. k_splits > 1 splits K over that many work items per
 *   tile which add into the zeroed output. Any shape up to 2^30 per
 *   dimension.
 * lce_test_gemm_bf16_unmet_dependency: the CTA-pair GEMM in its dX form
 *   (A K-major [M, K], B MN-major [K, N]) with its side job's dependency
 *   made unsatisfiable: counters[0] (claimed work chunks, preset by the
 *   caller to a value >= ceil(M / 512), e.g. 1 << 20) lets no chunk run and counters[1] (finished
 *   units, preset to 0) never reaches the count the producer waits for. The
 *   producer's bounded wait (about 2 s of SM clock) gives up, every role of
 *   the kernel unwinds through its own bounded waits, and dev_status
 *   receives the timeout bit (2); the context stays usable. For tests of
 *   the failure path only; out is left unspecified.
 * Return an lce_status_e code.
 *
 * Host-only planning entry points (no device needed; nothing is launched):
 * lce_test_row_slabs: the row slabs a chunk of `rows` rows is cut into on
 *   the CTA-pair backward path (used there when rows >= 1024): slab k is
 *   [slab_off[k], slab_off[k + 1]). slab_off is a host array of 5; returns
 *   the number of slabs (at most 4), or -1 on a NULL array or rows < 0.
 * lce_test_plan: the workspace plan a loss call with these arguments makes
 *   for a workspace of ws_bytes (op LCE_OP_FORWARD, LCE_OP_FORWARD_BACKWARD
 *   or LCE_OP_BACKWARD; the fastest plan that fits, as the calls choose it).
 *   Writes LCE_TEST_PLAN_FIELDS int64 values to the host array out: chunk
 *   rows, chunk count, total bytes, padded class count, (max, sum-exp)
 *   segments per row, then the byte offsets of the regions in workspace
 *   order: counters, row losses, target logits, target columns, target
 *   gradients, (max, sum-exp) pairs, the [chunk rows, Cb] P~ / G buffer,
 *   fp32 dW accumulator, db accumulator, fp16 row weights, fp16 weight sum,
 *   fp16 scaled X, rows' lse and G weights of recomputed classes, fp32 dX
 *   accumulator, then the TF32 parts W hi, W lo, X hi, X lo, G lo; then
 *   Cb (buffer columns), Cs (classes whose G the forward sweep stores) and
 *   the number of class chunks recomputed after it. A region a call does
 *   not use has the next region's offset (zero length). Returns
 *   LCE_TEST_PLAN_FIELDS, 0 when no plan fits ws_bytes, -1 on invalid
 *   arguments.
 */
#ifndef LCE_TESTING_H_
#define LCE_TESTING_H_

#include <stddef.h>
#include <stdint.h>

#ifndef LCE_API
#if defined(__GNUC__)
#define LCE_API __attribute__((visibility("default")))
#else
#define LCE_API
#endif
#endif

#ifdef __cplusplus
extern "C" {
#endif

LCE_API int lce_test_gemm_bf16(const void* A, const void* B, float* out, int64_t M, int64_t N,
                       int64_t K, int a_mn_major, int b_mn_major, int cta_pair, int* dev_status,
                       void* stream);

LCE_API int lce_test_gemm_f32(const float* A, const float* B, float* out, int64_t M, int64_t N,
                      int64_t K, int a_mn_major, int b_mn_major, void* stream);

LCE_API int lce_test_gemm_bf16_unmet_dependency(const void* A, const void* B, float* out, int64_t M,
                                        int64_t N, int64_t K, int* counters, int* dev_status,
                                        void* stream);

#define LCE_TEST_PLAN_FIELDS 28

LCE_API int lce_test_row_slabs(int64_t rows, int64_t* slab_off);

LCE_API int lce_test_plan(int op, int64_t N, int64_t D, int64_t C, int dtype, int grad_dtype,
                          int want_dx, int want_dw, int want_db, size_t ws_bytes, int64_t* out,
                          int n_out);

LCE_API int lce_test_gemm_tf32x3(const float* A, const float* B, float* out, int64_t M, int64_t N,
                         int64_t K, int a_mn_major, int b_mn_major, int k_splits, void* workspace,
                         size_t ws_bytes, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LCE_TESTING_H_ */
