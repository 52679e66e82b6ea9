/*
 * lce.h -- C ABI of liblce.so: fused linear + cross-entropy loss on GB300.
 *
 * The operation (PyTorch source torch/nn/modules/linear_cross_entropy.py,
 * the batch-chunked implementation; PyTorch commit ddfa80bd "Fix NJT
 * linear_backward() memory usage" for the gradient formulas):
 *
 *   z[n, j]  = sum_d X[n, d] W[j, d] + b[j]          n < N, j < C, d < D
 *   lse_n    = log sum_j exp z[n, j]
 *   loss_n   = lse_n - z[n, t_n]   (0 when t_n == ignore_index)
 *   loss     = none: loss_n | sum: sum_n loss_n | mean: sum_n loss_n / n_valid
 *   G[n, j]  = w_n (softmax(z_n)_j - [j == t_n]),
 *              w_n = 0 on ignored rows, else g / n_valid (mean), g (sum),
 *                    g_n (none), with g the upstream gradient
 *   dX = G W,  dW = G^T X,  db = sum_n G[n, :]
 *
 * and cross entropy on logits the caller already holds, whose gradient
 * replaces the logits in place (Liger-Kernel issue #343, "cross entropy
 * kernel: inplace modification of input").
 *
 * Conventions shared by every entry point
 *  - Every pointer named X, W, b, target, logits, dX, dW, db, grad_out,
 *    loss_out, lse_out and workspace is a DEVICE pointer on the current
 *    CUDA device; stream is a cudaStream_t (NULL = legacy default stream).
 *    All work is enqueued asynchronously on that stream; the call returns
 *    before the GPU finishes.
 *  - Matrices are dense row-major: X [N, D], W [C, D], dX [N, D],
 *    dW [C, D], logits [N, V]; vectors b, db [C]; target [N] int64;
 *    loss_out [1] (sum, mean) or [N] (none); lse_out [N] fp32.
 *  - The caller owns and allocates every buffer, including the workspace
 *    (size from lce_workspace_size). The library allocates no device
 *    memory and keeps no state between calls (except the optional
 *    profiling records below). Inputs are never written, except
 *    logits_inout of lce_cross_entropy_from_logits.
 *  - Gradients are the full result, WRITTEN into the caller's buffers
 *    (not accumulated into them).
 *  - Host-side argument errors return a nonzero status synchronously and
 *    enqueue nothing. Errors found by the kernels (a target that is neither
 *    ignore_index nor in [0, C), an internal wait that timed out) are
 *    recorded in the workspace and read back with lce_read_device_status;
 *    rows with such a target get loss 0 and gradient 0 and do not count
 *    toward n_valid.
 *  - Types: dtype LCE_F32, LCE_BF16 or LCE_F16 for X, W, b (or for
 *    logits); acc_dtype must be LCE_F32 (accumulation is always fp32);
 *    grad_dtype (dX, dW, db) LCE_F32, LCE_BF16 or LCE_F16. Loss and lse
 *    are fp32.
 *  - LCE_BF16 and LCE_F16 inputs run on the tcgen05 tensor cores and need
 *    D % 8 == 0 and 16-byte aligned X, W, dX, dW (else LCE_ERR_ALIGN).
 *    LCE_F32 inputs accept any shape and also run on the tensor cores, as
 *    three TF32 products per fp32 product (hi*hi + hi*lo + lo*hi with
 *    hi = x rounded to TF32 and lo the rounded remainder; partial sums
 *    folded in fp32 every 512 of K), which keeps the fp32 tolerances. Two
 *    environment variables, each read once per process, select other
 *    engines: LCE_F32_SIMT=1 runs LCE_F32 inputs with exact fp32 FMA on the
 *    CUDA cores instead; LCE_TC_PAIR=0 runs LCE_BF16 inputs on the one-CTA
 *    tcgen05 GEMM (128 x 256 tiles) instead of CTA pairs (256 x 256 tiles,
 *    cta_group::2). Results agree within the tolerances either way.
 *    With LCE_F16 the backward keeps the per-row weights w_n out of
 *    the 16-bit gradient tile (1/n_valid is below fp16's normal range for
 *    large batches; linear_cross_entropy.py keeps the per-row weight in
 *    fp32 for the same reason) and applies them in fp32 afterwards.
 *  - Device: compute capability 10.3 (GB300, sm_103a); else LCE_ERR_DEVICE.
 */
#ifndef LCE_H_
#define LCE_H_

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

/* Element types (linear_cross_entropy.py supports fp32 accumulation for
 * fp16/bf16 inputs, and accumulation in the input type otherwise). */
enum lce_dtype_e { LCE_F32 = 0, LCE_BF16 = 1, LCE_F16 = 2 };

/* Reductions accepted by linear_cross_entropy.py: "none", "sum", "mean". */
enum lce_reduction_e { LCE_RED_NONE = 0, LCE_RED_SUM = 1, LCE_RED_MEAN = 2 };

/* Operations, for lce_workspace_size. */
enum lce_op_e { LCE_OP_FORWARD = 0, LCE_OP_FORWARD_BACKWARD = 1, LCE_OP_CE_FROM_LOGITS = 2, LCE_OP_BACKWARD = 3 };

/* Status codes. */
enum lce_status_e {
  LCE_OK = 0,
  LCE_ERR_NULL = 1,         /* a required pointer is NULL */
  LCE_ERR_SHAPE = 2,        /* N < 0, D < 1, C < 1 or V < 1, or N or V > 2^40, D or C > 2^30 */
  LCE_ERR_DTYPE = 3,        /* unknown dtype, or acc_dtype != LCE_F32 */
  LCE_ERR_REDUCTION = 4,    /* reduction not one of none / sum / mean */
  LCE_ERR_GRAD_OUT = 5,     /* reduction none without a per-row upstream gradient */
  LCE_ERR_WORKSPACE = 6,    /* workspace NULL or smaller than needed for 128-row chunks */
  LCE_ERR_CUDA = 7,         /* a CUDA runtime call or kernel launch failed */
  LCE_ERR_TARGET_RANGE = 8, /* device: a target neither ignore_index nor in [0, C) */
  LCE_ERR_ALIGN = 9,        /* bf16 / fp16: D % 8 != 0 or a pointer not 16-byte aligned */
  LCE_ERR_TIMEOUT = 10,     /* device: an internal pipeline wait gave up */
  LCE_ERR_DEVICE = 11       /* current device is not compute capability 10.3 */
};

/*
 * Workspace bytes needed by one call.
 *   op          LCE_OP_FORWARD, LCE_OP_FORWARD_BACKWARD, LCE_OP_BACKWARD or
 *               LCE_OP_CE_FROM_LOGITS
 *   N, D, C     problem sizes (for CE_FROM_LOGITS pass D = 1 and C = V)
 *   dtype       input type; grad_dtype: gradient type (ignored for FORWARD)
 *   chunk_rows  0: the default plan, whose gradient buffer is bounded by
 *               1 GiB (below). > 0: batch chunks of that many rows (rounded
 *               down to 128 * 2^k, or all N rows), each with one buffer for
 *               every class: [rows, ceil(C/256)*256] of the input type, plus
 *               an fp32 [C, D] accumulator for a bf16 / fp16 dW when there
 *               is more than one chunk. chunk_rows >= N gives the plan with
 *               the whole [N, C] buffer, which does no recomputation.
 *
 * The backward keeps the softmax of a [rows, classes] block of logits in a
 * buffer of the input type (the batch-chunked buffer of
 * linear_cross_entropy.py; the full [N, C] logits are never held unless
 * they fit the budget). Under the default 1 GiB budget, on the bf16 / fp16
 * path, the buffer keeps all N rows and as many classes Cb as fit (at
 * least D rounded up to 256): the forward sweep stores its exp values for
 * classes [0, Cb); classes [Cb, C) are recomputed in chunks of Cb (their
 * logits computed a second time, 2 N D Cb flop each, formed straight into
 * gradient tiles); dX is summed over the class chunks in an fp32 [N, D]
 * accumulator and each chunk's rows of dW are complete when written (no
 * [C, D] scratch). Only when even D classes of all rows exceed the budget
 * does it also split the rows into batch chunks. fp32 inputs split rows only.
 * E.g. N = 8192, C = 128256 (bf16): Cb = 65536, one recomputed chunk, total
 * work 7 N D C instead of 6 N D C, buffer 1 GiB instead of 2.1 GB.
 *
 * The size depends only on these arguments. A call given any ws_bytes uses
 * the fastest plan that fits: all rows and all classes; else all rows and
 * the widest class chunk (a multiple of 256, at least D rounded up) that
 * fits; else the same for the largest batch chunk of 128 * 2^k rows that
 * fits. Returns 0 on invalid arguments.
 */
LCE_API size_t lce_workspace_size(int op, int64_t N, int64_t D, int64_t C, int dtype,
                          int reduction, int grad_dtype, int64_t chunk_rows);

/*
 * The batch chunk size of linear_cross_entropy.py's "aspect_ratio" chunking
 * method (LinearCrossEntropyOptions docs: each chunk's [rows, C] logits
 * buffer about as large as the [N, D] input): next_pow2(ceil(N /
 * ceil(C / D))), divided by divisor for "aspect_ratio:divisor", at least 1.
 * Pass it as chunk_rows to lce_workspace_size to size a workspace with that
 * page's policy (batch chunks, every class per chunk, an fp32 [C, D] dW
 * accumulator across them). Returns 0 on invalid arguments.
 */
LCE_API int64_t lce_aspect_ratio_chunk_rows(int64_t N, int64_t D, int64_t C, int64_t divisor);

/*
 * Workspace bytes of the plan whose gradient buffer fits buffer_bytes (the
 * rule of the default plan above with that budget; 0 means the default
 * 1 GiB; (size_t)-1 gives the whole [N, C] buffer). The smallest plan keeps
 * min(N, 256) rows and the minimum class chunk (D rounded up to 256, at
 * most every class): a budget below that block's bytes gets that block.
 * Same arguments as lce_workspace_size otherwise; 0 on invalid arguments.
 */
LCE_API size_t lce_workspace_size_for_buffer(int op, int64_t N, int64_t D, int64_t C, int dtype,
                                             int reduction, int grad_dtype, size_t buffer_bytes);

/*
 * Loss only (linear_cross_entropy.py: the chunked forward and the
 * reduction="none" loss-only branch).
 *   X [N, D], W [C, D] of dtype; b [C] of dtype or NULL; target [N] int64.
 *   loss_out: [1] for sum / mean, [N] for none. mean with no valid row
 *   (N == 0 or every row ignored) gives NaN; sum over no row gives 0.
 *   lse_out: NULL or [N] fp32, receives log sum_j exp z[n, j].
 */
LCE_API int lce_forward(const void* X, const void* W, const void* b, const int64_t* target,
                int64_t N, int64_t D, int64_t C, int dtype, int acc_dtype,
                int reduction, int64_t ignore_index,
                float* loss_out, float* lse_out,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * Loss and gradients in one call.
 *   grad_out: sum / mean: NULL (= 1.0) or a device fp32 scalar g; the
 *             gradients are those of the loss times g (the scalar-reduction
 *             ops of linear_cross_entropy.py precompute the gradients and
 *             scale them by grad_output in the backward).
 *             none: required, [N] fp32 per-row upstream gradient; the
 *             gradients are the vector-Jacobian product (grad_output folded
 *             into neg_weight_target).
 *   loss_out: as lce_forward (the forward loss, not multiplied by g).
 *   dX [N, D], dW [C, D], db [C] of grad_dtype; a NULL pointer skips that
 *   gradient (like compute_input_grad / compute_linear_weight_grad /
 *   compute_linear_bias_grad). db is only computed when b is given.
 *   mean with every row ignored gives NaN loss and NaN gradients
 *   (neg_weight_target divides by NaN when the valid count is 0).
 *   A bias of -inf masks classes: they get probability 0, so dW rows and db
 *   entries 0 (any block of them, including whole 256-class tiles).
 */
LCE_API int lce_forward_backward(const void* X, const void* W, const void* b, const int64_t* target,
                         int64_t N, int64_t D, int64_t C, int dtype, int acc_dtype,
                         int reduction, int64_t ignore_index, const float* grad_out,
                         float* loss_out, void* dX, void* dW, void* db, int grad_dtype,
                         void* workspace, size_t ws_bytes, void* stream);

/*
 * Gradients only, from the row log-sum-exp a forward call returned (its
 * lse_out): the backward of reduction="none" in linear_cross_entropy.py,
 * which saves the inputs and recomputes the logits chunk by chunk in its
 * backward. Same arguments as lce_forward_backward, without loss_out and
 * with lse [N] fp32 (device): it must be the lse of these X, W, b.
 * On the bf16 / fp16 path every class's logits are recomputed once
 * (2 N D C flop) and formed straight into gradient tiles, so the call does
 * 6 N D C flop and no forward sweep; an lce_forward + lce_backward pair is
 * the 8 N D C of the page's none op.
 * fp32 inputs do not use lse: the call computes the row statistics itself
 * (its own forward sweep) and returns the same gradients.
 * Workspace: lce_workspace_size(LCE_OP_BACKWARD, ...).
 */
LCE_API int lce_backward(const void* X, const void* W, const void* b, const int64_t* target,
                         const float* lse, int64_t N, int64_t D, int64_t C, int dtype,
                         int acc_dtype, int reduction, int64_t ignore_index, const float* grad_out,
                         void* dX, void* dW, void* db, int grad_dtype, void* workspace,
                         size_t ws_bytes, void* stream);

/*
 * Cross entropy on given logits [N, V] (dtype LCE_F32, LCE_BF16 or
 * LCE_F16); the gradient w_n (softmax - onehot) REPLACES the logits in
 * place, in the logits' own type (a PyTorch wrapper must declare the tensor
 * dirty).
 *   grad_out: as lce_forward_backward (NULL = 1.0 for sum / mean: no extra
 *   scaling; required [N] for none). loss_out: [1] or [N].
 *   Logits of -inf (a masked vocabulary) get probability 0 and gradient 0;
 *   a row's target must then be a finite logit, else its loss is +inf.
 * Liger-Kernel issue #343: loss and gradient in one pass, gradient written
 * into the input buffer, so no separate gradient pass or accumulation runs.
 */
LCE_API int lce_cross_entropy_from_logits(void* logits_inout, const int64_t* target,
                                  int64_t N, int64_t V, int dtype, int reduction,
                                  int64_t ignore_index, const float* grad_out,
                                  float* loss_out, void* workspace, size_t ws_bytes,
                                  void* stream);

/*
 * Allocation-free variant of lce_cross_entropy_from_logits. The source pages
 * have no counterpart; it exists for callers that cannot allocate device
 * memory when they need the loss (code running inside a caching allocator's
 * own hooks, where allocating would re-enter the allocator, or an embedded
 * runtime that reserves a fixed memory budget up front and passes only the
 * buffers it owns). Same arguments and results as
 * lce_cross_entropy_from_logits, except:
 *  - no workspace: the call uses a fixed scratch array inside the library's
 *    device image (256 B + 4 B per row for at most LCE_NOALLOC_MAX_ROWS
 *    rows, i.e. 4 MiB + 256 B), reserved on every GPU that loads the library
 *    until the process exits. N > LCE_NOALLOC_MAX_ROWS returns LCE_ERR_SHAPE.
 *  - device_status: NULL or a device int; after the kernels it receives the
 *    device status bits of this call (1 = a target out of range, 2 = a wait
 *    timed out), copied on the stream.
 *  - every call shares that one array, which keeps the last call's contents
 *    (the call clears the part that must start at zero itself): calls that
 *    overlap on the GPU, on different streams or from different threads,
 *    race and give wrong results. Serialise them on one stream.
 *  - the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current. CUDA loads device
 *    code lazily by default, so that first call may also load the library's
 *    module and reserve the array then. Make that first call before any
 *    stream capture on the device and outside any region where memory must
 *    not be reserved (e.g. at start-up).
 *  - the address is cached per device until the process exits: resetting
 *    the device (cudaDeviceReset or a primary-context reset) while the
 *    library is loaded is not supported by this entry point.
 * The call allocates nothing (no cudaMalloc / cudaFree, no allocating
 * library routine).
 */
#define LCE_NOALLOC_MAX_ROWS (1 << 20)
LCE_API int lce_cross_entropy_from_logits_noalloc(void* logits_inout, const int64_t* target,
                                                  int64_t N, int64_t V, int dtype, int reduction,
                                                  int64_t ignore_index, const float* grad_out,
                                                  float* loss_out, int* device_status, void* stream);

/*
 * Per-class weights and a given mean denominator. Same as lce_forward /
 * lce_forward_backward / lce_backward / lce_cross_entropy_from_logits with
 * two more inputs:
 *  - class_weight: NULL (no class weights) or a device fp32 [C] (or [V])
 *    array (the page's `weight` argument of cross entropy). A valid row n
 *    then has loss weight c_n = class_weight[target_n]:
 *    loss_n = c_n (lse_n - z[n, target_n]), and the gradients carry c_n in
 *    w_n (linear_cross_entropy.py, neg_weight_target: the per-row weight is
 *    the class weight of the target, divided by their sum for mean).
 *  - denominator: NULL, or a device fp32 scalar d that replaces the mean's
 *    denominator (otherwise the number of valid rows, or the sum of c_n over
 *    them with class weights; the page's d). Only reduction mean reads it;
 *    d == 0 gives NaN as usual. It is what a data-parallel shard of one
 *    batch passes: with d the denominator of the WHOLE batch (the sum over
 *    the shards of lce_mean_denominator), each shard's loss and gradients
 *    are its exact share, so summing the shards' loss, dW and db (dX rows
 *    are disjoint) gives the whole batch's mean loss and gradients.
 */
LCE_API int lce_forward_ex(const void* X, const void* W, const void* b, const int64_t* target,
                           const float* class_weight, const float* denominator, int64_t N, int64_t D,
                           int64_t C, int dtype, int acc_dtype, int reduction, int64_t ignore_index,
                           float* loss_out, float* lse_out, void* workspace, size_t ws_bytes,
                           void* stream);
LCE_API int lce_forward_backward_ex(const void* X, const void* W, const void* b, const int64_t* target,
                                    const float* class_weight, const float* denominator, int64_t N,
                                    int64_t D, int64_t C, int dtype, int acc_dtype, int reduction,
                                    int64_t ignore_index, const float* grad_out, float* loss_out,
                                    void* dX, void* dW, void* db, int grad_dtype, void* workspace,
                                    size_t ws_bytes, void* stream);
LCE_API int lce_backward_ex(const void* X, const void* W, const void* b, const int64_t* target,
                            const float* class_weight, const float* denominator, const float* lse,
                            int64_t N, int64_t D, int64_t C, int dtype, int acc_dtype, int reduction,
                            int64_t ignore_index, const float* grad_out, void* dX, void* dW, void* db,
                            int grad_dtype, void* workspace, size_t ws_bytes, void* stream);
LCE_API int lce_cross_entropy_from_logits_ex(void* logits_inout, const int64_t* target,
                                             const float* class_weight, const float* denominator,
                                             int64_t N, int64_t V, int dtype, int reduction,
                                             int64_t ignore_index, const float* grad_out,
                                             float* loss_out, void* workspace, size_t ws_bytes,
                                             void* stream);

/*
 * The mean's denominator of these rows, into the device fp32 scalar
 * denominator_out: the number of rows whose target is neither ignore_index
 * nor out of [0, C), or the sum of class_weight[target] over them when
 * class_weight (device fp32 [C]) is given (linear_cross_entropy.py,
 * neg_weight_target's d). A data-parallel shard sums this over the shards
 * (an all-reduce) and passes the total as `denominator` above. workspace:
 * device, 16-byte aligned, at least 256 bytes. Targets out of range set the
 * device status (lce_read_device_status on this workspace).
 */
LCE_API int lce_mean_denominator(const int64_t* target, const float* class_weight, int64_t N,
                                 int64_t C, int64_t ignore_index, float* denominator_out,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * Gradients times a device scalar, in place: dX[:n_dx], dW[:n_dw] and
 * db[:n_db] (elements of grad_dtype; a NULL pointer or a count of 0 skips
 * that buffer) are multiplied by *grad_out (a device fp32 scalar). The
 * kernel reads *grad_out first and touches nothing when it is exactly 1, so
 * the caller needs no host-side test (and no synchronisation) to skip the
 * pass. This is the backward of the scalar-reduction ops of
 * linear_cross_entropy.py: their forward computes the gradients for an
 * upstream gradient of 1 and their backward multiplies them by
 * grad_output.
 */
LCE_API int lce_scale_gradients(void* dX, int64_t n_dx, void* dW, int64_t n_dw, void* db, int64_t n_db,
                                int grad_dtype, const float* grad_out, void* stream);

/* Human-readable text of a status code (static storage). */
LCE_API const char* lce_status_string(int status);

/*
 * Device-side status of the last call that used this workspace: waits for
 * the stream, then returns LCE_OK, LCE_ERR_TARGET_RANGE or LCE_ERR_TIMEOUT
 * (LCE_ERR_CUDA if the read itself fails). workspace is the device pointer
 * given to that call.
 */
LCE_API int lce_read_device_status(const void* workspace, void* stream);

/*
 * Kernel accounting (used by the benchmark; not needed for the math).
 * lce_launch_count: kernels this library has launched since it was loaded.
 * lce_profile_enable(1): from now on, bracket every launch with CUDA events
 * on the launching stream; lce_profile_enable(0) stops, and
 * lce_profile_reset clears the records. lce_profile_query waits for the
 * recorded events and returns, for one kernel id, the number of launches,
 * their summed duration in ms and (if total_work is not NULL) their summed
 * algorithmic work: flop for the gemm_* kernels (2 M N K per launch), bytes
 * that must cross HBM for the others. lce_kernel_name gives the id's name;
 * ids run from 0 to lce_num_kernel_ids() - 1. Not thread-safe.
 */
LCE_API int64_t lce_launch_count(void);
LCE_API int lce_profile_enable(int on);
LCE_API int lce_profile_reset(void);
LCE_API int lce_profile_query(int kernel_id, int64_t* launches, double* total_ms, double* total_work);
LCE_API const char* lce_kernel_name(int kernel_id);
LCE_API int lce_num_kernel_ids(void);

#ifdef __cplusplus
}
#endif

#endif /* LCE_H_ */
