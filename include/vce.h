/*
 * vce.h -- C ABI of the GB300 (sm_103a) vocabulary cross-entropy library (libvce.so).
 *
 * Two forms of large-vocabulary softmax cross entropy, neither of which keeps a
 * full-precision logit or gradient matrix:
 *
 *   logits form  ce_forward / ce_backward
 *       Follows Transformer Engine's parallel_cross_entropy (API card
 *       "Implementation:NVIDIA TransformerEngine Cross Entropy", sections
 *       "Signature" and "I/O Contract": inp, target, label_smoothing,
 *       reduce_loss, ignore_idx = -100, FP32 loss for BF16/FP32 input), minus the
 *       process group.  Forward saves per-row statistics (max, log-sum-exp)
 *       instead of the derivative, and backward rebuilds dlogits from them
 *       (pull request "Minimize the memory usage of the fused cross entropy
 *       kernel", section "Changes"); backward may write dlogits over the logits
 *       (same pull request, the destructive buffer-reuse mode).
 *
 *   linear form  lce_forward / lce_backward
 *       Loss from hidden states X [N, H] and classifier W [V, H]; the logits
 *       X W^T are produced tile by tile and never stored (Cut Cross-Entropy
 *       package card, "what_it_does"; Liger pull request "Add SM100
 *       tensor-parallel fused scaled cross entropy", sections "Summary",
 *       "Implementation": forward GEMM fused with NLL/LSE, backward = logits
 *       recomputation, dX and dW).
 *
 * Common conventions
 *   - Every pointer argument is a DEVICE pointer unless said otherwise; the
 *     caller owns every buffer and the stream.  The library never allocates,
 *     frees or synchronises, so calls can be captured in a CUDA graph once
 *     each entry point has run eagerly on the device: the first call of a
 *     kernel on a device may set that kernel's shared-memory limit, which is
 *     not a stream operation.
 *   - ``stream`` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - The math: for a row n with logits z[n, 0..V) and target y_n,
 *         lse_n  = log sum_v exp(z[n, v])
 *         loss_n = (1 - eps) (lse_n - z[n, y_n]) + eps (lse_n - (1/V) sum_v z[n, v])
 *         dz[n, v] = g_n (exp(z[n, v] - lse_n) - (1 - eps) [v = y_n] - eps / V)
 *     with eps = label_smoothing spread over all V classes (the convention of
 *     torch.nn.functional.cross_entropy, which the API card names as the op the
 *     function replaces).  Loss and gradient arithmetic is FP32 whatever the
 *     input dtype ("Description": "Loss and gradient computation in FP32").
 *   - Rows whose target equals ``ignore_idx`` give loss 0 and gradient 0.
 *   - ``reduce_loss``: VCE_REDUCE_MEAN (1): the loss is sum_n loss_n / N_v,
 *     N_v = number of rows whose target is not ignore_idx (NaN when N_v = 0),
 *     and backward uses g_n = grad_output[0] / N_v.  VCE_REDUCE_SUM (2): the
 *     loss is sum_n loss_n and g_n = grad_output[0].  VCE_REDUCE_NONE (0): the
 *     loss is per row and g_n = grad_output[n].  Other values are rejected.
 *   - Host-detectable errors return a status before any launch and write
 *     nothing.  Errors found on the device are ORed into ``*dev_status`` (a
 *     device int the caller zeroes and reads after its own synchronisation;
 *     may be NULL): VCE_DEVSTATUS_BAD_TARGET for a target outside [0, V) that
 *     is not ignore_idx (that row's loss is NaN and its gradient row 0),
 *     VCE_DEVSTATUS_TIMEOUT when a wait of a tensor-core or copy pipeline gave
 *     up (the outputs are then incomplete).
 *   - The library runs on compute capability 10.3 (GB300) only; on any other
 *     device every compute call returns VCE_ERR_ARCH.
 */
#ifndef VCE_H
#define VCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vce_status {
    VCE_OK = 0,
    VCE_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride/option */
    VCE_ERR_DTYPE = 2,       /* unsupported dtype code */
    VCE_ERR_ALIGN = 3,       /* pointer or leading dimension violates the stated alignment */
    VCE_ERR_WORKSPACE = 4,   /* workspace pointer NULL or smaller than required */
    VCE_ERR_ARCH = 5,        /* current device is not compute capability 10.3 */
    VCE_ERR_CUDA = 6         /* a CUDA runtime/driver call or a launch failed */
} vce_status;

typedef enum vce_dtype {
    VCE_BF16 = 0,
    VCE_F32 = 1
} vce_dtype;

#define VCE_DEVSTATUS_BAD_TARGET 1
#define VCE_DEVSTATUS_TIMEOUT 2
/* Set only by a library built with -DVCE_BOUNDS_CHECK (a debugging build; see
 * vce_bounds_check_build): an address a kernel computed fell outside the
 * element range, row or buffer it belongs to, or a bulk or tensor copy was not
 * 16-byte aligned; that access was skipped instead of made. */
#define VCE_DEVSTATUS_BOUNDS 4

/* reduce_loss values */
#define VCE_REDUCE_NONE 0 /* per-row loss */
#define VCE_REDUCE_MEAN 1 /* sum over rows / N_v (the API card's reduce_loss=True) */
#define VCE_REDUCE_SUM 2  /* sum over rows (the Cut Cross-Entropy card's reduction='sum') */

/* Human-readable name of a vce_status value (static string, never NULL). */
const char* vce_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int vce_version(void);

/* Number of kernels this library has launched in this process so far (a host-side
 * counter; diagnostics, e.g. counting the launches of a timed region). */
unsigned long long vce_kernel_launches(void);

/* 1 when this library was built with -DVCE_BOUNDS_CHECK: every kernel then checks
 * the addresses it computes (row element ranges, 16-byte vector and bulk-copy
 * alignment, tensor-copy coordinates, output and workspace indices) before it
 * uses them, ORs VCE_DEVSTATUS_BOUNDS into *dev_status and skips the access
 * when one fails.  It stands in for a memory checker where none can run, and
 * is slower; the normal build returns 0 and checks nothing. */
int vce_bounds_check_build(void);

/* ------------------------------------------------------------------------ */
/* logits form                                                              */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of device workspace ce_forward and ce_forward_backward need: n_rows * 4
 * (per-row losses, rounded up to 256 B) when reduce_loss != 0, else 0.
 */
size_t ce_workspace_size(int64_t n_rows, int64_t vocab, int reduce_loss);

/*
 * Forward of the logits form (API card "Signature"; pull request #3273
 * "Changes": single-GPU path, one kernel computes the loss and the statistics).
 *
 *   logits      [n_rows, vocab] row-major, element (n, v) at logits[n * row_stride + v];
 *               dtype BF16 or F32; must be aligned to its element size.  The
 *               (B, SQ, V) and (SQ, B, V) layouts are both passed flattened to
 *               n_rows = B * SQ rows, targets flattened in the same order.
 *   row_stride  elements between rows, >= vocab.
 *   target      [n_rows] int64.
 *   label_smoothing in [0, 1].
 *   loss        F32: [1] when reduce_loss != 0, else [n_rows] (0 for ignored rows).
 *   stats       F32 [n_rows, 2]: (max_v z, lse) per row, the only state backward
 *               needs.  Rows with target == ignore_idx are never read and get (0, 0).
 *   n_valid     int64 [1]: N_v, written when non-NULL; required for VCE_REDUCE_MEAN
 *               (backward reads it).
 *   ws/ws_bytes workspace of at least ce_workspace_size(...) bytes, 256-B aligned
 *               (may be NULL when that size is 0).
 */
vce_status ce_forward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                      int64_t row_stride, const int64_t* target, float label_smoothing,
                      int reduce_loss, int64_t ignore_idx, float* loss, float* stats,
                      int64_t* n_valid, void* ws, size_t ws_bytes, int* dev_status,
                      void* stream);

/*
 * Backward of the logits form: rebuilds dlogits from the logits and the saved
 * statistics (pull request #3273 "Changes" and its sequence diagram: backward
 * reads the saved input, targets, stats and grad_output).
 *
 *   logits, dtype, n_rows, vocab, row_stride, target, label_smoothing,
 *   reduce_loss, ignore_idx: as passed to ce_forward.
 *   stats       F32 [n_rows, 2] from ce_forward (only the lse column is read).
 *   n_valid     int64 [1] from ce_forward (read only for VCE_REDUCE_MEAN).
 *   grad_output F32 [1] when reduce_loss != 0, else [n_rows].
 *   dlogits     same dtype and layout (row_stride) as logits; MAY EQUAL logits,
 *               in which case the logits are overwritten by their gradient (the
 *               pull request's destructive mode: no extra buffer).  Any other
 *               overlap is undefined.  Its address must have the same offset
 *               modulo 16 bytes as logits (else VCE_ERR_ALIGN); buffers of
 *               equal layout from one allocator always do.  Ignored rows are
 *               written as zeros.
 */
vce_status ce_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                       int64_t row_stride, const int64_t* target, const float* stats,
                       const int64_t* n_valid, const float* grad_output,
                       float label_smoothing, int reduce_loss, int64_t ignore_idx,
                       void* dlogits, int* dev_status, void* stream);

/*
 * Forward and backward of the logits form in one pass, for a caller that knows
 * the upstream gradient before the loss is computed (the usual training step:
 * the loss is the objective and grad_output is 1 or a loss scale).  This takes
 * the pull request's destructive buffer reuse ("Minimize the memory usage of
 * the fused cross entropy kernel", opt-in mode that reuses the input storage)
 * one step further: each logit row is read from HBM once, its statistics are
 * formed, and the same row, still in L2, is turned into its gradient and
 * written once, so the pair costs one read and one write per logit instead of
 * two reads and one write.
 *
 *   Arguments are those of ce_forward and ce_backward combined; the results are
 *   those of ce_forward followed by ce_backward with the same grad_output (loss,
 *   stats, n_valid, dlogits): bit for bit for rows of at most 16 KiB, BF16
 *   rows of 48 to 64 KiB and of 112 to 448 KiB, and FP32 rows of 16 to 56 KiB
 *   and of 64 to 400 KiB, where both calls give every thread the same elements
 *   in the same order; for other rows this call splits a row's sum
 *   differently, so lse and the loss agree to FP32 rounding (row maxima,
 *   n_valid and ignored rows exactly).  BF16 rows above 448 KiB and FP32 rows
 *   above 400 KiB are each split between the two CTAs of a cluster on two
 *   SMs.  For rows above 16 KiB the
 *   call uses up to about 226 KiB of shared memory per SM and raises its
 *   kernels' dynamic shared-memory limit on the first call on each device.  A
 *   timeout of its internal copy pipeline (not expected) sets
 *   VCE_DEVSTATUS_TIMEOUT and leaves the outputs undefined.  dlogits MAY EQUAL
 *   logits (in place), with the same 16-byte offset rule as ce_backward.
 *   grad_output F32 [1] when reduce_loss != 0, else [n_rows].
 *   ws/ws_bytes: ce_workspace_size(n_rows, vocab, reduce_loss) bytes.
 */
vce_status ce_forward_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                               int64_t row_stride, const int64_t* target, float label_smoothing,
                               int reduce_loss, int64_t ignore_idx, const float* grad_output,
                               float* loss, float* stats, int64_t* n_valid, void* dlogits, void* ws,
                               size_t ws_bytes, int* dev_status, void* stream);

/*
 * ce_forward for callers that cannot allocate device memory.  The pages have no
 * counterpart of this call; it exists for callers that are handed only their
 * inputs and outputs (a plugin inside another runtime's execution plan, or a
 * deployment that forbids device allocation once it has started) and so cannot
 * provide the workspace ce_forward asks for when reduce_loss != 0.
 *
 * Arguments and results are those of ce_forward without ws/ws_bytes.  The
 * per-row loss scratch is a fixed array compiled into the library
 * (VCE_NOALLOC_MAX_ROWS floats = 4 MiB), present on every GPU that loads the
 * library until the process exits.  With reduce_loss != 0, n_rows above
 * VCE_NOALLOC_MAX_ROWS returns VCE_ERR_WORKSPACE before any launch.  The call
 * allocates and frees nothing.  The first call on each device looks up the
 * array's device address (with that device current); make that first call
 * before any stream capture.  The address is cached with the id of its
 * context, so the first call after cudaDeviceReset looks it up again (make
 * that one before any capture too).  All calls share the array: each call writes
 * every slot it reads, so nothing needs clearing, but calls that overlap on
 * the GPU (different streams or host threads) race on it.
 */
#define VCE_NOALLOC_MAX_ROWS 1048576
vce_status ce_forward_noalloc(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                              int64_t row_stride, const int64_t* target, float label_smoothing,
                              int reduce_loss, int64_t ignore_idx, float* loss, float* stats,
                              int64_t* n_valid, int* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* linear form (X, W and the gradients are BF16; accumulation is FP32)      */
/* ------------------------------------------------------------------------ */

/* The dZ slab cap that max_slab_bytes = 0 selects: 256 MiB. */
#define VCE_DEFAULT_SLAB_BYTES ((size_t)256 << 20)
/* max_slab_bytes for no cap: one slab covers the whole vocabulary. */
#define VCE_SLAB_UNCAPPED ((size_t)-1)

/*
 * Bytes of device workspace lce_forward and lce_backward need.
 *
 * Backward recomputes the logits one vocabulary slab at a time and keeps that
 * slab's gradient dZ [n, slab] in BF16; ``max_slab_bytes`` caps that buffer.
 * 0 selects VCE_DEFAULT_SLAB_BYTES (256 MiB): at N = H = 4096, V = 131072 that
 * is four slabs, whose step measured 0.2-0.4% slower than one slab's with 1.0
 * GB less workspace; at 8192 tokens of H = 2048-7168, V = 129280-202048 it is
 * 8-13 slabs and 3.4-4.3% slower, with 336-503 MB against 2.1-3.8 GB (each
 * extra slab adds an FP32 pass over the dX partials and its own GEMM
 * launches).  VCE_SLAB_UNCAPPED lets one slab cover the whole
 * vocabulary (an N x V BF16 buffer).  The slab is at least 256 vocabulary
 * rows.  dX = dZ W has few output tiles, so its vocabulary
 * range is cut into 1-4 chunks (chosen from the tile count and the SM count
 * of the current device); unless one slab and one chunk let dX be written
 * directly, each chunk keeps an FP32 [n, h] partial sum inside the workspace.
 * The forward part holds per-tile softmax partials (16 B per token per 256
 * vocabulary ids: max, sum of exp, sum of logits, entropy term), the
 * per-token target logit and, when reducing, the per-token losses.  Both
 * parts end with 256 bytes for the GEMMs' work-unit counter, which the
 * library zeroes with a one-thread kernel on the call's stream before each
 * GEMM.  The same size passed to lce_backward on the same device selects the
 * same slab.
 */
size_t lce_workspace_size(int64_t n, int64_t h, int64_t v, int reduce_loss,
                          size_t max_slab_bytes);

/*
 * Forward of the linear form: loss and lse from X and W without storing X W^T
 * (Cut Cross-Entropy card "what_it_does"; Liger pull request "Implementation",
 * "Forward": classifier GEMM whose epilogue folds each vocabulary tile into a
 * running max and sum).
 *
 *   X  BF16 [n, h] row-major; W BF16 [v, h] row-major.  h must be a multiple of 8
 *      and both pointers 16-byte aligned (tensor-memory-access descriptors).
 *   target int64 [n].
 *   loss   F32 [1] (reduce_loss) or [n].
 *   lse    F32 [n]: log-sum-exp of every row (ignored rows included), the state
 *          lce_backward needs.
 *   entropy F32 [n] or NULL: per-token entropy of the softmax,
 *          H_n = -sum_v p_v log p_v = lse_n - sum_v p_v z[n, v], for every row
 *          (the Liger pull request's optional entropy output, "Summary").
 *   n_valid int64 [1], written when non-NULL; required for VCE_REDUCE_MEAN.
 *   ws/ws_bytes at least lce_workspace_size(n, h, v, reduce_loss, *) bytes,
 *          256-B aligned.
 */
vce_status lce_forward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                       const int64_t* target, float label_smoothing, int reduce_loss,
                       int64_t ignore_idx, float* loss, float* lse, float* entropy,
                       int64_t* n_valid, void* ws, size_t ws_bytes, int* dev_status,
                       void* stream);

/*
 * Backward of the linear form (Liger pull request "Implementation", "Backward":
 * dZ from recomputed logits, then dX = dZ W and dW = dZ^T X with FP32
 * accumulation).
 *
 *   X, W, n, h, v, target, label_smoothing, reduce_loss, ignore_idx: as forward.
 *   lse        F32 [n] from lce_forward.
 *   n_valid    int64 [1] from lce_forward (read only for VCE_REDUCE_MEAN).
 *   grad_output F32 [1] (reduce_loss != 0) or [n].
 *   dX         BF16 [n, h], 16-byte aligned; fully written.
 *   dW         BF16 [v, h], 16-byte aligned; fully written.
 *   ws/ws_bytes at least lce_workspace_size(n, h, v, reduce_loss, 0, a cap or
 *              VCE_SLAB_UNCAPPED); the largest slab that fits in ws_bytes is used.
 */
vce_status lce_backward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                        const int64_t* target, const float* lse, const int64_t* n_valid,
                        const float* grad_output, float label_smoothing, int reduce_loss,
                        int64_t ignore_idx, void* dX, void* dW, void* ws, size_t ws_bytes,
                        int* dev_status, void* stream);

/*
 * Targets for causal language modelling with token shifting (Cut
 * Cross-Entropy package card, "what_it_does": optional support for
 * token-shifting).  With sequences of ``seq_len`` positions stored one after
 * another (the (B, SQ) layout flattened), position t of a sequence is to be
 * scored against the label at t + 1 of the same sequence:
 *     shifted[i] = target[i + 1], or ignore_idx where i is the last position
 *     of its sequence (i mod seq_len == seq_len - 1) or of the array.
 * The result is passed as ``target`` to any entry point above; the row
 * layout of the logits / hidden states does not change, and the last
 * position of every sequence contributes no loss and no gradient.
 *
 *   target   int64 [n] (device); shifted int64 [n] (device), not overlapping target.
 *   seq_len  >= 1.  A trailing partial sequence follows the same rule.
 */
vce_status shift_targets(const int64_t* target, int64_t n, int64_t seq_len, int64_t ignore_idx,
                         int64_t* shifted, void* stream);

/* ------------------------------------------------------------------------ */
/* diagnostics                                                              */
/* ------------------------------------------------------------------------ */

/*
 * Failure-detection self-test of the bounded wait that every tensor-core
 * pipeline wait of lce_forward / lce_backward uses.  The pages have no
 * counterpart of this call.  One thread waits on an mbarrier that nothing
 * arrives on; after ``timeout_ns`` (1 ns .. 2 s) the wait gives up and
 * VCE_DEVSTATUS_TIMEOUT is ORed into *dev_status (device int).  When
 * ``waited_ns`` (device, may be NULL) is given it receives the measured wait.
 * The kernel returns normally and the context stays usable.
 */
vce_status vce_selftest_wait_timeout(uint64_t timeout_ns, int* dev_status,
                                     unsigned long long* waited_ns, void* stream);

/*
 * Failure-detection self-tests of the timeout exits of the two pipelined
 * kernels.  The pages have no counterpart of these calls.  Each runs the real
 * kernel with every wait limited to ``timeout_ns`` (1 us .. 2 s) and its work
 * held back, so that each role's first wait runs out while no copy or MMA is
 * in flight; the kernel then takes its timeout exit (abort flag shared by the
 * roles, drain of anything issued, tensor memory released) and ORs
 * VCE_DEVSTATUS_TIMEOUT into *dev_status.  The kernels return normally and
 * the context stays usable; the numeric outputs of these calls are undefined.
 *
 * vce_selftest_lce_forward_timeout: lce_forward's tensor-core GEMM, whose
 *   work-unit scheduler publishes no unit.  Arguments as lce_forward with
 *   label_smoothing 0, VCE_REDUCE_NONE, ignore_idx -100, no entropy or n_valid;
 *   ws of lce_workspace_size(n, h, v, VCE_REDUCE_NONE, 0) bytes.
 * vce_selftest_ce_fused_timeout: ce_forward_backward's ring kernel, whose copy
 *   producer issues no copy.  Arguments as ce_forward_backward with
 *   label_smoothing 0, VCE_REDUCE_NONE (grad_output [n_rows]), ignore_idx -100,
 *   no n_valid or workspace.  Only rows of more than 16 KiB go through the
 *   ring; shorter rows return VCE_ERR_INVALID_ARG.
 */
vce_status vce_selftest_lce_forward_timeout(const void* X, const void* W, int64_t n, int64_t h,
                                            int64_t v, const int64_t* target, uint64_t timeout_ns,
                                            float* loss, float* lse, void* ws, size_t ws_bytes,
                                            int* dev_status, void* stream);
vce_status vce_selftest_ce_fused_timeout(const void* logits, int dtype, int64_t n_rows,
                                         int64_t vocab, int64_t row_stride, const int64_t* target,
                                         const float* grad_output, uint64_t timeout_ns, float* loss,
                                         float* stats, void* dlogits, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VCE_H */
