/*
 * ce.h -- C ABI of the GB300 (sm_103a) softmax cross-entropy library (libce.so).
 *
 * The operation: for a [n_rows, vocab] logits matrix X (row stride ld
 * elements), targets t, optional class weights w, label smoothing eps and a
 * reduction, compute the cross-entropy loss and its gradient with respect to
 * X, writing the gradient over X. Per valid row i (t_i != ignore_index and
 * 0 <= t_i < vocab):
 *
 *   loss_i = (1-eps) * w_{t_i} * (LSE_i - x_{i,t_i})
 *          + (eps/V) * sum_c w_c * (LSE_i - x_ic),   LSE_i = log sum_c exp(x_ic)
 *   dX_ic  = s_i * [ (1-eps) * w_{t_i} * (p_ic - [c == t_i])
 *                    + (eps/V) * (p_ic * W_all - w_c) ],  p = softmax(x_i)
 *
 * with W_all = sum_c w_c, W_y = sum over valid rows of w_{t_i} (the
 * non-ignored count when unweighted), s_i = g / W_y for mean, g for sum and
 * g_i for none. Rows that are not valid contribute loss 0 and gradient 0.
 * Unweighted this is (softmax - (1-eps) onehot - eps/V) * g / N.
 *
 * Sources: Liger-Kernel PR "perf(ce): single-shot dx_y gradient correction
 * - #1268" (review diff: the eps/V term and the weighted true-class term;
 * the #1329 commit message quoted there: dx_y recomputed once in fp32 and
 * stored once, the logits buffer holding the gradient; the #1290 commit
 * message: gradient scaled in place, peak memory one logits tensor);
 * Liger-Kernel PR "perf(flce): drop host syncs that do not feed the
 * computation - #1622" (Summary: normalisers, reductions, device-side
 * grad_output == 1 skip, no host syncs); TransformerEngine PR #2325 "change
 * fused cross entropy backward grad to fp32 and reduce one read/write"
 * (forward saves per-row m, d, X_y and the smoothing sum; backward forms the
 * gradient in fp32 from them).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device (or managed) memory owned by
 *    the caller. The library allocates nothing and keeps no pointer after a
 *    call returns.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Every call
 *    only enqueues work on it and returns; nothing waits for the GPU, except
 *    ce_get_status, which synchronises `stream` explicitly.
 *  - The return code reports host-side argument checks and launch errors.
 *    On an error nothing has been enqueued (argument errors) or the CUDA
 *    error of the failed launch is reported (CE_ERR_CUDA, see
 *    ce_last_cuda_error). Data errors found on the device (a target outside
 *    [0, vocab) that is not ignore_index) set bits in the workspace status
 *    word; such rows are treated as ignored.
 *  - The workspace is scratch owned by the caller, at least
 *    ce_workspace_size() bytes, 256-byte aligned. Calls that share a
 *    workspace must be ordered on one stream (or otherwise serialised).
 *    Its contents need no initialisation.
 */
#ifndef CE_H
#define CE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CE_OK = 0,
    CE_ERR_INVALID_ARG = 1,   /* a pointer, size, stride or enum is invalid */
    CE_ERR_UNSUPPORTED = 2,   /* valid but not supported (e.g. misaligned for the asked variant) */
    CE_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    CE_ERR_WORKSPACE = 4      /* workspace missing, too small or misaligned */
} ce_status;

typedef enum { CE_RED_NONE = 0, CE_RED_MEAN = 1, CE_RED_SUM = 2 } ce_reduction;

/* storage type of the logits / gradient buffer */
typedef enum { CE_DT_F32 = 0, CE_DT_BF16 = 1, CE_DT_F16 = 2 } ce_dtype;

/* bits of the device status word (ce_get_status) */
#define CE_FLAG_TARGET_OUT_OF_RANGE 0x1u /* some target was neither ignore_index nor in [0, vocab) */
#define CE_FLAG_NO_VALID_ROWS 0x2u       /* mean over zero valid rows: loss and gradient set to 0 */
#define CE_FLAG_WAIT_TIMEOUT 0x4u        /* a device-side wait gave up (results invalid) */

/* ce_params.variant: which kernels ce_fwd_bwd uses */
#define CE_VARIANT_AUTO 0   /* the library picks (ce_select_variant) */
#define CE_VARIANT_SPLIT 1  /* ce_forward then ce_backward kernels (row read twice) */
#define CE_VARIANT_FUSED 2  /* fused kernel; CE_ERR_UNSUPPORTED if the rows do not allow it */
#define CE_VARIANT_ROWPASS 3 /* one kernel, each row read twice, the second read from L2 */
#define CE_VARIANT_STREAM 4  /* as ROWPASS, the two passes streamed through a shared-memory
                                ring by bulk copies (any row alignment: the part of a row
                                before its first and after its last 16-byte boundary goes
                                through plain accesses) */
/* bits 8..15 of variant: fused-kernel cluster size override, or CTAs per SM
 * of the row-pass and stream kernels (0 = automatic) */
#define CE_VARIANT_CLUSTER_SHIFT 8
/* the workspace already holds this batch's normalisers from ce_prepare (same
 * target, weights, n_rows and reduction): ce_forward / ce_backward /
 * ce_fwd_bwd skip their own normaliser kernel */
#define CE_VARIANT_PREPARED 0x10000
/* bits 20..30 of variant: stream-kernel tuning (0 = the library's choice):
 * 1 = 16 consumer warps and one CTA per SM, 2 = second pass over each row's
 * chunks in reverse order, 4 = first pass without the L2 evict-last policy,
 * 8 = a cluster of two CTAs per row (each streams half the row),
 * 16 = three CTAs per SM with a smaller ring, 32 = with 16: a cluster of four
 * CTAs per row (each streams a quarter), 64 = with 16, for class-weighted
 * label smoothing on bf16 / f16 rows: the class weights of the second pass
 * bulk-copied into a shared-memory ring (other rows ignore the bit);
 * bits 7..9 of the tuning value (128 x k, k = 0..7): the first k/8 of the
 * first-pass chunks of each row part carry an L2 evict-first hint (useful
 * with 2, where the rows waiting for their second pass exceed the L2);
 * 1024 = with 64 and one CTA per row: the weight ring at two CTAs per SM
 * with a deeper logits ring */
#define CE_VARIANT_TUNE_SHIFT 20

typedef struct ce_params {
    int64_t n_rows;             /* BT >= 0 */
    int64_t vocab;              /* V >= 1 */
    int64_t ld;                 /* row stride of logits in elements, >= vocab; the logits
                                   pointer is aligned to its element size, else
                                   CE_ERR_INVALID_ARG (rows need no other alignment) */
    int64_t ignore_index;       /* targets equal to this are ignored (torch default -100) */
    const float *class_weight;  /* device [vocab] fp32, or NULL for all ones */
    float label_smoothing;      /* eps in [0, 1] */
    int32_t dtype;              /* ce_dtype of the logits buffer */
    int32_t reduction;          /* ce_reduction */
    int32_t target_is_int32;    /* 0: int64 targets, 1: int32 targets */
    int32_t variant;            /* CE_VARIANT_* (ce_fwd_bwd only) */
    int32_t reserved;           /* must be 0 */
    /* Options named next to the method on the Liger-Kernel #1268 page (its CE
     * suite: "class weights, softcap, label smoothing, z-loss"; its dx_y
     * correction keeps the "softcap factors") without a definition there;
     * this library takes the plain ones. Supported by ce_forward /
     * ce_backward and ce_fwd_bwd's stream, row-pass and split paths, and by
     * flce_fwd_bwd (softcap applied to the GEMM's logits); the cluster
     * variants (CE_VARIANT_FUSED, CE_FLCE_CE_CLUSTER) and
     * ce_fwd_bwd_from_host return CE_ERR_UNSUPPORTED with an option set. */
    float softcap;              /* c > 0: every logit becomes c*tanh(x/c); 0 = off */
    float z_loss;               /* lambda >= 0: loss_i += lambda*LSE_i^2 on valid rows */
    float *accuracy;            /* device fp32 [1] or NULL: share of valid rows whose argmax
                                   (first column of the row maximum) is the target */
} ce_params; /* 80 bytes */

/* Library version string, e.g. "ce-gb300 1.0". */
const char *ce_version(void);

/* Human-readable name of a status code. */
const char *ce_status_string(ce_status status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char *ce_last_cuda_error(void);

/*
 * Bytes of workspace the calls below need for these parameters: O(n_rows),
 * independent of vocab (20 bytes per row plus at most 512 bytes).
 */
ce_status ce_workspace_size(const ce_params *p, size_t *bytes);

/*
 * Batch normalisers into the workspace: the number of valid rows, W_y (the
 * target-weight sum, the mean's divisor), W_all (the class-weight sum, used
 * with label smoothing), and the target check (CE_FLAG_TARGET_OUT_OF_RANGE).
 * Every other call runs this itself unless p->variant has
 * CE_VARIANT_PREPARED. One single-block kernel; no host synchronisation
 * (Liger-Kernel #1622: the count and weight sums stay on the device).
 *   target device [n_rows] int64 / int32.
 */
ce_status ce_prepare(const ce_params *p, const void *target, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * Forward: one online-softmax pass over each row (TransformerEngine #2325's
 * forward; the row statistics it saves are the pages' m_d_X_y).
 *   logits    device [n_rows, ld] of p->dtype, read only.
 *   target    device [n_rows] int64 (or int32 with target_is_int32).
 *   loss      device fp32: [1] for mean/sum, [n_rows] for none (written).
 *   stats     device fp32 [n_rows][4] or NULL. Row i gets
 *             {m_i, s_i, x_{i,t_i}, r_i}: m_i = max_c x_ic;
 *             s_i = sum_{c != t_i} exp(x_ic - m_i) (all c on invalid rows),
 *             so that d_i = s_i + exp(x_{i,t_i} - m_i); x_{i,t_i} (0 on invalid
 *             rows); r_i = sum_c w_c (x_ic - m_i). The target term is kept out
 *             of s_i so that the backward forms 1 - p_y = s/d without
 *             cancellation.
 */
ce_status ce_forward(const ce_params *p, const void *logits, const void *target, float *loss,
                     float *stats, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward from saved statistics: reads each row once more and writes the
 * fp32 gradient, rounded once to p->dtype, over it (TransformerEngine
 * #2325's backward; dx_y recomputed once in fp32 and stored once, as in
 * Liger-Kernel #1329).
 *   logits_inout device [n_rows, ld]: logits in, gradient out (columns >= vocab untouched).
 *   stats        device fp32 [n_rows][4] from ce_forward on the same logits.
 *   grad_output  device fp32 [1] for mean/sum, [n_rows] for none, or NULL for 1.0.
 * The logits are consumed: call it once per forward.
 */
ce_status ce_backward(const ce_params *p, void *logits_inout, const void *target,
                      const float *stats, const float *grad_output, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * Forward and backward in one call: loss as ce_forward, gradient as
 * ce_backward, written over the logits. With the fused variant each row is
 * read from HBM once and written once (the row is held in the shared memory
 * of a thread-block cluster); the split variant reads it twice. Peak memory
 * is the logits buffer plus the workspace.
 *   grad_output device fp32 ([1] or [n_rows] for none) or NULL for 1.0. It is
 *               applied inside the gradient pass (single rounding).
 */
ce_status ce_fwd_bwd(const ce_params *p, void *logits_inout, const void *target, float *loss,
                     const float *grad_output, void *workspace, size_t workspace_bytes,
                     void *stream);

/* Largest n_rows ce_fwd_bwd_noalloc accepts (its fixed scratch, about
 * 1.3 MB, is sized for this many rows). */
#define CE_NOALLOC_MAX_ROWS 65536

/*
 * ce_fwd_bwd without a workspace argument, for callers that cannot allocate
 * device memory: hosts that give their extensions no allocator, such as a
 * runtime that reserves all device memory for its own pool up front, or a
 * plugin interface that hands an entry point only its inputs and outputs.
 * The pages this library follows have no counterpart to this entry point.
 * Same arguments, results and error behaviour as ce_fwd_bwd; the caller
 * still passes every input and output buffer.
 *  - Scratch: a fixed array of about 1.3 MB in the library's own device
 *    memory, present on every GPU that loads the library until the process
 *    exits. Nothing is allocated by this call.
 *  - n_rows above CE_NOALLOC_MAX_ROWS returns CE_ERR_WORKSPACE with nothing
 *    enqueued.
 *  - p->variant with CE_VARIANT_PREPARED returns CE_ERR_INVALID_ARG: the
 *    normalisers must be computed by this call, since no caller can run
 *    ce_prepare on the library's scratch.
 *  - The first call on a device looks up the array's device address (a
 *    runtime query with that device current; with lazy module loading the
 *    driver places the array in device memory at that moment), and so does
 *    the first call after the device's context was replaced
 *    (cudaDeviceReset); make those calls before any stream capture. Later
 *    calls change no device memory in use.
 *  - Every call on a device shares the one array, and the array keeps the
 *    last call's contents (each call runs its own normaliser kernel first,
 *    which resets every counter and sum that the later kernels read).
 *    Calls whose GPU work overlaps (different streams, or different host
 *    threads without ordering) race on it: serialise them, e.g. on one
 *    stream. Status bits are read with ce_get_status only through a
 *    caller-provided workspace, so this variant offers none.
 */
ce_status ce_fwd_bwd_noalloc(const ce_params *p, void *logits_inout, const void *target, float *loss,
                             const float *grad_output, void *stream);

/*
 * ce_fwd_bwd for logits that start in host memory: the rows are copied to
 * logits_dev in n_parts blocks on copy_stream, and each block's forward +
 * backward (the stream kernel, with the whole batch's normalisers computed
 * first on `stream`) runs on `stream` as soon as its copy has landed, so the
 * transfer and the kernels overlap (Liger-Kernel #1622 counts the
 * host-device traffic around the loss; this call hides the kernels under
 * it). Same results as ce_fwd_bwd on the device copy.
 *   logits_host  host [n_rows, ld] of p->dtype, page-locked (cudaHostAlloc
 *                or registered) for the copies to be asynchronous; it must
 *                stay valid and unchanged until `stream` has passed this call.
 *   logits_dev   device [n_rows, ld]: receives the logits, then the gradient.
 *   target, loss, grad_output, workspace: as in ce_fwd_bwd.
 *   copy_stream  a stream other than `stream` (not the legacy default
 *                stream, which would serialise the two); it first waits for
 *                the work already queued on `stream`.
 *   n_parts      >= 1 blocks of rows (clamped to n_rows); 8 is a good choice.
 * p->variant must be 0; softcap, z-loss and accuracy give
 * CE_ERR_UNSUPPORTED. Allocates no device memory; creates and releases CUDA
 * events.
 */
ce_status ce_fwd_bwd_from_host(const ce_params *p, const void *logits_host, void *logits_dev, const void *target,
                               float *loss, const float *grad_output, void *workspace, size_t workspace_bytes,
                               void *stream, void *copy_stream, int32_t n_parts);

/*
 * Scale a gradient already written with grad_output = 1 (ce_fwd_bwd with
 * grad_output NULL) by the grad_output that arrives later: row i is
 * multiplied by g ([1]) or g_i ([n_rows], reduction none). With a [1]
 * grad_output equal to 1.0 every block returns after reading it (the
 * device-side skip of Liger-Kernel #1622). The product is rounded again to
 * the buffer dtype; callers that know grad_output before the gradient pass
 * should pass it to ce_fwd_bwd / ce_backward instead (one rounding).
 *   grad_inout device [n_rows, ld] of p->dtype (columns < vocab are scaled).
 */
ce_status ce_scale_grad(const ce_params *p, void *grad_inout, const float *grad_output,
                        void *stream);

/*
 * The fused-kernel launch the library picks for these parameters (host
 * query, no GPU work): cluster size, CTAs per cluster row slice, clusters
 * in the grid and slice bytes per CTA. Returns CE_ERR_UNSUPPORTED when the
 * fused kernel cannot take these rows (ce_fwd_bwd then runs split).
 */
ce_status ce_fused_plan(const ce_params *p, int32_t *cluster_size, int32_t *n_clusters,
                        int32_t *ctas_per_sm, int64_t *slice_bytes);

/*
 * The kernel path ce_fwd_bwd takes for p->variant == CE_VARIANT_AUTO (host
 * query, no GPU work): one of the CE_VARIANT_* paths in *variant. `logits`
 * is only inspected for alignment.
 */
ce_status ce_select_variant(const ce_params *p, const void *logits, int32_t *variant);

/*
 * Self-test of the device-side bounded wait every kernel of this library
 * uses on its mbarriers: one block waits on an mbarrier that nothing ever
 * arrives on, gives up after about limit_ns nanoseconds, and writes
 * CE_FLAG_WAIT_TIMEOUT to *device_flags (device uint32). Lets a caller
 * check that a failed wait ends with a status instead of a hang, and that
 * the context stays usable. limit_ns in [1e6, 5e9].
 */
ce_status ce_selftest_wait_timeout(uint64_t limit_ns, uint32_t *device_flags, void *stream);

/*
 * Synchronises `stream`, then copies the workspace status word (CE_FLAG_*
 * bits of the most recent call that used this workspace) to *flags. The
 * only call that waits for the GPU.
 */
ce_status ce_get_status(const void *workspace, uint32_t *flags, void *stream);

/* ------------------------------------------------------------------------
 * Fused-linear cross-entropy (Liger-Kernel PR "perf(flce): drop host syncs
 * that do not feed the computation - #1622": logits = hidden x weight^T
 * formed chunk by chunk, cross-entropy forward and backward on each chunk,
 * then the gradient GEMMs; the full logits are never materialised and the
 * host never waits).
 * ------------------------------------------------------------------------ */

/* CE_GEMM_* output modes of ce_gemm_bf16 */
#define CE_GEMM_F32_STORE 0   /* D = A B (+ bias[n]) in fp32 */
#define CE_GEMM_F32_ACCUM 1   /* D += A B in fp32 */
#define CE_GEMM_BF16_STORE 2  /* D = A B rounded once to bf16 */

/*
 * D[M,N] = A[M,K] x B[K,N] on the tcgen05 tensor cores: bf16 operands,
 * fp32 accumulation in tensor memory, 128 x 256 tiles fed by TMA. The GEMM
 * the fused-linear path is built from, exposed for direct use and testing.
 *   A  device bf16. a_mn_major = 0: stored [M, K] row-major (row stride
 *      lda >= K); 1: stored [K, M] (lda >= M).
 *   B  device bf16. b_mn_major = 0: stored [N, K] (ldb >= K); 1: stored
 *      [K, N] (ldb >= N).
 *   D  device fp32 or bf16 (out_kind) [M, N], row stride ldd elements.
 *   bias device fp32 [N] added in CE_GEMM_F32_STORE mode, or NULL.
 * Base pointers (A, B and bias) 16-byte aligned and lda/ldb multiples of 8
 * (TMA rules), else CE_ERR_INVALID_ARG.
 */
ce_status ce_gemm_bf16(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int32_t a_mn_major,
                       const void *B, int64_t ldb, int32_t b_mn_major, int32_t out_kind, void *D,
                       int64_t ldd, const float *bias, void *stream);

/* ce_params.variant of flce_fwd_bwd (bits, 0 = the defaults):
 * CE_FLCE_DENSE runs every row through every GEMM instead of compacting the
 * valid rows first; CE_FLCE_CE_CLUSTER runs each chunk's cross-entropy with
 * the cluster kernel (row held in shared memory) instead of the default:
 * row statistics formed in the logits GEMM's epilogue, then one streaming
 * map from the fp32 logits to dZ. */
#define CE_FLCE_DENSE 1
#define CE_FLCE_CE_CLUSTER 2

/* Workspace bytes of flce_fwd_bwd for these sizes (the fp32 logits chunk,
 * the bf16 logits-gradient chunk and the cross-entropy workspace; with
 * compaction also a compacted copy of hidden, BT x H bf16, and 24 bytes per
 * row of maps, targets and grad_output). */
ce_status flce_workspace_size(const ce_params *p, int64_t hidden_dim, int64_t chunk_rows, size_t *bytes);

/*
 * Fused-linear cross-entropy forward and backward.
 *   p            n_rows = BT, vocab = V, dtype = CE_DT_BF16 (hidden and
 *                weight), ignore_index, class_weight, label_smoothing,
 *                reduction; variant a combination of the CE_FLCE_*
 *                bits (else CE_ERR_INVALID_ARG); ld is ignored.
 *   hidden       device bf16 [BT, H] row-major.
 *   weight       device bf16 [V, H] row-major (the lm head).
 *   bias         device fp32 [V] (16-byte aligned) or NULL.
 *   target       device [BT] int64 / int32.
 *   loss         device fp32 [1] (mean/sum) or [BT] (none).
 *   grad_output  device fp32 [1] / [BT] or NULL for 1.0, applied to dZ.
 *   grad_hidden  device bf16 [BT, H] (written).
 *   grad_weight  device fp32 [V, H] (written: the sum over all chunks).
 *   grad_bias    device fp32 [V] or NULL (written when bias is given).
 *   chunk_rows   rows per chunk (> 0); the logits of one chunk,
 *                chunk_rows x V fp32, are the largest intermediate.
 * Per chunk: Z = hidden_c W^T (+ b) in fp32; the fused cross-entropy kernel
 * turns Z into dZ (bf16, one rounding) with the batch's normalisers;
 * grad_hidden_c = dZ W; grad_weight (+)= dZ^T hidden_c. H and V multiples
 * of 8.
 * Ignored rows (target == ignore_index, or out of range: status bit) add
 * nothing to the loss or grad_weight and get zero grad_hidden rows. By
 * default they are also skipped, without a host sync (the device-side form
 * of Liger-Kernel PR #1554's ignored-row skip): one kernel gathers the valid
 * rows of hidden and their targets to the front of the workspace, and the
 * GEMMs and the chunk kernels read the valid-row count from device memory,
 * so chunks and tiles past it do no work. The host still launches every
 * chunk. Results equal the dense path's up to the order of fp32 sums.
 */
ce_status flce_fwd_bwd(const ce_params *p, int64_t hidden_dim, const void *hidden, const void *weight,
                       const float *bias, const void *target, float *loss, const float *grad_output,
                       void *grad_hidden, float *grad_weight, float *grad_bias, int64_t chunk_rows,
                       void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CE_H */
