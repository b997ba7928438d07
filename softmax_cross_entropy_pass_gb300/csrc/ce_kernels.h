// ce_kernels.h -- host-visible kernel argument blocks and launchers of the
// cross-entropy library (shared by the C-ABI layer and the kernel files).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ce.h"

namespace ce {

struct WsCtl;

constexpr int kPrepThreads = 256;
constexpr int kRowThreads = 256;
constexpr int kRowpassThreads = 512;

struct PrepArgs {
    const void *target;
    int tgt32;
    int reduction;
    int64_t n_rows, vocab, ignore_index;
    const float *weight;
    int need_w_all;
    WsCtl *ctl;
};

// arguments of the split-path row kernels (stats, grad)
struct RowArgs {
    const void *logits;        // stats kernel input
    void *grad;                // grad kernel in/out (in place)
    int64_t n_rows, vocab, ld;
    const void *target;
    int tgt32;
    int reduction;
    int64_t ignore_index;
    const float *weight;
    float eps;
    const float *grad_output;  // NULL = 1.0
    float *loss;               // [1] or [n_rows]
    float *stats;              // [n_rows][4] (stats: out, grad: in)
    float *row_loss;           // workspace per-row loss (mean / sum)
    WsCtl *ctl;
    float softcap;             // > 0: logits become c tanh(x / c)
    float z_loss;              // lambda of lambda LSE^2
    float *accuracy;           // token accuracy out [1] or NULL
    int32_t no_finalize;       // stream kernel: leave the batch reduction to a later kernel
};

struct ScaleArgs {
    void *grad;
    int64_t n_rows, vocab, ld;
    const float *grad_output;
    int per_row;
};

// fused single-read forward + backward (thread-block cluster per row)
struct FusedArgs {
    void *x;                   // logits in, gradient out
    int64_t n_rows, vocab, ld;
    const void *target;
    int tgt32;
    int reduction;
    int64_t ignore_index;
    const float *weight;
    float eps;
    const float *grad_output;
    float *loss;
    float *row_loss;
    WsCtl *ctl;
    int64_t slice_elems;       // columns per CTA of a cluster (multiple of 8)
    int32_t chunk_bytes;       // bulk-copy chunk (multiple of 16)
    int32_t n_chunks;          // chunks per slice (<= kMaxChunks)
    void *out;                 // gradient destination (== x for in place)
    int64_t ld_out;            // row stride of out in elements of the output dtype
    int32_t finalize;          // 1: the last CTA reduces the row losses into loss[0]
    // Device-side row count (NULL: n_rows). The kernel handles rows
    // [0, min(n_rows, round_up(max(0, *row_limit - row_limit_off), 64))):
    // rows past the count but inside its 64-row block are expected to carry
    // ignored targets and come out as zero gradient rows, so a GEMM that
    // reduces over them in 64-row steps sees zeros.
    const int *row_limit;
    int64_t row_limit_off;
};

constexpr int kFusedConsumerWarps = 8;
constexpr int kFusedThreads = (kFusedConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kMaxChunks = 32;
constexpr int kMaxCluster = 16;

// smem bytes of the fused kernel besides the row slice
constexpr int kFusedSmemFixed = 2048;

cudaError_t launch_prep(const PrepArgs &a, cudaStream_t s);
cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int *flags, cudaStream_t s);
cudaError_t launch_stats(const RowArgs &a, int dtype, int mode, int grid, cudaStream_t s);
cudaError_t launch_grad(const RowArgs &a, int dtype, int mode, int grid, cudaStream_t s);
// true when softcap, z-loss or token accuracy is asked for (row-pass / split kernels only)
inline bool row_features(const RowArgs &a) { return a.softcap > 0.f || a.z_loss > 0.f || a.accuracy; }
cudaError_t launch_scale(const ScaleArgs &a, int dtype, int grid, cudaStream_t s);
// one-kernel forward + backward, two passes per row (second from L2)
cudaError_t launch_rowpass(const RowArgs &a, int dtype, int mode, int ctas_per_sm, cudaStream_t s);
// the same two passes streamed through a shared-memory ring by bulk copies
// (16-byte aligned rows only)
// loss[0] = sum of row_loss[0, n) in fp64 (divided by the workspace's W_y for
// mean), one block; for the row kernels launched with no_finalize.
cudaError_t launch_reduce_row_losses(const float *row_loss, int64_t n, int reduction, const WsCtl *ctl, float *loss,
                                     cudaStream_t s);
cudaError_t launch_stream(const RowArgs &a, int dtype, int mode, int ctas_per_sm, int tune, bool after_prep,
                          cudaStream_t s);
// The forward only (row statistics and losses) by the stream kernel's first
// pass: every row read once through the bulk-copy ring, one CTA per row.
// a.grad holds the logits (read only), a.stats the [n_rows][4] output or
// NULL. `mode` 0 or 1 (no class-weighted smoothing), no options.
cudaError_t launch_stream_forward(const RowArgs &a, int dtype, int mode, bool after_prep, cudaStream_t s);

// Fused kernel plan / launch. `mode`: 0 no smoothing, 1 smoothing, 2 weighted smoothing.
struct FusedPlan {
    int cluster;
    int n_clusters;
    int ctas_per_sm;
    int64_t slice_elems;
    int chunk_bytes;
    int n_chunks;
    size_t smem_bytes;
};
cudaError_t fused_plan(int dtype, int mode, int64_t n_rows, int64_t vocab, int cluster_override,
                       FusedPlan *plan, bool *supported);
cudaError_t launch_fused(const FusedArgs &a, const FusedPlan &plan, int dtype, int mode,
                         cudaStream_t s, bool after_prep);
// fp32 logits in, bf16 gradient out to a separate buffer (fused-linear chunks)
cudaError_t launch_fused_f32_to_bf16(const FusedArgs &a, const FusedPlan &plan, int mode,
                                     cudaStream_t s);
cudaError_t fused_plan_f32_to_bf16(int mode, int64_t n_rows, int64_t vocab, FusedPlan *plan,
                                   bool *supported);

}  // namespace ce
