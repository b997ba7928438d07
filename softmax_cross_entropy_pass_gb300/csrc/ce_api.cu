// ce_api.cu -- the C ABI of libce.so (declared in include/ce.h): argument
// checks, workspace layout, kernel selection and launches. Host code only;
// it never allocates device memory and never waits for the GPU (except in
// ce_get_status, whose job is to wait).
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "ce.h"
#include "ce_device.cuh"
#include "ce_kernels.h"

using namespace ce;

namespace {

thread_local std::string g_last_cuda_error;

ce_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
    return CE_ERR_CUDA;
}

int64_t elem_bytes(int32_t dtype) { return dtype == CE_DT_F32 ? 4 : 2; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

ce_status check_params(const ce_params *p) {
    if (!p) return CE_ERR_INVALID_ARG;
    if (p->n_rows < 0 || p->vocab < 1 || p->ld < p->vocab) return CE_ERR_INVALID_ARG;
    if (p->vocab > (int64_t(1) << 31) - 1) return CE_ERR_UNSUPPORTED;
    if (p->dtype != CE_DT_F32 && p->dtype != CE_DT_BF16 && p->dtype != CE_DT_F16) return CE_ERR_INVALID_ARG;
    if (p->reduction != CE_RED_NONE && p->reduction != CE_RED_MEAN && p->reduction != CE_RED_SUM)
        return CE_ERR_INVALID_ARG;
    if (!(p->label_smoothing >= 0.f && p->label_smoothing <= 1.f)) return CE_ERR_INVALID_ARG;
    if (p->target_is_int32 != 0 && p->target_is_int32 != 1) return CE_ERR_INVALID_ARG;
    if (p->reserved != 0) return CE_ERR_INVALID_ARG;
    if (p->class_weight && !aligned(p->class_weight, 4)) return CE_ERR_INVALID_ARG;
    if (!(p->softcap >= 0.f && p->softcap < INFINITY) || !(p->z_loss >= 0.f && p->z_loss < INFINITY))
        return CE_ERR_INVALID_ARG;
    if (p->accuracy && !aligned(p->accuracy, 4)) return CE_ERR_INVALID_ARG;
    return CE_OK;
}

// softcap, z-loss or token accuracy asked for
bool has_options(const ce_params *p) { return p->softcap > 0.f || p->z_loss > 0.f || p->accuracy; }

size_t workspace_bytes_for(int64_t n_rows) { return ws_bytes(n_rows); }

ce_status check_ws(const ce_params *p, const void *ws, size_t ws_bytes) {
    if (!ws || !aligned(ws, 256)) return CE_ERR_WORKSPACE;
    if (ws_bytes < workspace_bytes_for(p->n_rows)) return CE_ERR_WORKSPACE;
    return CE_OK;
}

int smoothing_mode(const ce_params *p) {
    if (p->label_smoothing <= 0.f) return 0;
    return p->class_weight ? 2 : 1;
}

cudaError_t run_prep(const ce_params *p, const void *target, void *ws, cudaStream_t s);

int row_grid(int64_t n_rows) {
    const int64_t cap = int64_t(1) << 20;
    return static_cast<int>(n_rows < 1 ? 1 : (n_rows < cap ? n_rows : cap));
}

cudaError_t enqueue_prep(const ce_params *p, const void *target, void *ws, cudaStream_t s) {
    if (p->variant & CE_VARIANT_PREPARED) return cudaSuccess;
    return run_prep(p, target, ws, s);
}

cudaError_t run_prep(const ce_params *p, const void *target, void *ws, cudaStream_t s) {
    PrepArgs a{};
    a.target = target;
    a.tgt32 = p->target_is_int32;
    a.reduction = p->reduction;
    a.n_rows = p->n_rows;
    a.vocab = p->vocab;
    a.ignore_index = p->ignore_index;
    a.weight = p->class_weight;
    a.need_w_all = p->label_smoothing > 0.f ? 1 : 0;
    a.ctl = reinterpret_cast<WsCtl *>(ws);
    return launch_prep(a, s);
}

RowArgs row_args(const ce_params *p, const void *target, void *ws) {
    RowArgs a{};
    a.n_rows = p->n_rows;
    a.vocab = p->vocab;
    a.ld = p->ld;
    a.target = target;
    a.tgt32 = p->target_is_int32;
    a.reduction = p->reduction;
    a.ignore_index = p->ignore_index;
    a.weight = p->class_weight;
    a.eps = p->label_smoothing;
    a.row_loss = ws_row_loss(ws);
    a.ctl = reinterpret_cast<WsCtl *>(ws);
    a.softcap = p->softcap;
    a.z_loss = p->z_loss;
    a.accuracy = p->accuracy;
    return a;
}

// The forward (row statistics and losses) of ce_forward and the split path:
// the stream kernel's first pass (bulk-copy ring: the bytes in flight are
// not limited by registers) where it applies, the register row kernel for
// class-weighted smoothing and the options.
cudaError_t launch_forward(const RowArgs &a0, const ce_params *p, cudaStream_t s) {
    const int mode = smoothing_mode(p);
    if (mode != 2 && !has_options(p)) {
        RowArgs a = a0;
        a.grad = const_cast<void *>(a0.logits);  // read only in this kernel
        return launch_stream_forward(a, p->dtype, mode, (p->variant & CE_VARIANT_PREPARED) == 0, s);
    }
    return launch_stats(a0, p->dtype, mode, row_grid(p->n_rows), s);
}

// ---------------------------------------------------------------- fused plan cache
std::mutex g_plan_mu;
std::map<std::tuple<int, int, int, int64_t, int64_t, int>, std::pair<bool, FusedPlan>> g_plans;

cudaError_t get_plan(const ce_params *p, FusedPlan *plan, bool *ok) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int mode = smoothing_mode(p);
    const int cl = (p->variant >> CE_VARIANT_CLUSTER_SHIFT) & 0xff;
    auto key = std::make_tuple(dev, p->dtype, mode, p->vocab, p->n_rows, cl);
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            *ok = it->second.first;
            *plan = it->second.second;
            return cudaSuccess;
        }
    }
    FusedPlan pl{};
    bool sup = false;
    e = fused_plan(p->dtype, mode, p->n_rows, p->vocab, cl, &pl, &sup);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans[key] = std::make_pair(sup, pl);
    *ok = sup;
    *plan = pl;
    return cudaSuccess;
}

// the rows allow the fused kernel: 16-byte aligned row starts and weights
bool fused_layout_ok(const ce_params *p, const void *x) {
    const int64_t esz = elem_bytes(p->dtype);
    if (!aligned(x, 16)) return false;
    if (p->n_rows > 1 && ((p->ld * esz) & 15) != 0) return false;
    if (p->class_weight && !aligned(p->class_weight, 16)) return false;
    return true;
}

// The path of CE_VARIANT_AUTO: the stream kernel (HBM read once, the second
// read served by L2 through a bulk-copy ring) is the fastest measured path
// on GB300 for every row size, takes any row alignment (the unaligned head
// and tail of a row go through plain accesses) and carries the options; the
// row pass and the split path remain for callers that ask for them.
int auto_path(const ce_params *, const void *) { return CE_VARIANT_STREAM; }

}  // namespace

extern "C" {

ce_status ce_select_variant(const ce_params *p, const void *logits, int32_t *variant) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if (!variant) return CE_ERR_INVALID_ARG;
    const int path = p->variant & 0xff;
    *variant = path == CE_VARIANT_AUTO ? auto_path(p, logits) : path;
    return CE_OK;
}

const char *ce_version(void) { return "ce-gb300 1.0 (sm_103a)"; }

const char *ce_status_string(ce_status s) {
    switch (s) {
    case CE_OK: return "CE_OK";
    case CE_ERR_INVALID_ARG: return "CE_ERR_INVALID_ARG";
    case CE_ERR_UNSUPPORTED: return "CE_ERR_UNSUPPORTED";
    case CE_ERR_CUDA: return "CE_ERR_CUDA";
    case CE_ERR_WORKSPACE: return "CE_ERR_WORKSPACE";
    default: return "CE_ERR_UNKNOWN";
    }
}

const char *ce_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

ce_status ce_workspace_size(const ce_params *p, size_t *bytes) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if (!bytes) return CE_ERR_INVALID_ARG;
    *bytes = workspace_bytes_for(p->n_rows);
    return CE_OK;
}

ce_status ce_prepare(const ce_params *p, const void *target, void *ws, size_t ws_bytes, void *stream) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != CE_OK) return st;
    if (p->n_rows > 0 && !target) return CE_ERR_INVALID_ARG;
    cudaError_t e = run_prep(p, target, ws, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

ce_status ce_forward(const ce_params *p, const void *logits, const void *target, float *loss,
                     float *stats, void *ws, size_t ws_bytes, void *stream) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != CE_OK) return st;
    if (!loss || (p->n_rows > 0 && (!logits || !target))) return CE_ERR_INVALID_ARG;
    if (!aligned(logits, elem_bytes(p->dtype))) return CE_ERR_INVALID_ARG;
    if (stats && !aligned(stats, 16)) return CE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = enqueue_prep(p, target, ws, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (p->n_rows == 0) {
        if (p->reduction != CE_RED_NONE && (e = cudaMemsetAsync(loss, 0, sizeof(float), s)) != cudaSuccess)
            return cuda_fail(e);
        return CE_OK;
    }
    RowArgs a = row_args(p, target, ws);
    a.logits = logits;
    a.loss = loss;
    a.stats = stats;
    e = launch_forward(a, p, s);
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

ce_status ce_backward(const ce_params *p, void *logits_inout, const void *target, const float *stats,
                      const float *grad_output, void *ws, size_t ws_bytes, void *stream) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != CE_OK) return st;
    if (p->n_rows > 0 && (!logits_inout || !target || !stats)) return CE_ERR_INVALID_ARG;
    if (!aligned(logits_inout, elem_bytes(p->dtype))) return CE_ERR_INVALID_ARG;
    if (stats && !aligned(stats, 16)) return CE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = enqueue_prep(p, target, ws, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (p->n_rows == 0) return CE_OK;
    RowArgs a = row_args(p, target, ws);
    a.grad = logits_inout;
    a.stats = const_cast<float *>(stats);
    a.grad_output = grad_output;
    e = launch_grad(a, p->dtype, smoothing_mode(p), row_grid(p->n_rows), s);
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

ce_status ce_fwd_bwd(const ce_params *p, void *logits_inout, const void *target, float *loss,
                     const float *grad_output, void *ws, size_t ws_bytes, void *stream) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != CE_OK) return st;
    if (!loss || (p->n_rows > 0 && (!logits_inout || !target))) return CE_ERR_INVALID_ARG;
    if (!aligned(logits_inout, elem_bytes(p->dtype))) return CE_ERR_INVALID_ARG;
    int path = p->variant & 0xff;
    if (p->variant & ~(0xffff | CE_VARIANT_PREPARED | (0x7ff << CE_VARIANT_TUNE_SHIFT))) return CE_ERR_INVALID_ARG;
    if (path == CE_VARIANT_AUTO) path = auto_path(p, logits_inout);
    if (path != CE_VARIANT_AUTO && path != CE_VARIANT_SPLIT && path != CE_VARIANT_FUSED &&
        path != CE_VARIANT_ROWPASS && path != CE_VARIANT_STREAM)
        return CE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (path == CE_VARIANT_FUSED && has_options(p)) return CE_ERR_UNSUPPORTED;
    if (path == CE_VARIANT_STREAM) {
        cudaError_t e = enqueue_prep(p, target, ws, s);
        if (e != cudaSuccess) return cuda_fail(e);
        if (p->n_rows == 0) {
            if (p->reduction != CE_RED_NONE && (e = cudaMemsetAsync(loss, 0, sizeof(float), s)) != cudaSuccess)
                return cuda_fail(e);
            return CE_OK;
        }
        RowArgs a = row_args(p, target, ws);
        a.grad = logits_inout;
        a.loss = loss;
        a.grad_output = grad_output;
        e = launch_stream(a, p->dtype, smoothing_mode(p), (p->variant >> CE_VARIANT_CLUSTER_SHIFT) & 0xff,
                          (p->variant >> CE_VARIANT_TUNE_SHIFT) & 0x7ff, (p->variant & CE_VARIANT_PREPARED) == 0, s);
        return e == cudaSuccess ? CE_OK : cuda_fail(e);
    }

    if (path == CE_VARIANT_ROWPASS) {
        cudaError_t e = enqueue_prep(p, target, ws, s);
        if (e != cudaSuccess) return cuda_fail(e);
        if (p->n_rows == 0) {
            if (p->reduction != CE_RED_NONE && (e = cudaMemsetAsync(loss, 0, sizeof(float), s)) != cudaSuccess)
                return cuda_fail(e);
            return CE_OK;
        }
        RowArgs a = row_args(p, target, ws);
        a.grad = logits_inout;
        a.loss = loss;
        a.grad_output = grad_output;
        e = launch_rowpass(a, p->dtype, smoothing_mode(p), (p->variant >> CE_VARIANT_CLUSTER_SHIFT) & 0xff, s);
        return e == cudaSuccess ? CE_OK : cuda_fail(e);
    }

    bool use_fused = false;
    FusedPlan plan{};
    if (path != CE_VARIANT_SPLIT && p->n_rows > 0) {
        bool ok = false;
        if (fused_layout_ok(p, logits_inout)) {
            cudaError_t e = get_plan(p, &plan, &ok);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        if (!ok && path == CE_VARIANT_FUSED) return CE_ERR_UNSUPPORTED;
        use_fused = ok;
    } else if (path == CE_VARIANT_FUSED) {
        if (!fused_layout_ok(p, logits_inout)) return CE_ERR_UNSUPPORTED;
    }

    if (!use_fused) {
        // split: statistics pass, then the gradient pass rereading each row;
        // the row statistics live in the workspace between the two
        cudaError_t e = enqueue_prep(p, target, ws, s);
        if (e != cudaSuccess) return cuda_fail(e);
        if (p->n_rows == 0) {
            if (p->reduction != CE_RED_NONE && (e = cudaMemsetAsync(loss, 0, sizeof(float), s)) != cudaSuccess)
                return cuda_fail(e);
            return CE_OK;
        }
        RowArgs a = row_args(p, target, ws);
        a.logits = logits_inout;
        a.loss = loss;
        a.stats = ws_stats(ws, p->n_rows);
        e = launch_forward(a, p, s);
        if (e != cudaSuccess) return cuda_fail(e);
        a.grad = logits_inout;
        a.grad_output = grad_output;
        e = launch_grad(a, p->dtype, smoothing_mode(p), row_grid(p->n_rows), s);
        return e == cudaSuccess ? CE_OK : cuda_fail(e);
    }

    cudaError_t e = enqueue_prep(p, target, ws, s);
    if (e != cudaSuccess) return cuda_fail(e);
    FusedArgs a{};
    a.x = logits_inout;
    a.n_rows = p->n_rows;
    a.vocab = p->vocab;
    a.ld = p->ld;
    a.target = target;
    a.tgt32 = p->target_is_int32;
    a.reduction = p->reduction;
    a.ignore_index = p->ignore_index;
    a.weight = p->class_weight;
    a.eps = p->label_smoothing;
    a.grad_output = grad_output;
    a.loss = loss;
    a.row_loss = ws_row_loss(ws);
    a.ctl = reinterpret_cast<WsCtl *>(ws);
    a.out = logits_inout;
    a.ld_out = p->ld;
    a.finalize = 1;
    e = launch_fused(a, plan, p->dtype, smoothing_mode(p), s, (p->variant & CE_VARIANT_PREPARED) == 0);
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

ce_status ce_fwd_bwd_from_host(const ce_params *p, const void *logits_host, void *logits_dev, const void *target,
                               float *loss, const float *grad_output, void *ws, size_t ws_bytes, void *stream,
                               void *copy_stream, int32_t n_parts) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != CE_OK) return st;
    if (n_parts < 1 || p->variant != 0) return CE_ERR_INVALID_ARG;
    if (has_options(p)) return CE_ERR_UNSUPPORTED;
    if (!loss || (p->n_rows > 0 && (!logits_host || !logits_dev || !target))) return CE_ERR_INVALID_ARG;
    const int64_t esz = elem_bytes(p->dtype);
    if (!aligned(logits_dev, esz) || !aligned(logits_host, esz)) return CE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);
    if (cs == s) return CE_ERR_INVALID_ARG;  // the copies must run beside the kernels
    const int64_t R = p->n_rows;
    cudaError_t e = run_prep(p, target, ws, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (R == 0) {
        if (p->reduction != CE_RED_NONE && (e = cudaMemsetAsync(loss, 0, sizeof(float), s)) != cudaSuccess)
            return cuda_fail(e);
        return CE_OK;
    }
    const int64_t parts = n_parts < R ? n_parts : R;
    const int64_t per = (R + parts - 1) / parts;
    // events: one for the work already queued on `stream` (the copies must not
    // overwrite logits_dev under an earlier call's kernels), one per part;
    // destroyed once queued (the runtime releases them when they complete)
    cudaEvent_t ev_start = nullptr;
    if ((e = cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
    e = cudaEventRecord(ev_start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev_start, 0);
    cudaEventDestroy(ev_start);
    if (e != cudaSuccess) return cuda_fail(e);
    const int tb = p->target_is_int32 ? 4 : 8;
    for (int64_t r0 = 0; r0 < R; r0 += per) {
        const int64_t n = (R - r0) < per ? (R - r0) : per;
        const size_t off = static_cast<size_t>(r0 * p->ld * esz);
        const size_t bytes = static_cast<size_t>(((n - 1) * p->ld + p->vocab) * esz);  // not past the last row
        e = cudaMemcpyAsync(static_cast<char *>(logits_dev) + off, static_cast<const char *>(logits_host) + off, bytes,
                            cudaMemcpyHostToDevice, cs);
        if (e != cudaSuccess) return cuda_fail(e);
        cudaEvent_t ev = nullptr;
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
        e = cudaEventRecord(ev, cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev, 0);
        cudaEventDestroy(ev);
        if (e != cudaSuccess) return cuda_fail(e);
        // this block's rows, with the batch normalisers from the kernel above
        RowArgs a = row_args(p, static_cast<const char *>(target) + r0 * tb, ws);
        a.n_rows = n;
        a.grad = static_cast<char *>(logits_dev) + off;
        a.row_loss = ws_row_loss(ws) + r0;
        a.loss = p->reduction == CE_RED_NONE ? loss + r0 : loss;
        a.grad_output = grad_output ? (p->reduction == CE_RED_NONE ? grad_output + r0 : grad_output) : nullptr;
        a.no_finalize = 1;
        if ((e = launch_stream(a, p->dtype, smoothing_mode(p), 0, 0, false, s)) != cudaSuccess) return cuda_fail(e);
    }
    if (p->reduction != CE_RED_NONE) {
        e = launch_reduce_row_losses(ws_row_loss(ws), R, p->reduction, reinterpret_cast<const WsCtl *>(ws), loss, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return CE_OK;
}

ce_status ce_scale_grad(const ce_params *p, void *grad_inout, const float *grad_output, void *stream) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    if (!grad_output || (p->n_rows > 0 && !grad_inout)) return CE_ERR_INVALID_ARG;
    if (p->n_rows == 0) return CE_OK;
    ScaleArgs a{};
    a.grad = grad_inout;
    a.n_rows = p->n_rows;
    a.vocab = p->vocab;
    a.ld = p->ld;
    a.grad_output = grad_output;
    a.per_row = p->reduction == CE_RED_NONE ? 1 : 0;
    cudaError_t e = launch_scale(a, p->dtype, row_grid(p->n_rows), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

ce_status ce_fused_plan(const ce_params *p, int32_t *cluster_size, int32_t *n_clusters,
                        int32_t *ctas_per_sm, int64_t *slice_bytes) {
    ce_status st = check_params(p);
    if (st != CE_OK) return st;
    FusedPlan plan{};
    bool ok = false;
    cudaError_t e = get_plan(p, &plan, &ok);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!ok) return CE_ERR_UNSUPPORTED;
    if (cluster_size) *cluster_size = plan.cluster;
    if (n_clusters) *n_clusters = plan.n_clusters;
    if (ctas_per_sm) *ctas_per_sm = plan.ctas_per_sm;
    if (slice_bytes) *slice_bytes = plan.slice_elems * elem_bytes(p->dtype);
    return CE_OK;
}

ce_status ce_selftest_wait_timeout(uint64_t limit_ns, uint32_t *device_flags, void *stream) {
    if (!device_flags || !aligned(device_flags, 4)) return CE_ERR_INVALID_ARG;
    if (limit_ns < 1000000ull || limit_ns > 5000000000ull) return CE_ERR_INVALID_ARG;
    cudaError_t e = launch_wait_selftest(limit_ns, device_flags, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CE_OK : cuda_fail(e);
}

ce_status ce_get_status(const void *ws, uint32_t *flags, void *stream) {
    if (!ws || !flags) return CE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t v = 0;
    e = cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    *flags = v;
    return CE_OK;
}

}  // extern "C"
