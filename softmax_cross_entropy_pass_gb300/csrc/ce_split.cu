// ce_split.cu -- the forward/backward split of softmax cross-entropy:
//   ce_prep_kernel    normalisers (valid count, target-weight sum, class-weight
//                     sum) and target validation, on the device, no host sync
//                     (Liger-Kernel #1622, Summary);
//   ce_stats_kernel   one online-softmax pass per row writing the row
//                     statistics and the row loss (TransformerEngine #2325's
//                     forward), with a last-block deterministic reduction;
//   ce_grad_kernel    rereads each row once and writes the fp32 gradient,
//                     rounded once, over it; dx_y formed once per row and
//                     stored once (Liger-Kernel #1329 quoted on #1268);
//   ce_scale_kernel   grad_output scaling in place with the device-side
//                     skip when grad_output == 1 (Liger-Kernel #1622).
// Rows may start at any element alignment: each row is walked as a scalar
// head up to the first 16-byte boundary, 16-byte vectors, and a scalar tail.
#include "ce_device.cuh"
#include "ce_kernels.h"

namespace ce {

// ------------------------------------------------------------------ prep
// The normalisers written to the control block (the status word, counters
// reset for the call).
__device__ inline void prep_write_ctl(const PrepArgs &a, double c, double y, double w, unsigned bad) {
    WsCtl *ctl = a.ctl;
    unsigned status = bad ? CE_FLAG_TARGET_OUT_OF_RANGE : 0u;
    if (a.reduction == CE_RED_MEAN && y == 0.0) status |= CE_FLAG_NO_VALID_ROWS;
    ctl->status = status;
    ctl->done = 0u;
    ctl->n_correct = 0u;
    ctl->n_valid = static_cast<float>(c);
    ctl->w_y = static_cast<float>(y);
    ctl->w_all = a.weight ? static_cast<float>(w) : static_cast<float>(a.vocab);
}

// Small blocks (they share SMs with the next kernel's CTAs, which may start
// before they end): every thread keeps 8 target loads in flight. Without
// class weights one block writes the normalisers; with them kPrepParts
// blocks each write a partial (the weight gathers and the sum over the
// vocabulary spread over SMs) and ce_prep_finish_kernel combines them.
__global__ void __launch_bounds__(kPrepThreads) ce_prep_kernel(PrepArgs a) {
    pdl_launch_dependents();
    __shared__ double sh[3][kPrepThreads / 32];
    __shared__ unsigned sh_bad;
    constexpr int U = 8;
    if (threadIdx.x == 0) sh_bad = 0;
    __syncthreads();
    double cnt = 0.0, wy = 0.0, wall = 0.0;
    unsigned bad = 0;
    const int64_t nt = static_cast<int64_t>(gridDim.x) * blockDim.x;  // threads of the grid
    const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i0 = gt; i0 < a.n_rows; i0 += nt * U) {
        int64_t t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + static_cast<int64_t>(u) * nt;
            t[u] = i < a.n_rows ? load_target(a.target, a.tgt32, i) : a.ignore_index;
        }
        float w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool ok = target_valid(t[u], a.ignore_index, a.vocab);
            w[u] = ok ? (a.weight ? __ldg(a.weight + t[u]) : 1.f) : 0.f;
            cnt += ok ? 1.0 : 0.0;
            bad |= (!ok && t[u] != a.ignore_index) ? 1u : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) wy += static_cast<double>(w[u]);
    }
    if (a.weight && a.need_w_all) {
        const int64_t n4 = (reinterpret_cast<uintptr_t>(a.weight) & 15u) ? 0 : a.vocab / 4;
        const float4 *w4 = reinterpret_cast<const float4 *>(a.weight);
        for (int64_t c0 = gt; c0 < n4; c0 += nt * U) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + static_cast<int64_t>(u) * nt;
                v[u] = c < n4 ? __ldg(w4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // 32 weights summed in fp32 (a fixed tree), then one fp64 add: the
            // fp64 rate of this GPU is a small fraction of its fp32 rate
            float ps = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) ps += (v[u].x + v[u].y) + (v[u].z + v[u].w);
            wall += static_cast<double>(ps);
        }
        for (int64_t c = 4 * n4 + gt; c < a.vocab; c += nt) wall += __ldg(a.weight + c);
    }
    // fixed-order block reduction (deterministic)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        wy += __shfl_xor_sync(0xffffffffu, wy, off);
        wall += __shfl_xor_sync(0xffffffffu, wall, off);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sh[0][warp] = cnt; sh[1][warp] = wy; sh[2][warp] = wall; }
    if (bad) atomicOr(&sh_bad, 1u);
    __syncthreads();
    if (threadIdx.x == 0) {
        double c = 0.0, y = 0.0, w = 0.0;
        for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) { c += sh[0][k]; y += sh[1][k]; w += sh[2][k]; }
        if (gridDim.x == 1) {
            prep_write_ctl(a, c, y, w, sh_bad);
        } else {
            a.ctl->prep_part[blockIdx.x][0] = c;
            a.ctl->prep_part[blockIdx.x][1] = y;
            a.ctl->prep_part[blockIdx.x][2] = w;
            a.ctl->prep_bad[blockIdx.x] = sh_bad;
        }
    }
}

// The partials of the kPrepParts normaliser blocks, combined in block order
// (deterministic) once those blocks have finished.
__global__ void __launch_bounds__(32) ce_prep_finish_kernel(PrepArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    if (threadIdx.x == 0) {
        double c = 0.0, y = 0.0, w = 0.0;
        unsigned bad = 0u;
        for (int k = 0; k < kPrepParts; ++k) {
            c += a.ctl->prep_part[k][0];
            y += a.ctl->prep_part[k][1];
            w += a.ctl->prep_part[k][2];
            bad |= a.ctl->prep_bad[k];
        }
        prep_write_ctl(a, c, y, w, bad);
    }
}

// ------------------------------------------------------------------ shared helpers
// Column handled by thread `tid` among the scalar columns of a row: the head
// [0, head) (at most 7 elements) then the tail [tail0, V) (at most 7); -1
// when the thread has none. Threads 0..head-1 take the head, the next ones
// the tail.
__device__ inline int64_t scalar_col(unsigned tid, int64_t head, int64_t tail0, int64_t V) {
    const int64_t t = static_cast<int64_t>(tid);
    if (t < head) return t;
    const int64_t k = t - head;
    return (k < V - tail0) ? tail0 + k : -1;
}

__device__ inline float grad_scale(const RowArgs &a, const WsCtl *ctl, int64_t row) {
    float g = a.grad_output ? __ldg(a.grad_output + (a.reduction == CE_RED_NONE ? row : 0)) : 1.f;
    if (a.reduction == CE_RED_MEAN) {
        float wy = ctl->w_y;
        return wy != 0.f ? g / wy : 0.f;
    }
    return g;
}

// Last block to finish reduces the per-row losses in a fixed order (double
// accumulation) and resets the counter. Thread 0 of each block must have
// written its rows' losses before calling.
__device__ inline void finish_accuracy(const RowArgs &a, WsCtl *ctl);

__device__ inline void finish_loss(const RowArgs &a, WsCtl *ctl, unsigned n_blocks) {
    __shared__ unsigned sh_last;
    __shared__ double sh_sum[32];
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned prev = atomicAdd(&ctl->done, 1u);
        sh_last = (prev == n_blocks - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!sh_last) return;
    __threadfence();
    finish_accuracy(a, ctl);
    if (a.reduction == CE_RED_NONE) {
        if (threadIdx.x == 0) ctl->done = 0u;
        return;
    }
    const float *rl = a.row_loss;
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < a.n_rows; i += blockDim.x) s += static_cast<double>(__ldcg(rl + i));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((threadIdx.x & 31) == 0) sh_sum[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) tot += sh_sum[k];
        if (a.reduction == CE_RED_MEAN) {
            float wy = ctl->w_y;
            tot = wy != 0.f ? tot / static_cast<double>(wy) : 0.0;
        }
        a.loss[0] = static_cast<float>(tot);
        ctl->done = 0u;
    }
}

// Last-block token accuracy: correct rows over valid rows (0 with none).
__device__ inline void finish_accuracy(const RowArgs &a, WsCtl *ctl) {
    if (threadIdx.x == 0 && a.accuracy) {
        const float n = ctl->n_valid;
        a.accuracy[0] = n > 0.f ? static_cast<float>(__ldcg(&ctl->n_correct)) / n : 0.f;
    }
}

// Statistics of one vector with the options on: the logits are capped
// first (the statistics describe the capped logits z), the argmax follows
// the raw logits (tanh is monotonic, so it is the same column).
template <int VEC, bool SMOOTH>
__device__ inline void feat_add(RowState &st, ArgMax &am, const float *xraw, int64_t col0, int skip,
                                const float *w, float cap, bool want_am) {
    float z[VEC];
    float zmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        z[j] = cap > 0.f ? softcap_logit(xraw[j], cap) : xraw[j];
        zmax = fmaxf(zmax, z[j]);
    }
    if (want_am) {
#pragma unroll
        for (int j = 0; j < VEC; ++j) am = argmax_merge(am, ArgMax{xraw[j], static_cast<int>(col0 + j)});
    }
    row_state_add<VEC, SMOOTH>(st, z, zmax, skip, w);
}

// Block-wide argmax; the result is valid in thread 0.
__device__ inline ArgMax block_argmax(ArgMax am, ArgMax *sh /*[32]*/) {
    am = warp_argmax(am);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) sh[warp] = am;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        am = lane < nw ? sh[lane] : ArgMax{-INFINITY, 0x7fffffff};
        am = warp_argmax(am);
    }
    return am;
}

// Block-wide merge of per-thread states; the result is valid in thread 0.
__device__ inline RowState block_merge(RowState st, RowState *sh /*[32]*/) {
    st = warp_merge(st);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sh[warp] = st;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        st = lane < nw ? sh[lane] : row_state_empty();
        st = warp_merge(st);
    }
    return st;
}

// ------------------------------------------------------------------ forward: row statistics
template <int DT, int MODE, bool FEAT>
__global__ void __launch_bounds__(kRowThreads, 3) ce_stats_kernel(RowArgs a) {
    using F = Fmt<DT>;
    constexpr int VEC = F::kVec;
    constexpr bool SMOOTH = MODE != 0;
    constexpr int UNROLL = 4;
    __shared__ RowState sh[32];
    __shared__ ArgMax sh_am[32];
    const float cap = FEAT ? a.softcap : 0.f;
    const bool want_am = FEAT && a.accuracy != nullptr;
    WsCtl *ctl = a.ctl;
    const float inv_v = 1.f / static_cast<float>(a.vocab);
    // the normalisers (and the zeroed counters) of the normaliser kernel are
    // waited for where they are first read, so the logits stream starts at once
    bool have_norm = false;

    for (int64_t row = blockIdx.x; row < a.n_rows; row += gridDim.x) {
        const char *rowp = reinterpret_cast<const char *>(a.logits) + row * a.ld * F::kBytes;
        const int64_t t = load_target(a.target, a.tgt32, row);
        const bool valid = target_valid(t, a.ignore_index, a.vocab);
        const int64_t y = valid ? t : -1;
        const int64_t V = a.vocab;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
        int64_t head = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) / F::kBytes);
        if (head > V) head = V;
        const int64_t nvec = (V - head) / VEC;
        const int64_t tail0 = head + nvec * VEC;

        RowState st = row_state_empty();
        ArgMax am{-INFINITY, 0x7fffffff};
        // scalar head (< 16 bytes before the first aligned vector) and tail
        if (const int64_t c = scalar_col(threadIdx.x, head, tail0, V); c >= 0) {
            float x = F::load1(rowp, c);
            float w = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
            if constexpr (FEAT) feat_add<1, SMOOTH>(st, am, &x, c, (c == y) ? 0 : -1, MODE == 2 ? &w : nullptr, cap, want_am);
            else row_state_add<1, SMOOTH>(st, &x, x, (c == y) ? 0 : -1, MODE == 2 ? &w : nullptr);
        }
        // 16-byte vectors
        const uint4 *vp = reinterpret_cast<const uint4 *>(rowp + head * F::kBytes);
        for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += static_cast<int64_t>(blockDim.x) * UNROLL) {
            uint4 raw[UNROLL];
            bool ok[UNROLL];
            bool has_y = false;  // does one of these vectors hold the target column?
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
                ok[u] = v < nvec;
                if (ok[u]) raw[u] = ld_stream_ro(vp + v);
                has_y |= ok[u] && static_cast<uint64_t>(y - (head + v * VEC)) < static_cast<uint64_t>(VEC);
            }
            if (MODE != 2 && !FEAT && !has_y) {
                // one maximum for the group, then the exp-sum over packed fp32 pairs in
                // two independent accumulators (and the smoothing sum likewise)
                float gm = -INFINITY;
                int nok = 0;
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    if (!ok[u]) continue;
                    gm = fmaxf(gm, F::vmax(raw[u]));
                    ++nok;
                }
                if (gm > st.m) {
                    if (st.m != -INFINITY) st.s *= ex2_hw((st.m - gm) * kLog2e);
                    st.m = gm;
                }
                const float mL = st.m * kLog2e;
                const F2 l2 = f2(kLog2e, kLog2e), nm = f2(-mL, -mL);
                F2 acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)}, racc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    if (!ok[u]) continue;
                    float x[VEC];
                    F::unpack(raw[u], x);
#pragma unroll
                    for (int p = 0; p < VEC / 2; ++p) {
                        const F2 xx = f2(x[2 * p], x[2 * p + 1]);
                        if (SMOOTH) racc[p & 1] = f2_add(racc[p & 1], xx);
                        acc[p & 1] = f2_add(acc[p & 1], f2_ex2(f2_fma(xx, l2, nm)));
                    }
                }
                float a0, a1, a2, a3;
                if (SMOOTH) {
                    f2_split(racc[0], a0, a1);
                    f2_split(racc[1], a2, a3);
                    st.r += (a0 + a1) + (a2 + a3);
                    st.n += static_cast<float>(nok * VEC);
                }
                if (st.m != -INFINITY) {  // every value so far -inf: nothing to add
                    f2_split(acc[0], a0, a1);
                    f2_split(acc[1], a2, a3);
                    st.s += (a0 + a1) + (a2 + a3);
                }
                continue;
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
                if (v >= nvec) break;
                float x[VEC];
                F::unpack(raw[u], x);
                const int64_t base = head + v * VEC;
                const int skip = (static_cast<uint64_t>(y - base) < static_cast<uint64_t>(VEC)) ? static_cast<int>(y - base) : -1;
                float w[VEC];
                if (MODE == 2) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) w[j] = __ldg(a.weight + base + j);
                }
                if constexpr (FEAT) feat_add<VEC, SMOOTH>(st, am, x, base, skip, MODE == 2 ? w : nullptr, cap, want_am);
                else row_state_add<VEC, SMOOTH>(st, x, F::vmax(raw[u]), skip, MODE == 2 ? w : nullptr);
            }
        }
        if constexpr (FEAT) {
            if (want_am) am = block_argmax(am, sh_am);
        }
        st = block_merge(st, sh);
        if (threadIdx.x == 0) {
            if (!have_norm) {
                pdl_wait();
                have_norm = true;
            }
            float xy = valid ? F::load1(rowp, y) : 0.f;
            if (FEAT && cap > 0.f) xy = softcap_logit(xy, cap);
            const float wy = valid ? (a.weight ? __ldg(a.weight + y) : 1.f) : 0.f;
            // the loss needs no gradient scale
            const float rrel = SMOOTH ? row_state_rel_sum(st) : 0.f;
            RowScalars rs = make_row_scalars(st.m, st.s, xy, rrel, valid, y, wy, ctl->w_all,
                                             a.eps, inv_v, 1.f, FEAT ? a.z_loss : 0.f);
            if (want_am && valid && am.i == y) atomicAdd(&ctl->n_correct, 1u);
            if (a.stats) {
                float4 s4 = make_float4(st.m, st.s, xy, rrel);
                reinterpret_cast<float4 *>(a.stats)[row] = s4;
            }
            if (a.reduction == CE_RED_NONE) a.loss[row] = rs.loss;
            else a.row_loss[row] = rs.loss;
        }
        __syncthreads();
    }
    if (a.reduction != CE_RED_NONE || (FEAT && a.accuracy)) {
        pdl_wait();
        finish_loss(a, ctl, gridDim.x);
    }
}

// ------------------------------------------------------------------ backward: gradient in place
template <int DT, int MODE, bool FEAT>
__global__ void __launch_bounds__(kRowThreads, 3) ce_grad_kernel(RowArgs a) {
    using F = Fmt<DT>;
    constexpr int VEC = F::kVec;
    constexpr int UNROLL = 4;
    const float cap = FEAT ? a.softcap : 0.f;
    const WsCtl *ctl = a.ctl;
    const float inv_v = 1.f / static_cast<float>(a.vocab);
    pdl_wait();
    const float w_all = ctl->w_all;

    for (int64_t row = blockIdx.x; row < a.n_rows; row += gridDim.x) {
        char *rowp = reinterpret_cast<char *>(a.grad) + row * a.ld * F::kBytes;
        const int64_t t = load_target(a.target, a.tgt32, row);
        const bool valid = target_valid(t, a.ignore_index, a.vocab);
        const int64_t y = valid ? t : -1;
        const float4 s4 = __ldg(reinterpret_cast<const float4 *>(a.stats) + row);
        const float wy = valid ? (a.weight ? __ldg(a.weight + y) : 1.f) : 0.f;
        const RowScalars rs = make_row_scalars(s4.x, s4.y, s4.z, s4.w, valid, y, wy, w_all, a.eps,
                                               inv_v, grad_scale(a, ctl, row), FEAT ? a.z_loss : 0.f);
        const int64_t V = a.vocab;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
        int64_t head = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) / F::kBytes);
        if (head > V) head = V;
        const int64_t nvec = (V - head) / VEC;
        const int64_t tail0 = head + nvec * VEC;

        if (const int64_t c = scalar_col(threadIdx.x, head, tail0, V); c >= 0) {
            float g = 0.f;
            if (valid) {
                float wc = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
                float x = F::load1(rowp, c);
                if (FEAT && cap > 0.f) x = softcap_logit(x, cap);
                g = (c == y) ? rs.dxy : grad_elem(rs, x, wc);
                if (FEAT && cap > 0.f) g *= softcap_deriv(x, cap);
            }
            F::store1(rowp, c, g);
        }
        uint4 *vp = reinterpret_cast<uint4 *>(rowp + head * F::kBytes);
        if (!valid) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) st_stream(vp + v, z);
            continue;
        }
        for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += static_cast<int64_t>(blockDim.x) * UNROLL) {
            uint4 raw[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
                if (v < nvec) raw[u] = ld_stream(vp + v);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
                if (v >= nvec) break;
                float x[VEC], g[VEC];
                F::unpack(raw[u], x);
                const int64_t base = head + v * VEC;
                if (FEAT && cap > 0.f) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) x[j] = softcap_logit(x[j], cap);
                }
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    float wc = (MODE == 2) ? __ldg(a.weight + base + j) : 1.f;
                    g[j] = grad_elem(rs, x[j], wc);
                }
                if (static_cast<uint64_t>(y - base) < static_cast<uint64_t>(VEC)) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) g[e] = (base + e == y) ? rs.dxy : g[e];
                }
                if (FEAT && cap > 0.f) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) g[j] *= softcap_deriv(x[j], cap);
                }
                st_stream(vp + v, F::pack(g));
            }
        }
    }
}

// ------------------------------------------------------------------ one kernel, two passes per row
// Forward + backward in one kernel without cluster shared memory: each CTA
// owns whole rows; the statistics pass reads the row from HBM marking its
// lines evict-last in L2, and the gradient pass rereads it (from L2 while
// the lines survive) marking them evict-first and writes the gradient in
// place. HBM then sees one read and one write per element, as the fused
// cluster kernel does, at the price of the L2 holding the rows in flight
// (a few CTAs per SM x the row size).
__device__ inline uint4 ld_policy(const void *p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
    return v;
}
__device__ inline uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

template <int DT, int MODE, bool FEAT>
__global__ void __launch_bounds__(kRowpassThreads, 2) ce_rowpass_kernel(RowArgs a) {
    using F = Fmt<DT>;
    constexpr int VEC = F::kVec;
    constexpr bool SMOOTH = MODE != 0;
    constexpr int UNROLL = 4;
    __shared__ RowState sh[32];
    __shared__ ArgMax sh_am[32];
    __shared__ RowScalars sh_rs;
    const float cap = FEAT ? a.softcap : 0.f;
    const bool want_am = FEAT && a.accuracy != nullptr;
    WsCtl *ctl = a.ctl;
    const float inv_v = 1.f / static_cast<float>(a.vocab);
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    pdl_wait();
    const float w_all = ctl->w_all;

    for (int64_t row = blockIdx.x; row < a.n_rows; row += gridDim.x) {
        char *rowp = reinterpret_cast<char *>(a.grad) + row * a.ld * F::kBytes;
        const int64_t t = load_target(a.target, a.tgt32, row);
        const bool valid = target_valid(t, a.ignore_index, a.vocab);
        const int64_t y = valid ? t : -1;
        const int64_t V = a.vocab;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
        int64_t head = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) / F::kBytes);
        if (head > V) head = V;
        const int nvec = static_cast<int>((V - head) / VEC);
        const int64_t tail0 = head + static_cast<int64_t>(nvec) * VEC;
        uint4 *vp = reinterpret_cast<uint4 *>(rowp + head * F::kBytes);
        const int y_rel = valid ? static_cast<int>(y - head) : -(1 << 30);

        if (!valid) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int v = threadIdx.x; v < nvec; v += blockDim.x) st_stream(vp + v, z);
            if (const int64_t c = scalar_col(threadIdx.x, head, tail0, V); c >= 0) F::store1(rowp, c, 0.f);
            if (threadIdx.x == 0) {
                if (a.reduction == CE_RED_NONE) a.loss[row] = 0.f;
                else a.row_loss[row] = 0.f;
            }
            continue;
        }
        // ---------------------------------------------------------------- pass 1: statistics
        RowState st = row_state_empty();
        ArgMax am{-INFINITY, 0x7fffffff};
        if (const int64_t c = scalar_col(threadIdx.x, head, tail0, V); c >= 0) {
            float x = F::load1(rowp, c);
            float w = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
            if constexpr (FEAT) feat_add<1, SMOOTH>(st, am, &x, c, (c == y) ? 0 : -1, MODE == 2 ? &w : nullptr, cap, want_am);
            else row_state_add<1, SMOOTH>(st, &x, x, (c == y) ? 0 : -1, MODE == 2 ? &w : nullptr);
        }
        for (int v0 = threadIdx.x; v0 < nvec; v0 += blockDim.x * UNROLL) {
            uint4 raw[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v < nvec) raw[u] = ld_policy(vp + v, keep);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v >= nvec) break;
                float x[VEC];
                F::unpack(raw[u], x);
                const int vb = v * VEC;
                const int skip = (static_cast<unsigned>(y_rel - vb) < static_cast<unsigned>(VEC)) ? y_rel - vb : -1;
                float w[VEC];
                if (MODE == 2) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) w[j] = __ldg(a.weight + head + vb + j);
                }
                if constexpr (FEAT) feat_add<VEC, SMOOTH>(st, am, x, head + vb, skip, MODE == 2 ? w : nullptr, cap, want_am);
                else row_state_add<VEC, SMOOTH>(st, x, F::vmax(raw[u]), skip, MODE == 2 ? w : nullptr);
            }
        }
        if constexpr (FEAT) {
            if (want_am) am = block_argmax(am, sh_am);
        }
        st = block_merge(st, sh);
        if (threadIdx.x == 0) {
            float xy = F::load1(rowp, y);
            if (FEAT && cap > 0.f) xy = softcap_logit(xy, cap);
            const float wy = a.weight ? __ldg(a.weight + y) : 1.f;
            const float rrel = SMOOTH ? row_state_rel_sum(st) : 0.f;
            const float zl = FEAT ? a.z_loss : 0.f;
            const RowScalars rl = make_row_scalars(st.m, st.s, xy, rrel, true, y, wy, w_all, a.eps, inv_v, 1.f, zl);
            if (a.reduction == CE_RED_NONE) a.loss[row] = rl.loss;
            else a.row_loss[row] = rl.loss;
            sh_rs = make_row_scalars(st.m, st.s, xy, rrel, true, y, wy, w_all, a.eps, inv_v,
                                     grad_scale(a, ctl, row), zl);
            if (want_am && am.i == y) atomicAdd(&ctl->n_correct, 1u);
        }
        __syncthreads();
        const RowScalars rs = sh_rs;
        // ---------------------------------------------------------------- pass 2: gradient in place
        if (const int64_t c = scalar_col(threadIdx.x, head, tail0, V); c >= 0) {
            const float wc = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
            float x = F::load1(rowp, c);
            if (FEAT && cap > 0.f) x = softcap_logit(x, cap);
            float g = (c == y) ? rs.dxy : grad_elem(rs, x, wc);
            if (FEAT && cap > 0.f) g *= softcap_deriv(x, cap);
            F::store1(rowp, c, g);
        }
        for (int v0 = threadIdx.x; v0 < nvec; v0 += blockDim.x * UNROLL) {
            uint4 raw[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v < nvec) raw[u] = ld_policy(vp + v, drop);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v >= nvec) break;
                float x[VEC], g[VEC];
                F::unpack(raw[u], x);
                const int vb = v * VEC;
                if (FEAT && cap > 0.f) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) x[j] = softcap_logit(x[j], cap);
                }
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float wc = (MODE == 2) ? __ldg(a.weight + head + vb + j) : 1.f;
                    g[j] = grad_elem(rs, x[j], wc);
                }
                if (static_cast<unsigned>(y_rel - vb) < static_cast<unsigned>(VEC)) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) g[e] = (vb + e == y_rel) ? rs.dxy : g[e];
                }
                if (FEAT && cap > 0.f) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) g[j] *= softcap_deriv(x[j], cap);
                }
                st_stream(vp + v, F::pack(g));
            }
        }
        __syncthreads();  // sh / sh_rs are reused by the next row
    }
    if (a.reduction != CE_RED_NONE || (FEAT && a.accuracy)) finish_loss(a, ctl, gridDim.x);
}

// ------------------------------------------------------------------ grad_output scaling in place
template <int DT>
__global__ void __launch_bounds__(kRowThreads) ce_scale_kernel(ScaleArgs a) {
    using F = Fmt<DT>;
    constexpr int VEC = F::kVec;
    if (!a.per_row) {
        const float g = __ldg(a.grad_output);
        if (g == 1.f) return;  // device-side skip: nothing to scale
    }
    for (int64_t row = blockIdx.x; row < a.n_rows; row += gridDim.x) {
        const float g = __ldg(a.grad_output + (a.per_row ? row : 0));
        char *rowp = reinterpret_cast<char *>(a.grad) + row * a.ld * F::kBytes;
        const int64_t V = a.vocab;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
        int64_t head = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) / F::kBytes);
        if (head > V) head = V;
        const int64_t nvec = (V - head) / VEC;
        const int64_t tail0 = head + nvec * VEC;
        if (const int64_t c = scalar_col(threadIdx.x, head, tail0, V); c >= 0)
            F::store1(rowp, c, F::load1(rowp, c) * g);
        uint4 *vp = reinterpret_cast<uint4 *>(rowp + head * F::kBytes);
        for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
            float x[VEC];
            F::unpack(ld_stream(vp + v), x);
#pragma unroll
            for (int j = 0; j < VEC; ++j) x[j] *= g;
            st_stream(vp + v, F::pack(x));
        }
    }
}

// ------------------------------------------------------------------ bounded-wait self-test
// Waits on an mbarrier that nothing arrives on; the bounded wait gives up
// after limit_ns and the block reports CE_FLAG_WAIT_TIMEOUT.
__global__ void ce_wait_selftest_kernel(uint64_t limit_ns, unsigned int *flags) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded<false>(smem_u32(&bar), 0u, &abort_flag, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0) *flags = (!ok || abort_flag) ? CE_FLAG_WAIT_TIMEOUT : 0u;
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int *flags, cudaStream_t s) {
    void *args[] = {&limit_ns, &flags};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&ce_wait_selftest_kernel), dim3(1), dim3(32), args, 0, s);
}

// ------------------------------------------------------------------ launchers
// cudaLaunchKernel reports the status of this launch itself (a <<<>>> launch
// followed by cudaGetLastError could return an earlier, unrelated error).
// Kernels that follow the normaliser kernel are launched with programmatic
// stream serialisation: they may start while it runs and wait for it inside.
template <typename Args>
static cudaError_t launch(const void *fn, int grid, int block, const Args &a, cudaStream_t s,
                          bool after_prep = true) {
    Args copy = a;
    void *args[] = {&copy};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prep ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int DT, bool FEAT>
static const void *stats_fn(int mode) {
    switch (mode) {
    case 0: return reinterpret_cast<const void *>(&ce_stats_kernel<DT, 0, FEAT>);
    case 1: return reinterpret_cast<const void *>(&ce_stats_kernel<DT, 1, FEAT>);
    default: return reinterpret_cast<const void *>(&ce_stats_kernel<DT, 2, FEAT>);
    }
}
template <int DT, bool FEAT>
static const void *grad_fn(int mode) {
    switch (mode) {
    case 0: return reinterpret_cast<const void *>(&ce_grad_kernel<DT, 0, FEAT>);
    case 1: return reinterpret_cast<const void *>(&ce_grad_kernel<DT, 1, FEAT>);
    default: return reinterpret_cast<const void *>(&ce_grad_kernel<DT, 2, FEAT>);
    }
}
template <bool FEAT>
static const void *stats_fn_dt(int dtype, int mode) {
    return dtype == CE_DT_F32 ? stats_fn<CE_DT_F32, FEAT>(mode)
         : dtype == CE_DT_BF16 ? stats_fn<CE_DT_BF16, FEAT>(mode) : stats_fn<CE_DT_F16, FEAT>(mode);
}
template <bool FEAT>
static const void *grad_fn_dt(int dtype, int mode) {
    return dtype == CE_DT_F32 ? grad_fn<CE_DT_F32, FEAT>(mode)
         : dtype == CE_DT_BF16 ? grad_fn<CE_DT_BF16, FEAT>(mode) : grad_fn<CE_DT_F16, FEAT>(mode);
}

cudaError_t launch_prep(const PrepArgs &a, cudaStream_t s) {
    if (!a.weight) return launch(reinterpret_cast<const void *>(&ce_prep_kernel), 1, kPrepThreads, a, s, false);
    // with class weights: kPrepParts blocks, then the finishing kernel in
    // stream order (the next kernel is its programmatic dependent)
    cudaError_t e = launch(reinterpret_cast<const void *>(&ce_prep_kernel), kPrepParts, kPrepThreads, a, s, false);
    if (e != cudaSuccess) return e;
    return launch(reinterpret_cast<const void *>(&ce_prep_finish_kernel), 1, 32, a, s, false);
}

cudaError_t launch_stats(const RowArgs &a, int dtype, int mode, int grid, cudaStream_t s) {
    const void *fn = row_features(a) ? stats_fn_dt<true>(dtype, mode) : stats_fn_dt<false>(dtype, mode);
    return launch(fn, grid, kRowThreads, a, s);
}

cudaError_t launch_grad(const RowArgs &a, int dtype, int mode, int grid, cudaStream_t s) {
    const void *fn = row_features(a) ? grad_fn_dt<true>(dtype, mode) : grad_fn_dt<false>(dtype, mode);
    return launch(fn, grid, kRowThreads, a, s);
}

template <int DT, bool FEAT>
static const void *rowpass_fn(int mode) {
    switch (mode) {
    case 0: return reinterpret_cast<const void *>(&ce_rowpass_kernel<DT, 0, FEAT>);
    case 1: return reinterpret_cast<const void *>(&ce_rowpass_kernel<DT, 1, FEAT>);
    default: return reinterpret_cast<const void *>(&ce_rowpass_kernel<DT, 2, FEAT>);
    }
}
template <bool FEAT>
static const void *rowpass_fn_dt(int dtype, int mode) {
    return dtype == CE_DT_F32 ? rowpass_fn<CE_DT_F32, FEAT>(mode)
         : dtype == CE_DT_BF16 ? rowpass_fn<CE_DT_BF16, FEAT>(mode) : rowpass_fn<CE_DT_F16, FEAT>(mode);
}

cudaError_t launch_rowpass(const RowArgs &a, int dtype, int mode, int ctas_per_sm, cudaStream_t s) {
    const void *fn = row_features(a) ? rowpass_fn_dt<true>(dtype, mode) : rowpass_fn_dt<false>(dtype, mode);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int64_t grid = static_cast<int64_t>(sms) * (ctas_per_sm > 0 ? ctas_per_sm : 2);
    if (grid > a.n_rows) grid = a.n_rows;
    if (grid < 1) grid = 1;
    return launch(fn, static_cast<int>(grid), kRowpassThreads, a, s);
}

cudaError_t launch_scale(const ScaleArgs &a, int dtype, int grid, cudaStream_t s) {
    const void *fn = dtype == CE_DT_F32 ? reinterpret_cast<const void *>(&ce_scale_kernel<CE_DT_F32>)
                   : dtype == CE_DT_BF16 ? reinterpret_cast<const void *>(&ce_scale_kernel<CE_DT_BF16>)
                                         : reinterpret_cast<const void *>(&ce_scale_kernel<CE_DT_F16>);
    return launch(fn, grid, kRowThreads, a, s);
}

}  // namespace ce
