// ce_fused.cu -- fused single-read softmax cross-entropy forward + backward.
//
// Each row of the logits is read from HBM once and the gradient written
// once, in place. A thread-block cluster of C CTAs owns one row at a time;
// CTA r of the cluster holds columns [r*S, (r+1)*S) of the row in its shared
// memory. Per row:
//   1. a producer warp streams the slice in with 1-D bulk async copies
//      (cp.async.bulk, no multicast) into a ring of chunks, each completing
//      on its own mbarrier;
//   2. eight consumer warps run the online-softmax pass over the chunks as
//      they land (max, off-target exp-sum, smoothing sum);
//   3. each CTA pushes its partial (m, s, r, n, x_y) into every CTA's shared
//      memory of the cluster (st.shared::cluster + a remote mbarrier
//      arrive); every CTA merges the C partials in rank order;
//   4. the consumers form the fp32 gradient from shared memory, patch the
//      target column with dx_y formed once from (m, d, x_y), round once and
//      store 16 bytes per thread; as each chunk is consumed its buffer is
//      handed back to the producer, which starts the next row's copy there.
//
// This replaces the pages' two passes over global memory (Liger-Kernel
// #1268's pass 1 / pass 2; TransformerEngine #2325's forward and backward
// kernels) by one read: the row is resident in cluster shared memory
// between the statistics and the gradient (the single-GPU counterpart of
// TransformerEngine's cross-rank merge of m_d_X_y).
//
// Every wait is bounded (about 2 s); a wait that gives up sets
// CE_FLAG_WAIT_TIMEOUT in the workspace status and lets the kernel finish.
#include "ce_device.cuh"
#include "ce_kernels.h"

namespace ce {

struct XSlot {            // one CTA's partial for one row (32 bytes)
    float m, s, r, n;
    float xy, pad0, pad1, pad2;
};

struct FusedSmem {        // fixed part, placed after the row slice
    uint64_t full[kMaxChunks];
    uint64_t empty[kMaxChunks];
    uint64_t xbar[2];
    XSlot slot[2][kMaxCluster];
    RowState red[kFusedConsumerWarps];
    int abort;
};
static_assert(sizeof(FusedSmem) <= kFusedSmemFixed, "fixed shared memory block too large");

__device__ inline void consumer_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(kFusedConsumerWarps * 32) : "memory");
}

// Writes one vector of gradients (VEC values of the input format) to the
// output row: 16 bytes when the output has the input's type, 8 bytes for
// fp32 -> bf16.
template <int DT, int ODT>
__device__ inline void store_grad_vec(char *outp, int base, const float *gr) {
    using F = Fmt<DT>;
    if constexpr (DT == ODT) {
        st_stream(outp + static_cast<uint32_t>(base) * F::kBytes, F::pack(gr));
    } else {
        static_assert(DT == CE_DT_F32 && ODT == CE_DT_BF16, "fp32 -> bf16 only");
        st_stream_v2(outp + static_cast<uint32_t>(base) * 2u, Fmt<CE_DT_BF16>::pack2(gr[0], gr[1]),
                     Fmt<CE_DT_BF16>::pack2(gr[2], gr[3]));
    }
}

template <int DT, int MODE, int ODT>
__global__ void __launch_bounds__(kFusedThreads, 3) ce_fused_kernel(FusedArgs a) {
    using F = Fmt<DT>;
    using FO = Fmt<ODT>;
    constexpr int VEC = F::kVec;
    constexpr bool SMOOTH = MODE != 0;
    constexpr int NCT = kFusedConsumerWarps * 32;

    extern __shared__ __align__(128) uint8_t smem[];
    const int64_t slice_bytes_alloc = ((a.slice_elems * F::kBytes + 127) / 128) * 128;
    FusedSmem &S = *reinterpret_cast<FusedSmem *>(smem + slice_bytes_alloc);
    const uint32_t buf = smem_u32(smem);

    const uint32_t rank = cluster_ctarank();
    const uint32_t C = cluster_nctarank();
    const uint32_t q = cluster_id_x();
    const uint32_t nq = nclusters_x();
    const int64_t V = a.vocab;
    const int64_t lo = static_cast<int64_t>(rank) * a.slice_elems;
    const int64_t hi = (lo + a.slice_elems < V) ? lo + a.slice_elems : V;
    const int64_t L = hi > lo ? hi - lo : 0;                  // columns of this CTA
    const int64_t Lb16 = (L * F::kBytes) & ~static_cast<int64_t>(15);  // bytes moved by bulk copies
    const int nvec = static_cast<int>(Lb16 / 16);             // 16-byte vectors in shared memory
    const int64_t tail0 = lo + Lb16 / F::kBytes;              // first column of the scalar tail
    const int ntail = static_cast<int>(hi - tail0);           // < 16 / element size
    const int nch = static_cast<int>((Lb16 + a.chunk_bytes - 1) / a.chunk_bytes);
    const int vec_per_chunk = a.chunk_bytes / 16;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int64_t n_rows = a.n_rows;
    if (a.row_limit) {
        const int64_t left = static_cast<int64_t>(__ldg(a.row_limit)) - a.row_limit_off;
        const int64_t blk = left > 0 ? (left + 63) / 64 * 64 : 0;
        n_rows = blk < n_rows ? blk : n_rows;
    }

    if (tid == 0) {
        for (int k = 0; k < nch; ++k) {
            mbar_init(smem_u32(&S.full[k]), 1);
            mbar_init(smem_u32(&S.empty[k]), kFusedConsumerWarps);
        }
        mbar_init(smem_u32(&S.xbar[0]), C);
        mbar_init(smem_u32(&S.xbar[1]), C);
        S.abort = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers exist before any remote arrive

    volatile int *abort = &S.abort;
    const size_t row_bytes = static_cast<size_t>(a.ld) * F::kBytes;
    char *const xbase = reinterpret_cast<char *>(a.x);
    const size_t out_row_bytes = static_cast<size_t>(a.ld_out) * FO::kBytes;
    char *const obase = reinterpret_cast<char *>(a.out);

    if (warp == kFusedConsumerWarps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t j = 0;
            for (int64_t row = q; row < n_rows; row += nq) {
                const int64_t t = load_target(a.target, a.tgt32, row);
                if (!target_valid(t, a.ignore_index, V)) continue;
                const char *src = xbase + row * row_bytes + lo * F::kBytes;
                for (int k = 0; k < nch; ++k) {
                    if (j > 0) mbar_wait_bounded<false>(smem_u32(&S.empty[k]), (j - 1) & 1u, abort);
                    const int64_t off = static_cast<int64_t>(k) * a.chunk_bytes;
                    const uint32_t bytes = static_cast<uint32_t>(
                        (Lb16 - off < a.chunk_bytes) ? (Lb16 - off) : a.chunk_bytes);
                    mbar_expect_tx(smem_u32(&S.full[k]), bytes);
                    bulk_g2s(buf + static_cast<uint32_t>(off), src + off, bytes, smem_u32(&S.full[k]), pol);
                }
                ++j;
            }
            // drain: the last copies have landed before the CTA may exit
            if (j > 0)
                for (int k = 0; k < nch; ++k) mbar_wait_bounded<false>(smem_u32(&S.full[k]), (j - 1) & 1u, abort);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- consumers
        const float inv_v = 1.f / static_cast<float>(V);
        const float eps = a.eps;
        float w_all = 0.f, w_y_sum = 0.f;   // batch normalisers, read after the normaliser kernel ends
        bool have_norm = false;
        uint32_t j = 0;
        for (int64_t row = q; row < n_rows; row += nq) {
            const int64_t t = load_target(a.target, a.tgt32, row);
            const bool valid = target_valid(t, a.ignore_index, V);
            char *rowp = xbase + row * row_bytes;
            char *outp = obase + row * out_row_bytes;
            if (!valid) {
                // ignored row: no read, zero gradient, zero loss
                const float zero[VEC] = {};
                char *const out_slice = outp + lo * FO::kBytes;
                for (int v = tid; v < nvec; v += NCT) store_grad_vec<DT, ODT>(out_slice, v * VEC, zero);
                if (tid < ntail) FO::store1(outp, tail0 + tid, 0.f);
                if (rank == 0 && tid == 0) {
                    if (a.reduction == CE_RED_NONE) a.loss[row] = 0.f;
                    else a.row_loss[row] = 0.f;
                }
                continue;
            }
            const int64_t y = t;
            // target column relative to this CTA's slice (outside: a value no vector matches)
            const int y_rel = (y >= lo && y < hi) ? static_cast<int>(y - lo) : -(1 << 30);
            // ------------------------------------------------ statistics pass over the slice
            RowState st = row_state_empty();
            for (int k = 0; k < nch; ++k) {
                mbar_wait_bounded<false>(smem_u32(&S.full[k]), j & 1u, abort);
                const int v1 = min(nvec, (k + 1) * vec_per_chunk);
                for (int v = k * vec_per_chunk + tid; v < v1; v += NCT) {
                    const uint4 raw = ld_shared_v4(buf + 16u * v);
                    float x[VEC];
                    F::unpack(raw, x);
                    const int vb = v * VEC;
                    const int skip = (static_cast<unsigned>(y_rel - vb) < static_cast<unsigned>(VEC)) ? y_rel - vb : -1;
                    float w[VEC];
                    if (MODE == 2) {
                        const float4 *wp = reinterpret_cast<const float4 *>(a.weight + lo + vb);
#pragma unroll
                        for (int h = 0; h < VEC / 4; ++h) {
                            float4 w4 = __ldg(wp + h);
                            w[4 * h] = w4.x; w[4 * h + 1] = w4.y; w[4 * h + 2] = w4.z; w[4 * h + 3] = w4.w;
                        }
                    }
                    row_state_add<VEC, SMOOTH>(st, x, F::vmax(raw), skip, MODE == 2 ? w : nullptr);
                }
            }
            if (tid < ntail) {
                const int64_t c = tail0 + tid;
                float x = F::load1(rowp, c);
                float w = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
                row_state_add<1, SMOOTH>(st, &x, x, (c == y) ? 0 : -1, MODE == 2 ? &w : nullptr);
            }
            st = warp_merge(st);
            if (lane == 0) S.red[warp] = st;
            consumer_sync();
            // ------------------------------------------------ cluster exchange
            const uint32_t par = j & 1u;
            if (warp == 0) {
                st = lane < kFusedConsumerWarps ? S.red[lane] : row_state_empty();
                st = warp_merge(st);
                if (lane == 0) {
                    float xy = 0.f;
                    if (y >= lo && y < hi) {
                        if (y < tail0) {
                            const uint32_t off = static_cast<uint32_t>((y - lo) * F::kBytes);
                            float tmp[VEC];
                            F::unpack(ld_shared_v4(buf + (off & ~15u)), tmp);
                            const int e_y = static_cast<int>((off & 15u) / F::kBytes);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) xy = (e == e_y) ? tmp[e] : xy;
                        } else {
                            xy = F::load1(rowp, y);
                        }
                    }
                    const uint32_t my_slot = smem_u32(&S.slot[par][rank]);
                    const uint32_t my_bar = smem_u32(&S.xbar[par]);
                    for (uint32_t d = 0; d < C; ++d) {
                        const uint32_t rs = mapa_shared(my_slot, d);
                        st_cluster_v4(rs, st.m, st.s, st.r, st.n);
                        st_cluster_v4(rs + 16u, xy, 0.f, 0.f, 0.f);
                        mbar_arrive_remote(mapa_shared(my_bar, d));
                    }
                }
            }
            mbar_wait_bounded<true>(smem_u32(&S.xbar[par]), (j >> 1) & 1u, abort);
            RowState tot = row_state_empty();
            for (uint32_t d = 0; d < C; ++d) {
                const XSlot &xs = S.slot[par][d];
                tot = row_state_merge(tot, RowState{xs.m, xs.s, xs.r, xs.n});
            }
            const uint32_t owner = static_cast<uint32_t>(y / a.slice_elems);
            const float xy = S.slot[par][owner].xy;
            // ------------------------------------------------ row scalars and loss
            if (!have_norm) {
                pdl_wait();
                w_all = a.ctl->w_all;
                w_y_sum = a.ctl->w_y;
                have_norm = true;
            }
            const float wy = a.weight ? __ldg(a.weight + y) : 1.f;
            float g = a.grad_output ? __ldg(a.grad_output + (a.reduction == CE_RED_NONE ? row : 0)) : 1.f;
            float scale = g;
            if (a.reduction == CE_RED_MEAN) scale = (w_y_sum != 0.f) ? g / w_y_sum : 0.f;
            const float rrel = row_state_rel_sum(tot);
            const RowScalars rs = make_row_scalars(tot.m, tot.s, xy, rrel, true, y, wy, w_all,
                                                   eps, inv_v, scale);
            if (rank == 0 && tid == 0) {
                // loss_i without the gradient scale
                const RowScalars rl = make_row_scalars(tot.m, tot.s, xy, rrel, true, y, wy, w_all,
                                                       eps, inv_v, 1.f);
                if (a.reduction == CE_RED_NONE) a.loss[row] = rl.loss;
                else a.row_loss[row] = rl.loss;
            }
            // ------------------------------------------------ gradient pass from shared memory
            char *const out_slice = outp + lo * FO::kBytes;
            for (int k = 0; k < nch; ++k) {
                const int v1 = min(nvec, (k + 1) * vec_per_chunk);
                for (int v = k * vec_per_chunk + tid; v < v1; v += NCT) {
                    float x[VEC], gr[VEC];
                    F::unpack(ld_shared_v4(buf + 16u * v), x);
                    const int vb = v * VEC;
                    if (MODE == 2) {
                        const float4 *wp = reinterpret_cast<const float4 *>(a.weight + lo + vb);
#pragma unroll
                        for (int h = 0; h < VEC / 4; ++h) {
                            float4 w4 = __ldg(wp + h);
                            gr[4 * h] = grad_elem(rs, x[4 * h], w4.x);
                            gr[4 * h + 1] = grad_elem(rs, x[4 * h + 1], w4.y);
                            gr[4 * h + 2] = grad_elem(rs, x[4 * h + 2], w4.z);
                            gr[4 * h + 3] = grad_elem(rs, x[4 * h + 3], w4.w);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) gr[e] = grad_elem(rs, x[e], 1.f);
                    }
                    if (static_cast<unsigned>(y_rel - vb) < static_cast<unsigned>(VEC)) {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) gr[e] = (vb + e == y_rel) ? rs.dxy : gr[e];
                    }
                    store_grad_vec<DT, ODT>(out_slice, vb, gr);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.empty[k]));
            }
            if (tid < ntail) {
                const int64_t c = tail0 + tid;
                const float wc = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
                FO::store1(outp, c, (c == y) ? rs.dxy : grad_elem(rs, F::load1(rowp, c), wc));
            }
            ++j;
        }
        // ---------------------------------------------------- batch reduction (last CTA)
        if (a.reduction != CE_RED_NONE && a.finalize) {
            __shared__ unsigned sh_last;
            __shared__ double sh_sum[kFusedConsumerWarps];
            if (!have_norm) {
                pdl_wait();
                w_y_sum = a.ctl->w_y;
            }
            consumer_sync();
            if (tid == 0) {
                __threadfence();
                const unsigned prev = atomicAdd(&a.ctl->done, 1u);
                sh_last = (prev == gridDim.x - 1) ? 1u : 0u;
            }
            consumer_sync();
            if (sh_last) {
                __threadfence();
                double s = 0.0;
                for (int64_t i = tid; i < n_rows; i += NCT) s += static_cast<double>(__ldcg(a.row_loss + i));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (lane == 0) sh_sum[warp] = s;
                consumer_sync();
                if (tid == 0) {
                    double tot = 0.0;
                    for (int k = 0; k < kFusedConsumerWarps; ++k) tot += sh_sum[k];
                    if (a.reduction == CE_RED_MEAN)
                        tot = (w_y_sum != 0.f) ? tot / static_cast<double>(w_y_sum) : 0.0;
                    a.loss[0] = static_cast<float>(tot);
                    a.ctl->done = 0u;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0 && S.abort) {
        pdl_wait();  // the status word is rewritten by the normaliser kernel
        atomicOr(&a.ctl->status, CE_FLAG_WAIT_TIMEOUT);
    }
    cluster_sync_all();  // no CTA leaves while a peer may still write into it
}

// ------------------------------------------------------------------ host side: plan and launch
template <int DT, int MODE, int ODT = DT>
static const void *fused_fn() {
    return reinterpret_cast<const void *>(&ce_fused_kernel<DT, MODE, ODT>);
}

static const void *fused_kernel_ptr(int dtype, int mode) {
    switch (dtype * 3 + mode) {
    case CE_DT_F32 * 3 + 0: return fused_fn<CE_DT_F32, 0>();
    case CE_DT_F32 * 3 + 1: return fused_fn<CE_DT_F32, 1>();
    case CE_DT_F32 * 3 + 2: return fused_fn<CE_DT_F32, 2>();
    case CE_DT_BF16 * 3 + 0: return fused_fn<CE_DT_BF16, 0>();
    case CE_DT_BF16 * 3 + 1: return fused_fn<CE_DT_BF16, 1>();
    case CE_DT_BF16 * 3 + 2: return fused_fn<CE_DT_BF16, 2>();
    case CE_DT_F16 * 3 + 0: return fused_fn<CE_DT_F16, 0>();
    case CE_DT_F16 * 3 + 1: return fused_fn<CE_DT_F16, 1>();
    default: return fused_fn<CE_DT_F16, 2>();
    }
}

static const void *fused_f32_to_bf16_ptr(int mode) {
    switch (mode) {
    case 0: return fused_fn<CE_DT_F32, 0, CE_DT_BF16>();
    case 1: return fused_fn<CE_DT_F32, 1, CE_DT_BF16>();
    default: return fused_fn<CE_DT_F32, 2, CE_DT_BF16>();
    }
}

// Largest row slice one CTA holds; three such CTAs share an SM.
constexpr int64_t kTargetSliceBytes = 64 * 1024;
constexpr int64_t kMaxSliceBytes = 200 * 1024;
constexpr int kMinChunkBytes = 8192;

static cudaError_t plan_for(const void *fn, int dtype, int64_t n_rows, int64_t vocab,
                            int cluster_override, FusedPlan *plan, bool *supported) {
    *supported = false;
    const int64_t esz = dtype == CE_DT_F32 ? 4 : 2;
    const int64_t vec = 16 / esz;
    int C = 1;
    if (cluster_override > 0) {
        C = cluster_override;
    } else {
        while (C < 8 && ((vocab + C - 1) / C) * esz > kTargetSliceBytes) ++C;
        if (((vocab + C - 1) / C) * esz > kTargetSliceBytes) C = 16;
    }
    if (C < 1 || C > kMaxCluster) return cudaSuccess;
    int64_t slice = (vocab + C - 1) / C;
    slice = ((slice + vec - 1) / vec) * vec;
    if (slice * (C - 1) >= vocab && C > 1) return cudaSuccess;  // a CTA would own no column
    const int64_t slice_bytes = slice * esz;
    if (slice_bytes > kMaxSliceBytes) return cudaSuccess;
    int n_chunks = static_cast<int>((slice_bytes + kMinChunkBytes - 1) / kMinChunkBytes);
    if (n_chunks > kMaxChunks) n_chunks = kMaxChunks;
    if (n_chunks < 1) n_chunks = 1;
    int chunk = static_cast<int>((slice_bytes + n_chunks - 1) / n_chunks);
    chunk = ((chunk + 15) / 16) * 16;
    if (chunk < 16) chunk = 16;
    const size_t smem = static_cast<size_t>(((slice_bytes + 127) / 128) * 128) + kFusedSmemFixed;

    // The attribute belongs to the kernel function, not to a launch: set it
    // to the largest slice any plan may use, so that every cached plan of
    // this function stays launchable.
    const size_t smem_cap = static_cast<size_t>(((kMaxSliceBytes + 127) / 128) * 128) + kFusedSmemFixed;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_cap));
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kFusedThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * sms * per_sm), 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&n_clusters, fn, &cfg);
    if (e != cudaSuccess) return e;
    if (n_clusters < 1) return cudaSuccess;
    if (n_rows > 0 && n_clusters > n_rows) n_clusters = static_cast<int>(n_rows);
    plan->cluster = C;
    plan->n_clusters = n_clusters;
    plan->ctas_per_sm = per_sm;
    plan->slice_elems = slice;
    plan->chunk_bytes = chunk;
    plan->n_chunks = n_chunks;
    plan->smem_bytes = smem;
    *supported = true;
    return cudaSuccess;
}

cudaError_t fused_plan(int dtype, int mode, int64_t n_rows, int64_t vocab, int cluster_override,
                       FusedPlan *plan, bool *supported) {
    return plan_for(fused_kernel_ptr(dtype, mode), dtype, n_rows, vocab, cluster_override, plan, supported);
}

cudaError_t fused_plan_f32_to_bf16(int mode, int64_t n_rows, int64_t vocab, FusedPlan *plan,
                                   bool *supported) {
    return plan_for(fused_f32_to_bf16_ptr(mode), CE_DT_F32, n_rows, vocab, 0, plan, supported);
}

// `after_prep`: the previous kernel on the stream is the normaliser kernel,
// which writes nothing this kernel reads before its griddepcontrol.wait, so
// the launch may overlap it. Any other predecessor (for instance the GEMM
// that writes the logits) must complete first: the producer warp reads the
// logits at once.
static cudaError_t launch_plan(const void *fn, const FusedArgs &a0, const FusedPlan &plan, cudaStream_t s,
                               bool after_prep) {
    FusedArgs a = a0;
    a.slice_elems = plan.slice_elems;
    a.chunk_bytes = plan.chunk_bytes;
    a.n_chunks = plan.n_chunks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.cluster * plan.n_clusters), 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = plan.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the normaliser kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prep ? 2 : 1;
    void *args[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_fused(const FusedArgs &a, const FusedPlan &plan, int dtype, int mode, cudaStream_t s,
                         bool after_prep) {
    return launch_plan(fused_kernel_ptr(dtype, mode), a, plan, s, after_prep);
}

cudaError_t launch_fused_f32_to_bf16(const FusedArgs &a, const FusedPlan &plan, int mode, cudaStream_t s) {
    return launch_plan(fused_f32_to_bf16_ptr(mode), a, plan, s, false);
}

}  // namespace ce
