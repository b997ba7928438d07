// ce_stream.cu -- launch of the streaming forward + backward kernel
// (ce_stream.cuh) and its instantiations for 16-byte aligned rows.
#include <mutex>

#include "ce_host.h"
#include "ce_stream.cuh"

namespace ce {

// Per (kernel, context): the dynamic shared memory attribute has been set
// and the SM count read, so a launch makes neither call again (they were a
// few microseconds of host time per call, which dominates at small batches).
static cudaError_t stream_fn_ready(const void *fn, int smem, int *dev_out, int *sms_out) {
    struct Entry {
        const void *fn;
        unsigned long long ctx;
        int dev, sms;
    };
    static Entry cache[256];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = current_context_id();
    if (ctx != 0) {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].fn == fn && cache[i].ctx == ctx && cache[i].dev == dev) {
                *dev_out = dev;
                *sms_out = cache[i].sms;
                return cudaSuccess;
            }
    }
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const unsigned long long ctx2 = current_context_id();  // current now, if it was not before
    if (ctx2 != 0) {
        std::lock_guard<std::mutex> lk(mu);
        if (used < 256) cache[used++] = Entry{fn, ctx2, dev, sms};
    }
    *dev_out = dev;
    *sms_out = sms;
    return cudaSuccess;
}

// SM count and L2 size of the current device, asked once per device.
static cudaError_t device_sms_l2(int *sms_out, int64_t *l2_out) {
    struct Entry {
        int sms, l2;
    };
    constexpr int kMaxDev = 64;
    static Entry cache[kMaxDev] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    Entry *c = dev >= 0 && dev < kMaxDev ? &cache[dev] : nullptr;
    if (!c || c->sms == 0) {
        Entry n{};
        if ((e = cudaDeviceGetAttribute(&n.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&n.l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return e;
        if (!c) {
            *sms_out = n.sms;
            *l2_out = n.l2;
            return cudaSuccess;
        }
        *c = n;
    }
    *sms_out = c->sms;
    *l2_out = c->l2;
    return cudaSuccess;
}

// The first-pass evict-first share (in sixteenths) of a launch whose second
// pass walks each row part last chunk first: the bytes waiting in L2 for
// their second pass are F = (CTAs in flight) x (bytes of a row part), and
// when F exceeds what the L2 keeps of them (about 0.8 of its size C; the
// rest holds the written gradient lines) the first 1 - 0.8 C / F of each
// part -- the chunks read again last -- are loaded under evict-first, so the
// L2 keeps the parts' later chunks, which the second pass reads first.
// GB300 (L2 135.5 MB), class-weight ring, kernel alone, CUDA events, best
// share in sixteenths against the rule's: three CTAs per SM, 456 x 500 KB
// waiting (16384 x 256000) 6-8 (flat to 10) against 9 (3.492 ms against
// 3.547 with none), 456 x 1 MB (4096 x 524288) 10-12 against 12 (1.864
// against 1.891), 456 x 320 KB 0-5 (flat) against 4, 456 x 250 KB 0-2
// against 1; two CTAs per SM, 304 x 500 KB 4-5 (flat 3-6) against 5 (3.436
// against 3.486 with none). The share is applied in eighths.
static int first_pass_drop8(int64_t ctas, int64_t part_bytes, int64_t l2) {
    const double f = static_cast<double>(ctas) * static_cast<double>(part_bytes);
    const double kept = 0.8 * static_cast<double>(l2);
    if (l2 <= 0 || f <= kept) return 0;
    const int k = static_cast<int>(8.0 * (1.0 - kept / f) + 0.5);
    return k < 0 ? 0 : (k > 7 ? 7 : k);
}

// Resident clusters of a kernel on a device (0 if unknown), asked once per
// kernel and device.
static int max_active_clusters(const void *fn, int dev, const cudaLaunchConfig_t &cfg) {
    struct Entry {
        const void *fn;
        int dev, n;
    };
    static Entry cache[128];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev) return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    (void)cudaGetLastError();
    if (used < 128) cache[used++] = Entry{fn, dev, n};
    return n;
}

// The class-weight ring shapes (SHAPE 3 and 4): aligned bf16 / f16 rows
// with class-weighted smoothing and no options.
template <int SHAPE, int CL>
static const void *stream_kernel_wring(int dtype) {
    return dtype == CE_DT_BF16 ? reinterpret_cast<const void *>(&ce_stream_kernel<CE_DT_BF16, 2, SHAPE, CL, false, 0>)
         : dtype == CE_DT_F16  ? reinterpret_cast<const void *>(&ce_stream_kernel<CE_DT_F16, 2, SHAPE, CL, false, 0>)
                               : nullptr;
}

template <int SHAPE, int CL>
static cudaError_t launch_stream_shape(const RowArgs &a0, int dtype, int mode, int ctas_per_sm, int tune,
                                       bool after_prep, cudaStream_t s, bool fwd = false) {
    using SH = StreamShape<SHAPE>;
    RowArgs a = a0;
    // rows that all start on a 16-byte boundary take the fixed-geometry instantiation
    const int64_t esz = dtype == CE_DT_F32 ? 4 : 2;
    const bool ragged = (reinterpret_cast<uintptr_t>(a.grad) & 15u) != 0 || (a.n_rows > 1 && ((a.ld * esz) & 15) != 0);
    const bool opts = a.softcap > 0.f || a.z_loss > 0.f || a.accuracy;
    const void *fn = nullptr;
    if (fwd) {
        if (SHAPE != 2 || CL != 1 || mode == 2 || opts) return cudaErrorInvalidValue;
        fn = stream_kernel_forward(dtype, mode, ragged);
    } else if constexpr (SHAPE == 3 || SHAPE == 4) {
        // the weight ring copies whole 32-byte weight vectors from 16-byte aligned weights
        const bool ok = mode == 2 && !ragged && !opts && dtype != CE_DT_F32 && a.weight &&
                        (reinterpret_cast<uintptr_t>(a.weight) & 15u) == 0;
        if (!ok) return launch_stream_shape<2, CL>(a0, dtype, mode, ctas_per_sm, tune, after_prep, s);
        fn = stream_kernel_wring<SHAPE, CL>(dtype);
    } else {
        fn = a.softcap > 0.f ? stream_kernel_softcap(dtype, mode, SHAPE, CL, ragged)
           : opts ? stream_kernel_options(dtype, mode, SHAPE, CL, ragged)
           : ragged ? stream_kernel_ragged(dtype, mode, SHAPE, CL) : stream_kernel_for<false>(dtype, mode, SHAPE, CL);
    }
    if (!fn) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = stream_fn_ready(fn, SH::kSmem, &dev, &sms);
    if (e != cudaSuccess) return e;
    int64_t grid = static_cast<int64_t>(sms) * (ctas_per_sm > 0 ? ctas_per_sm : SH::kCtasPerSm);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(SH::kThreads);
    cfg.dynamicSmemBytes = SH::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute cl_attr;
    if (CL > 1) {
        // the kernel is persistent: no more clusters than can be resident at once
        // (clusters are placed within a GPC, so fewer may fit than SMs x CTAs per SM)
        cl_attr.id = cudaLaunchAttributeClusterDimension;
        cl_attr.val.clusterDim.x = CL;
        cl_attr.val.clusterDim.y = 1;
        cl_attr.val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(grid / CL * CL));
        cfg.attrs = &cl_attr;
        cfg.numAttrs = 1;
        const int max_clusters = max_active_clusters(fn, dev, cfg);
        if (max_clusters > 0 && static_cast<int64_t>(max_clusters) * CL < grid)
            grid = static_cast<int64_t>(max_clusters) * CL;
    }
    if (grid > a.n_rows * CL) grid = a.n_rows * CL;
    grid = grid / CL * CL;
    if (grid < CL) grid = CL;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (CL > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = CL;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (after_prep) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    void *args[] = {&a, &tune};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// The forward only: one CTA per row and three CTAs per SM (rows are read
// once, so nothing waits in L2 and a pair's exchange would only add work).
cudaError_t launch_stream_forward(const RowArgs &a, int dtype, int mode, bool after_prep, cudaStream_t s) {
    return launch_stream_shape<2, 1>(a, dtype, mode, 0, kTuneThree | kTuneNoKeep, after_prep, s, true);
}

cudaError_t launch_stream(const RowArgs &a, int dtype, int mode, int ctas_per_sm, int tune, bool after_prep,
                          cudaStream_t s) {
    // Library choice by row size (GB300 measurements, CUDA events, L2 flushed):
    //  rows <= 176 KB: three CTAs per SM, one CTA per row (4096 x 32000 bf16:
    //    0.102 ms vs 0.121 ms with two CTAs per SM; 8192 x 50257: 0.300 vs
    //    0.398 ms for pairs, x 64000 0.372 vs 0.441, x 80000 0.484 vs 0.502,
    //    x 88000 0.545 vs 0.549, x 96000 0.611 vs 0.587);
    //  rows <= 384 KB: three CTAs per SM, a pair of CTAs per row, so the
    //    second pass is served by L2, walking each half row last chunk first
    //    (8192 x 128256 bf16: 0.746 ms; 0.749 ms first chunk first; 0.775 ms
    //    unpaired; 0.827 ms paired at two CTAs per SM);
    //  bf16 / f16 rows <= 512 KB (<= 640 KB without class-weighted
    //    smoothing; with it from 288 KB: 8192 x 150000 1.39 vs 1.48 ms for
    //    pairs, x 180000 1.60 vs 1.81, x 196608 1.64 vs 1.98, kernel alone;
    //    x 128256 1.25 vs 1.01): three CTAs per SM, a cluster of four per row, each
    //    streaming a quarter, second pass last chunk first: the 114 rows in
    //    flight keep 58 MB waiting in L2 at 512 KB (16384 x 256000 bf16 with
    //    class weights: 4.42 ms vs 4.63 ms for 16-warp pairs; 8192 x 256000:
    //    1.513 vs 1.675 ms; 8192 x 320000: 1.878 vs 2.013 ms; with class
    //    weights at 640 KB 4.80 vs 4.45 ms, whose pass-2 weight loads add to
    //    the L2 traffic; 8192 x 256000 with softcap 30: 2.673 vs 2.907 ms,
    //    with z-loss and accuracy 1.626 vs 1.930 ms; 16384 x 256000 with
    //    class weights and softcap 30: 7.087 vs 7.045 ms);
    //  larger rows, and fp32 rows over 384 KB: one 16-warp CTA per SM, a
    //    pair per row: the half rows waiting in L2 for their second pass fit
    //    with room to spare (8192 x 448000: 2.708 ms vs 2.728 for quads;
    //    fp32 8192 x 128256: 1.408 ms vs 1.455 for quads, fewer elements per
    //    byte needing fewer warps; three CTAs per SM in pairs at 16384 x
    //    256000: 117 MB waiting, bimodal 4.3 / 5.4 ms).
    //  In every case the first pass carries no L2 evict-last hint: with the
    //  hint the second pass missed more (8192 x 128256: 9.5% reads over the
    //  algorithmic bytes against 5.3%; 16384 x 256000: 4.93 ms against 4.50),
    //  while the second pass keeps its evict-first hint (without it 0.762 ms).
    const bool opts = a.softcap > 0.f || a.z_loss > 0.f || a.accuracy;
    // Class-weighted smoothing on aligned bf16 / f16 rows: the class weights
    // of the second pass go through the shared-memory weight ring, one CTA
    // per row, the second pass last chunk first, at every row size (GB300,
    // CUDA events, kernel alone: 8192 x 64000 0.525 ms against 0.538 for the
    // per-lane loads; 8192 x 128256 0.995 against 1.020 (per-lane pairs);
    // 8192 x 163840 1.195 against 1.246 for ring pairs, x 196608 1.439
    // against 1.479, x 229376 1.672 against 1.713; 16384 x 256000 3.695
    // against 3.819 for ring pairs, 4.25 for ring quads, 4.14 for per-lane
    // quads; 8192 x 320000 2.371 against 2.414 for ring pairs; 4096 x 400000
    // 1.501 against 1.513 for ring pairs and 2.183 for 16-warp per-lane
    // pairs, x 524288 1.941 against 1.953 and 3.094). Its second pass misses
    // L2 more (456 rows wait there), but a row needs no exchange between CTAs.
    // The ring runs at two CTAs per SM with two weight vectors per thread in a
    // weight slot (304 rows waiting, half the weight-slot hand-overs; kernel
    // alone, with the evict-first share, against three CTAs per SM with one:
    // 8192 x 64000 0.440 ms against 0.457, x 128256 0.839 against 0.899,
    // 16384 x 256000 3.339 against 3.476, 4096 x 393216 1.347 against 1.386,
    // x 524288 1.810 against 1.852).
    const int64_t esz = dtype == CE_DT_F32 ? 4 : 2;
    const bool ragged = (reinterpret_cast<uintptr_t>(a.grad) & 15u) != 0 || (a.n_rows > 1 && ((a.ld * esz) & 15) != 0);
    const bool wring_ok = mode == 2 && !opts && dtype != CE_DT_F32 && !ragged && a.weight &&
                          (reinterpret_cast<uintptr_t>(a.weight) & 15u) == 0;
    const bool auto_tune = tune == 0;
    if (tune == 0 && wring_ok) {
        tune = kTuneThree | kTuneNoKeep | kTuneReverse | kTuneWRing | kTuneWRing2;
    }
    if (tune == 0) {
        const int64_t row_bytes = a.vocab * (dtype == CE_DT_F32 ? 4 : 2);
        const int64_t quad_max = (mode == 2 ? 512 : 640) * 1024;
        // class-weighted smoothing leaves the pairs earlier (its pass-2 weight
        // loads hold each row longer in L2)
        const int64_t pair_max = (mode == 2 ? 288 : 384) * 1024;
        tune = row_bytes <= 176 * 1024 ? (kTuneThree | kTuneNoKeep)
             : row_bytes <= pair_max ? (kTuneThree | kTuneCluster2 | kTuneNoKeep | kTuneReverse)
             : (dtype != CE_DT_F32 && row_bytes <= quad_max) ? (kTuneThree | kTuneCluster4 | kTuneNoKeep | kTuneReverse)
                                     : (kTuneWide | kTuneCluster2 | kTuneNoKeep);
    }
    const int vec = dtype == CE_DT_F32 ? 4 : 8;
    const bool pair = (tune & kTuneCluster2) && a.vocab >= 2 * vec;
    const bool quad = (tune & kTuneCluster4) && a.vocab >= 4 * vec;
    if (auto_tune && (tune & kTuneReverse)) {
        int sms = 0;
        int64_t l2 = 0;
        if (device_sms_l2(&sms, &l2) == cudaSuccess) {
            const int cl = quad ? 4 : (pair ? 2 : 1);
            const bool ring = (tune & kTuneThree) && (tune & kTuneWRing) && wring_ok;
            const int per_sm = ctas_per_sm > 0 ? ctas_per_sm
                             : (tune & kTuneWide) ? StreamShape<1>::kCtasPerSm
                             : (ring && (tune & kTuneWRing2) && cl == 1) ? StreamShape<4>::kCtasPerSm
                             : ring ? StreamShape<3>::kCtasPerSm
                             : (tune & kTuneThree) ? StreamShape<2>::kCtasPerSm : StreamShape<0>::kCtasPerSm;
            int64_t ctas = static_cast<int64_t>(sms) * per_sm;
            if (ctas > a.n_rows * cl) ctas = a.n_rows * cl;
            const int64_t part = ((a.vocab + cl - 1) / cl) * esz;
            tune |= first_pass_drop8(ctas, part, l2) << kTuneDropShift;
        }
    }
    if (opts) {
        // the options are built for the four shapes the library picks by row size
        if ((tune & kTuneWide) && pair) return launch_stream_shape<1, 2>(a, dtype, mode, ctas_per_sm, tune, after_prep, s);
        return quad ? launch_stream_shape<2, 4>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
             : pair ? launch_stream_shape<2, 2>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
                    : launch_stream_shape<2, 1>(a, dtype, mode, ctas_per_sm, tune, after_prep, s);
    }
    if (tune & kTuneWide)
        return pair ? launch_stream_shape<1, 2>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
                    : launch_stream_shape<1, 1>(a, dtype, mode, ctas_per_sm, tune, after_prep, s);
    if ((tune & kTuneThree) && (tune & kTuneWRing))
        return quad ? launch_stream_shape<3, 4>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
             : (!pair && (tune & kTuneWRing2)) ? launch_stream_shape<4, 1>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
             : pair ? launch_stream_shape<3, 2>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
                    : launch_stream_shape<3, 1>(a, dtype, mode, ctas_per_sm, tune, after_prep, s);
    if (tune & kTuneThree)
        return quad ? launch_stream_shape<2, 4>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
             : pair ? launch_stream_shape<2, 2>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
                    : launch_stream_shape<2, 1>(a, dtype, mode, ctas_per_sm, tune, after_prep, s);
    return pair ? launch_stream_shape<0, 2>(a, dtype, mode, ctas_per_sm, tune, after_prep, s)
                : launch_stream_shape<0, 1>(a, dtype, mode, ctas_per_sm, tune, after_prep, s);
}

}  // namespace ce
