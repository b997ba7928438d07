// ce_stream.cuh -- streaming forward + backward: each CTA (or CTA pair) owns
// whole rows and a producer warp streams every row through a ring of
// shared-memory chunks twice, with 1-D bulk async copies:
//   pass 1 (statistics): the row comes from HBM (no L2 hint by default; an
//          evict-last hint is a tuning bit, measured slower);
//   pass 2 (gradient):   the same bytes again, now served by L2 under an
//          evict-first hint (in the one-CTA and pair shapes the last four
//          chunks of a row part stay in the ring and are read there), while
//          the consumer warps write the fp32 gradient, rounded once, over
//          the logits.
// The ring is not tied to a row: while the consumers merge a row's
// statistics, the producer keeps copying (the row's pass-2 chunks and the
// next row's pass-1 chunks), so the memory system never idles between
// phases, and the bytes in flight are set by the ring, not by registers.
// HBM sees one read and one write per element; the L2 holds about one row
// per CTA pair between the passes.
//
// With a cluster of two (or four) CTAs per row, each CTA streams half (a
// quarter) of the row and the parts' statistics are exchanged through
// distributed shared memory (st.shared::cluster + a remote mbarrier arrive),
// which divides the bytes each CTA keeps waiting in L2 for its second pass.
//
// Rows at any alignment: the part of a row before its first 16-byte boundary
// and after its last goes through plain accesses (RAG instantiations). The
// options (softcap, z-loss, token accuracy) have their own instantiations
// (OPT). Every wait is bounded.
#pragma once

#include <type_traits>

#include "ce_device.cuh"
#include "ce_kernels.h"

namespace ce {

// Five shapes: 8 consumer warps and a 6-slot ring (two CTAs per SM);
// 16 consumer warps and a 12-slot ring (one CTA per SM, half the rows
// waiting in L2 for their second pass); 8 consumer warps and a 4-slot ring
// (three CTAs per SM, more warps to cover a cluster exchange); and, for
// bf16 / f16 rows with class-weighted smoothing, a 3-slot ring plus a 3-slot
// ring of class weights, at three CTAs per SM with one weight vector per
// consumer thread in a weight slot (SHAPE 3, 8 KB slots) or at two CTAs per
// SM with two (SHAPE 4, 16 KB slots: a third fewer rows waiting in L2 for
// their second pass and half the weight-slot hand-overs; the library's
// choice at every row size). A second producer lane bulk-copies the fp32 weights of
// each second-pass chunk into shared memory, so the gradient loop reads them
// from shared memory instead of waiting on per-lane loads.
constexpr int kStreamChunk = 16384;  // bytes per ring slot
constexpr int kStreamMaxSlots = 12;
constexpr int kStreamCtlBytes = 2048;  // control block after the rings
constexpr int kStreamWSlots = 3;  // class-weight slots (at most)
constexpr float kFoldMax = 32.f;  // |c| below which the gradient's exponent folds m into one FMA (below)
// Suspend-time hints of the kernel's mbarrier waits (0: spin). The
// producer sleeps while it waits for a free slot: a spinning producer takes
// issue slots from the consumer warps of its scheduler (GB300, CUDA events:
// 8192 x 128256 bf16 0.749 -> 0.745 ms, 4096 x 32000 0.102 -> 0.100 ms).
// The consumers spin on data and on the cluster exchange (sleeping there
// cost 8192 x 128256 2%: a sleeping warp wakes late), except with the
// class-weight ring, whose consumers wait on it once per weight vector and
// gain from sleeping (16384 x 256000 weighted pairs 3.92 -> 3.87 ms).
#ifndef CE_STREAM_PRODUCER_WAIT_NS
#define CE_STREAM_PRODUCER_WAIT_NS 5000
#endif
#ifndef CE_STREAM_CONSUMER_WAIT_NS
#define CE_STREAM_CONSUMER_WAIT_NS 0
#endif
#ifndef CE_STREAM_WRING_CONSUMER_WAIT_NS
#define CE_STREAM_WRING_CONSUMER_WAIT_NS 5000
#endif
constexpr uint32_t kStreamSleepP = CE_STREAM_PRODUCER_WAIT_NS;
constexpr uint32_t kStreamSleepConsumer = CE_STREAM_CONSUMER_WAIT_NS;
constexpr uint32_t kStreamSleepConsumerW = CE_STREAM_WRING_CONSUMER_WAIT_NS;
template <int SHAPE> struct StreamShape {
    static constexpr int kWarps = SHAPE == 1 ? 16 : 8;
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kSlots = SHAPE == 0 ? 6 : (SHAPE == 1 ? 12 : (SHAPE == 2 ? 4 : 3));
    static constexpr int kCtasPerSm = SHAPE == 0 ? 2 : (SHAPE == 1 ? 1 : (SHAPE == 4 ? 2 : 3));
    static constexpr int kWSlots = SHAPE >= 3 ? kStreamWSlots : 0;  // class-weight ring
    // weight vectors per consumer thread in one class-weight slot (a piece)
    static constexpr int kWVecs = SHAPE == 4 ? 2 : 1;
    static constexpr int kWSlotBytes = kWVecs * kWarps * 32 * 32;  // one 32-byte weight vector per thread
    static constexpr int kSmem = kSlots * kStreamChunk + kWSlots * kWSlotBytes + kStreamCtlBytes;
};

struct StreamXSlot {      // one CTA's partial of one row (32 bytes)
    float m, s, r, n;
    float xy, pad0, pad1, pad2;
};

struct StreamSmem {
    uint64_t full[kStreamMaxSlots];
    uint64_t empty[kStreamMaxSlots];
    uint64_t wfull[kStreamWSlots];   // class-weight ring (SHAPE 3)
    uint64_t wempty[kStreamWSlots];
    uint64_t xbar[2];
    StreamXSlot slot[2][4];  // [row parity][CTA of the cluster]
    // per row parity: a warp may write the next row's values while a slower
    // warp still reads this row's (never further ahead: the row's barrier
    // waits for every warp)
    RowState red[2][16];    // per-warp partial states of pass 1
    float2 defer[2][16];    // class-weighted smoothing: per-warp {sum w x, sum w} of pass 2
    ArgMax am[2][16];       // token accuracy: per-warp first column of the row maximum
    float xy[2];            // the target logit
    int abort;
    double cta_sum;         // this CTA's row losses (first CTA of a cluster; thread 0 only)
};
static_assert(sizeof(StreamSmem) <= kStreamCtlBytes, "stream control block too large");

// tuning bits (ce_params.variant >> CE_VARIANT_TUNE_SHIFT)
constexpr int kTuneWide = 1;       // 16 consumer warps, one CTA per SM
constexpr int kTuneReverse = 2;    // second pass walks the row's chunks last to first
constexpr int kTuneNoKeep = 4;     // first pass without the L2 evict-last policy
constexpr int kTuneCluster2 = 8;   // a cluster of two CTAs per row, each streaming half
constexpr int kTuneThree = 16;     // three CTAs per SM with a 4-slot ring
constexpr int kTuneCluster4 = 32;  // a cluster of four CTAs per row (three CTAs per SM)
constexpr int kTuneWRing = 64;     // with 16, class-weighted smoothing: weights through a shared-memory ring
// bits 7..9: how many eighths of each row part's first-pass chunks (the
// first ones, which a reversed second pass reads last) carry an L2
// evict-first hint, so that where the rows waiting for their second pass
// exceed the L2 the lines given up are those least likely to be read again
constexpr int kTuneDropShift = 7;
constexpr int kTuneWRing2 = 1024;  // with 64 and one CTA per row: the weight ring at two CTAs per SM

template <int NCW>
__device__ inline void stream_consumer_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(NCW * 32) : "memory");
}

__device__ inline void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}
__device__ inline uint64_t createpolicy_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ inline uint64_t policy_keep() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Where one row's slice [lo, lo + L) sits against 16-byte boundaries: the
// head (columns before the first boundary, at most 15 bytes) and the tail
// (after the last) are read and written with plain accesses; the interior
// [vlo, tail0) moves with bulk copies and 16-byte vectors. Rows whose start
// is 16-byte aligned have no head.
struct RowGeom {
    int64_t vlo, tail0;  // first column of the interior, first column of the tail
    int nhead, ntail, nvec, nch;
    int64_t bytes;       // interior bytes (a multiple of 16)
};
template <int KB>
__device__ inline RowGeom row_geom(const char *slice, int64_t lo, int64_t L) {
    RowGeom g;
    const int64_t hb = static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(slice) & 15u)) & 15u);
    const int64_t nh = hb / KB < L ? hb / KB : L;
    g.nhead = static_cast<int>(nh);
    g.vlo = lo + nh;
    g.bytes = ((L - nh) * KB) & ~static_cast<int64_t>(15);
    g.nvec = static_cast<int>(g.bytes / 16);
    g.tail0 = g.vlo + g.bytes / KB;
    g.ntail = static_cast<int>(lo + L - g.tail0);
    g.nch = static_cast<int>((g.bytes + kStreamChunk - 1) / kStreamChunk);
    return g;
}

// the same for a slice that starts on a 16-byte boundary
template <int KB>
__device__ inline RowGeom row_geom_aligned(int64_t lo, int64_t L) {
    RowGeom g;
    g.nhead = 0;
    g.vlo = lo;
    g.bytes = (L * KB) & ~static_cast<int64_t>(15);
    g.nvec = static_cast<int>(g.bytes / 16);
    g.tail0 = g.vlo + g.bytes / KB;
    g.ntail = static_cast<int>(lo + L - g.tail0);
    g.nch = static_cast<int>((g.bytes + kStreamChunk - 1) / kStreamChunk);
    return g;
}

// 4 class weights starting at column c (c a multiple of 4 when vec4)
__device__ inline float4 load_w4(const float *w, int64_t c, bool vec4) {
    if (vec4) return __ldg(reinterpret_cast<const float4 *>(w + c));
    return make_float4(__ldg(w + c), __ldg(w + c + 1), __ldg(w + c + 2), __ldg(w + c + 3));
}
// 8 class weights at a 32-byte aligned address, one 256-bit read-only load
// (one full sector per lane instead of two half-sector loads)
__device__ inline void load_w8(const float *p, float4 &lo, float4 &hi) {
    asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z), "=f"(hi.w)
                 : "l"(p));
}

// A row's loss: stored per row for reduction none (and, for a batch
// reduction left to a later kernel, in the workspace), else added in fp64 to
// the CTA's sum, in row order; the CTA's sum goes to the workspace at the end
// and the last CTA adds those up. Called by the first CTA of the row only.
__device__ inline void put_row_loss(const RowArgs &a, int64_t row, float loss, double &cta_sum) {
    if (a.reduction == CE_RED_NONE) a.loss[row] = loss;
    else if (a.no_finalize) a.row_loss[row] = loss;
    else cta_sum += static_cast<double>(loss);
}

// The loss of a row whose class-weighted smoothing sum (r = sum w x over the
// whole row) arrived after its gradient pass; the weight sum over the row is
// W_all, the normaliser kernel's (fp64) sum of the class weights.
__device__ inline float deferred_loss(float m, float s, float xy, float r, int yg, float wy, float w_all, float eps,
                                      float inv_v, float z_loss) {
    const float rrel = w_all > 0.f ? __fsub_rn(r, __fmul_rn(w_all, m)) : 0.f;
    return make_row_scalars(m, s, xy, rrel, true, yg, wy, w_all, eps, inv_v, 1.f, z_loss).loss;
}

// RAG: rows may start off a 16-byte boundary (per-row head and tail);
// without it every row of the launch is 16-byte aligned and the geometry is
// fixed for the whole launch. OPT 1: z-loss and token accuracy (the argmax
// of the raw logits, the same column as that of the capped ones since tanh
// is increasing); OPT 2: the same plus softcap (every logit becomes
// c tanh(x / c), the gradient gains the factor 1 - (z / c)^2). Softcap has
// its own instantiations: its tanh evaluation, inlined into the element
// loops, costs instruction-cache room even when it is not taken.
template <int DT, int MODE, int SHAPE, int CL, bool RAG, int OPT = 0>
__global__ void __launch_bounds__(StreamShape<SHAPE>::kThreads, StreamShape<SHAPE>::kCtasPerSm)
ce_stream_kernel(RowArgs a, int tune) {
    using F = Fmt<DT>;
    using SH = StreamShape<SHAPE>;
    constexpr int NCW = SH::kWarps;
    constexpr int VEC = F::kVec;
    constexpr bool SMOOTH = MODE != 0;
    // Class-weighted smoothing needs sum_c w_c x_c, which only the loss uses:
    // it is summed in pass 2 (where w_c is loaded for the gradient anyway)
    // instead of pass 1, and the row's loss is completed at the next row's
    // merge (or after the last row), so pass 1 reads no weights.
    constexpr bool DEFER = MODE == 2;
    constexpr bool P1S = SMOOTH && !DEFER;   // smoothing sums in pass 1
    constexpr int kStreamConsumerWarps = NCW;
    constexpr int kStreamSlots = SH::kSlots;
    constexpr int kWS = SH::kWSlots;
    constexpr int kWV = SH::kWVecs;
    constexpr bool WR = kWS > 0;  // class weights of pass 2 through the weight ring
    constexpr uint32_t kStreamSleepC = WR ? kStreamSleepConsumerW : kStreamSleepConsumer;
    static_assert(!WR || (MODE == 2 && !RAG && VEC == 8 && OPT == 0),
                  "the class-weight ring serves aligned bf16 / f16 rows with class-weighted smoothing");
    constexpr int NCT = NCW * 32;
    constexpr int VPC = kStreamChunk / 16;          // vectors per full chunk
    constexpr int VPT = VPC / NCT;                  // vectors per thread per full chunk
    static_assert(VPC % NCT == 0, "chunk must split evenly over the consumers");
    static_assert(CL == 1 || CL == 2 || CL == 4, "one, two or four CTAs per row");
    static_assert((NCW & (NCW - 1)) == 0 && NCW <= 32, "the warp partials merge in groups of NCW lanes");

    extern __shared__ __align__(128) uint8_t smem[];
    StreamSmem &S = *reinterpret_cast<StreamSmem *>(smem + kStreamSlots * kStreamChunk + kWS * SH::kWSlotBytes);
    const uint32_t ring = smem_u32(smem);
    const uint32_t wring = ring + kStreamSlots * kStreamChunk;  // class-weight slots (SHAPE 3)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t V = a.vocab;
    // this CTA's columns [lo, hi) of every row: all of it, or one half
    const uint32_t rank = CL == 1 ? 0u : cluster_ctarank();
    const int64_t q0 = CL == 1 ? blockIdx.x : cluster_id_x();
    const int64_t nq = CL == 1 ? gridDim.x : nclusters_x();
    // columns per CTA (a multiple of the vector width, so every part starts on a vector)
    const int64_t half = CL == 1 ? V : ((V + CL - 1) / CL + VEC - 1) / VEC * VEC;
    const int64_t lo = rank * half;
    const int64_t hi = (lo + half < V) ? lo + half : V;
    const int64_t L = hi > lo ? hi - lo : 0;
    const size_t row_bytes = static_cast<size_t>(a.ld) * F::kBytes;
    char *const xbase = reinterpret_cast<char *>(a.grad);
    // weights as float4 when the base allows it (each row's interior start decides the rest)
    const bool w_base16 = (reinterpret_cast<uintptr_t>(a.weight) & 15u) == 0;
    const bool w_base32 = (reinterpret_cast<uintptr_t>(a.weight) & 31u) == 0;
    const RowGeom g_aligned = row_geom_aligned<F::kBytes>(lo, L);
    // OPT 3: the forward only (ce_forward): one pass over every row, ignored
    // rows included, writing the row statistics and losses; no options
    constexpr bool FWD = OPT == 3;
    constexpr bool FEAT = OPT == 1 || OPT == 2;
    constexpr bool CAPF = OPT == 2;
    constexpr bool TGT_AFTER = !CAPF && CL == 1;  // the target element stored after the gradient loop
    // one CTA or a pair per row in the three-per-SM shape: the last
    // kStreamSlots chunks of a row part (all of a part of at most that many)
    // stay in the ring between the passes; the second pass reads them there
    // first, then the earlier chunks copied again from L2
    constexpr bool KEEPABLE = CL <= 2 && SHAPE == 2 && OPT == 0;
    static_assert(!FWD || (MODE != 2 && CL == 1), "the forward-only kernel: one CTA per row, no class-weighted smoothing");
    const float cap = CAPF ? a.softcap : 0.f;
    const float inv_cap = CAPF && cap > 0.f ? 1.f / cap : 0.f;
    const float nic2 = -(inv_cap * inv_cap);
    const float zl = FEAT ? a.z_loss : 0.f;
    const bool want_am = FEAT && a.accuracy != nullptr;
    // weight pieces are bulk-copied from the weights' 16-byte aligned start
    // plus whole 32-byte vectors of the (aligned) part
    const bool wr = WR && w_base16;

    if (tid == 0) {
        for (int s = 0; s < kStreamSlots; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);
            mbar_init(smem_u32(&S.empty[s]), kStreamConsumerWarps);
        }
        for (int s = 0; s < kWS; ++s) {
            mbar_init(smem_u32(&S.wfull[s]), 1);
            mbar_init(smem_u32(&S.wempty[s]), kStreamConsumerWarps);
        }
        mbar_init(smem_u32(&S.xbar[0]), CL);
        mbar_init(smem_u32(&S.xbar[1]), CL);
        S.abort = 0;
        S.cta_sum = 0.0;
        fence_mbar_init_cluster();
    }
    __syncthreads();
    if (CL > 1) cluster_sync_all();  // the peer's barriers exist before any remote arrive
    volatile int *abort = &S.abort;

    const bool reverse = (tune & kTuneReverse) != 0;
    if (warp == kStreamConsumerWarps) {
        // -------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t drop = policy_evict_first();
            const uint64_t keep = (tune & kTuneNoKeep) ? createpolicy_normal() : policy_keep();
            const int drop8 = (tune >> kTuneDropShift) & 7;
            const uint64_t hold = policy_keep();  // evict-last
            uint32_t it = 0;
            // each row's target is loaded one row ahead, so its latency hides under the previous row
            int64_t t_next = q0 < a.n_rows ? load_target(a.target, a.tgt32, q0) : 0;
            for (int64_t row = q0; row < a.n_rows; row += nq) {
                const int64_t t = t_next;
                if (row + nq < a.n_rows) t_next = load_target(a.target, a.tgt32, row + nq);
                if (!FWD && !target_valid(t, a.ignore_index, V)) continue;
                const char *slice = xbase + row * row_bytes + lo * F::kBytes;
                const RowGeom gm = RAG ? row_geom<F::kBytes>(slice, lo, L) : g_aligned;
                const char *src = slice + static_cast<int64_t>(gm.nhead) * F::kBytes;
                const int nch = gm.nch;
                const int ndrop = (nch * drop8) >> 3;
                const int nkeep = KEEPABLE ? min(nch, kStreamSlots) : 0;  // chunks the second pass reads in the ring
                for (int pass = 0; pass < (FWD ? 1 : 2); ++pass) {
                    for (int k = 0; k < (pass == 0 ? nch : nch - nkeep); ++k, ++it) {
                        const int c = (pass == 1 && reverse) ? nch - nkeep - 1 - k : k;
                        // evict-first for the second pass and the evict-first share; with
                        // chunks kept in the ring, evict-last for the earlier ones, which
                        // the second pass copies again from L2
                        const uint64_t pol = pass == 1 || c < ndrop ? drop : (nkeep > 0 && c < nch - nkeep ? hold : keep);
                        const uint32_t s = it % kStreamSlots, r = it / kStreamSlots;
                        if (r > 0) mbar_wait_bounded<false, kStreamSleepP>(smem_u32(&S.empty[s]), (r - 1) & 1u, abort);
                        const int64_t off = static_cast<int64_t>(c) * kStreamChunk;
                        const uint32_t bytes =
                            static_cast<uint32_t>(gm.bytes - off < kStreamChunk ? gm.bytes - off : kStreamChunk);
                        mbar_expect_tx(smem_u32(&S.full[s]), bytes);
                        bulk_g2s_hint(ring + s * kStreamChunk, src + off, bytes, smem_u32(&S.full[s]), pol);
                    }
                }
            }
            // drain: every issued copy has landed before the CTA may exit
            for (uint32_t k = 0; k < kStreamSlots && k < it; ++k) {
                const uint32_t i = it - 1 - k;
                mbar_wait_bounded<false, kStreamSleepP>(smem_u32(&S.full[i % kStreamSlots]), (i / kStreamSlots) & 1u, abort);
            }
        } else if (WR && lane == 1 && wr) {
            // class-weight producer: for every second-pass chunk, in the consumers'
            // order, the weights of its vectors in pieces of kWV vectors per consumer
            // thread (kWV x 8 KB), kept in L2 (every row reads them again)
            const uint64_t wpol = policy_keep();
            uint32_t wi = 0;
            int64_t t_next = q0 < a.n_rows ? load_target(a.target, a.tgt32, q0) : 0;
            const int nch = g_aligned.nch, nvec = g_aligned.nvec;
            const float *wsrc = a.weight + g_aligned.vlo;
            for (int64_t row = q0; row < a.n_rows; row += nq) {
                const int64_t t = t_next;
                if (row + nq < a.n_rows) t_next = load_target(a.target, a.tgt32, row + nq);
                if (!target_valid(t, a.ignore_index, V)) continue;
                for (int k = 0; k < nch; ++k) {
                    const int c = reverse ? nch - 1 - k : k;
                    const int v0 = c * VPC;
                    const int nv = min(VPC, nvec - v0);
                    for (int q = 0; q * NCT * kWV < nv; ++q, ++wi) {
                        const uint32_t s = wi % kWS, r = wi / kWS;
                        if (r > 0) mbar_wait_bounded<false, kStreamSleepP>(smem_u32(&S.wempty[s]), (r - 1) & 1u, abort);
                        const int nvq = min(NCT * kWV, nv - q * NCT * kWV);
                        const uint32_t bytes = static_cast<uint32_t>(nvq * VEC * 4);
                        mbar_expect_tx(smem_u32(&S.wfull[s]), bytes);
                        bulk_g2s_hint(wring + s * SH::kWSlotBytes, wsrc + static_cast<int64_t>(v0 + q * NCT * kWV) * VEC,
                                      bytes, smem_u32(&S.wfull[s]), wpol);
                    }
                }
            }
            for (uint32_t k = 0; k < static_cast<uint32_t>(kWS) && k < wi; ++k) {
                const uint32_t i = wi - 1 - k;
                mbar_wait_bounded<false, kStreamSleepP>(smem_u32(&S.wfull[i % kWS]), (i / kWS) & 1u, abort);
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------- consumers
        const float inv_v = 1.f / static_cast<float>(V);
        const float eps = a.eps;
        bool have_norm = false;
        float w_all = 0.f, w_y_sum = 0.f, g_all = 1.f;  // batch constants, read once
        // the row whose loss still waits for its deferred smoothing sums (class weights)
        bool pend = false;
        int64_t pend_row = 0;
        float pend_m = 0.f, pend_s = 0.f, pend_xy = 0.f, pend_wy = 0.f;
        int pend_yg = 0;
        uint32_t it = 0, j = 0;  // ring position; valid rows done (exchange parity)
        uint32_t wsl = 0, wph = 0;  // class-weight ring slot and phase (SHAPE 3 and 4)
        double &cta_sum = S.cta_sum;  // kept in shared memory: no registers to spare
        int64_t t_next = q0 < a.n_rows ? load_target(a.target, a.tgt32, q0) : 0;  // one row ahead
        for (int64_t row = q0; row < a.n_rows; row += nq) {
            const int64_t t = t_next;
            if (row + nq < a.n_rows) t_next = load_target(a.target, a.tgt32, row + nq);
            const bool valid = target_valid(t, a.ignore_index, V);
            char *rowp = xbase + row * row_bytes;
            const RowGeom gm = RAG ? row_geom<F::kBytes>(rowp + lo * F::kBytes, lo, L) : g_aligned;
            const int nvec = gm.nvec, nch = gm.nch, nedge = gm.nhead + gm.ntail;
            const int64_t vlo = gm.vlo;
            // the column a plain-access thread owns: head columns first, then the tail
            const int64_t edge_c = tid < gm.nhead ? lo + tid : gm.tail0 + (tid - gm.nhead);
            uint4 *vp = reinterpret_cast<uint4 *>(rowp + vlo * F::kBytes);
            const bool w4 = w_base16 && (vlo & 3) == 0;
            const bool w8 = VEC == 8 && w_base32 && (vlo & 7) == 0;  // 8 weights per vector, one load
            if (!valid && !FWD) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int v = tid; v < nvec; v += NCT) st_stream(vp + v, z);
                if (tid < nedge) F::store1(rowp, edge_c, 0.f);
                if (tid == 0 && rank == 0) put_row_loss(a, row, 0.f, cta_sum);
                continue;
            }
            // (the forward-only kernel reads ignored rows too: no target column there)
            const int yg = valid ? static_cast<int>(t) : 0;     // target column in the row
            const uint32_t rp = j & 1u;                         // parity of this row
            // target column relative to the interior (far outside when it is not in it)
            const int y = (valid && t >= vlo && t < gm.tail0) ? static_cast<int>(t - vlo) : -(1 << 30);
            // per-row values the merge needs, fetched now so their latency hides under pass 1
            const float g_row = (a.grad_output && a.reduction == CE_RED_NONE) ? __ldg(a.grad_output + row) : 0.f;
            const float wy = (valid && a.weight) ? __ldg(a.weight + yg) : 1.f;
            // ------------------------------------------------ pass 1: statistics
            RowState st = row_state_empty();
            ArgMax am{-INFINITY, 0x7fffffff};
            uint64_t cap_forms = 0;  // softcap: the form of chunk c (c < 32) in bits 2c, 2c+1
            const int nkeep = KEEPABLE ? min(nch, kStreamSlots) : 0;  // last chunks kept in the ring
            const uint32_t it_row = it;                               // the row's first ring position
            for (int c = 0; c < nch; ++c, ++it) {
                const uint32_t s = it % kStreamSlots;
                mbar_wait_bounded<false, kStreamSleepC>(smem_u32(&S.full[s]), (it / kStreamSlots) & 1u, abort);
                const uint32_t base_s = ring + s * kStreamChunk;
                const int v0 = c * VPC;
                const int nv = min(VPC, nvec - v0);
                // does one of this thread's vectors hold the target column?
                const unsigned q = static_cast<unsigned>(y / VEC - v0 - tid);
                const bool mine = q < static_cast<unsigned>(VPT * NCT) && (q % NCT) == 0;
                // softcap: a form (softcap_form) that covers this thread's vectors of the
                // chunk, taken on the full-chunk path, kept for the second pass over the
                // same vectors (the partial and target chunks take the general form here)
                unsigned form = 0u;
                // the unrolled path takes the full chunks of a thread without the
                // target column and, with one CTA per row and no class-weighted
                // smoothing or softcap, its partial chunk too: vectors past the end
                // read as -inf, which adds exactly 0 to the exp-sum, and are left out
                // of the smoothing sums (4096 x 32000: 0.1009 -> 0.0989 ms; in the pair
                // and ring shapes the extra registers cost more than it saves)
                const bool fullc = nv == VPC;
                constexpr bool PARTIAL = CL == 1 && MODE != 2 && !CAPF;
                if (!mine && (fullc || PARTIAL)) {
                    // no target: one max per chunk, four independent sums
                    uint4 raw[VPT];
                    bool okv[VPT];
                    int nok = 0;  // this thread's vectors in the chunk
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        okv[k] = !PARTIAL || fullc || tid + k * NCT < nv;
                        const uint32_t ninf = F::kNegInfWord;
                        raw[k] = okv[k] ? ld_shared_v4(base_s + 16u * (tid + k * NCT)) : make_uint4(ninf, ninf, ninf, ninf);
                        nok += okv[k] ? 1 : 0;
                    }
                    if (CAPF && cap > 0.f) {
                        float ax = 0.f;
#pragma unroll
                        for (int k = 0; k < VPT; ++k) ax = fmaxf(ax, F::vabsmax(raw[k]));
                        form = softcap_form(ax, cap);
                    }
                    float vm[VPT];
#pragma unroll
                    for (int k = 0; k < VPT; ++k) vm[k] = F::vmax(raw[k]);
                    float cm = vm[0];
#pragma unroll
                    for (int k = 1; k < VPT; ++k) cm = fmaxf(cm, vm[k]);
                    if (FEAT && want_am && cm > am.v) {
                        // a new maximum: its first column among this thread's vectors of the
                        // chunk (earlier chunks hold smaller columns, so ties keep those)
                        int kk = VPT - 1;
#pragma unroll
                        for (int k = VPT - 1; k >= 0; --k) kk = (vm[k] == cm) ? k : kk;
                        uint4 rk = raw[0];
#pragma unroll
                        for (int k = 1; k < VPT; ++k) rk = (k == kk) ? raw[k] : rk;
                        float xk[VEC];
                        F::unpack(rk, xk);
                        int e0 = VEC - 1;
#pragma unroll
                        for (int e = VEC - 1; e >= 0; --e) e0 = (xk[e] == cm) ? e : e0;
                        am = ArgMax{cm, static_cast<int>(vlo + (v0 + tid + kk * NCT) * VEC + e0)};
                    }
                    // softcap is increasing: the chunk's capped maximum is that of its raw
                    // maximum (up to the rounding of the two evaluations, which the online
                    // sum absorbs)
                    const float zm = (CAPF && cap > 0.f) ? softcap_fast(cm, cap, inv_cap) : cm;
                    if (zm > st.m) {
                        if (st.m != -INFINITY) st.s *= ex2_hw((st.m - zm) * kLog2e);
                        st.m = zm;
                    }
                    if (st.m != -INFINITY) {
                        // four accumulators, column j into sum j mod 4, held as two packed
                        // pairs {0,1} {2,3}: the pair ops round each lane as the scalar ops do
                        const float mL = st.m * kLog2e;
                        const F2 l2 = f2(kLog2e, kLog2e), nm = f2(-mL, -mL);
                        F2 acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)}, racc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                        for (int k = 0; k < VPT; ++k) {
                            float x[VEC];
                            F::unpack(raw[k], x);
                            if (CAPF && cap > 0.f) softcap_vec_form<VEC>(x, x, cap, inv_cap, form);
#pragma unroll
                            for (int p = 0; p < VEC / 2; ++p) {
                                const F2 xx = f2(x[2 * p], x[2 * p + 1]);
                                acc[p & 1] = f2_add(acc[p & 1], f2_ex2(f2_fma(xx, l2, nm)));
                                if (P1S && okv[k]) racc[p & 1] = f2_add(racc[p & 1], xx);
                            }
                        }
                        float a0, a1, a2, a3;
                        f2_split(acc[0], a0, a1);
                        f2_split(acc[1], a2, a3);
                        st.s += (a0 + a1) + (a2 + a3);
                        if (P1S) {
                            f2_split(racc[0], a0, a1);
                            f2_split(racc[1], a2, a3);
                            st.r += (a0 + a1) + (a2 + a3);
                            st.n += static_cast<float>(nok * VEC);
                        }
                    } else if (P1S) {
#pragma unroll
                        for (int k = 0; k < VPT; ++k) {
                            if (!okv[k]) continue;
                            float x[VEC];
                            F::unpack(raw[k], x);
                            if (CAPF && cap > 0.f) softcap_vec_form<VEC>(x, x, cap, inv_cap, form);
#pragma unroll
                            for (int j = 0; j < VEC; ++j) st.r += x[j];
                        }
                        st.n += static_cast<float>(nok * VEC);
                    }
                } else if (CAPF && cap > 0.f) {
                    // softcap, partial chunk or the target's: capped logits, first-maximum
                    // column of the raw logits
                    for (int v = tid; v < nv; v += NCT) {
                        const uint4 raw = ld_shared_v4(base_s + 16u * v);
                        const int vb = (v0 + v) * VEC;
                        float x[VEC], z[VEC];
                        F::unpack(raw, x);
                        form = max(form, softcap_form(F::vabsmax(raw), cap));
                        softcap_vec_form<VEC>(x, z, cap, inv_cap, 1u);  // general form: a rare path
                        float zmax = -INFINITY;
#pragma unroll
                        for (int j = 0; j < VEC; ++j) zmax = fmaxf(zmax, z[j]);
                        if (want_am) {
#pragma unroll
                            for (int j = 0; j < VEC; ++j)
                                am = argmax_merge(am, ArgMax{x[j], static_cast<int>(vlo + vb + j)});
                        }
                        const int skip = (static_cast<unsigned>(y - vb) < static_cast<unsigned>(VEC)) ? y - vb : -1;
                        if (skip >= 0) {
                            float zv = 0.f;
#pragma unroll
                            for (int j = 0; j < VEC; ++j) zv = (j == skip) ? z[j] : zv;
                            S.xy[rp] = zv;  // the capped target logit, for the merge
                        }
                        row_state_add<VEC, P1S>(st, z, zmax, skip, nullptr);
                    }
                } else {
                    for (int v = tid; v < nv; v += NCT) {
                        const uint4 raw = ld_shared_v4(base_s + 16u * v);
                        const int vb = (v0 + v) * VEC;
                        float x[VEC];
                        F::unpack(raw, x);
                        const int skip = (static_cast<unsigned>(y - vb) < static_cast<unsigned>(VEC)) ? y - vb : -1;
                        if (skip >= 0) {
                            float xv = 0.f;
#pragma unroll
                            for (int j = 0; j < VEC; ++j) xv = (j == skip) ? x[j] : xv;
                            S.xy[rp] = xv;  // the target logit, for the merge
                        }
                        const float vmx = F::vmax(raw);
                        if (FEAT && want_am && vmx > am.v) {
                            // vectors come in increasing column order: ties keep the earlier one
                            int e0 = VEC - 1;
#pragma unroll
                            for (int e = VEC - 1; e >= 0; --e) e0 = (x[e] == vmx) ? e : e0;
                            am = ArgMax{vmx, static_cast<int>(vlo + vb + e0)};
                        }
                        row_state_add<VEC, P1S>(st, x, vmx, skip, nullptr);
                    }
                }
                if (CAPF && c < 32) cap_forms |= static_cast<uint64_t>(form) << (2 * c);
                __syncwarp();
                if (lane == 0 && c < nch - nkeep) mbar_arrive(smem_u32(&S.empty[s]));
            }
            if (tid < nedge) {
                const int64_t c = edge_c;
                const float xr = F::load1(rowp, c);
                float x = (CAPF && cap > 0.f) ? softcap_fast(xr, cap, inv_cap) : xr;
                if (want_am) am = argmax_merge(am, ArgMax{xr, static_cast<int>(c)});
                if (valid && c == yg) S.xy[rp] = x;
                row_state_add<1, P1S>(st, &x, x, (valid && c == yg) ? 0 : -1, nullptr);
            }
            // ------------------------------------------------ merge and row scalars
            // Every warp merges the CTA's partials and forms the row scalars itself
            // (the same operations in the same order, so every thread holds the
            // same values): one barrier per row, no thread waits on another's
            // scalar work.
            st = warp_merge(st);
            if (lane == 0) S.red[rp][warp] = st;
            if (want_am) {
                am = warp_argmax(am);
                if (lane == 0) S.am[rp][warp] = am;
            }
            stream_consumer_sync<NCW>();
            // each group of NCW lanes holds the NCW warp partials and merges them
            // (the same operations in every group)
            RowState m = S.red[rp][lane & (NCW - 1)];
            m = warp_merge<NCW>(m);
            float xy = valid ? S.xy[rp] : 0.f;
            if (want_am) {
                am = S.am[rp][lane & (NCW - 1)];
                am = warp_argmax<NCW>(am);
            }
            if (DEFER) {
                // r and n of this state carry the previous row's deferred sums (this CTA's
                // part, then both CTAs' after the exchange); pass 1 left them at 0
                float pr = 0.f, pn = 0.f;
                if (pend)
                    for (int k = 0; k < kStreamConsumerWarps; ++k) {
                        pr += S.defer[rp ^ 1u][k].x;
                        pn += S.defer[rp ^ 1u][k].y;
                    }
                m.r = pr;
                m.n = pn;
            }
            if (CL > 1) {
                // one thread pushes this half's partial into both CTAs; every thread
                // waits for both and merges them in rank order
                const uint32_t par = rp;
                const uint32_t my_bar = smem_u32(&S.xbar[par]);
                if (warp == 0 && lane == 0) {
                    const uint32_t my_slot = smem_u32(&S.slot[par][rank]);
                    for (uint32_t d = 0; d < static_cast<uint32_t>(CL); ++d) {
                        const uint32_t rs_addr = mapa_shared(my_slot, d);
                        st_cluster_v4(rs_addr, m.m, m.s, m.r, m.n);
                        st_cluster_v4(rs_addr + 16u, xy, am.v, __int_as_float(am.i), 0.f);
                        mbar_arrive_remote(mapa_shared(my_bar, d));
                    }
                }
                mbar_wait_bounded<true, kStreamSleepC>(my_bar, (j >> 1) & 1u, abort);
                RowState tot = row_state_empty();
                ArgMax amt{-INFINITY, 0x7fffffff};
                for (int d = 0; d < CL; ++d) {
                    const StreamXSlot &xs = S.slot[par][d];
                    tot = row_state_merge(tot, RowState{xs.m, xs.s, xs.r, xs.n});
                    if (want_am) amt = argmax_merge(amt, ArgMax{xs.pad0, __float_as_int(xs.pad1)});
                }
                m = tot;
                am = amt;
                xy = S.slot[par][yg / half].xy;
            }
            if (!have_norm) {
                pdl_wait();
                w_all = a.ctl->w_all;
                w_y_sum = a.ctl->w_y;
                g_all = a.grad_output ? __ldg(a.grad_output) : 1.f;
                have_norm = true;
            }
            float rrel = SMOOTH ? row_state_rel_sum(m) : 0.f;
            const bool writer = warp == 0 && lane == 0;
            if (DEFER) {
                if (writer) {
                    if (pend && rank == 0)
                        put_row_loss(a, pend_row,
                                     deferred_loss(pend_m, pend_s, pend_xy, m.r, pend_yg, pend_wy, w_all, eps, inv_v, zl),
                                     cta_sum);
                    pend_row = row; pend_m = m.m; pend_s = m.s; pend_xy = xy; pend_yg = yg; pend_wy = wy;
                }
                rrel = 0.f;  // the gradient does not use it; this row's loss waits for pass 2
            }
            const float g = a.reduction == CE_RED_NONE ? (a.grad_output ? g_row : 1.f) : g_all;
            float scale = g;
            if (a.reduction == CE_RED_MEAN) scale = w_y_sum != 0.f ? g / w_y_sum : 0.f;
            if (writer && rank == 0 && !DEFER) {
                const RowScalars rl = make_row_scalars(m.m, m.s, xy, rrel, valid, yg, wy, w_all, eps, inv_v, 1.f, zl);
                put_row_loss(a, row, rl.loss, cta_sum);
                // the row statistics {m, s without the target column, x_y, sum w (x - m)}
                if (FWD && a.stats) reinterpret_cast<float4 *>(a.stats)[row] = make_float4(m.m, m.s, xy, rrel);
            }
            if (FWD) {
                ++j;
                continue;  // no second pass
            }
            if (want_am && writer && rank == 0 && am.i == yg) atomicAdd(&a.ctl->n_correct, 1u);
            const RowScalars rs = make_row_scalars(m.m, m.s, xy, rrel, true, yg, wy, w_all, eps, inv_v, scale, zl);
            // grad_elem over packed pairs: p = 2^((x - m) log2e - log2 d), g = a p - b w
            const F2 rs_m = f2(rs.m, rs.m), rs_l2 = f2(kLog2e, kLog2e), rs_nl = f2(rs.neg_log2d, rs.neg_log2d);
            const F2 rs_a = f2(rs.a, rs.a), rs_nb = f2(-rs.b, -rs.b);
            // On 16-bit rows the exponent takes one packed FMA a pair, x log2e + c
            // with c = -m log2e - log2 d (= -log2e LSE) rounded once, instead of the
            // exact difference x - m and an FMA, while |c| < kFoldMax: rounding c then
            // moves the exponent by at most 2^-20, no more than the rounding of the
            // exponent itself already does where p is near the smoothing term (p ~
            // eps / V, exponent in [-32, -16)). Other rows, fp32 gradients and softcap
            // (whose instantiations have no registers to spare for a second loop) keep
            // the exact form.
            // With class-weighted smoothing on aligned rows and a > 0, log2 a joins c
            // as well (form 2): a p = 2^(x log2e + c + log2 a) and the gradient is one FMA,
            // w (-b) + a p. Its two further roundings (of log2 d - log2 a, then of
            // the sum with -m log2e) keep the exponent within about 2^-18 in all;
            // the smoothing term b w then dominates every element whose a p
            // leaves fp32's normal range and flushes to 0.
            const float fold_c = fmaf(-rs.m, kLog2e, rs.neg_log2d);
            const float fold_ca = MODE == 2 && rs.a > 0.f ? fmaf(-rs.m, kLog2e, rs.neg_log2d + log2f(rs.a)) : INFINITY;
            const F2 rs_c = f2(fold_c, fold_c), rs_ca = f2(fold_ca, fold_ca);
            F2 dr[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};  // deferred smoothing sum of w x
            // ------------------------------------------------ pass 2: gradient in place
            // form 0: exact x - m; 1: m folded into c; 2: m and a folded (class weights)
            auto pass2 = [&](auto form_tag) {
                constexpr int FORM = decltype(form_tag)::value;
                auto exp_arg = [&](F2 xx) {
                    if constexpr (FORM == 2) return f2_fma(xx, rs_l2, rs_ca);
                    else if constexpr (FORM == 1) return f2_fma(xx, rs_l2, rs_c);
                    else return f2_fma(f2_sub(xx, rs_m), rs_l2, rs_nl);
                };
                // the kept chunks first, from the slots the first pass filled (they go
                // back to the producer in ring order), then the earlier ones copied again
                for (int k = 0; k < nch; ++k) {
                    const bool in_ring = k < nkeep;
                    const int c = in_ring ? nch - nkeep + k : (reverse ? nch - 1 - k : k - nkeep);
                    const uint32_t s = (in_ring ? it_row + static_cast<uint32_t>(c) : it) % kStreamSlots;
                    if (!in_ring) {
                        mbar_wait_bounded<false, kStreamSleepC>(smem_u32(&S.full[s]), (it / kStreamSlots) & 1u, abort);
                        ++it;
                    }
                    const uint32_t base_s = ring + s * kStreamChunk;
                    const int v0 = c * VPC;
                    const int nv = min(VPC, nvec - v0);
                    const unsigned form = c < 32 ? static_cast<unsigned>(cap_forms >> (2 * c)) & 3u : 2u;
                    // class-weighted element math of one vector: p, the gradient a p - b w,
                    // and the deferred smoothing sums (the same operations whichever way
                    // the weights arrive)
                    auto weighted_vec = [&](const float *x, const float4 *wq, float *gr) {
#pragma unroll
                        for (int h = 0; h < VEC / 4; ++h) {
                            const float4 wv = wq[h];
                            const F2 w01 = f2(wv.x, wv.y), w23 = f2(wv.z, wv.w);
                            const F2 x01 = f2(x[4 * h], x[4 * h + 1]), x23 = f2(x[4 * h + 2], x[4 * h + 3]);
                            if constexpr (FORM == 2) {  // a p directly
                                const F2 ap0 = f2_ex2(exp_arg(x01));
                                const F2 ap1 = f2_ex2(exp_arg(x23));
                                dr[0] = f2_fma(w01, x01, dr[0]);
                                dr[1] = f2_fma(w23, x23, dr[1]);
                                f2_split(f2_fma(w01, rs_nb, ap0), gr[4 * h], gr[4 * h + 1]);
                                f2_split(f2_fma(w23, rs_nb, ap1), gr[4 * h + 2], gr[4 * h + 3]);
                            } else {
                                const F2 nbw0 = f2_mul(rs_nb, w01), nbw1 = f2_mul(rs_nb, w23);
                                const F2 p0 = f2_ex2(exp_arg(x01));
                                const F2 p1 = f2_ex2(exp_arg(x23));
                                dr[0] = f2_fma(w01, x01, dr[0]);
                                dr[1] = f2_fma(w23, x23, dr[1]);
                                f2_split(f2_fma(p0, rs_a, nbw0), gr[4 * h], gr[4 * h + 1]);
                                f2_split(f2_fma(p1, rs_a, nbw1), gr[4 * h + 2], gr[4 * h + 3]);
                            }
                        }
                    };
                    if (WR && wr) {
                        // weights from the weight ring: piece q holds the weights of vectors
                        // [q kWV NCT, (q + 1) kWV NCT) of the chunk, those of vector
                        // (q kWV + u) NCT + tid at 32 (u NCT + tid) bytes
                        for (int q = 0; q * NCT * kWV < nv; ++q) {
                            mbar_wait_bounded<false, kStreamSleepC>(smem_u32(&S.wfull[wsl]), wph, abort);
#pragma unroll
                            for (int u = 0; u < kWV; ++u) {
                                const int v = (q * kWV + u) * NCT + tid;
                                if (v < nv) {
                                    float x[VEC], gr[VEC];
                                    F::unpack(ld_shared_v4(base_s + 16u * v), x);
                                    const int vb = (v0 + v) * VEC;
                                    const uint32_t wa = wring + wsl * SH::kWSlotBytes + 32u * (u * NCT + tid);
                                    const uint4 wlo = ld_shared_v4(wa), whi = ld_shared_v4(wa + 16u);
                                    const float4 wq[2] = {
                                        make_float4(__uint_as_float(wlo.x), __uint_as_float(wlo.y), __uint_as_float(wlo.z),
                                                    __uint_as_float(wlo.w)),
                                        make_float4(__uint_as_float(whi.x), __uint_as_float(whi.y), __uint_as_float(whi.z),
                                                    __uint_as_float(whi.w))};
                                    weighted_vec(x, wq, gr);
                                    if (!TGT_AFTER && static_cast<unsigned>(y - vb) < static_cast<unsigned>(VEC)) {
#pragma unroll
                                        for (int e = 0; e < VEC; ++e) gr[e] = (vb + e == y) ? rs.dxy : gr[e];
                                    }
                                    st_stream(vp + v0 + v, F::pack(gr));
                                }
                            }
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(&S.wempty[wsl]));
                            if (++wsl == static_cast<uint32_t>(kWS)) {
                                wsl = 0;
                                wph ^= 1u;
                            }
                        }
                    } else {
                    for (int v = tid; v < nv; v += NCT) {
                        float x[VEC], gr[VEC];
                        F::unpack(ld_shared_v4(base_s + 16u * v), x);
                        const int vb = (v0 + v) * VEC;
                        // softcap: the capped logits replace the raw ones; dz/dx scales below
                        if (CAPF && cap > 0.f) softcap_vec_form<VEC>(x, x, cap, inv_cap, form);
                        if (MODE == 2) {
                            float4 wq[VEC / 4];
                            if (VEC == 8 && w8) {
                                load_w8(a.weight + vlo + vb, wq[0], wq[VEC / 4 - 1]);
                            } else {
#pragma unroll
                                for (int h = 0; h < VEC / 4; ++h) wq[h] = load_w4(a.weight, vlo + vb + 4 * h, w4);
                            }
                            weighted_vec(x, wq, gr);
                        } else {
#pragma unroll
                            for (int p = 0; p < VEC / 2; ++p) {
                                const F2 pp = f2_ex2(exp_arg(f2(x[2 * p], x[2 * p + 1])));
                                f2_split(f2_fma(pp, rs_a, rs_nb), gr[2 * p], gr[2 * p + 1]);
                            }
                        }
                        if (!TGT_AFTER && static_cast<unsigned>(y - vb) < static_cast<unsigned>(VEC)) {
#pragma unroll
                            for (int e = 0; e < VEC; ++e) gr[e] = (vb + e == y) ? rs.dxy : gr[e];
                        }
                        if (CAPF && cap > 0.f) softcap_deriv_vec<VEC>(gr, x, nic2);
                        st_stream(vp + v0 + v, F::pack(gr));  // vp points at this CTA's slice
                    }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&S.empty[s]));
                }
            };
            if (F::kBytes == 2 && !CAPF && !RAG && MODE == 2 && fabsf(fold_ca) < kFoldMax)
                pass2(std::integral_constant<int, 2>{});
            else if (F::kBytes == 2 && !CAPF && MODE != 2 && fabsf(fold_c) < kFoldMax)
                pass2(std::integral_constant<int, 1>{});
            else
                pass2(std::integral_constant<int, 0>{});
            // With one CTA per row and no softcap the target column of the interior
            // is written after the row's loop, not tested for in every vector: the
            // thread that stored its vector (vector y / VEC of a chunk belongs to
            // thread (y / VEC) mod NCT, VPC being a multiple of NCT) overwrites that
            // element, after its vector store in program order (4096 x 32000: fewer
            // instructions; in the pair shapes the compiler then took two more
            // registers and the loop ran slower).
            if (TGT_AFTER && y >= 0 && (y / VEC) % NCT == tid) F::store1(rowp, vlo + y, rs.dxy);
            float er = 0.f;
            if (tid < nedge) {
                const int64_t c = edge_c;
                const float wc = (MODE == 2) ? __ldg(a.weight + c) : 1.f;
                const float xr = F::load1(rowp, c);
                const float xe = (CAPF && cap > 0.f) ? softcap_fast(xr, cap, inv_cap) : xr;
                er = wc * xe;
                float ge = (c == yg) ? rs.dxy : grad_elem(rs, xe, wc);
                if (CAPF && cap > 0.f) ge *= fmaf(xe * xe, nic2, 1.f);
                F::store1(rowp, c, ge);
            }
            if (DEFER) {
                // this thread's, then this warp's, deferred sum (fixed order), for the next merge
                float r0, r1, r2, r3;
                f2_split(dr[0], r0, r1);
                f2_split(dr[1], r2, r3);
                float rr = ((r0 + r1) + (r2 + r3)) + er;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) rr += __shfl_xor_sync(0xffffffffu, rr, off);
                if (lane == 0) S.defer[rp][warp] = make_float2(rr, 0.f);
            }
            pend = true;
            ++j;
        }
        // ---------------------------------------------------- the last row's deferred loss
        if (DEFER && pend) {
            stream_consumer_sync<NCW>();  // every warp's sums of the last row are in S.defer
            if (warp == 0 && lane == 0) {
                float pr = 0.f, pn = 0.f;
                const uint32_t lp = (j - 1u) & 1u;  // parity of the last row
                for (int k = 0; k < kStreamConsumerWarps; ++k) { pr += S.defer[lp][k].x; pn += S.defer[lp][k].y; }
                if (CL > 1) {
                    // one more exchange (the next parity) carrying only the sums
                    const uint32_t par = j & 1u;
                    const uint32_t my_slot = smem_u32(&S.slot[par][rank]);
                    const uint32_t my_bar = smem_u32(&S.xbar[par]);
                    for (uint32_t d = 0; d < static_cast<uint32_t>(CL); ++d) {
                        const uint32_t rs_addr = mapa_shared(my_slot, d);
                        st_cluster_v4(rs_addr, -INFINITY, 0.f, pr, pn);
                        st_cluster_v4(rs_addr + 16u, 0.f, 0.f, 0.f, 0.f);
                        mbar_arrive_remote(mapa_shared(my_bar, d));
                    }
                    mbar_wait_bounded<true, kStreamSleepC>(my_bar, (j >> 1) & 1u, abort);
                    RowState tot = row_state_empty();
                    for (int d = 0; d < CL; ++d) {
                        const StreamXSlot &xs = S.slot[par][d];
                        tot = row_state_merge(tot, RowState{xs.m, xs.s, xs.r, xs.n});
                    }
                    pr = tot.r;
                    pn = tot.n;
                }
                if (rank == 0)
                    put_row_loss(a, pend_row, deferred_loss(pend_m, pend_s, pend_xy, pr, pend_yg, pend_wy, w_all, eps,
                                                            inv_v, zl),
                                 cta_sum);
            }
        }
        // ---------------------------------------------------- batch reduction (last CTA)
        if ((a.reduction != CE_RED_NONE || want_am) && !a.no_finalize) {
            __shared__ unsigned sh_last;
            __shared__ double sh_sum[kStreamConsumerWarps];
            if (!have_norm) pdl_wait();
            stream_consumer_sync<NCW>();
            if (tid == 0) {
                // this CTA's (cluster's) sum of its rows' losses, in the slot of its first row
                // (the index read again here rather than kept in a register through the rows)
                if (a.reduction != CE_RED_NONE && (CL == 1 || cluster_ctarank() == 0))
                    a.row_loss[CL == 1 ? ctaid_x_fresh() : cluster_id_x()] = static_cast<float>(cta_sum);
                __threadfence();
                const unsigned prev = atomicAdd(&a.ctl->done, 1u);
                sh_last = (prev == gridDim.x - 1) ? 1u : 0u;
            }
            stream_consumer_sync<NCW>();
            if (sh_last && want_am && tid == 0) {
                __threadfence();
                const float nv = a.ctl->n_valid;
                a.accuracy[0] = nv > 0.f ? static_cast<float>(__ldcg(&a.ctl->n_correct)) / nv : 0.f;
            }
            if (sh_last && a.reduction == CE_RED_NONE && tid == 0) a.ctl->done = 0u;
            if (sh_last && a.reduction != CE_RED_NONE) {
                __threadfence();
                double sum = 0.0;
                // the CTAs' (clusters') sums in CTA order, then a fixed tree
                const int n_part = static_cast<int>(CL == 1 ? nctaid_x_fresh() : nclusters_x());
                for (int i = tid; i < n_part; i += NCT) sum += static_cast<double>(__ldcg(a.row_loss + i));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                if (lane == 0) sh_sum[warp] = sum;
                stream_consumer_sync<NCW>();
                if (tid == 0) {
                    double tot = 0.0;
                    for (int k = 0; k < kStreamConsumerWarps; ++k) tot += sh_sum[k];
                    if (a.reduction == CE_RED_MEAN) {
                        const float wys = a.ctl->w_y;  // after the normaliser kernel (waited above)
                        tot = wys != 0.f ? tot / static_cast<double>(wys) : 0.0;
                    }
                    a.loss[0] = static_cast<float>(tot);
                    a.ctl->done = 0u;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0 && S.abort) {
        pdl_wait();
        atomicOr(&a.ctl->status, CE_FLAG_WAIT_TIMEOUT);
    }
    if (CL > 1) cluster_sync_all();  // no CTA leaves while its peer may still write into it
}

// Kernel entry of one instantiation (the aligned ones are compiled in
// ce_stream.cu, the ragged ones in ce_stream_ragged.cu).
template <int DT, int SHAPE, int CL, bool RAG, int OPT = 0>
const void *stream_fn(int mode) {
    switch (mode) {
    case 0: return reinterpret_cast<const void *>(&ce_stream_kernel<DT, 0, SHAPE, CL, RAG, OPT>);
    case 1: return reinterpret_cast<const void *>(&ce_stream_kernel<DT, 1, SHAPE, CL, RAG, OPT>);
    default: return reinterpret_cast<const void *>(&ce_stream_kernel<DT, 2, SHAPE, CL, RAG, OPT>);
    }
}

#define CE_STREAM_PICK(S, C, R, OP)                                                                          \
    if (shape == S && cl == C)                                                                               \
        return dtype == CE_DT_F32 ? stream_fn<CE_DT_F32, S, C, R, OP>(mode)                                  \
             : dtype == CE_DT_BF16 ? stream_fn<CE_DT_BF16, S, C, R, OP>(mode) : stream_fn<CE_DT_F16, S, C, R, OP>(mode);

template <bool RAG>
const void *stream_kernel_for(int dtype, int mode, int shape, int cl) {
    CE_STREAM_PICK(0, 1, RAG, 0) CE_STREAM_PICK(0, 2, RAG, 0) CE_STREAM_PICK(1, 1, RAG, 0)
    CE_STREAM_PICK(1, 2, RAG, 0) CE_STREAM_PICK(2, 1, RAG, 0) CE_STREAM_PICK(2, 2, RAG, 0)
    CE_STREAM_PICK(2, 4, RAG, 0)
    return nullptr;
}

// With the options: the four shapes the library picks by row size (three
// CTAs per SM, alone, in pairs or in quads; one wide CTA per SM in pairs).
template <bool RAG, int OPT>
const void *stream_kernel_options_for(int dtype, int mode, int shape, int cl) {
    CE_STREAM_PICK(2, 1, RAG, OPT) CE_STREAM_PICK(2, 2, RAG, OPT) CE_STREAM_PICK(2, 4, RAG, OPT)
    CE_STREAM_PICK(1, 2, RAG, OPT)
    return nullptr;
}
#undef CE_STREAM_PICK

// defined in ce_stream_ragged.cu, ce_stream_options.cu, ce_stream_options_ragged.cu,
// ce_stream_softcap.cu, ce_stream_softcap_ragged.cu and ce_stream_forward.cu
const void *stream_kernel_ragged(int dtype, int mode, int shape, int cl);
const void *stream_kernel_options(int dtype, int mode, int shape, int cl, bool ragged);
const void *stream_kernel_options_ragged(int dtype, int mode, int shape, int cl);
const void *stream_kernel_softcap(int dtype, int mode, int shape, int cl, bool ragged);
const void *stream_kernel_softcap_ragged(int dtype, int mode, int shape, int cl);
const void *stream_kernel_forward(int dtype, int mode, bool ragged);

}  // namespace ce
