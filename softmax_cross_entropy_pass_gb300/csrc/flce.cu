// flce.cu -- fused-linear cross-entropy: the lm-head GEMMs on the 5th
// generation tensor cores and the chunk loop around the cross-entropy
// kernel (Liger-Kernel PR #1622's FLCE: logits computed chunk by chunk,
// never materialised for the whole batch, no host syncs).
//
// GEMM kernel: D[M,N] (fp32 in TMEM) = A[M,K] * B[K,N], bf16 operands,
// 128 x 256 x 64 tiles, persistent CTAs (one per SM), warp-specialised:
//   warp 0      TMA producer: 2-D tiled bulk tensor loads (128-byte swizzle)
//               into a 4-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators) and issues tcgen05.mma (one elected thread),
//               releasing each stage with tcgen05.commit;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per
//               thread), optional bias, then fp32 store, fp32 accumulate or
//               bf16 store; the accumulator is handed back so the next
//               tile's MMAs overlap this epilogue.
// Either operand may be K-major or MN-major in memory, so the three FLCE
// products need no transposed copies:
//   Z      = h W^T      A = h (K-major), B = W (K-major)
//   dh     = dZ W       A = dZ (K-major), B = W (MN-major)
//   dW    += dZ^T h     A = dZ (MN-major), B = h (MN-major)
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ce_device.cuh"
#include "ce_kernels.h"
#include "flce.h"
#include "tc_device.cuh"

namespace ce {

constexpr int GB_M = 128, GB_N = 256, GB_K = 64, GB_STAGES = 4;
static_assert(GB_N == kGemmTileN, "the row statistics are kept per 256-column tile");
constexpr int GB_A_BYTES = GB_M * GB_K * 2;  // 16 KB
constexpr int GB_B_BYTES = GB_N * GB_K * 2;  // 32 KB
constexpr int GB_THREADS = 192;
constexpr int GB_TMEM_COLS = 512;
constexpr size_t GB_SMEM = 1024 + GB_STAGES * (GB_A_BYTES + GB_B_BYTES) + 256;

enum { OUT_F32_STORE = 0, OUT_F32_ACCUM = 1, OUT_BF16_STORE = 2 };

struct GemmArgs {
    int M, N, K;
    int a_mn, b_mn;        // 1: operand is MN-major in memory
    int out_kind;
    void *out;
    int64_t ldo;           // elements
    const float *bias;     // [N] (fp32 store only) or NULL
    int tiles_m, tiles_n;
    int m_fastest;         // tile order: consecutive tiles step along M
    unsigned int *status;
    // Device-side size (NULL: the sizes above). The kernel reads
    // n = clamp(*dyn_count - dyn_off, 0, size) and uses it as M (dyn_dim 0)
    // or K (dyn_dim 1); the launch must be stream-ordered after the kernel
    // that writes the count.
    const int *dyn_count;
    int dyn_off, dyn_dim;
    const int *row_map;    // output row r is stored at row row_map[r] (NULL: r)
    // Split-K: every output tile is computed as ksplit partial products over
    // consecutive K ranges; partial s is stored (fp32) split_stride elements
    // after partial s - 1 (ksplit 1: one product, the usual output).
    int ksplit;
    int64_t split_stride;
    // Row statistics of the fp32 output (logits GEMM of the fused-linear
    // path): per row and column tile, the running softmax state of the tile's
    // columns {max m, exp-sum s without the target column, smoothing sum r,
    // weight sum n}, stored at part[row * tiles_n + tile].
    float4 *part;
    float2 *pam;           // token accuracy: per row and tile {raw maximum, its first column}, or NULL
    float st_cap, st_inv_cap;  // softcap c (0: off): the stored logits are c tanh(x / c)
    const void *st_target;
    int st_tgt32;
    int64_t st_ignore;
    const float *st_weight;
};

__device__ inline void tile_coords(const GemmArgs &g, int t, int &tm, int &tn) {
    if (g.m_fastest) { tm = t % g.tiles_m; tn = t / g.tiles_m; }
    else { tn = t % g.tiles_n; tm = t / g.tiles_n; }
}

// One thread's 32 consecutive accumulator columns of one output row.
// `orow` is the row of the output the tile row `row` is stored at.
__device__ inline void epilogue_store(const GemmArgs &g, int row, int orow, int col0, const uint32_t (&v)[32],
                                      int64_t base = 0) {
    if (row >= g.M) return;
    const bool full = col0 + 32 <= g.N;
    if (g.out_kind == OUT_BF16_STORE) {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(g.out) + base + static_cast<int64_t>(orow) * g.ldo + col0;
        if (full && (g.ldo % 8) == 0) {
            uint4 *o4 = reinterpret_cast<uint4 *>(o);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = Fmt<CE_DT_BF16>::pack2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
                w.y = Fmt<CE_DT_BF16>::pack2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
                w.z = Fmt<CE_DT_BF16>::pack2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
                w.w = Fmt<CE_DT_BF16>::pack2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
                o4[q] = w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < g.N) o[j] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
        return;
    }
    float *o = reinterpret_cast<float *>(g.out) + base + static_cast<int64_t>(orow) * g.ldo + col0;
    const bool accum = g.out_kind == OUT_F32_ACCUM;
    if (full && (g.ldo % 4) == 0) {
        float4 *o4 = reinterpret_cast<float4 *>(o);
        const float4 *b4 = reinterpret_cast<const float4 *>(g.bias + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 w = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            if (g.bias) {
                const float4 bb = __ldg(b4 + q);
                w.x += bb.x; w.y += bb.y; w.z += bb.z; w.w += bb.w;
            }
            if (accum) {
                const float4 old = o4[q];
                w.x += old.x; w.y += old.y; w.z += old.z; w.w += old.w;
            }
            o4[q] = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (col0 + j < g.N) {
                float w = __uint_as_float(v[j]) + (g.bias ? __ldg(g.bias + col0 + j) : 0.f);
                o[j] = accum ? o[j] + w : w;
            }
        }
    }
}

// Statistics epilogue: store 32 fp32 logits (+ bias; capped to c tanh(x / c)
// with a softcap) of one row and fold them into the row's softmax state over
// the current column tile. `skip` is the target's position among the 32
// columns (-1: not among them). With `pam`, `am` follows the first column
// of the raw maximum (columns arrive in increasing order, so a strictly
// greater value is needed to move it). SMODE 0: no smoothing sums; 1: sum of
// the logits; 2: class-weighted sum.
template <int SMODE>
__device__ inline void epilogue_stats(const GemmArgs &g, int row, int col0, const uint32_t (&v)[32], RowState &st,
                                      int skip, ArgMax &am) {
    const int nv = g.N - col0;
    if (nv <= 0) return;
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
    float *o = reinterpret_cast<float *>(g.out) + static_cast<int64_t>(row) * g.ldo + col0;
    if (nv >= 32 && (g.ldo % 4) == 0) {
        if (g.bias) {
            const float4 *b4 = reinterpret_cast<const float4 *>(g.bias + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 bb = __ldg(b4 + q);
                x[4 * q] += bb.x; x[4 * q + 1] += bb.y; x[4 * q + 2] += bb.z; x[4 * q + 3] += bb.w;
            }
        }
        if (g.pam) {
            float rmax = x[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) rmax = fmaxf(rmax, x[j]);
            if (rmax > am.v) {
                int e0 = 31;
#pragma unroll
                for (int j = 31; j >= 0; --j) e0 = (x[j] == rmax) ? j : e0;
                am = ArgMax{rmax, col0 + e0};
            }
        }
        if (g.st_cap > 0.f) {
#pragma unroll
            for (int q = 0; q < 4; ++q) softcap_vec<8>(x + 8 * q, x + 8 * q, g.st_cap, g.st_inv_cap);
        }
        float4 *o4 = reinterpret_cast<float4 *>(o);
#pragma unroll
        for (int q = 0; q < 8; ++q) o4[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        float vmax = x[0];
#pragma unroll
        for (int j = 1; j < 32; ++j) vmax = fmaxf(vmax, x[j]);
        float w[32];
        if (SMODE == 2) {
            const float4 *w4 = reinterpret_cast<const float4 *>(g.st_weight + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 ww = __ldg(w4 + q);
                w[4 * q] = ww.x; w[4 * q + 1] = ww.y; w[4 * q + 2] = ww.z; w[4 * q + 3] = ww.w;
            }
        }
        row_state_add<32, SMODE != 0>(st, x, vmax, skip, SMODE == 2 ? w : nullptr);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < nv) {
                float xv = x[j] + (g.bias ? __ldg(g.bias + col0 + j) : 0.f);
                if (g.pam) am = argmax_merge(am, ArgMax{xv, col0 + j});
                if (g.st_cap > 0.f) xv = softcap_fast(xv, g.st_cap, g.st_inv_cap);
                o[j] = xv;
                float wj = SMODE == 2 ? __ldg(g.st_weight + col0 + j) : 1.f;
                row_state_add<1, SMODE != 0>(st, &xv, xv, skip == j ? 0 : -1, SMODE == 2 ? &wj : nullptr);
            }
        }
    }
}

// EPI 0: the plain epilogue (epilogue_store); 1..3: fp32 store with row
// statistics (epilogue_stats, smoothing mode EPI - 1).
template <int EPI>
__global__ void __launch_bounds__(GB_THREADS, 1)
flce_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs g) {
    if (g.dyn_count) {
        int n = __ldg(g.dyn_count) - g.dyn_off;
        if (g.dyn_dim == 0) {
            g.M = n < 0 ? 0 : (n < g.M ? n : g.M);
            g.tiles_m = (g.M + GB_M - 1) / GB_M;
        } else {
            g.K = n < 0 ? 0 : (n < g.K ? n : g.K);
        }
    }
    const int ksplit = g.ksplit > 1 ? g.ksplit : 1;
    // tiles run K part by K part (all output tiles of part 0, then part 1, ...), so
    // the CTAs of a wave share one K range of the operands in L2
    const int mn_tiles = g.tiles_m * g.tiles_n;
    const int num_tiles = mn_tiles * ksplit;
    const int kiters = (g.K + GB_K - 1) / GB_K;
    const int kper = (kiters + ksplit - 1) / ksplit;   // K steps of one split (the last may have fewer)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (num_tiles == 0) return;
    if (kiters == 0) {
        // empty reduction: D = 0 (+ bias) in the store modes, nothing to add in accumulate mode
        if (g.out_kind != OUT_F32_ACCUM && warp >= 2) {
            const int q = warp & 3;
            const uint32_t zero[32] = {};
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                int tm, tn;
                tile_coords(g, t % mn_tiles, tm, tn);
                const int row = tm * GB_M + q * 32 + lane;
                const int orow = (g.row_map && row < g.M) ? __ldg(g.row_map + row) : row;
                const int64_t base = static_cast<int64_t>(t / mn_tiles) * g.split_stride;
                for (int c0 = 0; c0 < GB_N; c0 += 32) epilogue_store(g, row, orow, tn * GB_N + c0, zero, base);
            }
        }
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128-byte swizzle atoms need 1 KB alignment
    uint8_t *basep = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + GB_STAGES * GB_A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(basep + GB_STAGES * (GB_A_BYTES + GB_B_BYTES));
    uint64_t *full = bars, *empty = bars + GB_STAGES, *tfull = bars + 2 * GB_STAGES, *tempty = bars + 2 * GB_STAGES + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * GB_STAGES + 4);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *abort = abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GB_STAGES; ++s) { mbar_init(smem_u32(&full[s]), 1); mbar_init(smem_u32(&empty[s]), 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(smem_u32(&tfull[a]), 1); mbar_init(smem_u32(&tempty[a]), 4); }
        *abort_flag = 0;
        fence_mbar_init_cluster();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), GB_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t it = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                int tm, tn;
                tile_coords(g, t % mn_tiles, tm, tn);
                const int kb = (t / mn_tiles) * kper, ke = min(kiters, kb + kper);
                for (int k = kb; k < ke; ++k, ++it) {
                    const uint32_t s = it % GB_STAGES, r = it / GB_STAGES;
                    if (r > 0) mbar_wait_bounded<false>(smem_u32(&empty[s]), (r - 1) & 1u, abort);
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_expect_tx(fb, GB_A_BYTES + GB_B_BYTES);
                    const uint32_t a_dst = sA + s * GB_A_BYTES, b_dst = sB + s * GB_B_BYTES;
                    if (!g.a_mn) tma_load_2d(a_dst, &tmA, k * GB_K, tm * GB_M, fb);
                    else for (int j = 0; j < GB_M / 64; ++j) tma_load_2d(a_dst + j * 8192, &tmA, tm * GB_M + 64 * j, k * GB_K, fb);
                    if (!g.b_mn) tma_load_2d(b_dst, &tmB, k * GB_K, tn * GB_N, fb);
                    else for (int j = 0; j < GB_N / 64; ++j) tma_load_2d(b_dst + j * 8192, &tmB, tn * GB_N + 64 * j, k * GB_K, fb);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(GB_M, GB_N, g.a_mn, g.b_mn);
            // K-major: the 16-wide K step is 32 bytes inside the swizzle atom, 8-row groups 1 KB apart.
            // MN-major: the K step is 16 rows of 128 bytes; 64-element MN blocks are 8 KB apart
            // (one TMA box each), 8-row K groups 1 KB apart.
            const uint32_t a_kstep = g.a_mn ? 2048u : 32u, b_kstep = g.b_mn ? 2048u : 32u;
            const uint32_t a_lbo = g.a_mn ? 8192u : 16u, b_lbo = g.b_mn ? 8192u : 16u;
            uint32_t it = 0, lt = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++lt) {
                const uint32_t acc = lt & 1u, u = lt >> 1;
                if (u > 0) mbar_wait_bounded<false>(smem_u32(&tempty[acc]), (u - 1) & 1u, abort);
                tc_fence_after();
                const uint32_t d = tmem + acc * GB_N;
                const int kb = (t / mn_tiles) * kper, ke = min(kiters, kb + kper);
                for (int k = kb; k < ke; ++k, ++it) {
                    const uint32_t s = it % GB_STAGES, r = it / GB_STAGES;
                    mbar_wait_bounded<false>(smem_u32(&full[s]), r & 1u, abort);
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < GB_K / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(sA + s * GB_A_BYTES + kk * a_kstep, a_lbo, 1024);
                        const uint64_t bd = smem_desc_sw128(sB + s * GB_B_BYTES + kk * b_kstep, b_lbo, 1024);
                        mma_bf16(d, ad, bd, idesc, (k > kb || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&empty[s]));
                }
                mma_commit(smem_u32(&tfull[acc]));
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2..5)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint32_t lt = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++lt) {
            int tm, tn;
            tile_coords(g, t % mn_tiles, tm, tn);
            const int64_t base = static_cast<int64_t>(t / mn_tiles) * g.split_stride;
            const uint32_t acc = lt & 1u, u = lt >> 1;
            mbar_wait_bounded<false>(smem_u32(&tfull[acc]), u & 1u, abort);
            tc_fence_after();
            const int row = tm * GB_M + q * 32 + lane;
            const int orow = (g.row_map && row < g.M) ? __ldg(g.row_map + row) : row;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * GB_N;
            RowState st = row_state_empty();
            ArgMax am{-INFINITY, 0x7fffffff};
            int y_rel = -(1 << 30);   // target column relative to the tile (none: far outside)
            if (EPI != 0 && row < g.M) {
                const int64_t y = load_target(g.st_target, g.st_tgt32, row);
                if (target_valid(y, g.st_ignore, g.N)) y_rel = static_cast<int>(y - static_cast<int64_t>(tn) * GB_N);
            }
#pragma unroll 1
            for (int c0 = 0; c0 < GB_N; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + c0, v);
                tmem_ld_wait();
                if (EPI == 0) {
                    epilogue_store(g, row, orow, tn * GB_N + c0, v, base);
                } else if (row < g.M) {
                    const int skip = (static_cast<unsigned>(y_rel - c0) < 32u) ? y_rel - c0 : -1;
                    epilogue_stats<(EPI > 0 ? EPI - 1 : 0)>(g, row, tn * GB_N + c0, v, st, skip, am);
                }
            }
            if (EPI != 0 && row < g.M) {
                g.part[static_cast<int64_t>(row) * g.tiles_n + tn] = make_float4(st.m, st.s, st.r, st.n);
                if (g.pam) g.pam[static_cast<int64_t>(row) * g.tiles_n + tn] = make_float2(am.v, __int_as_float(am.i));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, GB_TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag && g.status) atomicOr(g.status, CE_FLAG_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ CTA-pair GEMM
// The same product with a pair of CTAs (a cluster of 2, one CTA per SM) per
// 256 x 256 tile: the even CTA issues tcgen05.mma.cta_group::2; each CTA
// loads its 128 rows of A and its 128 columns of B per 64-deep K stage
// (32 KB instead of 48 KB per SM), and holds its 128 accumulator rows in its
// own tensor memory. Stage barriers: `full` in the even CTA counts both
// CTAs' bytes (TMA loads of the odd CTA complete on it), `empty` in each CTA
// is signalled by the MMA's multicast commit, `tfull` likewise, and `tempty`
// in the even CTA collects the 8 epilogue warps of the pair.
constexpr int GP_M = 256, GP_N = 256, GP_STAGES = 6;
constexpr int GP_A_BYTES = 128 * GB_K * 2;   // 16 KB: this CTA's half of A
constexpr int GP_B_BYTES = 128 * GB_K * 2;   // 16 KB: this CTA's half of B
constexpr size_t GP_SMEM = 1024 + GP_STAGES * (GP_A_BYTES + GP_B_BYTES) + 256;

template <int EPI>
__global__ void __launch_bounds__(GB_THREADS, 1)
flce_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs g) {
    if (g.dyn_count) {
        int n = __ldg(g.dyn_count) - g.dyn_off;
        if (g.dyn_dim == 0) {
            g.M = n < 0 ? 0 : (n < g.M ? n : g.M);
            g.tiles_m = (g.M + GP_M - 1) / GP_M;
        } else {
            g.K = n < 0 ? 0 : (n < g.K ? n : g.K);
        }
    }
    const int ksplit = g.ksplit > 1 ? g.ksplit : 1;
    const int mn_tiles = g.tiles_m * g.tiles_n;
    const int num_tiles = mn_tiles * ksplit;
    const int kiters = (g.K + GB_K - 1) / GB_K;
    const int kper = (kiters + ksplit - 1) / ksplit;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(nclusters_x());
    // both CTAs of a pair see the same sizes, so they leave here together
    if (num_tiles == 0) return;
    if (kiters == 0) {
        if (g.out_kind != OUT_F32_ACCUM && warp >= 2) {
            const int q = warp & 3;
            const uint32_t zero[32] = {};
            for (int t = cid; t < num_tiles; t += ncl) {
                int tm, tn;
                tile_coords(g, t % mn_tiles, tm, tn);
                const int row = tm * GP_M + static_cast<int>(rank) * 128 + q * 32 + lane;
                const int orow = (g.row_map && row < g.M) ? __ldg(g.row_map + row) : row;
                const int64_t base = static_cast<int64_t>(t / mn_tiles) * g.split_stride;
                for (int c0 = 0; c0 < GP_N; c0 += 32) epilogue_store(g, row, orow, tn * GP_N + c0, zero, base);
            }
        }
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // the same offsets in both CTAs of the pair
    uint8_t *basep = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + GP_STAGES * GP_A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(basep + GP_STAGES * (GP_A_BYTES + GP_B_BYTES));
    uint64_t *full = bars, *empty = bars + GP_STAGES, *tfull = bars + 2 * GP_STAGES, *tempty = bars + 2 * GP_STAGES + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * GP_STAGES + 4);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *abort = abort_flag;

    if (threadIdx.x == 0) {
        for (int st = 0; st < GP_STAGES; ++st) {
            mbar_init(smem_u32(&full[st]), 1);
            mbar_init(smem_u32(&empty[st]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 8);
        }
        *abort_flag = 0;
        fence_mbar_init_cluster();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or copy
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), GB_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            uint32_t it = 0;
            for (int t = cid; t < num_tiles; t += ncl) {
                int tm, tn;
                tile_coords(g, t % mn_tiles, tm, tn);
                const int kb = (t / mn_tiles) * kper, ke = min(kiters, kb + kper);
                const int row0 = tm * GP_M + static_cast<int>(rank) * 128, col0 = tn * GP_N + static_cast<int>(rank) * 128;
                for (int k = kb; k < ke; ++k, ++it) {
                    const uint32_t st = it % GP_STAGES, r = it / GP_STAGES;
                    if (r > 0) mbar_wait_bounded<false>(smem_u32(&empty[st]), (r - 1) & 1u, abort);
                    const uint32_t fb = mapa_shared(smem_u32(&full[st]), 0);  // the even CTA's barrier
                    if (rank == 0) mbar_expect_tx(smem_u32(&full[st]), 2 * (GP_A_BYTES + GP_B_BYTES));
                    const uint32_t a_dst = sA + st * GP_A_BYTES, b_dst = sB + st * GP_B_BYTES;
                    if (!g.a_mn) tma_load_2d_pair(a_dst, &tmA, k * GB_K, row0, fb);
                    else for (int j = 0; j < 2; ++j) tma_load_2d_pair(a_dst + j * 8192, &tmA, row0 + 64 * j, k * GB_K, fb);
                    if (!g.b_mn) tma_load_2d_pair(b_dst, &tmB, k * GB_K, col0, fb);
                    else for (int j = 0; j < 2; ++j) tma_load_2d_pair(b_dst + j * 8192, &tmB, col0 + 64 * j, k * GB_K, fb);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer (even CTA)
            const uint32_t idesc = idesc_bf16_f32(GP_M, GP_N, g.a_mn, g.b_mn);
            const uint32_t a_kstep = g.a_mn ? 2048u : 32u, b_kstep = g.b_mn ? 2048u : 32u;
            const uint32_t a_lbo = g.a_mn ? 8192u : 16u, b_lbo = g.b_mn ? 8192u : 16u;
            uint32_t it = 0, lt = 0;
            for (int t = cid; t < num_tiles; t += ncl, ++lt) {
                const uint32_t acc = lt & 1u, u = lt >> 1;
                if (u > 0) mbar_wait_bounded<false>(smem_u32(&tempty[acc]), (u - 1) & 1u, abort);
                tc_fence_after();
                const uint32_t d = tmem + acc * GP_N;
                const int kb = (t / mn_tiles) * kper, ke = min(kiters, kb + kper);
                for (int k = kb; k < ke; ++k, ++it) {
                    const uint32_t st = it % GP_STAGES, r = it / GP_STAGES;
                    mbar_wait_bounded<false>(smem_u32(&full[st]), r & 1u, abort);
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < GB_K / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(sA + st * GP_A_BYTES + kk * a_kstep, a_lbo, 1024);
                        const uint64_t bd = smem_desc_sw128(sB + st * GP_B_BYTES + kk * b_kstep, b_lbo, 1024);
                        mma_bf16_pair(d, ad, bd, idesc, (k > kb || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_pair_mc(smem_u32(&empty[st]), 0x3);
                }
                mma_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2..5, both CTAs)
        const int q = warp & 3;
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
        uint32_t lt = 0;
        for (int t = cid; t < num_tiles; t += ncl, ++lt) {
            int tm, tn;
            tile_coords(g, t % mn_tiles, tm, tn);
            const int64_t obase = static_cast<int64_t>(t / mn_tiles) * g.split_stride;
            const uint32_t acc = lt & 1u, u = lt >> 1;
            mbar_wait_bounded<false>(smem_u32(&tfull[acc]), u & 1u, abort);
            tc_fence_after();
            const int row = tm * GP_M + static_cast<int>(rank) * 128 + q * 32 + lane;
            const int orow = (g.row_map && row < g.M) ? __ldg(g.row_map + row) : row;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * GP_N;
            RowState stt = row_state_empty();
            ArgMax am{-INFINITY, 0x7fffffff};
            int y_rel = -(1 << 30);
            if (EPI != 0 && row < g.M) {
                const int64_t y = load_target(g.st_target, g.st_tgt32, row);
                if (target_valid(y, g.st_ignore, g.N)) y_rel = static_cast<int>(y - static_cast<int64_t>(tn) * GP_N);
            }
#pragma unroll 1
            for (int c0 = 0; c0 < GP_N; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + c0, v);
                tmem_ld_wait();
                if (EPI == 0) {
                    epilogue_store(g, row, orow, tn * GP_N + c0, v, obase);
                } else if (row < g.M) {
                    const int skip = (static_cast<unsigned>(y_rel - c0) < 32u) ? y_rel - c0 : -1;
                    epilogue_stats<(EPI > 0 ? EPI - 1 : 0)>(g, row, tn * GP_N + c0, v, stt, skip, am);
                }
            }
            if (EPI != 0 && row < g.M) {
                g.part[static_cast<int64_t>(row) * g.tiles_n + tn] = make_float4(stt.m, stt.s, stt.r, stt.n);
                if (g.pam) g.pam[static_cast<int64_t>(row) * g.tiles_n + tn] = make_float2(am.v, __int_as_float(am.i));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(smem_u32(&tempty[acc]));
                else mbar_arrive_remote(tempty0 + acc * 8u);
            }
        }
    }
    __syncthreads();
    cluster_sync_all();  // every MMA of the pair has completed and both CTAs have read their accumulators
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, GB_TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag && g.status) atomicOr(g.status, CE_FLAG_WAIT_TIMEOUT);
    cluster_sync_all();  // no CTA leaves while its peer may still signal one of its barriers
}

// ------------------------------------------------------------------ small kernels
// Rows past a device-side count are skipped: n = clamp(*count - off, 0, n).
__device__ inline int64_t dyn_rows(int64_t n, const int *count, int64_t off) {
    if (!count) return n;
    const int64_t left = static_cast<int64_t>(__ldg(count)) - off;
    return left < 0 ? 0 : (left < n ? left : n);
}

// grad_bias[c] (+)= sum over rows of dZ[r, c]
__global__ void flce_colsum_kernel(const __nv_bfloat16 *dz, int64_t ldd, int rows, int64_t V, float *gb, int accumulate,
                                   const int *count, int off) {
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= V) return;
    const int n = static_cast<int>(dyn_rows(rows, count, off));
    float s = 0.f;
    for (int r = 0; r < n; ++r) s += __bfloat162float(dz[static_cast<int64_t>(r) * ldd + c]);
    gb[c] = accumulate ? gb[c] + s : s;
}

// Ignored-row compaction (the device-side form of Liger-Kernel PR #1554's
// skip of ignored rows: no host sync). One block scans the targets in order
// and writes, for the n rows whose target is valid, idx[k] = the k-th valid
// row and tgt_c[k] = its target; pos[i] = k for a valid row i, -1 otherwise;
// tgt_c[k] = ignore_index for k >= n; *count = n.
constexpr int kCompactThreads = 1024;
__global__ void __launch_bounds__(kCompactThreads) flce_compact_kernel(const void *target, int tgt32, int64_t n_rows,
                                                                      int64_t vocab, int64_t ignore_index, int *idx,
                                                                      int *pos, int64_t *tgt_c, int *count) {
    __shared__ int warp_off[kCompactThreads / 32];
    __shared__ int total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int base = 0;
    for (int64_t r0 = 0; r0 < n_rows; r0 += kCompactThreads) {
        const int64_t i = r0 + tid;
        int64_t t = 0;
        bool v = false;
        if (i < n_rows) {
            t = load_target(target, tgt32, i);
            v = target_valid(t, ignore_index, vocab);
        }
        const unsigned b = __ballot_sync(0xffffffffu, v);
        if (lane == 0) warp_off[warp] = __popc(b);
        __syncthreads();
        if (warp == 0) {
            const int c = warp_off[lane];
            int x = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += y;
            }
            warp_off[lane] = x - c;  // exclusive prefix over warps
            if (lane == 31) total = x;
        }
        __syncthreads();
        const int k = base + warp_off[warp] + __popc(b & ((1u << lane) - 1u));
        if (i < n_rows) {
            if (v) {
                idx[k] = static_cast<int>(i);
                tgt_c[k] = t;
            }
            pos[i] = v ? k : -1;
        }
        base += total;
        __syncthreads();  // warp_off and total are rewritten by the next tile
    }
    for (int64_t k = base + tid; k < n_rows; k += kCompactThreads) {
        tgt_c[k] = ignore_index;
        idx[k] = -1;
    }
    if (tid == 0) *count = base;
}

// h_c[k] = hidden[idx[k]] for k < n and 0 beyond (so that a GEMM reducing
// over the compacted rows in 64-row steps meets zeros past n); the gradient
// rows of the rows left out are zeroed; for reduction none the per-row
// grad_output is gathered the same way.
__global__ void __launch_bounds__(256) flce_gather_kernel(const uint4 *hidden, int64_t row16, int64_t n_rows,
                                                          const int *idx, const int *pos, const int *count, uint4 *hc,
                                                          uint4 *grad_hidden, const float *g_in, float *g_c) {
    const int64_t n = __ldg(count);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
        uint4 *dst = hc + r * row16;
        if (r < n) {
            const uint4 *src = hidden + static_cast<int64_t>(__ldg(idx + r)) * row16;
            for (int64_t j = threadIdx.x; j < row16; j += blockDim.x) dst[j] = __ldg(src + j);
        } else {
            for (int64_t j = threadIdx.x; j < row16; j += blockDim.x) dst[j] = zero;
        }
        if (__ldg(pos + r) < 0) {
            uint4 *gh = grad_hidden + r * row16;
            for (int64_t j = threadIdx.x; j < row16; j += blockDim.x) gh[j] = zero;
        }
        if (g_in && threadIdx.x == 0) g_c[r] = r < n ? __ldg(g_in + __ldg(idx + r)) : 0.f;
    }
}

// reduction none after compaction: loss[i] = the compacted row's loss, 0 for rows left out
__global__ void flce_scatter_loss_kernel(const int *pos, const float *row_loss_c, int64_t n_rows, float *loss) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n_rows) return;
    const int k = __ldg(pos + i);
    loss[i] = k >= 0 ? __ldg(row_loss_c + k) : 0.f;
}

// ------------------------------------------------------------------ cross-entropy on a logits chunk
// The rows a chunk kernel handles: all n rows, or with a device-side count
// only min(n, round_up(max(0, *count - off), 64)) (the rows past the count
// in that 64-row block carry ignored targets and become zero rows, which the
// grad_weight GEMM's 64-row K steps then read).
__device__ inline int64_t chunk_rows_64(int64_t n, const int *count, int64_t off) {
    if (!count) return n;
    const int64_t left = static_cast<int64_t>(__ldg(count)) - off;
    const int64_t blk = left > 0 ? (left + 63) / 64 * 64 : 0;
    return blk < n ? blk : n;
}

// What the map kernel needs of one row (32 bytes): p = 2^((z - m) log2e +
// neg_log2d), gradient a p - b w_c off the target, dxy at the target column
// y; y = -1 marks a row whose gradient is all zeros.
struct MapRow {
    float neg_log2d, m, a, b;
    float dxy;
    int y;
    float pad0, pad1;
};
static_assert(sizeof(MapRow) == 32, "two 16-byte loads per row");

struct ChunkArgs {
    const float *z;            // logits chunk [n_rows, ldz] fp32
    int64_t ldz;
    const float4 *part;        // [n_rows, tiles] partial row states of the logits GEMM
    int tiles;
    int64_t n_rows, vocab;
    const void *target;
    int tgt32;
    int64_t ignore_index;
    const float *weight;
    float eps;
    int reduction;
    const float *grad_output;  // [1], or [n_rows] for none, or NULL
    float *loss;               // reduction none: [n_rows]
    float *row_loss;           // mean / sum: [n_rows]
    WsCtl *ctl;
    MapRow *rows;
    float cap, inv_cap;        // softcap (0: off); the logits chunk holds the capped logits
    float z_loss;
    const float2 *pam;         // token accuracy: the logits GEMM's per-tile argmax, or NULL
    __nv_bfloat16 *out;        // dZ [n_rows, ld_out] bf16
    int64_t ld_out;
    const int *row_limit;
    int64_t row_limit_off;
};

// One warp per row: merge the row's tile states, read x_y from the logits,
// form the loss and the gradient scalars.
__global__ void __launch_bounds__(256) flce_row_scalars_kernel(ChunkArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n = chunk_rows_64(a.n_rows, a.row_limit, a.row_limit_off);
    const int64_t V = a.vocab;
    const float inv_v = 1.f / static_cast<float>(V);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp; row < n; row += static_cast<int64_t>(gridDim.x) * 8) {
        const int64_t t = load_target(a.target, a.tgt32, row);
        const bool valid = target_valid(t, a.ignore_index, V);
        RowState st = row_state_empty();
        ArgMax am{-INFINITY, 0x7fffffff};
        if (valid) {
            const float4 *pp = a.part + row * a.tiles;
            for (int j = lane; j < a.tiles; j += 32) {
                const float4 q = __ldg(pp + j);
                st = row_state_merge(st, RowState{q.x, q.y, q.z, q.w});
            }
            st = warp_merge(st);
            if (a.pam) {
                const float2 *pa = a.pam + row * a.tiles;
                for (int j = lane; j < a.tiles; j += 32) {
                    const float2 q = __ldg(pa + j);
                    am = argmax_merge(am, ArgMax{q.x, __float_as_int(q.y)});
                }
                am = warp_argmax(am);
            }
        }
        if (lane != 0) continue;
        MapRow mr{};
        float loss = 0.f;
        mr.y = -1;
        if (valid) {
            const float xy = __ldg(a.z + row * a.ldz + t);
            const float w_all = a.ctl->w_all, w_y_sum = a.ctl->w_y;
            const float wy = a.weight ? __ldg(a.weight + t) : 1.f;
            const float g = a.grad_output ? __ldg(a.grad_output + (a.reduction == CE_RED_NONE ? row : 0)) : 1.f;
            float scale = g;
            if (a.reduction == CE_RED_MEAN) scale = (w_y_sum != 0.f) ? g / w_y_sum : 0.f;
            const float rrel = row_state_rel_sum(st);
            const RowScalars rs =
                make_row_scalars(st.m, st.s, xy, rrel, true, t, wy, w_all, a.eps, inv_v, scale, a.z_loss);
            loss = make_row_scalars(st.m, st.s, xy, rrel, true, t, wy, w_all, a.eps, inv_v, 1.f, a.z_loss).loss;
            if (a.pam && am.i == static_cast<int>(t)) atomicAdd(&a.ctl->n_correct, 1u);
            mr.neg_log2d = rs.neg_log2d; mr.m = rs.m; mr.a = rs.a; mr.b = rs.b; mr.dxy = rs.dxy;
            mr.y = static_cast<int>(t);
        }
        a.rows[row] = mr;
        if (a.reduction == CE_RED_NONE) a.loss[row] = loss;
        else a.row_loss[row] = loss;
    }
}

// dZ = the gradient of every element, rounded once to bf16: a flat map over
// the chunk's 8-element vectors (every thread two vectors per step), logits
// read once with streaming loads, dZ written with streaming stores.
template <bool WEIGHTED>
__device__ inline uint4 map_vec(const ChunkArgs &a, uint32_t row, uint32_t col, const MapRow &mr, const uint4 &u0,
                                const uint4 &u1) {
    float x[8] = {__uint_as_float(u0.x), __uint_as_float(u0.y), __uint_as_float(u0.z), __uint_as_float(u0.w),
                  __uint_as_float(u1.x), __uint_as_float(u1.y), __uint_as_float(u1.z), __uint_as_float(u1.w)};
    float w[8];
    if (WEIGHTED) {
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(a.weight + col));
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(a.weight + col) + 1);
        w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w; w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
    }
    RowScalars rs;
    rs.neg_log2d = mr.neg_log2d; rs.m = mr.m; rs.a = mr.a; rs.b = mr.b;
    const int yr = mr.y - static_cast<int>(col);
    float gr[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        gr[e] = grad_elem(rs, x[e], WEIGHTED ? w[e] : 1.f);
        gr[e] = (e == yr) ? mr.dxy : gr[e];
    }
    if (a.cap > 0.f) {
        // softcap: the chunk holds z = c tanh(x / c); dz/dx = 1 - (z / c)^2
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float te = x[e] * a.inv_cap;
            gr[e] *= fmaf(-te, te, 1.f);
        }
    }
    return Fmt<CE_DT_BF16>::pack(gr);
}

template <bool WEIGHTED>
__global__ void __launch_bounds__(256) flce_map_kernel(ChunkArgs a) {
    const int64_t n = chunk_rows_64(a.n_rows, a.row_limit, a.row_limit_off);
    const uint32_t vpr = static_cast<uint32_t>(a.vocab / 8);
    const uint32_t total = static_cast<uint32_t>(n) * vpr;   // < 2^31 (host check)
    const uint32_t stride = gridDim.x * blockDim.x;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += 2u * stride) {
        const uint32_t i1 = i + stride;
        const bool has1 = i1 < total;
        const uint32_t r0 = i / vpr, c0 = (i - r0 * vpr) * 8u;
        const uint32_t r1 = has1 ? i1 / vpr : r0, c1 = has1 ? (i1 - r1 * vpr) * 8u : c0;
        const float4 *m0p = reinterpret_cast<const float4 *>(a.rows + r0);
        const float4 *m1p = reinterpret_cast<const float4 *>(a.rows + r1);
        const float4 p0a = __ldg(m0p), p0b = __ldg(m0p + 1);
        const float4 p1a = __ldg(m1p), p1b = __ldg(m1p + 1);
        const MapRow mr0{p0a.x, p0a.y, p0a.z, p0a.w, p0b.x, __float_as_int(p0b.y), 0.f, 0.f};
        const MapRow mr1{p1a.x, p1a.y, p1a.z, p1a.w, p1b.x, __float_as_int(p1b.y), 0.f, 0.f};
        const float *z0 = a.z + static_cast<int64_t>(r0) * a.ldz + c0;
        const float *z1 = a.z + static_cast<int64_t>(r1) * a.ldz + c1;
        uint4 u00 = zero, u01 = zero, u10 = zero, u11 = zero;
        if (mr0.y >= 0) { u00 = ld_stream_ro(z0); u01 = ld_stream_ro(z0 + 4); }
        if (has1 && mr1.y >= 0) { u10 = ld_stream_ro(z1); u11 = ld_stream_ro(z1 + 4); }
        const uint4 o0 = mr0.y >= 0 ? map_vec<WEIGHTED>(a, r0, c0, mr0, u00, u01) : zero;
        st_stream(a.out + static_cast<int64_t>(r0) * a.ld_out + c0, o0);
        if (has1) {
            const uint4 o1 = mr1.y >= 0 ? map_vec<WEIGHTED>(a, r1, c1, mr1, u10, u11) : zero;
            st_stream(a.out + static_cast<int64_t>(r1) * a.ld_out + c1, o1);
        }
    }
}

// token accuracy = correct rows / valid rows (counted by the row-scalars kernels)
__global__ void flce_accuracy_kernel(const WsCtl *ctl, float *acc) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        const float n = ctl->n_valid;
        acc[0] = n > 0.f ? static_cast<float>(__ldcg(&ctl->n_correct)) / n : 0.f;
    }
}

// grad_hidden rows from the split-K partials of dZ W: the parts summed in
// fp32 in a fixed order, rounded once to bf16, stored at row_map[r] (or r)
// for the rows below the device-side count.
__global__ void __launch_bounds__(256) flce_splitk_sum_kernel(const float *part, int ksplit, int64_t split_stride,
                                                              int64_t n_rows, int64_t H, const int *count, int64_t off,
                                                              const int *row_map, __nv_bfloat16 *out, int64_t ldo) {
    const int64_t n = dyn_rows(n_rows, count, off);
    const int64_t vpr = H / 8;
    const int64_t total = n * vpr;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / vpr, c = (i - r * vpr) * 8;
        const float *p = part + r * H + c;
        float4 a = __ldcs(reinterpret_cast<const float4 *>(p)), b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
        for (int k = 1; k < ksplit; ++k) {
            const float4 *q = reinterpret_cast<const float4 *>(p + k * split_stride);
            const float4 a2 = __ldcs(q), b2 = __ldcs(q + 1);
            a.x += a2.x; a.y += a2.y; a.z += a2.z; a.w += a2.w;
            b.x += b2.x; b.y += b2.y; b.z += b2.z; b.w += b2.w;
        }
        using FB = Fmt<CE_DT_BF16>;
        const uint4 o = make_uint4(FB::pack2(a.x, a.y), FB::pack2(a.z, a.w), FB::pack2(b.x, b.y), FB::pack2(b.z, b.w));
        const int64_t orow = row_map ? static_cast<int64_t>(__ldg(row_map + r)) : r;
        st_stream(out + orow * ldo + c, o);
    }
}

// loss[0] = sum of the row losses (/ W_y for mean), fixed order, fp64; with
// `count`, only the first *count row losses (the compacted rows).
__global__ void __launch_bounds__(256) flce_reduce_kernel(const float *row_loss, int64_t n0, int reduction,
                                                          const WsCtl *ctl, float *loss, const int *count) {
    __shared__ double sh[8];
    const int64_t n = dyn_rows(n0, count, 0);
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s += static_cast<double>(row_loss[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int k = 0; k < 8; ++k) tot += sh[k];
        if (reduction == CE_RED_MEAN) {
            const float wy = ctl->w_y;
            tot = wy != 0.f ? tot / static_cast<double>(wy) : 0.0;
        }
        loss[0] = static_cast<float>(tot);
    }
}

cudaError_t launch_reduce_row_losses(const float *row_loss, int64_t n, int reduction, const WsCtl *ctl, float *loss,
                                     cudaStream_t s) {
    const int *none = nullptr;
    void *args[] = {&row_loss, &n, &reduction, &ctl, &loss, &none};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&flce_reduce_kernel), dim3(1), dim3(256), args, 0, s);
}

// ------------------------------------------------------------------ host: tensor maps and launch
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 row-major matrix [rows, cols] with row stride ld (elements), box
// of box_cols x box_rows, 128-byte swizzle, zero fill out of bounds.
static cudaError_t make_tmap(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                             uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n < 1) n = 1;
    }
    return n;
}

int gemm_fit_ksplit(int K, int ksplit) {
    const int kiters = (K + GB_K - 1) / GB_K;
    if (ksplit > kiters) ksplit = kiters > 0 ? kiters : 1;
    while (ksplit > 1) {
        const int kper = (kiters + ksplit - 1) / ksplit;
        if ((ksplit - 1) * kper < kiters) break;  // the last part is not empty
        --ksplit;
    }
    return ksplit;
}

// Resident CTA pairs of a pair kernel on a device (0 if unknown), asked once.
static int pair_clusters(const void *fn, int dev) {
    static const void *fns[8];
    static int devs[8], vals[8], used = 0;
    for (int i = 0; i < used; ++i)
        if (fns[i] == fn && devs[i] == dev) return vals[i];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 128);
    cfg.blockDim = dim3(GB_THREADS);
    cfg.dynamicSmemBytes = GP_SMEM;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    (void)cudaGetLastError();
    if (used < 8) { fns[used] = fn; devs[used] = dev; vals[used] = n; ++used; }
    return n;
}

// D[M,N] = A[M,K] B[K,N]. A: K-major = memory [M, K] (lda >= K); MN-major =
// memory [K, M] (lda >= M). B: K-major = memory [N, K]; MN-major = memory [K, N].
cudaError_t gemm_bf16(int M, int N, int K, const void *A, int64_t lda, int a_mn, const void *B, int64_t ldb,
                      int b_mn, int out_kind, void *out, int64_t ldo, const float *bias, unsigned int *status,
                      cudaStream_t s, const GemmDyn *dyn, const GemmStats *stats, int ksplit,
                      int64_t split_stride, int mode) {
    if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
    if (stats && out_kind != OUT_F32_STORE) return cudaErrorInvalidValue;
    if (ksplit < 1) ksplit = 1;
    if (ksplit > 1 && (out_kind != OUT_F32_STORE || stats || (dyn && dyn->dim == 1) || bias ||
                       gemm_fit_ksplit(K, ksplit) != ksplit))
        return cudaErrorInvalidValue;
    if (mode < GEMM_AUTO || mode > GEMM_PAIR) return cudaErrorInvalidValue;
    // CTA pairs (256 x 256 tiles) when both sides span at least two pair tiles
    const bool pair = mode == GEMM_PAIR || (mode == GEMM_AUTO && M >= 2 * GP_M && N >= 2 * GP_N);
    CUtensorMap ta, tb;
    cudaError_t e;
    if (!a_mn) e = make_tmap(&ta, A, M, K, lda, GB_K, GB_M);          // 128 rows per CTA in both kernels
    else e = make_tmap(&ta, A, K, M, lda, 64, GB_K);
    if (e != cudaSuccess) return e;
    if (!b_mn) e = make_tmap(&tb, B, N, K, ldb, GB_K, pair ? 128 : GB_N);
    else e = make_tmap(&tb, B, K, N, ldb, 64, GB_K);
    if (e != cudaSuccess) return e;
    GemmArgs g{};
    g.M = M; g.N = N; g.K = K;
    g.a_mn = a_mn; g.b_mn = b_mn;
    g.out_kind = out_kind; g.out = out; g.ldo = ldo; g.bias = bias;
    g.tiles_m = (M + (pair ? GP_M : GB_M) - 1) / (pair ? GP_M : GB_M);
    g.tiles_n = (N + GB_N - 1) / GB_N;                                 // 256 columns in both kernels
    g.m_fastest = g.tiles_m <= g.tiles_n ? 1 : 0;  // the operand of the short side stays in L2
    g.status = status;
    g.ksplit = ksplit;
    g.split_stride = split_stride;
    if (dyn) {
        g.dyn_count = dyn->count;
        g.dyn_off = dyn->off;
        g.dyn_dim = dyn->dim;
        g.row_map = dyn->row_map;
    }
    int epi = 0;
    if (stats) {
        g.part = stats->part;
        g.st_target = stats->target;
        g.st_tgt32 = stats->tgt32;
        g.st_ignore = stats->ignore_index;
        g.st_weight = stats->weight;
        g.st_cap = stats->cap > 0.f ? stats->cap : 0.f;
        g.st_inv_cap = stats->cap > 0.f ? 1.f / stats->cap : 0.f;
        g.pam = stats->pam;
        epi = 1 + stats->smooth_mode;
        if (stats->smooth_mode < 0 || stats->smooth_mode > 2 || (stats->smooth_mode == 2 && !stats->weight))
            return cudaErrorInvalidValue;
    }
    static const void *const kernels[2][4] = {
        {reinterpret_cast<const void *>(&flce_gemm_kernel<0>), reinterpret_cast<const void *>(&flce_gemm_kernel<1>),
         reinterpret_cast<const void *>(&flce_gemm_kernel<2>), reinterpret_cast<const void *>(&flce_gemm_kernel<3>)},
        {reinterpret_cast<const void *>(&flce_gemm_pair_kernel<0>),
         reinterpret_cast<const void *>(&flce_gemm_pair_kernel<1>),
         reinterpret_cast<const void *>(&flce_gemm_pair_kernel<2>),
         reinterpret_cast<const void *>(&flce_gemm_pair_kernel<3>)}};
    const void *fn = kernels[pair ? 1 : 0][epi];
    const size_t smem = pair ? GP_SMEM : GB_SMEM;
    // the shared-memory limit is a per-device attribute of each kernel: set it once per device
    static uint64_t attr_set[2][4] = {};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(attr_set[pair ? 1 : 0][epi] & bit)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[pair ? 1 : 0][epi] |= bit;
    }
    const int tiles = g.tiles_m * g.tiles_n * ksplit;
    void *args[] = {&ta, &tb, &g};
    if (!pair) {
        const int grid = tiles < sm_count() ? tiles : sm_count();
        return cudaLaunchKernel(fn, dim3(grid), dim3(GB_THREADS), args, GB_SMEM, s);
    }
    // persistent pairs: no more clusters than can be resident at once
    int clusters = pair_clusters(fn, dev);
    if (clusters < 1) clusters = sm_count() / 2 > 0 ? sm_count() / 2 : 1;
    if (clusters > tiles) clusters = tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.blockDim = dim3(GB_THREADS);
    cfg.dynamicSmemBytes = GP_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace ce

// ------------------------------------------------------------------ C ABI
using namespace ce;

namespace {

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

struct FlceLayout {
    size_t ce_ws, z_off, dz_off, total;
    int64_t ldz, ldd;
    // ignored-row compaction: compacted hidden rows, the maps, the compacted
    // targets and per-row grad_output, the valid-row count
    size_t hc_off, idx_off, pos_off, tgt_off, gc_off, cnt_off;
    // statistics path: the logits GEMM's per-tile row states (and argmax), the per-row map scalars
    size_t part_off, pam_off, rows_off;
    int tiles;
    // split-K parts of grad_hidden = dZ W (fp32, dh_splits x chunk x H)
    size_t dhp_off;
    int dh_splits;
};

// Split count of the grad_hidden GEMM: its output has few tiles (chunk x H)
// and a long K (V), so one product per tile leaves the last of few waves
// mostly idle; 4 parts below 1024 tiles, 2 below 2048 (host rule, no device
// query, so the workspace size is a function of the sizes alone).
int flce_dh_splits(int64_t chunk, int64_t H, int64_t V) {
    const int64_t tiles = ((chunk + 127) / 128) * ((H + 255) / 256);
    const int want = tiles >= 2048 ? 1 : (tiles >= 1024 ? 2 : 4);
    return gemm_fit_ksplit(static_cast<int>(V), want);
}

FlceLayout flce_layout(int64_t n_rows, int64_t vocab, int64_t chunk, int64_t hidden, bool compact, bool map_ce) {
    FlceLayout L{};
    L.ce_ws = round_up(static_cast<int64_t>(ws_bytes(n_rows)), 1024);
    L.ldz = round_up(vocab, 4);
    L.ldd = round_up(vocab, 8);
    L.z_off = L.ce_ws;
    L.dz_off = L.z_off + round_up(chunk * L.ldz * 4, 1024);
    L.total = L.dz_off + round_up(chunk * L.ldd * 2, 1024);
    if (compact) {
        L.hc_off = L.total;
        L.idx_off = L.hc_off + round_up(n_rows * hidden * 2, 1024);
        L.pos_off = L.idx_off + round_up(n_rows * 4, 256);
        L.tgt_off = L.pos_off + round_up(n_rows * 4, 256);
        L.gc_off = L.tgt_off + round_up(n_rows * 8, 256);
        L.cnt_off = L.gc_off + round_up(n_rows * 4, 256);
        L.total = L.cnt_off + 256;
    }
    L.dh_splits = flce_dh_splits(chunk, hidden, vocab);
    if (L.dh_splits > 1) {
        L.dhp_off = L.total;
        L.total = L.dhp_off + round_up(static_cast<int64_t>(L.dh_splits) * chunk * hidden * 4, 1024);
    }
    if (map_ce) {
        L.tiles = static_cast<int>((vocab + kGemmTileN - 1) / kGemmTileN);
        L.part_off = L.total;
        L.pam_off = L.part_off + round_up(chunk * L.tiles * 16, 1024);
        L.rows_off = L.pam_off + round_up(chunk * L.tiles * 8, 1024);
        L.total = L.rows_off + round_up(chunk * static_cast<int64_t>(sizeof(MapRow)), 1024);
    }
    return L;
}

bool flce_compacts(const ce_params *p) { return (p->variant & CE_FLCE_DENSE) == 0; }

// The cross-entropy of each chunk runs as the logits GEMM's statistics
// epilogue + a row-scalar kernel + a flat map, unless the caller asks for
// the cluster kernel or the chunk has 2^31 or more 8-element vectors.
bool flce_maps(const ce_params *p, int64_t chunk) {
    return (p->variant & CE_FLCE_CE_CLUSTER) == 0 && chunk * (p->vocab / 8) < (static_cast<int64_t>(1) << 31);
}

ce_status flce_cuda_fail(cudaError_t e) {
    (void)cudaGetLastError();
    return e == cudaSuccess ? CE_OK : CE_ERR_CUDA;
}

}  // namespace

extern "C" {

ce_status ce_gemm_bf16(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int32_t a_mn, const void *B,
                       int64_t ldb, int32_t b_mn, int32_t out_kind, void *D, int64_t ldd, const float *bias,
                       void *stream) {
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return CE_ERR_INVALID_ARG;
    if ((a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1)) return CE_ERR_INVALID_ARG;
    if (out_kind < CE_GEMM_F32_STORE || out_kind > CE_GEMM_BF16_STORE) return CE_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return CE_OK;
    if (!A || !B || !D || !al16(A) || !al16(B)) return CE_ERR_INVALID_ARG;
    if ((lda % 8) || (ldb % 8) || lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldd < N) return CE_ERR_INVALID_ARG;
    if (bias && (out_kind != CE_GEMM_F32_STORE || !al16(bias))) return CE_ERR_INVALID_ARG;
    if (K == 0) return CE_ERR_UNSUPPORTED;
    cudaError_t e = gemm_bf16(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), A, lda, a_mn, B, ldb,
                              b_mn, out_kind, D, ldd, bias, nullptr, reinterpret_cast<cudaStream_t>(stream));
    return flce_cuda_fail(e);
}

ce_status flce_workspace_size(const ce_params *p, int64_t hidden_dim, int64_t chunk_rows, size_t *bytes) {
    if (!p || !bytes || p->n_rows < 0 || p->vocab < 1 || hidden_dim < 1 || chunk_rows < 1) return CE_ERR_INVALID_ARG;
    int64_t chunk = chunk_rows < p->n_rows ? chunk_rows : (p->n_rows > 0 ? p->n_rows : 1);
    *bytes = flce_layout(p->n_rows, p->vocab, chunk, hidden_dim, flce_compacts(p), flce_maps(p, chunk)).total;
    return CE_OK;
}

ce_status flce_fwd_bwd(const ce_params *p, int64_t H, const void *hidden, const void *weight, const float *bias,
                       const void *target, float *loss, const float *grad_output, void *grad_hidden,
                       float *grad_weight, float *grad_bias, int64_t chunk_rows, void *ws, size_t ws_bytes,
                       void *stream) {
    if (!p || p->n_rows < 0 || p->vocab < 1 || H < 1 || chunk_rows < 1) return CE_ERR_INVALID_ARG;
    if (p->dtype != CE_DT_BF16 || (H % 8) || (p->vocab % 8)) return CE_ERR_UNSUPPORTED;
    if (p->reduction != CE_RED_NONE && p->reduction != CE_RED_MEAN && p->reduction != CE_RED_SUM)
        return CE_ERR_INVALID_ARG;
    if (!(p->label_smoothing >= 0.f && p->label_smoothing <= 1.f) || p->reserved != 0) return CE_ERR_INVALID_ARG;
    if (p->target_is_int32 != 0 && p->target_is_int32 != 1) return CE_ERR_INVALID_ARG;
    if (p->class_weight && (reinterpret_cast<uintptr_t>(p->class_weight) & 15u)) return CE_ERR_INVALID_ARG;
    if (!(p->softcap >= 0.f && p->softcap < INFINITY) || !(p->z_loss >= 0.f && p->z_loss < INFINITY))
        return CE_ERR_INVALID_ARG;
    if (p->accuracy && (reinterpret_cast<uintptr_t>(p->accuracy) & 3u)) return CE_ERR_INVALID_ARG;
    if ((p->variant & ~(CE_FLCE_DENSE | CE_FLCE_CE_CLUSTER)) != 0) return CE_ERR_INVALID_ARG;
    if (bias && !al16(bias)) return CE_ERR_INVALID_ARG;
    if (!loss || !ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CE_ERR_INVALID_ARG;
    const int64_t BT = p->n_rows, V = p->vocab;
    if (BT > INT32_MAX || V > INT32_MAX || H > INT32_MAX) return CE_ERR_UNSUPPORTED;
    const int64_t C = chunk_rows < BT ? chunk_rows : (BT > 0 ? BT : 1);
    const bool compact = flce_compacts(p);
    const bool map_ce = flce_maps(p, C);
    const bool options = p->softcap > 0.f || p->z_loss > 0.f || p->accuracy;
    if (options && !map_ce) return CE_ERR_UNSUPPORTED;  // the options live in the statistics path
    const FlceLayout L = flce_layout(BT, V, C, H, compact, map_ce);
    if (ws_bytes < L.total) return CE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (BT > 0 && (!hidden || !weight || !target || !grad_hidden || !grad_weight)) return CE_ERR_INVALID_ARG;
    if (BT > 0 && (!al16(hidden) || !al16(weight) || !al16(grad_hidden) || !al16(grad_weight))) return CE_ERR_INVALID_ARG;
    if (bias && !grad_bias) return CE_ERR_INVALID_ARG;

    WsCtl *ctl = reinterpret_cast<WsCtl *>(ws);
    char *wsb = reinterpret_cast<char *>(ws);
    float *Z = reinterpret_cast<float *>(wsb + L.z_off);
    __nv_bfloat16 *dZ = reinterpret_cast<__nv_bfloat16 *>(wsb + L.dz_off);
    float *row_loss = ws_row_loss(ws);
    const bool none = p->reduction == CE_RED_NONE;

    // batch normalisers over every row (the mean's W_y spans all chunks)
    PrepArgs pa{};
    pa.target = target; pa.tgt32 = p->target_is_int32; pa.reduction = p->reduction;
    pa.n_rows = BT; pa.vocab = V; pa.ignore_index = p->ignore_index; pa.weight = p->class_weight;
    pa.need_w_all = p->label_smoothing > 0.f ? 1 : 0; pa.ctl = ctl;
    cudaError_t e = launch_prep(pa, s);
    if (e != cudaSuccess) return flce_cuda_fail(e);
    if (BT == 0) {
        if (!none && (e = cudaMemsetAsync(loss, 0, sizeof(float), s)) != cudaSuccess)
            return flce_cuda_fail(e);
        if ((e = cudaMemsetAsync(grad_weight, 0, static_cast<size_t>(V) * H * 4, s)) != cudaSuccess)
            return flce_cuda_fail(e);
        if (grad_bias && (e = cudaMemsetAsync(grad_bias, 0, static_cast<size_t>(V) * 4, s)) != cudaSuccess)
            return flce_cuda_fail(e);
        if (p->accuracy && (e = cudaMemsetAsync(p->accuracy, 0, sizeof(float), s)) != cudaSuccess)
            return flce_cuda_fail(e);
        return CE_OK;
    }
    const int mode = p->label_smoothing <= 0.f ? 0 : (p->class_weight ? 2 : 1);
    FusedPlan plan{};
    if (!map_ce) {
        bool ok = false;
        if ((e = fused_plan_f32_to_bf16(mode, C, V, &plan, &ok)) != cudaSuccess) return flce_cuda_fail(e);
        if (!ok) return CE_ERR_UNSUPPORTED;
    }

    // Rows whose target is ignored (or out of range) add nothing to the loss
    // or to grad_weight and have a zero grad_hidden row. With compaction the
    // valid rows are gathered to the front on the device, every kernel of the
    // chunk loop reads the valid-row count from device memory, and the work
    // past it is skipped; the host never learns the count.
    const void *h_src = hidden;
    const void *tgt_src = target;
    int tgt32 = p->target_is_int32;
    const float *g_rows = grad_output;     // reduction none: per-row grad_output in chunk row order
    float *loss_rows = loss;               // reduction none: per-row loss in chunk row order
    const int *count = nullptr, *idx = nullptr, *pos = nullptr;
    if (compact) {
        int *idx_w = reinterpret_cast<int *>(wsb + L.idx_off);
        int *pos_w = reinterpret_cast<int *>(wsb + L.pos_off);
        int64_t *tgt_c = reinterpret_cast<int64_t *>(wsb + L.tgt_off);
        float *g_c = reinterpret_cast<float *>(wsb + L.gc_off);
        int *cnt = reinterpret_cast<int *>(wsb + L.cnt_off);
        {
            const void *tg = target;
            int t32 = p->target_is_int32;
            int64_t n = BT, vv = V, ign = p->ignore_index;
            void *args[] = {&tg, &t32, &n, &vv, &ign, &idx_w, &pos_w, &tgt_c, &cnt};
            e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_compact_kernel), dim3(1),
                                 dim3(kCompactThreads), args, 0, s);
            if (e != cudaSuccess) return flce_cuda_fail(e);
        }
        uint4 *hc = reinterpret_cast<uint4 *>(wsb + L.hc_off);
        {
            const uint4 *hid = reinterpret_cast<const uint4 *>(hidden);
            int64_t row16 = H * 2 / 16, n = BT;
            const int *ci = idx_w, *cp = pos_w, *cc = cnt;
            uint4 *gh = reinterpret_cast<uint4 *>(grad_hidden);
            const float *gi = (none && grad_output) ? grad_output : nullptr;
            float *gc = g_c;
            void *args[] = {&hid, &row16, &n, &ci, &cp, &cc, &hc, &gh, &gi, &gc};
            const int64_t want = static_cast<int64_t>(sm_count()) * 8;
            const int blocks = static_cast<int>(BT < want ? BT : want);
            e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_gather_kernel), dim3(blocks), dim3(256), args,
                                 0, s);
            if (e != cudaSuccess) return flce_cuda_fail(e);
        }
        h_src = hc;
        tgt_src = tgt_c;
        tgt32 = 0;
        if (none && grad_output) g_rows = g_c;
        if (none) loss_rows = row_loss;
        count = cnt;
        idx = idx_w;
        pos = pos_w;
    }
    const int tgt_bytes = tgt32 ? 4 : 8;

    for (int64_t r0 = 0; r0 < BT; r0 += C) {
        const int64_t c = (BT - r0) < C ? (BT - r0) : C;
        const char *h_c = reinterpret_cast<const char *>(h_src) + r0 * H * 2;
        const GemmDyn rows_m{count, static_cast<int>(r0), 0, nullptr};
        const GemmDyn rows_k{count, static_cast<int>(r0), 1, nullptr};
        const GemmDyn rows_out{count, static_cast<int>(r0), 0, idx ? idx + r0 : nullptr};
        const void *tgt_chunk = reinterpret_cast<const char *>(tgt_src) + r0 * tgt_bytes;
        if (map_ce) {
            // Z = h_c W^T (+ b), fp32, with the per-tile row states; then the
            // row scalars and the flat map to dZ (bf16) and the row losses
            float4 *part = reinterpret_cast<float4 *>(wsb + L.part_off);
            float2 *pam = p->accuracy ? reinterpret_cast<float2 *>(wsb + L.pam_off) : nullptr;
            const GemmStats gs{part, tgt_chunk, tgt32, p->ignore_index, mode, p->class_weight, p->softcap, pam};
            e = gemm_bf16(static_cast<int>(c), static_cast<int>(V), static_cast<int>(H), h_c, H, 0, weight, H, 0,
                          0, Z, L.ldz, bias, &ctl->status, s, compact ? &rows_m : nullptr, &gs);
            if (e != cudaSuccess) return flce_cuda_fail(e);
            ChunkArgs ca{};
            ca.z = Z; ca.ldz = L.ldz; ca.part = part; ca.tiles = L.tiles;
            ca.n_rows = c; ca.vocab = V; ca.target = tgt_chunk; ca.tgt32 = tgt32; ca.ignore_index = p->ignore_index;
            ca.weight = p->class_weight; ca.eps = p->label_smoothing; ca.reduction = p->reduction;
            ca.grad_output = g_rows ? (none ? g_rows + r0 : g_rows) : nullptr;
            ca.loss = none ? loss_rows + r0 : loss;
            ca.row_loss = row_loss + r0;
            ca.ctl = ctl;
            ca.cap = p->softcap > 0.f ? p->softcap : 0.f;
            ca.inv_cap = p->softcap > 0.f ? 1.f / p->softcap : 0.f;
            ca.z_loss = p->z_loss;
            ca.pam = pam;
            ca.rows = reinterpret_cast<MapRow *>(wsb + L.rows_off);
            ca.out = dZ; ca.ld_out = L.ldd;
            ca.row_limit = count; ca.row_limit_off = r0;
            void *cargs[] = {&ca};
            const int64_t want = static_cast<int64_t>(sm_count()) * 8;
            const int64_t sblk = (c + 7) / 8;
            e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_row_scalars_kernel),
                                 dim3(static_cast<unsigned>(sblk < want ? sblk : want)), dim3(256), cargs, 0, s);
            if (e != cudaSuccess) return flce_cuda_fail(e);
            const void *mk = mode == 2 ? reinterpret_cast<const void *>(&flce_map_kernel<true>)
                                              : reinterpret_cast<const void *>(&flce_map_kernel<false>);
            e = cudaLaunchKernel(mk, dim3(static_cast<unsigned>(want)), dim3(256), cargs, 0, s);
            if (e != cudaSuccess) return flce_cuda_fail(e);
        } else {
            // Z = h_c W^T (+ b), fp32
            e = gemm_bf16(static_cast<int>(c), static_cast<int>(V), static_cast<int>(H), h_c, H, 0, weight, H, 0,
                          0, Z, L.ldz, bias, &ctl->status, s, compact ? &rows_m : nullptr);
            if (e != cudaSuccess) return flce_cuda_fail(e);
            // cross-entropy forward + backward on the chunk: dZ (bf16) and row losses
            FusedArgs a{};
            a.x = Z; a.n_rows = c; a.vocab = V; a.ld = L.ldz;
            a.target = tgt_chunk;
            a.tgt32 = tgt32; a.reduction = p->reduction; a.ignore_index = p->ignore_index;
            a.weight = p->class_weight; a.eps = p->label_smoothing;
            a.grad_output = g_rows ? (none ? g_rows + r0 : g_rows) : nullptr;
            a.loss = none ? loss_rows + r0 : loss;
            a.row_loss = row_loss + r0;
            a.ctl = ctl;
            a.out = dZ; a.ld_out = L.ldd; a.finalize = 0;
            a.row_limit = count; a.row_limit_off = r0;
            FusedPlan pl = plan;
            if (pl.n_clusters > c) pl.n_clusters = static_cast<int>(c);
            if ((e = launch_fused_f32_to_bf16(a, pl, mode, s)) != cudaSuccess) return flce_cuda_fail(e);
        }
        // grad_hidden rows = dZ W   (A = dZ K-major, B = W stored [V, H] = [K, N]: MN-major);
        // compacted rows are stored back at their own rows
        void *gh = compact ? grad_hidden : reinterpret_cast<char *>(grad_hidden) + r0 * H * 2;
        if (L.dh_splits > 1) {
            // split-K parts in fp32, then one kernel sums them (fixed order), rounds once
            // to bf16 and stores each row at its own position
            float *dhp = reinterpret_cast<float *>(wsb + L.dhp_off);
            const int64_t stride = c * H;
            e = gemm_bf16(static_cast<int>(c), static_cast<int>(H), static_cast<int>(V), dZ, L.ldd, 0, weight, H, 1,
                          0, dhp, H, nullptr, &ctl->status, s, compact ? &rows_m : nullptr, nullptr, L.dh_splits,
                          stride);
            if (e != cudaSuccess) return flce_cuda_fail(e);
            const float *pp = dhp;
            int ks = L.dh_splits;
            int64_t st = stride, nr = c, hh = H, off = r0, ldo = H;
            const int *cc = count;
            const int *rm = compact ? idx + r0 : nullptr;
            __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(gh);
            void *args[] = {&pp, &ks, &st, &nr, &hh, &cc, &off, &rm, &o, &ldo};
            e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_splitk_sum_kernel),
                                 dim3(static_cast<unsigned>(sm_count() * 8)), dim3(256), args, 0, s);
        } else {
            e = gemm_bf16(static_cast<int>(c), static_cast<int>(H), static_cast<int>(V), dZ, L.ldd, 0, weight, H, 1,
                          2, gh, H, nullptr, &ctl->status, s, compact ? &rows_out : nullptr);
        }
        if (e != cudaSuccess) return flce_cuda_fail(e);
        // grad_weight (+)= dZ^T h_c   (A = dZ stored [c, V] = [K, M]: MN-major; B = h_c [K, N]: MN-major)
        e = gemm_bf16(static_cast<int>(V), static_cast<int>(H), static_cast<int>(c), dZ, L.ldd, 1, h_c, H, 1,
                      r0 == 0 ? 0 : 1, grad_weight, H, nullptr, &ctl->status, s, compact ? &rows_k : nullptr);
        if (e != cudaSuccess) return flce_cuda_fail(e);
        if (grad_bias) {
            const int threads = 256;
            const int blocks = static_cast<int>((V + threads - 1) / threads);
            const __nv_bfloat16 *dzc = dZ;
            int64_t ldd = L.ldd;
            int rows = static_cast<int>(c);
            int64_t vv = V;
            int accum = r0 == 0 ? 0 : 1;
            const int *cc = count;
            int off = static_cast<int>(r0);
            void *args[] = {&dzc, &ldd, &rows, &vv, &grad_bias, &accum, &cc, &off};
            e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_colsum_kernel), dim3(blocks), dim3(threads),
                                 args, 0, s);
            if (e != cudaSuccess) return flce_cuda_fail(e);
        }
    }
    if (p->accuracy) {
        const WsCtl *cc = ctl;
        float *acc = p->accuracy;
        void *args[] = {&cc, &acc};
        e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_accuracy_kernel), dim3(1), dim3(32), args, 0, s);
        if (e != cudaSuccess) return flce_cuda_fail(e);
    }
    if (!none) {
        const float *rl = row_loss;
        int64_t n = BT;
        int red = p->reduction;
        const WsCtl *cc = ctl;
        const int *cnt = count;
        void *args[] = {&rl, &n, &red, &cc, &loss, &cnt};
        e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_reduce_kernel), dim3(1), dim3(256), args, 0, s);
        if (e != cudaSuccess) return flce_cuda_fail(e);
    } else if (compact) {
        const int *pp = pos;
        const float *rl = row_loss;
        int64_t n = BT;
        void *args[] = {&pp, &rl, &n, &loss};
        e = cudaLaunchKernel(reinterpret_cast<const void *>(&flce_scatter_loss_kernel),
                             dim3(static_cast<unsigned>((BT + 255) / 256)), dim3(256), args, 0, s);
        if (e != cudaSuccess) return flce_cuda_fail(e);
    }
    return CE_OK;
}

}  // extern "C"
