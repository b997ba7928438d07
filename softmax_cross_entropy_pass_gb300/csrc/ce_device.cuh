// ce_device.cuh -- device-side building blocks shared by the cross-entropy
// kernels: element formats, vector loads/stores with cache hints, the
// online (max, sum) state and its merge, the per-row scalars of the
// gradient, and thin inline-PTX wrappers for mbarriers, bulk async copies
// and cluster shared memory (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ce.h"

namespace ce {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ workspace
// Control block at the start of the workspace (the rest holds per-row loss).
constexpr size_t kWsCtlBytes = 256;
constexpr int kPrepParts = 8;  // blocks of the normaliser pass with class weights
struct WsCtl {
    unsigned int status;      // CE_FLAG_* bits of the current call
    unsigned int done;        // blocks finished (last-block reduction)
    unsigned int n_correct;   // rows whose argmax is the target (token accuracy)
    unsigned int pad0;
    float n_valid;            // number of valid rows
    float w_y;                // sum of w_{t_i} over valid rows (n_valid when unweighted)
    float w_all;              // sum_c w_c (vocab when unweighted)
    float pad1;
    // per-block partials of the class-weighted normaliser pass, combined in
    // block order by its finishing kernel
    unsigned int prep_bad[kPrepParts];
    double prep_part[kPrepParts][3];  // valid rows, sum w_{t_i}, sum w_c
};
static_assert(sizeof(WsCtl) <= kWsCtlBytes, "workspace control block too large");

// Workspace layout: [control block 256 B][row loss: n_rows fp32, padded to
// 256 B][row statistics: n_rows x 4 fp32 (split ce_fwd_bwd only)].
__host__ __device__ inline size_t ws_row_loss_bytes(int64_t n_rows) {
    return (static_cast<size_t>(n_rows) * sizeof(float) + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ inline size_t ws_bytes(int64_t n_rows) {
    return kWsCtlBytes + ws_row_loss_bytes(n_rows) + static_cast<size_t>(n_rows) * 4 * sizeof(float);
}
__host__ __device__ inline float *ws_row_loss(void *ws) {
    return reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + kWsCtlBytes);
}
__host__ __device__ inline float *ws_stats(void *ws, int64_t n_rows) {
    return reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + kWsCtlBytes + ws_row_loss_bytes(n_rows));
}

// ------------------------------------------------------------------ element formats
// 16-byte vectors: 4 fp32 or 8 bf16 / f16 elements.
template <int DT> struct Fmt;
template <> struct Fmt<CE_DT_F32> {
    static constexpr int kVec = 4;
    static constexpr int kBytes = 4;
    static constexpr uint32_t kNegInfWord = 0xff800000u;  // one -inf
    __device__ static inline void unpack(const uint4 &v, float *x) {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
    __device__ static inline uint4 pack(const float *g) {
        return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]),
                          __float_as_uint(g[2]), __float_as_uint(g[3]));
    }
    __device__ static inline float load1(const void *p, int64_t i) {
        return reinterpret_cast<const float *>(p)[i];
    }
    __device__ static inline void store1(void *p, int64_t i, float g) {
        reinterpret_cast<float *>(p)[i] = g;
    }
    // max of a vector (no packed max for fp32)
    __device__ static inline float vmax(const uint4 &v) {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    // max of the magnitudes (sign bits cleared)
    __device__ static inline float vabsmax(const uint4 &v) {
        const uint32_t m = 0x7fffffffu;
        return vmax(make_uint4(v.x & m, v.y & m, v.z & m, v.w & m));
    }
};
template <> struct Fmt<CE_DT_BF16> {
    static constexpr int kVec = 8;
    static constexpr int kBytes = 2;
    static constexpr uint32_t kNegInfWord = 0xff80ff80u;  // two -inf (bf16)
    __device__ static inline void unpack2(uint32_t u, float &lo, float &hi) {
        lo = __uint_as_float(u << 16);
        hi = __uint_as_float(u & 0xffff0000u);
    }
    __device__ static inline void unpack(const uint4 &v, float *x) {
        unpack2(v.x, x[0], x[1]); unpack2(v.y, x[2], x[3]);
        unpack2(v.z, x[4], x[5]); unpack2(v.w, x[6], x[7]);
    }
    __device__ static inline uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // one RNE rounding each
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static inline uint4 pack(const float *g) {
        return make_uint4(pack2(g[0], g[1]), pack2(g[2], g[3]), pack2(g[4], g[5]), pack2(g[6], g[7]));
    }
    __device__ static inline float load1(const void *p, int64_t i) {
        uint16_t b = reinterpret_cast<const uint16_t *>(p)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    __device__ static inline void store1(void *p, int64_t i, float g) {
        reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(g);
    }
    __device__ static inline uint32_t hmax2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&a),
                                   *reinterpret_cast<__nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    // max of 8 elements via packed bf16x2 max, then one unpack
    __device__ static inline float vmax(const uint4 &v) {
        uint32_t m = hmax2(hmax2(v.x, v.y), hmax2(v.z, v.w));
        float lo, hi;
        unpack2(m, lo, hi);
        return fmaxf(lo, hi);
    }
    // max of the magnitudes (sign bits cleared)
    __device__ static inline float vabsmax(const uint4 &v) {
        const uint32_t m = 0x7fff7fffu;
        return vmax(make_uint4(v.x & m, v.y & m, v.z & m, v.w & m));
    }
};
template <> struct Fmt<CE_DT_F16> {
    static constexpr int kVec = 8;
    static constexpr int kBytes = 2;
    static constexpr uint32_t kNegInfWord = 0xfc00fc00u;  // two -inf (f16)
    __device__ static inline void unpack2(uint32_t u, float &lo, float &hi) {
        float2 f = __half22float2(*reinterpret_cast<__half2 *>(&u));
        lo = f.x; hi = f.y;
    }
    __device__ static inline void unpack(const uint4 &v, float *x) {
        unpack2(v.x, x[0], x[1]); unpack2(v.y, x[2], x[3]);
        unpack2(v.z, x[4], x[5]); unpack2(v.w, x[6], x[7]);
    }
    __device__ static inline uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static inline uint4 pack(const float *g) {
        return make_uint4(pack2(g[0], g[1]), pack2(g[2], g[3]), pack2(g[4], g[5]), pack2(g[6], g[7]));
    }
    __device__ static inline float load1(const void *p, int64_t i) {
        return __half2float(reinterpret_cast<const __half *>(p)[i]);
    }
    __device__ static inline void store1(void *p, int64_t i, float g) {
        reinterpret_cast<__half *>(p)[i] = __float2half_rn(g);
    }
    __device__ static inline uint32_t hmax2(uint32_t a, uint32_t b) {
        __half2 r = __hmax2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    __device__ static inline float vmax(const uint4 &v) {
        uint32_t m = hmax2(hmax2(v.x, v.y), hmax2(v.z, v.w));
        float lo, hi;
        unpack2(m, lo, hi);
        return fmaxf(lo, hi);
    }
    // max of the magnitudes (sign bits cleared)
    __device__ static inline float vabsmax(const uint4 &v) {
        const uint32_t m = 0x7fff7fffu;
        return vmax(make_uint4(v.x & m, v.y & m, v.z & m, v.w & m));
    }
};

// ------------------------------------------------------------------ memory ops
__device__ inline uint4 ld_stream_ro(const void *p) {  // read-only, no L1 allocation
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ inline uint4 ld_stream(const void *p) {     // coherent, no L1 allocation
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ inline void st_stream(void *p, const uint4 &v) {  // streaming store (evict first)
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ inline void st_stream_v2(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(a), "r"(b) : "memory");
}
__device__ inline uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ inline uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ targets
__device__ inline int64_t load_target(const void *target, int is32, int64_t i) {
    return is32 ? static_cast<int64_t>(reinterpret_cast<const int32_t *>(target)[i])
                : reinterpret_cast<const int64_t *>(target)[i];
}
__device__ inline bool target_valid(int64_t t, int64_t ignore_index, int64_t vocab) {
    return t != ignore_index && t >= 0 && t < vocab;
}

// ------------------------------------------------------------------ exponentials
// 2^x on the hardware exponential unit (MUFU ex2, approximate, flushing
// subnormal inputs and results to zero): every exponential of the kernels
// has x <= 0 and a result in (0, 1]; results under 2^-126 become 0.
__device__ inline float ex2_hw(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ packed fp32 pairs
// Two fp32 values in one 64-bit register pair, operated on by the packed
// fp32 instructions of sm_100-class GPUs (add / sub / fma .rn.f32x2): each
// lane is rounded exactly as the scalar instruction would round it, so a
// loop rewritten over pairs gives bit-identical results with half the FP32
// instructions.
struct F2 {
    uint64_t v;
};
__device__ inline F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ inline void f2_split(F2 a, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ inline F2 f2_add(F2 a, F2 b) {
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ inline F2 f2_sub(F2 a, F2 b) {
    F2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ inline F2 f2_mul(F2 a, F2 b) {
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ inline F2 f2_fma(F2 a, F2 b, F2 c) {
    F2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
__device__ inline F2 f2_ex2(F2 a) {
    float lo, hi;
    f2_split(a, lo, hi);
    return f2(ex2_hw(lo), ex2_hw(hi));
}

// ------------------------------------------------------------------ online softmax state
// One thread's (or block's) running statistics over a set of columns:
//   m = max x, s = sum exp(x - m) over non-target columns,
//   r = sum w_c x_c (the smoothing sum), n = sum w_c.
// r is kept as a plain sum; the statistics report r - n*m, the smoothing
// sum relative to m.
struct RowState {
    float m, s, r, n;
};
__device__ inline RowState row_state_empty() { return RowState{-INFINITY, 0.f, 0.f, 0.f}; }

// Merge two states onto the larger max.
__device__ inline RowState row_state_merge(const RowState &a, const RowState &b) {
    float M = fmaxf(a.m, b.m);
    RowState o;
    o.m = M;
    o.r = a.r + b.r;
    o.n = a.n + b.n;
    if (M == -INFINITY) { o.s = a.s + b.s; return o; }
    float fa = (a.m == -INFINITY) ? 0.f : ex2_hw((a.m - M) * kLog2e);
    float fb = (b.m == -INFINITY) ? 0.f : ex2_hw((b.m - M) * kLog2e);
    o.s = a.s * fa + b.s * fb;
    return o;
}

// Merge over groups of W lanes (W a power of two, at most 32): every lane
// ends with the merge of its group, in the same order in every group.
template <int W = 32>
__device__ inline RowState warp_merge(RowState st) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) {
        RowState o;
        o.m = __shfl_xor_sync(0xffffffffu, st.m, off);
        o.s = __shfl_xor_sync(0xffffffffu, st.s, off);
        o.r = __shfl_xor_sync(0xffffffffu, st.r, off);
        o.n = __shfl_xor_sync(0xffffffffu, st.n, off);
        st = row_state_merge(st, o);
    }
    return st;
}

// Fold the values of one vector into the state. `skip` (-1 for none) is the
// lane holding the target column, left out of s but kept in m and r.
// `SMOOTH` accumulates r and n (label smoothing); `w` is the class weight of
// each lane (nullptr for all ones). One FFMA and one MUFU ex2 per element
// for the exp-sum: exp(x - m) = 2^(x log2e - m log2e).
template <int VEC, bool SMOOTH>
__device__ inline void row_state_add(RowState &st, const float *x, float vmax, int skip,
                                     const float *w) {
    if (vmax > st.m) {
        if (st.m != -INFINITY) st.s *= ex2_hw((st.m - vmax) * kLog2e);
        st.m = vmax;
    }
    if (SMOOTH) {
        float racc = 0.f;
        if (w) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) { racc = fmaf(w[j], x[j], racc); st.n += w[j]; }
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) racc += x[j];
            st.n += static_cast<float>(VEC);
        }
        st.r += racc;
    }
    if (st.m == -INFINITY) return;  // every value seen so far is -inf: nothing to add
    const float mL = st.m * kLog2e;
    float acc = 0.f;
    if (skip < 0) {
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc += ex2_hw(fmaf(x[j], kLog2e, -mL));
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc += (j == skip) ? 0.f : ex2_hw(fmaf(x[j], kLog2e, -mL));
    }
    st.s += acc;
}

// the smoothing sum relative to the row max, as reported in the statistics
// (the product is rounded on its own, not fused into the subtraction, so a
// row of equal logits gives exactly 0)
__device__ inline float row_state_rel_sum(const RowState &st) {
    return st.n > 0.f ? __fsub_rn(st.r, __fmul_rn(st.n, st.m)) : 0.f;
}

// ------------------------------------------------------------------ softcap and argmax
// z = c tanh(x / c) with CUDA's accurate tanhf, for the row-pass and split
// kernels (the hardware tanh.approx, about 2^-11 relative, would move exp(z)
// by more than half a bf16 ulp), and dz/dx = 1 - (z / c)^2.
__device__ inline float softcap_logit(float x, float c) { return c * tanhf(x / c); }
__device__ inline float softcap_deriv(float z, float c) {
    const float u = z / c;
    return fmaf(-u, u, 1.f);
}

// The softcap z = c tanh(x / c) of the stream kernel and of the fused-linear
// epilogue, cheaper than c * tanhf(x / c). With u = x / c and w = u^2:
//   |u| < 0.3:  z = x (1 + n1 w + n2 w^2 + n3 w^3),
//   |u| < 0.8:  z = x (1 + c1 w + ... + c6 w^6),
//   otherwise:  z = c sign(u) (1 - 2 / (1 + e^(2|u|))), with the hardware
//               exponential and an approximate divide (no cancellation: the
//               result is above 0.66 c; the exponent is clamped at 126 so the
//               denominator stays in range, tanh being 1 in fp32 well before).
// The polynomials are least-squares fits (tanh_fit.py) of tanh(u) / u, within
// about 1.2 and 2.5 units in the last place of tanh in fp32; x p(w) stands for
// c u p(w) (the two differ by the rounding of c / c). NaN stays NaN.
constexpr float kTanhN1 = -0.33333057165145874f;
constexpr float kTanhN2 = 0.1331467479467392f;
constexpr float kTanhN3 = -0.05035468563437462f;
constexpr float kTanhC1 = -0.33333298563957214f;
constexpr float kTanhC2 = 0.13332220911979675f;
constexpr float kTanhC3 = -0.053852491080760956f;
constexpr float kTanhC4 = 0.021303808316588402f;
constexpr float kTanhC5 = -0.007411024998873472f;
constexpr float kTanhC6 = 0.0015856500249356031f;
constexpr float kTanhNarrowEdge = 0.3f;
constexpr float kTanhPolyEdge = 0.8f;

__device__ inline float tanh_poly_narrow(float w) {
    float p = fmaf(w, kTanhN3, kTanhN2);
    p = fmaf(p, w, kTanhN1);
    return fmaf(p, w, 1.f);
}
__device__ inline float tanh_poly(float w) {
    float p = fmaf(w, kTanhC6, kTanhC5);
    p = fmaf(p, w, kTanhC4);
    p = fmaf(p, w, kTanhC3);
    p = fmaf(p, w, kTanhC2);
    p = fmaf(p, w, kTanhC1);
    return fmaf(p, w, 1.f);
}
__device__ inline F2 tanh_poly_narrow2(F2 w) {
    F2 p = f2_fma(w, f2(kTanhN3, kTanhN3), f2(kTanhN2, kTanhN2));
    p = f2_fma(p, w, f2(kTanhN1, kTanhN1));
    return f2_fma(p, w, f2(1.f, 1.f));
}
__device__ inline F2 tanh_poly2(F2 w) {
    F2 p = f2_fma(w, f2(kTanhC6, kTanhC6), f2(kTanhC5, kTanhC5));
    p = f2_fma(p, w, f2(kTanhC4, kTanhC4));
    p = f2_fma(p, w, f2(kTanhC3, kTanhC3));
    p = f2_fma(p, w, f2(kTanhC2, kTanhC2));
    p = f2_fma(p, w, f2(kTanhC1, kTanhC1));
    return f2_fma(p, w, f2(1.f, 1.f));
}
__device__ inline float tanh_exp_form(float u) {
    const float e = ex2_hw(fminf(fabsf(u) * (2.f * kLog2e), 126.f));
    return copysignf(1.f - __fdividef(2.f, 1.f + e), u);
}

// One logit, its range chosen by its own |x| against 0.3 c and 0.8 c.
__device__ inline float softcap_fast(float x, float cap, float inv_cap) {
    const float a = fabsf(x);
    if (a >= kTanhPolyEdge * cap) return cap * tanh_exp_form(x * inv_cap);
    const float u = x * inv_cap, w = u * u;
    return x * (a < kTanhNarrowEdge * cap ? tanh_poly_narrow(w) : tanh_poly(w));
}

// The form softcap_vec_form takes for values with |x| <= a: 0 the narrow
// polynomial alone, 1 the general form (correct for any values).
__device__ inline unsigned softcap_form(float a, float cap) {
    return a < kTanhNarrowEdge * cap ? 0u : 1u;
}

// N logits (N even) in packed pairs, in the given form (one that covers every
// value of the vector, softcap_form): the narrow polynomial alone, or the wide
// polynomial and the exponential form for every value with a select (no
// divergence inside the vector). The stream kernel takes one form per thread
// and chunk and keeps it for the second pass, so logits of ordinary size never
// pay for the wider polynomial, an exponential or a divide; two forms only keep
// the inlined code small. The forms agree to about 2 units in the last place.
// x and z may alias.
template <int N>
__device__ inline void softcap_vec_form(const float *x, float *z, float cap, float inv_cap, unsigned form) {
    const F2 ic = f2(inv_cap, inv_cap);
    if (form == 0u) {
#pragma unroll
        for (int p = 0; p < N / 2; ++p) {
            const F2 xx = f2(x[2 * p], x[2 * p + 1]), u = f2_mul(xx, ic);
            f2_split(f2_mul(xx, tanh_poly_narrow2(f2_mul(u, u))), z[2 * p], z[2 * p + 1]);
        }
    } else {
        const float edge = kTanhPolyEdge * cap;
#pragma unroll
        for (int p = 0; p < N / 2; ++p) {
            const float x0 = x[2 * p], x1 = x[2 * p + 1];
            const F2 xx = f2(x0, x1), u = f2_mul(xx, ic);
            float q0, q1;
            f2_split(f2_mul(xx, tanh_poly2(f2_mul(u, u))), q0, q1);
            const float e0 = cap * tanh_exp_form(x0 * inv_cap), e1 = cap * tanh_exp_form(x1 * inv_cap);
            z[2 * p] = fabsf(x0) >= edge ? e0 : q0;
            z[2 * p + 1] = fabsf(x1) >= edge ? e1 : q1;
        }
    }
}

// The same with the form the vector's own largest |x| needs.
template <int N>
__device__ inline void softcap_vec(const float *x, float *z, float cap, float inv_cap) {
    float xmax = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) xmax = fmaxf(xmax, fabsf(x[j]));
    softcap_vec_form<N>(x, z, cap, inv_cap, softcap_form(xmax, cap));
}

// g *= dz/dx = 1 - (z / c)^2 for N values (N even), in packed pairs;
// nic2 = -1 / c^2.
template <int N>
__device__ inline void softcap_deriv_vec(float *g, const float *z, float nic2) {
    const F2 n2 = f2(nic2, nic2), one = f2(1.f, 1.f);
#pragma unroll
    for (int p = 0; p < N / 2; ++p) {
        const F2 zz = f2(z[2 * p], z[2 * p + 1]);
        f2_split(f2_mul(f2(g[2 * p], g[2 * p + 1]), f2_fma(f2_mul(zz, zz), n2, one)), g[2 * p], g[2 * p + 1]);
    }
}

// The first column holding the maximum (ties go to the smaller column).
struct ArgMax {
    float v;
    int i;
};
__device__ inline ArgMax argmax_merge(const ArgMax &a, const ArgMax &b) {
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}
template <int W = 32>
__device__ inline ArgMax warp_argmax(ArgMax a) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) {
        ArgMax o;
        o.v = __shfl_xor_sync(0xffffffffu, a.v, off);
        o.i = __shfl_xor_sync(0xffffffffu, a.i, off);
        a = argmax_merge(a, o);
    }
    return a;
}

// ------------------------------------------------------------------ per-row scalars
// Everything the gradient and the loss of one row need, formed once in fp32
// from the row statistics (m, s, x_y, r) and the batch normalisers.
struct RowScalars {
    float neg_log2d;  // -log2(d): p = exp2((x - m) * log2e - log2 d)
    float m;
    float a;          // scale * ((1-eps) w_y + (eps/V) W_all): coefficient of p
    float b;          // scale * eps / V: coefficient of -w_c
    float dxy;        // the gradient at the target column, formed once
    float loss;       // loss_i (0 on invalid rows)
    int64_t y;        // target column (-1 on invalid rows)
};

__device__ inline float softplus_f(float t) {
    return t > 0.f ? t + log1pf(expf(-t)) : log1pf(expf(t));
}

// m, s (off-target exp-sum), xy, r as in the stats layout; wy = w_{t_i};
// scale = s_i of the gradient; valid = row has a usable target.
__device__ inline RowScalars make_row_scalars(float m, float s, float xy, float r, bool valid,
                                              int64_t y, float wy, float w_all, float eps,
                                              float inv_v, float scale, float z_loss = 0.f) {
    RowScalars o;
    o.m = m;
    if (!valid) {
        o.neg_log2d = 0.f; o.a = 0.f; o.b = 0.f; o.dxy = 0.f; o.loss = 0.f; o.y = -1;
        return o;
    }
    const float e_y = expf(xy - m);     // <= 1
    const float d = s + e_y;            // >= 1
    const float log_d = logf(d);
    o.neg_log2d = -log_d * kLog2e;
    const float eps_v = eps * inv_v;
    o.a = scale * ((1.f - eps) * wy + eps_v * w_all);
    o.b = scale * eps_v;
    const float p_y = e_y / d;
    const float one_minus_py = s / d;   // no cancellation: s excludes the target
    o.dxy = scale * (-(1.f - eps) * wy * one_minus_py + eps_v * (p_y * w_all - wy));
    // LSE - x_y = log1p(s * exp(m - x_y)) = softplus(log s + m - x_y)
    const float nll = (s > 0.f) ? softplus_f(logf(s) + (m - xy)) : 0.f;
    o.loss = (1.f - eps) * wy * nll + eps_v * (w_all * log_d - r);
    if (z_loss > 0.f) {
        // lambda LSE^2: loss term, and 2 lambda LSE p in the gradient
        const float lse = m + log_d;
        o.loss += z_loss * lse * lse;
        const float zc = scale * 2.f * z_loss * lse;
        o.a += zc;
        o.dxy += zc * p_y;
    }
    o.y = y;
    return o;
}

// gradient of one off-target element
__device__ inline float grad_elem(const RowScalars &rs, float x, float wc) {
    float p = ex2_hw(fmaf(x - rs.m, kLog2e, rs.neg_log2d));
    return fmaf(p, rs.a, -rs.b * wc);
}

// ------------------------------------------------------------------ mbarrier / bulk copy / cluster
__device__ inline void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ inline void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}
__device__ inline void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
// arrive on an mbarrier of another CTA of the cluster (address from mapa),
// releasing this thread's earlier shared::cluster stores at cluster scope
__device__ inline void mbar_arrive_remote(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_bar) : "memory");
}
__device__ inline bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ inline bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// The same with a suspend-time hint: a thread whose phase is not complete
// sleeps in hardware until the phase completes or about hint_ns have passed,
// instead of returning at once and spinning (spinning warps take issue slots
// from the working warps of their scheduler).
__device__ inline bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}
__device__ inline bool mbar_try_wait_cluster_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}
__device__ inline uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after ~`limit_ns` and returns false. A wait that
// gives up marks `*abort` so that later waits of the CTA return at once.
// SLEEP_NS > 0: each try sleeps up to that long while the phase is not
// complete (mbar_try_wait_sleep), and the limit is checked after every try.
template <bool CLUSTER_SCOPE, uint32_t SLEEP_NS = 0>
__device__ inline bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort,
                                         uint64_t limit_ns = 2000000000ull) {
    if (SLEEP_NS > 0) {
        if (CLUSTER_SCOPE ? mbar_try_wait_cluster_sleep(bar, parity, SLEEP_NS) : mbar_try_wait_sleep(bar, parity, SLEEP_NS))
            return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (CLUSTER_SCOPE ? mbar_try_wait_cluster_sleep(bar, parity, SLEEP_NS)
                              : mbar_try_wait_sleep(bar, parity, SLEEP_NS))
                return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) { *abort = 1; return false; }
        }
    }
    if (CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))
            return true;
        if ((it & 255u) == 255u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) { *abort = 1; return false; }
        }
    }
}

// 1-D bulk async copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ inline void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
__device__ inline uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: the normaliser kernel lets the next kernel
// of the stream start at once; that kernel waits for the normalisers (the
// whole previous grid, with its memory visible) only where it reads them.
// Both are no-ops when the launch carries no programmatic dependency.
__device__ inline void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ inline uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ inline uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ inline uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %clusterid.x;" : "=r"(r));
    return r;
}
// the CTA's index and the grid's size along x read afresh (asm volatile: not
// merged with earlier reads, so no register holds them through a long loop)
__device__ inline uint32_t ctaid_x_fresh() {
    uint32_t r;
    asm volatile("mov.u32 %0, %ctaid.x;" : "=r"(r));
    return r;
}
__device__ inline uint32_t nctaid_x_fresh() {
    uint32_t r;
    asm volatile("mov.u32 %0, %nctaid.x;" : "=r"(r));
    return r;
}
__device__ inline uint32_t nclusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %nclusterid.x;" : "=r"(r));
    return r;
}
// address of the same shared-memory variable in CTA `rank` of the cluster
__device__ inline uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ inline void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ inline void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ inline void fence_mbar_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

}  // namespace ce
