// flce.h -- internal declarations of the tensor-core GEMM used by the
// fused-linear cross-entropy.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ce {

// D[M,N] (op)= A[M,K] B[K,N] with bf16 operands and fp32 accumulation.
// a_mn / b_mn: operand stored MN-major (A as [K, M], B as [K, N]) instead of
// K-major (A as [M, K], B as [N, K]). out_kind: 0 fp32 store (+ bias[N]),
// 1 fp32 accumulate, 2 bf16 store.
// `dyn` (optional) makes M or K a device-side value: the kernel uses
// clamp(*count - off, 0, M or K) (dim 0: M, 1: K), and `row_map` sends output
// row r to row row_map[r]. The sizes passed here are then upper bounds.
struct GemmDyn {
    const int *count;
    int off;
    int dim;
    const int *row_map;
};

// `ksplit` > 1 (fp32 store only, static K) computes every tile as ksplit
// partial products over consecutive K ranges, partial p stored at
// out + p * split_stride.
// `stats` (optional, fp32 store only) also writes, for every output row and
// 256-column tile, the tile's softmax state {max, exp-sum without the
// row's target column, smoothing sum, weight sum} to part[row * tiles + t]
// (tiles = ceil(N / 256)); smooth_mode 0: no smoothing sums, 1: plain sum
// of the logits, 2: class-weighted (weight[N]).
struct GemmStats {
    float4 *part;
    const void *target;
    int tgt32;
    int64_t ignore_index;
    int smooth_mode;
    const float *weight;
    float cap;      // softcap c > 0: the stored logits and the states are those of c tanh(x / c)
    float2 *pam;    // or NULL: per row and tile {raw maximum, its first column} (token accuracy)
};
constexpr int kGemmTileN = 256;

// `mode`: GEMM_AUTO (CTA pairs on 256 x 256 tiles when M and N both span at
// least two such tiles, else one CTA per 128 x 256 tile), GEMM_ONE_CTA,
// GEMM_PAIR.
enum { GEMM_AUTO = 0, GEMM_ONE_CTA = 1, GEMM_PAIR = 2 };

cudaError_t gemm_bf16(int M, int N, int K, const void *A, int64_t lda, int a_mn, const void *B,
                      int64_t ldb, int b_mn, int out_kind, void *out, int64_t ldo, const float *bias,
                      unsigned int *status, cudaStream_t s, const GemmDyn *dyn = nullptr,
                      const GemmStats *stats = nullptr, int ksplit = 1, int64_t split_stride = 0,
                      int mode = GEMM_AUTO);

// K steps of 64 per split-K part: ksplit parts over kiters steps, each
// non-empty (the split count actually used, <= ksplit).
int gemm_fit_ksplit(int K, int ksplit);

}  // namespace ce
