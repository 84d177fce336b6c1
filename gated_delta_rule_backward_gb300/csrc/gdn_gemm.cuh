// gdn_gemm.cuh -- block-level fp32 products from shared memory on the FP32 pipe.
//
// C[M][N] += A(m, k) B(k, n) over k < K, computed by the 256 threads (8 warps) of a CTA,
// every output element owned by exactly one thread and summed over k in increasing
// order (so a product's bits do not depend on how its outputs are spread over threads).
//
// Layouts (all in shared memory, leading dimensions in floats, multiples of 4; leading
// dimensions = 4 mod 32 keep the loads below free of bank conflicts):
//   A_KMAJOR = false : A(m, k) = A[m * lda + k]      (row-major A)
//   A_KMAJOR = true  : A(m, k) = A[k * lda + m]      (A stored transposed)
//   B_KMAJOR = false : B(k, n) = B[k * ldb + n]      (row-major B)
//   B_KMAJOR = true  : B(k, n) = B[n * ldb + k]      (B stored transposed)
//
// Thread mapping: the 8 warps tile the output as WGR x WGC warp tiles of
// (M / WGR) x (N / WGC); inside a warp the lanes form an 8 x 4 grid (lr = lane / 4,
// lc = lane % 4) and each thread owns TM x TN outputs:
//   rows    m = wr * (M / WGR) + lr + 8 i                        (i < TM)
//   columns n = wc * (N / WGC) + 4 lc + 16 c + e  (c < TN/4, e < 4)   row-major B
//           n = wc * (N / WGC) + lc + 4 j           (j < TN)          transposed B
// so a warp's A loads are 8 rows shared by 4 lanes each and its B loads 4 column groups
// shared by 8 lanes each.  M = WGR * 8 * TM, N = WGC * 4 * TN, WGR * WGC = 8.
#pragma once

#include <cuda_runtime.h>

namespace gdn {

template <int M, int N, int TM, int TN, bool B_KMAJOR>
struct GemmMap {
    static constexpr int WGR = M / (8 * TM);
    static constexpr int WGC = N / (4 * TN);
    static constexpr int WTM = M / WGR;
    static constexpr int WTN = N / WGC;
    static_assert(WGR * 8 * TM == M && WGC * 4 * TN == N, "tile");
    static_assert(WGR * WGC == 8, "the 8 warps must tile the output");
    static_assert(B_KMAJOR || TN % 4 == 0, "row-major B needs TN % 4 == 0");
    __device__ static int wr(int tid) { return (tid >> 5) / WGC; }
    __device__ static int wc(int tid) { return (tid >> 5) % WGC; }
    __device__ static int row(int tid, int i) { return wr(tid) * WTM + ((tid & 31) >> 2) + 8 * i; }
    __device__ static int col(int tid, int j)
    {
        const int lc = tid & 3;
        if (B_KMAJOR) return wc(tid) * WTN + lc + 4 * j;
        return wc(tid) * WTN + 4 * lc + 16 * (j >> 2) + (j & 3);
    }
};

// Fragment loads of one 4-wide k step.
template <int TM, bool A_KMAJOR>
__device__ __forceinline__ void frag_a(float (&a)[TM][4], const float* __restrict__ A, int lda,
                                       int mb, int k4)
{
    if constexpr (A_KMAJOR) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i][kk] = A[(k4 + kk) * lda + mb + 8 * i];
    } else {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float4 x = *reinterpret_cast<const float4*>(A + (mb + 8 * i) * lda + k4);
            a[i][0] = x.x;
            a[i][1] = x.y;
            a[i][2] = x.z;
            a[i][3] = x.w;
        }
    }
}

template <int TN, bool B_KMAJOR>
__device__ __forceinline__ void frag_b(float (&b)[4][TN], const float* __restrict__ B, int ldb,
                                       int nb, int k4)
{
    if constexpr (B_KMAJOR) {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const float4 x = *reinterpret_cast<const float4*>(B + (nb + 4 * j) * ldb + k4);
            b[0][j] = x.x;
            b[1][j] = x.y;
            b[2][j] = x.z;
            b[3][j] = x.w;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int c = 0; c < TN / 4; ++c) {
                const float4 x = *reinterpret_cast<const float4*>(B + (k4 + kk) * ldb + nb + 16 * c);
                b[kk][4 * c + 0] = x.x;
                b[kk][4 * c + 1] = x.y;
                b[kk][4 * c + 2] = x.z;
                b[kk][4 * c + 3] = x.w;
            }
    }
}

template <int TM, int TN>
__device__ __forceinline__ void frag_fma(float (&acc)[TM][TN], const float (&a)[TM][4],
                                         const float (&b)[4][TN])
{
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(a[i][kk], b[kk][j], acc[i][j]);
}

// First row / column a thread's fragments start from.
template <int M, int N, int TM, int TN, bool B_KMAJOR>
__device__ __forceinline__ void frag_origin(int tid, int& mb, int& nb)
{
    using Map = GemmMap<M, N, TM, TN, B_KMAJOR>;
    mb = Map::wr(tid) * Map::WTM + ((tid & 31) >> 2);
    nb = Map::wc(tid) * Map::WTN + (B_KMAJOR ? (tid & 3) : 4 * (tid & 3));
}

template <int M, int N, int TM, int TN, bool A_KMAJOR, bool B_KMAJOR>
__device__ __forceinline__ void block_gemm(float (&acc)[TM][TN], const float* __restrict__ A,
                                           int lda, const float* __restrict__ B, int ldb,
                                           int K, int tid)
{
    int mb, nb;
    frag_origin<M, N, TM, TN, B_KMAJOR>(tid, mb, nb);
#pragma unroll 2
    for (int k4 = 0; k4 < K; k4 += 4) {
        float a[TM][4], b[4][TN];
        frag_a<TM, A_KMAJOR>(a, A, lda, mb, k4);
        frag_b<TN, B_KMAJOR>(b, B, ldb, nb, k4);
        frag_fma(acc, a, b);
    }
}

// Two products sharing the B operand: C1 += A1 B, C2 += A2 B (same thread mapping as
// block_gemm with the same M, N, TM, TN, B layout).  Sharing B halves its smem traffic.
template <int M, int N, int TM, int TN, bool A1_KMAJOR, bool A2_KMAJOR, bool B_KMAJOR>
__device__ __forceinline__ void block_gemm_dual(float (&acc1)[TM][TN], const float* __restrict__ A1,
                                                int lda1, float (&acc2)[TM][TN],
                                                const float* __restrict__ A2, int lda2,
                                                const float* __restrict__ B, int ldb, int K, int tid)
{
    int mb, nb;
    frag_origin<M, N, TM, TN, B_KMAJOR>(tid, mb, nb);
#pragma unroll 2
    for (int k4 = 0; k4 < K; k4 += 4) {
        float a[TM][4], b[4][TN];
        frag_b<TN, B_KMAJOR>(b, B, ldb, nb, k4);
        frag_a<TM, A1_KMAJOR>(a, A1, lda1, mb, k4);
        frag_fma(acc1, a, b);
        frag_a<TM, A2_KMAJOR>(a, A2, lda2, mb, k4);
        frag_fma(acc2, a, b);
    }
}

template <int TM, int TN>
__device__ __forceinline__ void zero_acc(float (&acc)[TM][TN])
{
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
}

}  // namespace gdn
