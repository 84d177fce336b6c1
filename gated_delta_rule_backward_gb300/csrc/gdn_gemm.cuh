// gdn_gemm.cuh -- block-level fp32 products from shared memory on the FP32 pipe.
//
// C[M][N] += A(m, k) B(k, n) over k < K, computed by all NT threads of a CTA, every
// output element owned by exactly one thread and summed over k in increasing order (so
// a product's bits do not depend on how its outputs are spread over threads).
//
// Layouts (all in shared memory, leading dimensions in floats, multiples of 4):
//   A_KMAJOR = false : A(m, k) = A[m * lda + k]      (row-major A)
//   A_KMAJOR = true  : A(m, k) = A[k * lda + m]      (A stored transposed)
//   B_KMAJOR = false : B(k, n) = B[k * ldb + n]      (row-major B)
//   B_KMAJOR = true  : B(k, n) = B[n * ldb + k]      (B stored transposed)
// Thread (ty, tx), tx = tid % NX, ty = tid / NX, NX = N / TN, owns rows
// m = ty * TM + i (i < TM) and columns
//   n = 4 tx + 4 NX c + e   (c < TN/4, e < 4)   when B is row-major (float4 columns),
//   n = tx + NX j           (j < TN)            when B is stored transposed.
// K must be a multiple of 4 and the operands 16-byte aligned.
#pragma once

#include <cuda_runtime.h>

namespace gdn {

template <int M, int N, int TM, int TN, bool B_KMAJOR>
struct GemmMap {
    static constexpr int NX = N / TN;
    static constexpr int NY = M / TM;
    static_assert(M % TM == 0 && N % TN == 0, "tile");
    static_assert(B_KMAJOR || TN % 4 == 0, "row-major B needs TN % 4 == 0");
    __device__ static int row(int tid, int i) { return (tid / NX) * TM + i; }
    __device__ static int col(int tid, int j)
    {
        const int tx = tid % NX;
        if (B_KMAJOR) return tx + NX * j;
        return 4 * tx + 4 * NX * (j >> 2) + (j & 3);
    }
    __device__ static bool active(int tid) { return tid < NX * NY; }
};

// Fragment loads of one 4-wide k step.
template <int TM, bool A_KMAJOR>
__device__ __forceinline__ void frag_a(float (&a)[TM][4], const float* __restrict__ A, int lda,
                                       int m0, int k4)
{
    if constexpr (A_KMAJOR) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            if constexpr (TM % 4 == 0) {
#pragma unroll
                for (int i4 = 0; i4 < TM; i4 += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(A + (k4 + kk) * lda + m0 + i4);
                    a[i4 + 0][kk] = x.x;
                    a[i4 + 1][kk] = x.y;
                    a[i4 + 2][kk] = x.z;
                    a[i4 + 3][kk] = x.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i][kk] = A[(k4 + kk) * lda + m0 + i];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float4 x = *reinterpret_cast<const float4*>(A + (m0 + i) * lda + k4);
            a[i][0] = x.x;
            a[i][1] = x.y;
            a[i][2] = x.z;
            a[i][3] = x.w;
        }
    }
}

template <int TN, int NX, bool B_KMAJOR>
__device__ __forceinline__ void frag_b(float (&b)[4][TN], const float* __restrict__ B, int ldb,
                                       int tx, int k4)
{
    if constexpr (B_KMAJOR) {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const float4 x = *reinterpret_cast<const float4*>(B + (tx + NX * j) * ldb + k4);
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
                const float4 x =
                    *reinterpret_cast<const float4*>(B + (k4 + kk) * ldb + 4 * tx + 4 * NX * c);
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

template <int M, int N, int TM, int TN, bool A_KMAJOR, bool B_KMAJOR>
__device__ __forceinline__ void block_gemm(float (&acc)[TM][TN], const float* __restrict__ A,
                                           int lda, const float* __restrict__ B, int ldb,
                                           int K, int tid)
{
    using Map = GemmMap<M, N, TM, TN, B_KMAJOR>;
    constexpr int NX = Map::NX;
    if (!Map::active(tid)) return;
    const int tx = tid % NX, ty = tid / NX;
    const int m0 = ty * TM;
#pragma unroll 2
    for (int k4 = 0; k4 < K; k4 += 4) {
        float a[TM][4], b[4][TN];
        frag_a<TM, A_KMAJOR>(a, A, lda, m0, k4);
        frag_b<TN, NX, B_KMAJOR>(b, B, ldb, tx, k4);
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
    using Map = GemmMap<M, N, TM, TN, B_KMAJOR>;
    constexpr int NX = Map::NX;
    if (!Map::active(tid)) return;
    const int tx = tid % NX, ty = tid / NX;
    const int m0 = ty * TM;
#pragma unroll 2
    for (int k4 = 0; k4 < K; k4 += 4) {
        float a[TM][4], b[4][TN];
        frag_b<TN, NX, B_KMAJOR>(b, B, ldb, tx, k4);
        frag_a<TM, A1_KMAJOR>(a, A1, lda1, m0, k4);
        frag_fma(acc1, a, b);
        frag_a<TM, A2_KMAJOR>(a, A2, lda2, m0, k4);
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
