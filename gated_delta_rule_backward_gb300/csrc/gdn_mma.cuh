// gdn_mma.cuh -- block-level fp32 products on the tensor pipe: warp-level m16n8k8 tf32 MMAs
// (mma.sync) with the three-pass split of gdn_tc.cuh (x = hi + lo, a b ~= hi_a hi_b +
// hi_a lo_b + lo_a hi_b; the dropped lo lo term is below 2^-20 |a b|).
//
// C[M][N] += A(m, k) B(k, n) over k < K (K a multiple of 8), operands in shared memory with
// the layouts of gdn_gemm.cuh (A_KMAJOR / B_KMAJOR select the transposed storage), computed
// by the WR x WC warps of a CTA (2 x 4 = 8 by default; a 4 x 4 grid runs 16).  The warps
// tile the output WR x WC; a warp tile of (M / WR) x (N / WC) is MT x NT tiles of 16 x 8, and
// the accumulator of tile (mt, nt) is the m16n8 fragment acc[mt][nt][r] at
//   row    = wr (M / WR) + 16 mt + g + 8 (r / 2)
//   column = wc (N / WC) + 8 nt + 2 tq + (r % 2)
// (warp = WC wr + wc, g = lane / 4, tq = lane % 4): a row lives in the 4 lanes of one g and
// the WC warps of one wr, a column in the 8 lanes of one tq and the WR warps of one wc.
// Every output element is owned by one thread and its sum runs in a fixed order, so results
// do not change from run to run.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gdn_tc.cuh"

namespace gdn {

template <int M, int N, int WR_ = 2, int WC_ = 4>
struct MmaMap {
    static constexpr int WR = WR_, WC = WC_;
    static constexpr int WTM = M / WR, WTN = N / WC;
    static constexpr int MT = WTM / 16, NT = WTN / 8;
    static_assert(MT * 16 * WR == M && NT * 8 * WC == N, "tile");
    __device__ static int wr(int tid) { return (tid >> 5) / WC; }
    __device__ static int wc(int tid) { return (tid >> 5) % WC; }
    __device__ static int row(int tid, int mt, int r) { return wr(tid) * WTM + 16 * mt + ((tid & 31) >> 2) + 8 * (r >> 1); }
    __device__ static int col(int tid, int nt, int r) { return wc(tid) * WTN + 8 * nt + 2 * (tid & 3) + (r & 1); }
};

template <int M, int N, int WR = 2, int WC = 4>
using MmaAcc = float[MmaMap<M, N, WR, WC>::MT][MmaMap<M, N, WR, WC>::NT][4];

template <int M, int N, int WR = 2, int WC = 4>
__device__ __forceinline__ void zero_mma(MmaAcc<M, N, WR, WC>& acc)
{
#pragma unroll
    for (int i = 0; i < MmaMap<M, N, WR, WC>::MT; ++i)
#pragma unroll
        for (int j = 0; j < MmaMap<M, N, WR, WC>::NT; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;
}

template <int M, int N, bool A_KMAJOR, bool B_KMAJOR, int WR = 2, int WC = 4>
__device__ __forceinline__ void block_mma(MmaAcc<M, N, WR, WC>& acc, const float* __restrict__ A, int lda,
                                          const float* __restrict__ B, int ldb, int K, int tid)
{
    using Map = MmaMap<M, N, WR, WC>;
    const int lane = tid & 31, g = lane >> 2, tq = lane & 3;
    const int m0 = Map::wr(tid) * Map::WTM + g, n0 = Map::wc(tid) * Map::WTN + g;
    auto a_at = [&](int m, int k) { return A_KMAJOR ? A[k * lda + m] : A[m * lda + k]; };
    auto b_at = [&](int k, int n) { return B_KMAJOR ? B[n * ldb + k] : B[k * ldb + n]; };
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t ah[Map::MT][4], al[Map::MT][4], bh[Map::NT][2], bl[Map::NT][2];
#pragma unroll
        for (int i = 0; i < Map::MT; ++i) {
            const int m = m0 + 16 * i;
            tc::split_tf32(a_at(m, k0 + tq), ah[i][0], al[i][0]);
            tc::split_tf32(a_at(m + 8, k0 + tq), ah[i][1], al[i][1]);
            tc::split_tf32(a_at(m, k0 + tq + 4), ah[i][2], al[i][2]);
            tc::split_tf32(a_at(m + 8, k0 + tq + 4), ah[i][3], al[i][3]);
        }
#pragma unroll
        for (int j = 0; j < Map::NT; ++j) {
            const int n = n0 + 8 * j;
            tc::split_tf32(b_at(k0 + tq, n), bh[j][0], bl[j][0]);
            tc::split_tf32(b_at(k0 + tq + 4, n), bh[j][1], bl[j][1]);
        }
        // pass-major: the MT x NT independent tiles lie between two passes on one accumulator
        // (each element still sums hi hi, then hi lo, then lo hi)
#pragma unroll
        for (int i = 0; i < Map::MT; ++i)
#pragma unroll
            for (int j = 0; j < Map::NT; ++j) tc::mma_warp_tf32(acc[i][j], ah[i], bh[j]);
#pragma unroll
        for (int i = 0; i < Map::MT; ++i)
#pragma unroll
            for (int j = 0; j < Map::NT; ++j) tc::mma_warp_tf32(acc[i][j], ah[i], bl[j]);
#pragma unroll
        for (int i = 0; i < Map::MT; ++i)
#pragma unroll
            for (int j = 0; j < Map::NT; ++j) tc::mma_warp_tf32(acc[i][j], al[i], bh[j]);
    }
}

}  // namespace gdn
