// gdn_chunk.cu -- the gated delta rule in chunked (WY) form, scalar gate, on the FP32
// pipe of sm_103a.
//
// The recurrence ("metal: GATED_DELTA_NET_BACK", PR #16, row form; meTile "Recurrent
// delta attention", matrix form) is exact when regrouped by chunks of BC tokens.  In M
// layout (M = S^T, rows j = value index, columns i = key index), for a chunk with
// entering state M_c, log-decay cumsum G_t (inclusive), gamma_t = exp(G_t),
// Dm[t][tau] = exp(G_t - G_tau) (tau <= t):
//   L  = strict_lower(Dm (.) K K^T),   Z = (I + diag(beta) L)^-1,   T = Z diag(beta)
//   X  = V - diag(gamma) K M_c^T,      Delta = T X          (row t = delta_t)
//   Y  = scale (diag(gamma) Q M_c^T + (lower(Q K^T) (.) Dm) Delta)
//   M_end = gamma_last M_c + Delta^T diag(r) K,   r_tau = Dm[last][tau]
// and the backward is the chain rule through these products (dM chain across chunks in
// reverse, every other gradient chunk-local).  Every product is a dense fp32 GEMM on
// the FP32 pipe (gdn_gemm.cuh); nothing is approximated.
//
// Chunks are aligned to the checkpoint segments: segment s = tokens [s C, s C + C) is
// split into ceil(C / BC) chunks, the last one of each segment ragged (zero-padded:
// g = 0, beta = 0, q = k = v = gy = 0 in the padding, which leaves every real output
// unchanged).  Kernels:
//   gdn_chunk_prep_kernel    per (chunk, value head): T, lower(QK^T) (.) Dm, gamma, r
//                            and (when asked) W = T diag(gamma) K, U = T V
//   gdn_chunk_state_kernel   rows [p R, p R + R) of one head: forward mode walks every
//                            chunk (y, checkpoints, state_T); recompute mode rebuilds the
//                            chunk-entry states inside each segment for the backward
//   gdn_chunk_dstate_kernel  rows [p R, p R + R): the dM chain in reverse; parks dM at
//                            every chunk end, dDelta and dX for the gradient kernel
//   gdn_chunk_grad_kernel    per (chunk, key head), looping over the value heads it
//                            serves in ascending order: dq, dk, dv, dg, dbeta
#include <cuda_runtime.h>

#include "gdn_gemm.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

constexpr int CT = 256;        // threads per CTA (all chunk kernels)
constexpr int LDB = BC + 4;    // leading dimension of BC-wide shared rows
// Rows of M per CTA in the state kernels: 24 at head size 128 (6 CTAs per head, the last
// one 8 rows short; 48 heads then fill two CTAs per SM on 144 SMs), else 32.
template <int D>
struct Rows {
    static constexpr int RR = (D == 128) ? 24 : 32;
    static constexpr int P = (D + RR - 1) / RR;
};
constexpr unsigned kFullMask = 0xffffffffu;

template <int D>
struct Ld {
    static constexpr int v = D + 4;  // leading dimension of D-wide shared rows
};

struct ChunkPos {
    int t0, nb, seg, loc;
};

__device__ __forceinline__ ChunkPos chunk_pos(const ChunkArgs& A, int c)
{
    ChunkPos p;
    p.seg = c / A.cps;
    p.loc = c - p.seg * A.cps;
    const int s0 = p.seg * A.C;
    const int s1 = min(A.T, s0 + A.C);
    p.t0 = s0 + p.loc * BC;
    p.nb = min(BC, s1 - p.t0);
    return p;
}

// BC rows of `width` floats from global (row stride `stride`) into shared memory with
// leading dimension ld; rows >= nb are zero.  The scale (if non-null) multiplies row t.
__device__ __forceinline__ void load_rows_pad(float* dst, int ld, const float* src,
                                              long long stride, int nb, int width, bool vec,
                                              int tid, const float* row_scale = nullptr)
{
    const int per = width >> 2;
    for (int idx = tid; idx < BC * per; idx += CT) {
        const int t = idx / per, i4 = idx - t * per;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nb) {
            const float* p = src + t * stride + 4 * i4;
            if (vec) {
                x = __ldg(reinterpret_cast<const float4*>(p));
            } else {
                x = make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
            }
            if (row_scale) {
                const float s = row_scale[t];
                x = make_float4(__fmul_rn(s, x.x), __fmul_rn(s, x.y), __fmul_rn(s, x.z),
                                __fmul_rn(s, x.w));
            }
        }
        *reinterpret_cast<float4*>(dst + t * ld + 4 * i4) = x;
    }
}

// Register prefetch of one chunk's raw rows of a strided input (q or k): BC x D floats,
// NF = D / 32 float4 per thread, zero beyond the chunk's real rows.
template <int D>
__device__ __forceinline__ void pf_rows(float4 (&r)[D / 32], const float* src, long long stride,
                                        int nb, bool vec, int tid)
{
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
        const int f = tid + CT * kk, t = f / (D / 4), i4 = f - t * (D / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nb) {
            const float* p = src + t * stride + 4 * i4;
            x = vec ? __ldg(reinterpret_cast<const float4*>(p))
                    : make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
        }
        r[kk] = x;
    }
}

template <int D>
__device__ __forceinline__ void put_rows(float* dst, int ld, const float4 (&r)[D / 32], int tid)
{
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
        const int f = tid + CT * kk, t = f / (D / 4), i4 = f - t * (D / 4);
        *reinterpret_cast<float4*>(dst + t * ld + 4 * i4) = r[kk];
    }
}

// A dense [rows][width] block of the workspace (row stride = width) into shared memory.
__device__ __forceinline__ void load_ws(float* dst, int ld, const float* src, int rows, int width,
                                        int tid)
{
    const int per = width >> 2;
    for (int idx = tid; idx < rows * per; idx += CT) {
        const int t = idx / per, i4 = idx - t * per;
        *reinterpret_cast<float4*>(dst + t * ld + 4 * i4) =
            __ldg(reinterpret_cast<const float4*>(src + (long long)t * width) + i4);
    }
}

// A rows x width block stored in the unit layout (float4 unit (c / 4) * rows + row holds
// row `row`, columns c .. c + 3) into shared memory, row-major with leading dimension ld.
__device__ __forceinline__ void load_units(float* dst, int ld, const float* src, int rows, int width,
                                           int tid)
{
    for (int idx = tid; idx < rows * (width >> 2); idx += CT) {
        const int r = idx % rows, c4 = idx / rows;
        *reinterpret_cast<float4*>(dst + r * ld + 4 * c4) = __ldg(reinterpret_cast<const float4*>(src) + idx);
    }
}

// ---------------------------------------------------------------------------------
// [Q; K] K^T for one chunk: 64 x 32 outputs over k < D, rows [Q; K] of QKs (row stride
// ld), B(k, n) = K[n][k].  Each operand is split x = hi + lo (hi: the 13 low mantissa bits
// cleared; lo = x - hi, exact) and the product accumulated as hi hi + hi lo + lo hi, which
// is fp32-accurate (the terms dropped are below 2^-20 of |a b|).  Warp w owns rows
// 16 (w / 2) .. + 16 and the two 8-column tiles 2 (w % 2), 2 (w % 2) + 1; c[nt] is the
// m16n8 accumulator fragment (rows g, g + 8; columns 2 tq, 2 tq + 1; g = lane / 4,
// tq = lane % 4).  Row-stride ld = 4 mod 32 keeps the fragment loads free of bank
// conflicts.
template <int D>
__device__ __forceinline__ void qk_products(float (&c)[2][4], const float* QKs, const float* Ks, int ld, int tid)
{
    const int warp = tid >> 5, g = (tid & 31) >> 2, tq = tid & 3;
    const float* a0 = QKs + (16 * (warp >> 1) + g) * ld + tq;
    const float* a1 = a0 + 8 * ld;
    const float* b0 = Ks + (8 * (2 * (warp & 1)) + g) * ld + tq;
    const float* b1 = b0 + 8 * ld;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[nt][i] = 0.f;
    auto split = [](float x, uint32_t& hi, uint32_t& lo) {
        hi = __float_as_uint(x) & 0xffffe000u;
        lo = __float_as_uint(__fsub_rn(x, __uint_as_float(hi)));
    };
#pragma unroll 4
    for (int k0 = 0; k0 < D; k0 += 8) {
        uint32_t ah[4], al[4], bh[2][2], bl[2][2];
        split(a0[k0], ah[0], al[0]);
        split(a1[k0], ah[1], al[1]);
        split(a0[k0 + 4], ah[2], al[2]);
        split(a1[k0 + 4], ah[3], al[3]);
        split(b0[k0], bh[0][0], bl[0][0]);
        split(b0[k0 + 4], bh[0][1], bl[0][1]);
        split(b1[k0], bh[1][0], bl[1][0]);
        split(b1[k0 + 4], bh[1][1], bl[1][1]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            tc::mma_warp_tf32(c[nt], ah, bh[nt]);
            tc::mma_warp_tf32(c[nt], ah, bl[nt]);
            tc::mma_warp_tf32(c[nt], al, bh[nt]);
        }
    }
}

// C (32 x 128) = A (32 x 32) B (32 x 128) on the tensor pipe, three-pass tf32 as in
// qk_products: A(m, k) = A[m * lda + k], or A[k * lda + m] when A_T; B(k, n) = B[k * ldb + n].
// Warp w owns rows 16 (w % 2) .. + 16 and columns 32 (w / 2) .. + 32 (four 8-column
// tiles); c[nt] is the m16n8 accumulator fragment of tile nt (rows g, g + 8; columns
// 2 tq, 2 tq + 1).  rows_cols() gives a thread's first row and column.
template <bool A_T>
__device__ __forceinline__ void mma_32x128x32(float (&c)[4][4], const float* A, int lda, const float* B, int ldb,
                                              int tid)
{
    const int warp = tid >> 5, g = (tid & 31) >> 2, tq = tid & 3;
    const int m0 = 16 * (warp & 1), n0 = 32 * (warp >> 1);
    auto split = [](float x, uint32_t& hi, uint32_t& lo) {
        hi = __float_as_uint(x) & 0xffffe000u;
        lo = __float_as_uint(__fsub_rn(x, __uint_as_float(hi)));
    };
    auto a_at = [&](int m, int k) { return A_T ? A[k * lda + m] : A[m * lda + k]; };
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[nt][i] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) {
        uint32_t ah[4], al[4];
        split(a_at(m0 + g, k0 + tq), ah[0], al[0]);
        split(a_at(m0 + g + 8, k0 + tq), ah[1], al[1]);
        split(a_at(m0 + g, k0 + tq + 4), ah[2], al[2]);
        split(a_at(m0 + g + 8, k0 + tq + 4), ah[3], al[3]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            uint32_t bh[2], bl[2];
            split(B[(k0 + tq) * ldb + n0 + 8 * nt + g], bh[0], bl[0]);
            split(B[(k0 + tq + 4) * ldb + n0 + 8 * nt + g], bh[1], bl[1]);
            tc::mma_warp_tf32(c[nt], ah, bh);
            tc::mma_warp_tf32(c[nt], ah, bl);
            tc::mma_warp_tf32(c[nt], al, bh);
        }
    }
}
__device__ __forceinline__ void mma_32x128_origin(int tid, int& m, int& n)
{
    m = 16 * ((tid >> 5) & 1) + ((tid & 31) >> 2);
    n = 32 * (tid >> 6) + 2 * (tid & 3);
}

// Z = (I + A)^-1 for a strictly lower 32 x 32 A, and T = Z diag(beta).  On entry Ts holds
// A (row stride LDB), Zs is zero and the CTA is synchronised; Pw is a 32 x LDB tile whose
// strict upper half (columns > rows) is zero: it serves as scratch and is zero again on
// return.  Blockwise: [[I + A11, 0], [A21, I + A22]]^-1 = [[Z11, 0], [-Z22 A21 Z11, Z22]],
// from four 8 x 8 diagonal blocks (forward substitution) up to 32 x 32.  Leaves Z in Zs and
// T in Ts; ends with a __syncthreads.
__device__ void unit_lower_inverse(float* Ts, float* Zs, float* Pw, const float* bs, int tid)
{
    if (tid < 32) {  // diagonal 8 x 8 blocks: lane = 8 block + column
        const int r0 = (tid >> 3) * 8, j = r0 + (tid & 7);
        float z[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int row = r0 + t;
            float acc = 0.f;
#pragma unroll
            for (int tau = 0; tau < t; ++tau)
                if (r0 + tau >= j) acc = __fmaf_rn(Ts[row * LDB + r0 + tau], z[tau], acc);
            z[t] = (row < j) ? 0.f : (row == j ? 1.f : -acc);
            Zs[row * LDB + j] = z[t];
        }
    }
    __syncthreads();
    // level 16: blocks (1,0) and (3,2) of 8 x 8: Z_ij = -Z_ii A_ij Z_jj
    if (tid < 128) {
        const int b = tid >> 6, e = tid & 63, rr = e >> 3, cc = e & 7;
        const int i0 = 8 + 16 * b, j0 = 16 * b;  // block rows i0.., cols j0..
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = __fmaf_rn(Ts[(i0 + rr) * LDB + j0 + k], Zs[(j0 + k) * LDB + j0 + cc], acc);
        Pw[(j0 + cc) * LDB + i0 + rr] = acc;  // stored transposed in Pw's upper half
    }
    __syncthreads();
    if (tid < 128) {
        const int b = tid >> 6, e = tid & 63, rr = e >> 3, cc = e & 7;
        const int i0 = 8 + 16 * b, j0 = 16 * b;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = __fmaf_rn(Zs[(i0 + rr) * LDB + i0 + k], Pw[(j0 + cc) * LDB + i0 + k], acc);
        Zs[(i0 + rr) * LDB + j0 + cc] = -acc;
    }
    __syncthreads();
    // level 32: Z21 (rows 16..31, cols 0..15) = -Z22 A21 Z11
    {
        const int rr = tid >> 4, cc = tid & 15;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc = __fmaf_rn(Ts[(16 + rr) * LDB + k], Zs[k * LDB + cc], acc);
        Pw[cc * LDB + 16 + rr] = acc;  // transposed, in Pw's upper half
    }
    __syncthreads();
    {
        const int rr = tid >> 4, cc = tid & 15;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc = __fmaf_rn(Zs[(16 + rr) * LDB + 16 + k], Pw[cc * LDB + 16 + k], acc);
        Zs[(16 + rr) * LDB + cc] = -acc;
    }
    __syncthreads();
    // restore Pw's strict upper half to zero
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        if (tau > t) Pw[t * LDB + tau] = 0.f;
    }
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Ts[t * LDB + tau] = __fmul_rn(Zs[t * LDB + tau], bs[tau]);
    }
    __syncthreads();
}

// Chunk-local quantities from Q, K (shared, [Q; K] stacked, zero-padded rows), g, beta.
// Out: G (inclusive cumsum), gam = exp(G), Dm (lower incl), KKm = K K^T (strict lower),
// QKm = Q K^T (lower incl), Zs = (I + diag(beta) (Dm (.) KK))^-1, Ts = Zs diag(beta).
// Ends with a __syncthreads.
template <int D>
__device__ void chunk_prep(const float* QKs, const float* gs, const float* bs, float* Gs,
                           float* gam, float* Dm, float* KKm, float* QKm, float* Zs, float* Ts,
                           int tid)
{
    constexpr int ld = Ld<D>::v;
    const float* Ks = QKs + BC * ld;
    if (tid < 32) {  // inclusive scan of g over the BC = 32 tokens
        float x = gs[tid];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(kFullMask, x, o);
            if (tid >= o) x = __fadd_rn(x, y);
        }
        Gs[tid] = x;
        gam[tid] = expf(x);
    }
    {  // [QK; KK] = [Q; K] K^T, 64 x 32 x D, on the tensor pipe (tf32x3, warp-level MMA)
        float c[2][4];
        qk_products<D>(c, QKs, Ks, ld, tid);
        const int warp = tid >> 5, g = (tid & 31) >> 2, tq = tid & 3;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int m = 16 * (warp >> 1) + g + 8 * half;
                    const int n = 8 * (2 * (warp & 1) + nt) + 2 * tq + e;
                    const float v = c[nt][2 * half + e];
                    if (m < BC)
                        QKm[m * LDB + n] = (n <= m) ? v : 0.f;
                    else
                        KKm[(m - BC) * LDB + n] = (n < m - BC) ? v : 0.f;
                }
    }
    __syncthreads();
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Dm[t * LDB + tau] = (tau <= t) ? expf(__fsub_rn(Gs[t], Gs[tau])) : 0.f;
    }
    __syncthreads();
    // Z = (I + A)^-1 with A = diag(beta) (Dm (.) KK) strictly lower; Ts holds A meanwhile
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Ts[t * LDB + tau] = (tau < t) ? __fmul_rn(bs[t], __fmul_rn(Dm[t * LDB + tau], KKm[t * LDB + tau]))
                                      : 0.f;
        Zs[t * LDB + tau] = 0.f;
    }
    __syncthreads();
    unit_lower_inverse(Ts, Zs, Dm, bs, tid);  // Dm's strict upper half is zero
}

// L2 prefetches of [p, p + nf) (whole 128-byte lines), spread over the CTA's threads.
__device__ __forceinline__ void prefetch_span(const float* p, long long nf, int tid)
{
    for (long long o = 32LL * tid; o < nf; o += 32LL * CT) tc::prefetch_l2(p + o);
}

__device__ __forceinline__ void load_gate_beta(const ChunkArgs& A, int n, int h, const ChunkPos& cp,
                                               float* gs, float* bs, int tid)
{
    if (tid < BC) {
        const long long tok = (long long)n * A.T + cp.t0 + tid;
        const bool real = tid < cp.nb;
        gs[tid] = real ? __ldg(A.g + tok * A.H_v + h) : 0.f;
        bs[tid] = real ? __ldg(A.beta + tok * A.H_v + h) : 0.f;
    }
}

// Tensor-core operands of one (chunk, head) for the state chain at head size 128, in the
// bf16 operand layouts of gdn_tc.cuh: W = T diag(gamma) K (32 x 128, row-group-major; the key
// head's Q beside it when `first`), B23 = [scale QD; (r K)^T] (160 x 32) as bf16 hi then lo,
// and U^T (rows j, 32 tokens) in fp32, U = T V.  Vs holds V on entry and stages U afterwards.
template <int D>
__device__ void prep_tc_operands(const ChunkArgs& A, long long ch, long long ck, bool first,
                                 const float* QKs, float* Vs, const float* TG, const float* Ts,
                                 const float* QKm, const float* Dm, int tid)
{
    constexpr int ld = Ld<D>::v;
    const float* Ks = QKs + BC * ld;
    float* w1 = A.ws + A.o_W1 + ch * kTcWElems;
    float* q1 = A.ws + A.o_Q1 + ck * kTcQElems;
    float* b23 = A.ws + A.o_B23 + ch * kTcB23Elems;
    float* u = A.ws + A.o_U + ch * (BC * D);
    static_assert(D == 128, "tensor-core operands are built at head size 128");
    int fm, fn;
    mma_32x128_origin(tid, fm, fn);
    float c[4][4];
    mma_32x128x32<false>(c, Ts, LDB, Vs, ld, tid);  // U = T V
    __syncthreads();
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
            *reinterpret_cast<float2*>(Vs + (fm + 8 * hf) * ld + fn + 8 * nt) = make_float2(c[nt][2 * hf], c[nt][2 * hf + 1]);
    mma_32x128x32<false>(c, TG, LDB, Ks, ld, tid);  // W = T diag(gamma) K
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // rows t of W, 2 consecutive k (the first even) per thread
            const int off = tc::kmaj16_rg(fm + 8 * hf, fn + 8 * nt, D);
            uint32_t hi, lo;
            tc::split_bf16x2(c[nt][2 * hf], c[nt][2 * hf + 1], hi, lo);
            reinterpret_cast<uint32_t*>(w1)[off] = hi;
            reinterpret_cast<uint32_t*>(w1 + kTcWElems / 2)[off] = lo;
        }
    if (first) {  // Q, 16-byte unit u = (row group * 16 + k-chunk) * 8 + row % 8
        for (int u = tid; u < BC * (D / 8); u += CT) {
            const int t = ((u >> 7) << 3) + (u & 7), kc = (u >> 3) & 15;
            const float4 a = *reinterpret_cast<const float4*>(QKs + t * ld + 8 * kc);
            const float4 b = *reinterpret_cast<const float4*>(QKs + t * ld + 8 * kc + 4);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            tc::put_bf16x8(q1, kTcQElems / 2, u, x);
        }
    }
    for (int idx = tid; idx < 160 * (BC / 8); idx += CT) {  // B23, 16-byte unit = kc * 160 + row
        const int r = idx % 160, kc = idx / 160;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int tau = 8 * kc + e;
            x[e] = (r < BC) ? __fmul_rn(A.scale, __fmul_rn(QKm[r * LDB + tau], Dm[r * LDB + tau]))
                            : __fmul_rn(Dm[(BC - 1) * LDB + tau], Ks[tau * ld + r - BC]);
        }
        tc::put_bf16x8(b23, kTcB23Elems / 2, idx, x);
    }
    __syncthreads();
    for (int idx = tid; idx < (BC / 4) * D; idx += CT) {  // U^T, unit = b * 128 + j
        const int j = idx % D, b = idx / D;
        *reinterpret_cast<float4*>(u + 4 * idx) =
            make_float4(Vs[(4 * b) * ld + j], Vs[(4 * b + 1) * ld + j], Vs[(4 * b + 2) * ld + j],
                        Vs[(4 * b + 3) * ld + j]);
    }
}

// Tensor-core operands of one (chunk, head) for the dM chain at head size 128: the value
// head's block at o_DS and, when `first`, the key head's block at o_DK (layouts in
// gdn_internal.h; tiles in the operand layout of gdn_tc.cuh).  Vs and Zs are free on entry
// and are used for dY and QD.
template <int D>
__device__ void prep_tc_dstate_operands(const ChunkArgs& A, int n, int h, const ChunkPos& cp,
                                        long long ch, long long ck, bool first, const float* QKs,
                                        float* Vs, float* Zs, const float* Ts, const float* QKm,
                                        const float* Dm, const float* gam, int tid)
{
    constexpr int ld = Ld<D>::v;
    const float* Ks = QKs + BC * ld;
    float* blk = A.ws + A.o_DS + ch * kTcDsElems;
    float* kblk = A.ws + A.o_DK + ck * kTcDkElems;
    {
        const long long tg = (long long)n * A.gys0 + (long long)cp.t0 * A.gys1 + (long long)h * A.gys2;
        float4 r[D / 32];
        pf_rows<D>(r, A.gy + tg, A.gys1, cp.nb, A.vec_gy, tid);
        put_rows<D>(Vs, ld, r, tid);
    }
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Zs[t * LDB + tau] = __fmul_rn(QKm[t * LDB + tau], Dm[t * LDB + tau]);
    }
    __syncthreads();
    {  // E^T = scale QD^T dY (rows t), stored as E (rows j), fp32
        static_assert(D == 128, "tensor-core operands are built at head size 128");
        float c[4][4];
        mma_32x128x32<true>(c, Zs, LDB, Vs, ld, tid);
        int fm, fn;
        mma_32x128_origin(tid, fm, fn);
        float* e = blk + kDsE;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int t = fm + 8 * hf, j = fn + 8 * nt + x;
                    e[4 * ((t >> 2) * D + j) + (t & 3)] = __fmul_rn(A.scale, c[nt][2 * hf + x]);
                }
    }
    // bf16 tiles, k-chunk-major: 16-byte unit kc * R + row holds 8 consecutive K elements
    for (int idx = tid; idx < (BC / 8) * D; idx += CT) {  // scale gamma dY^T, unit kc * 128 + j
        const int j = idx % D, kc = idx / D;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            x[e] = __fmul_rn(__fmul_rn(A.scale, gam[8 * kc + e]), Vs[(8 * kc + e) * ld + j]);
        tc::put_bf16x8(blk + kDsG, 128 * 32 / 2, idx, x);
    }
    if (first) {
        for (int idx = tid; idx < (D / 8) * BC; idx += CT) {  // K rows t, unit kc * 32 + t
            const int t = idx % BC, kc = idx / BC;
            const float4 a = *reinterpret_cast<const float4*>(Ks + t * ld + 8 * kc);
            const float4 b = *reinterpret_cast<const float4*>(Ks + t * ld + 8 * kc + 4);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            tc::put_bf16x8(kblk + kDkKb, 32 * 128 / 2, idx, x);
        }
        for (int idx = tid; idx < (2 * BC / 8) * D; idx += CT) {  // [Q^T | K^T] rows i, unit kc * 128 + i
            const int i = idx % D, kc = idx / D;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = QKs[(8 * kc + e) * ld + i];
            tc::put_bf16x8(kblk + kDkQKT, 128 * 64 / 2, idx, x);
        }
    }
    for (int idx = tid; idx < (BC / 8) * BC; idx += CT) {  // T^T rows t: T[t'][t], unit kc * 32 + t
        const int t = idx % BC, kc = idx / BC;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = Ts[(8 * kc + e) * LDB + t];
        tc::put_bf16x8(blk + kDsTT, 32 * 32 / 2, idx, x);
    }
    if (tid < BC) {
        blk[kDsR + tid] = Dm[(BC - 1) * LDB + tid];
        blk[kDsGam + tid] = gam[tid];
    }
}

// ---------------------------------------------------------------------------------
// Prep: one CTA per (chunk, value head, sequence).
template <int D>
__global__ void __launch_bounds__(CT) gdn_chunk_prep_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    // blockIdx.x = (chunk - c_lo) * H_v + slot, the r value heads of one key head in adjacent
    // slots: they run together and read the key head's q and k rows through L2
    const int slot = blockIdx.x % A.H_v, c = A.c_lo + blockIdx.x / A.H_v, n = blockIdx.y, tid = threadIdx.x;
    const int h = (slot % (A.H_v / A.H_k)) * A.H_k + slot / (A.H_v / A.H_k);
    const int hk = h % A.H_k;
    const ChunkPos cp = chunk_pos(A, c);
    const long long ch = ((long long)n * A.H_v + h) * A.n_chunks + c;

    extern __shared__ __align__(16) float sm[];
    float* QKs = sm;                  // [Q; K]  2BC x ld
    float* Vs = QKs + 2 * BC * ld;    // BC x ld
    float* Dm = Vs + BC * ld;         // BC x LDB each
    float* KKm = Dm + BC * LDB;
    float* QKm = KKm + BC * LDB;
    float* Zs = QKm + BC * LDB;
    float* Ts = Zs + BC * LDB;
    float* TG = Zs;                   // T diag(gamma), once Z has been written out
    float* vec = Ts + BC * LDB;       // gs, bs, Gs, gam
    float *gs = vec, *bs = vec + BC, *Gs = vec + 2 * BC, *gam = vec + 3 * BC;

    const long long tq = (long long)(n / A.rep) * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
    const long long tk = (long long)(n / A.rep) * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
    {  // every load in flight before the first store
        float4 rq[D / 32], rk[D / 32], rv[D / 32];
        pf_rows<D>(rq, A.q + tq, A.qs1, cp.nb, A.vec_q, tid);
        pf_rows<D>(rk, A.k + tk, A.ks1, cp.nb, A.vec_k, tid);
        if (A.want_wu) {
            const long long tv = (long long)n * A.vs0 + (long long)cp.t0 * A.vs1 + (long long)h * A.vs2;
            pf_rows<D>(rv, A.v + tv, A.vs1, cp.nb, A.vec_v, tid);
        }
        load_gate_beta(A, n, h, cp, gs, bs, tid);
        put_rows<D>(QKs, ld, rq, tid);
        put_rows<D>(QKs + BC * ld, ld, rk, tid);
        if (A.want_wu) put_rows<D>(Vs, ld, rv, tid);
    }
    __syncthreads();
    chunk_prep<D>(QKs, gs, bs, Gs, gam, Dm, KKm, QKm, Zs, Ts, tid);

    // T^T, QD = lower(QK^T) (.) Dm, QD^T (the FP32 chain kernels' operands), gamma, r
    const bool fp32_chains = !(D == 128 && A.want_tc);
    float* wsTT = A.ws + A.o_T + ch * (BC * BC);
    float* wsQ = A.ws + A.o_QKD + ch * (BC * BC);
    float* wsQT = A.ws + A.o_QDT + ch * (BC * BC);
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        if (fp32_chains) {
            const float qd = __fmul_rn(QKm[t * LDB + tau], Dm[t * LDB + tau]);
            wsTT[tau * BC + t] = Ts[t * LDB + tau];
            wsQ[idx] = qd;
            wsQT[tau * BC + t] = qd;
        }
    }
    if (tid < BC) {
        A.ws[A.o_gam + ch * BC + tid] = gam[tid];
        A.ws[A.o_r + ch * BC + tid] = Dm[(BC - 1) * LDB + tid];
    }
    if (A.want_factors) {  // the gradient kernel's chunk factors, row-major BC x BC
        float* fT = A.ws + A.o_Tr + ch * (BC * BC);
        float* fZ = A.ws + A.o_Z + ch * (BC * BC);
        float* fK = A.ws + A.o_KK + ch * (BC * BC);
        float* fQ = A.ws + A.o_QK + ch * (BC * BC);
        float* fD = A.ws + A.o_Dm + ch * (BC * BC);
        for (int idx = tid; idx < BC * BC; idx += CT) {
            const int t = idx / BC, tau = idx - t * BC;
            fT[idx] = Ts[t * LDB + tau];
            fZ[idx] = Zs[t * LDB + tau];
            fK[idx] = KKm[t * LDB + tau];
            fQ[idx] = QKm[t * LDB + tau];
            fD[idx] = Dm[t * LDB + tau];
        }
    }
    __syncthreads();  // Z is out: its tile now holds T diag(gamma)
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        TG[t * LDB + tau] = __fmul_rn(Ts[t * LDB + tau], gam[tau]);
    }
    if constexpr (D == 128) {
        if (A.want_tc) {
            const long long ck = ((long long)n * A.H_k + hk) * A.n_chunks + c;
            const bool first = h < A.H_k;  // the key head's first value head writes its operands
            // the backward rebuilds only the states entering a segment's later chunks, so the
            // last chunk of a segment needs no state-chain operands there
            const bool seg_last = cp.t0 + BC >= min(A.T, cp.seg * A.C + A.C);
            if (A.want_wu && !(A.want_factors && seg_last)) {
                __syncthreads();
                prep_tc_operands<D>(A, ch, ck, first, QKs, Vs, TG, Ts, QKm, Dm, tid);
            }
            if (A.want_factors) {
                __syncthreads();
                prep_tc_dstate_operands<D>(A, n, h, cp, ch, ck, first, QKs, Vs, Zs, Ts, QKm, Dm, gam, tid);
            }
            return;
        }
    }
    if (!A.want_wu) return;
    __syncthreads();
    // W = T diag(gamma) K  (BC x D, row-major),  U^T = (T V)^T  (D x BC)
    constexpr int TM = D / 32;
    using Map = GemmMap<BC, D, TM, 4, false>;
    float acc[TM][4];
    zero_acc(acc);
    block_gemm<BC, D, TM, 4, false, false>(acc, TG, LDB, QKs + BC * ld, ld, BC, tid);
    float* wsW = A.ws + A.o_W + ch * (BC * D);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) wsW[Map::row(tid, i) * D + Map::col(tid, j)] = acc[i][j];
    zero_acc(acc);
    block_gemm<BC, D, TM, 4, false, false>(acc, Ts, LDB, Vs, ld, BC, tid);
    float* wsU = A.ws + A.o_U + ch * (BC * D);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) wsU[Map::col(tid, j) * BC + Map::row(tid, i)] = acc[i][j];
}

}  // namespace gdn

#include "gdn_kda_prep.cuh"

namespace gdn {

// ---------------------------------------------------------------------------------
// State chain, rows [p RR, p RR + RR) of M for one head.
//   forward  (grid: p, head, sequence): every chunk in order; writes the checkpoints at
//            segment starts, y, and state_T.
//   recompute(grid: p, segment, sequence * H_v + head): from ckpt[s] through the
//            segment's chunks but its last, parking each chunk-entry state.
// Per chunk (Delta^T and Y^T are kept transposed, rows j):
//   [W M^T; Q M^T]^T  ->  Delta^T = U^T - (W M^T)^T,   Y^T = gamma (.) (Q M^T)^T
//   Y^T += (QD Delta)^T,  y = scale Y
//   M   <- gamma_last M + (r (.) Delta)^T K
// The next chunk's operands are loaded into registers while the current one computes.
template <int D, bool FWD>
__global__ void __launch_bounds__(CT) gdn_chunk_state_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    constexpr int NF = D / 32;
    constexpr int RR = Rows<D>::RR;
    constexpr int TM1 = RR / 8;          // RR x (BC or 2BC) tiles: 8 x 32 threads
    constexpr int TM3 = RR * D / 1024;   // RR x D tile, float4 columns
    const int tid = threadIdx.x, p = blockIdx.x;
    int n, h, c_begin, c_end;
    if (FWD) {
        h = blockIdx.y;
        n = blockIdx.z;
        c_begin = 0;
        c_end = A.n_chunks;
    } else {
        const int hd = blockIdx.z;
        n = hd / A.H_v;
        h = hd - n * A.H_v;
        const int s = blockIdx.y;
        c_begin = s * A.cps;
        const int seg_len = min(A.T, s * A.C + A.C) - s * A.C;
        c_end = c_begin + (seg_len + BC - 1) / BC - 1;  // chunks whose end state is needed
        if (c_end <= c_begin) return;
    }
    const int hk = h % A.H_k;
    const long long head = (long long)n * A.H_v + h;
    const int row0 = p * RR;
    const int nr = min(RR, D - row0);  // real rows of this CTA
    extern __shared__ __align__(16) float sm[];
    float* Ms = sm;                   // RR x ld
    float* WQs = Ms + RR * ld;        // [W; Q]  2BC x ld
    float* Ks = WQs + 2 * BC * ld;    // BC x ld
    float* UT = Ks + BC * ld;         // RR x LDB each:
    float* QD = UT + RR * LDB;
    float* DT = QD + BC * LDB;
    float* DrT = DT + RR * LDB;
    float* YT = DrT + RR * LDB;
    float* vec = YT + RR * LDB;
    float *gam = vec, *rr = vec + BC;

    float4 pw[NF], pq[NF], pk[NF], pu, pqd, pgr;
    auto issue = [&](int c) {
        const ChunkPos cp = chunk_pos(A, c);
        const long long ch = head * A.n_chunks + c;
        const float* w = A.ws + A.o_W + ch * (BC * D);
#pragma unroll
        for (int kk = 0; kk < NF; ++kk) pw[kk] = __ldg(reinterpret_cast<const float4*>(w) + tid + CT * kk);
        const long long tk = (long long)(n / A.rep) * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
        pf_rows<D>(pk, A.k + tk, A.ks1, cp.nb, A.vec_k, tid);
        if (FWD) {
            const long long tq = (long long)(n / A.rep) * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
            pf_rows<D>(pq, A.q + tq, A.qs1, cp.nb, A.vec_q, tid);
            pqd = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_QKD + ch * (BC * BC)) + tid);
        }
        pu = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid < nr * (BC / 4))
            pu = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_U + ch * (BC * D) + row0 * BC) + tid);
        if (tid < 8)
            pgr = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_gam + ch * BC) + tid);
        else if (tid < 16)
            pgr = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_r + ch * BC) + tid - 8);
    };
    auto commit = [&]() {
        put_rows<D>(WQs, ld, pw, tid);
        put_rows<D>(Ks, ld, pk, tid);
        if (FWD) {
            put_rows<D>(WQs + BC * ld, ld, pq, tid);
            *reinterpret_cast<float4*>(QD + (tid >> 3) * LDB + 4 * (tid & 7)) = pqd;
        }
        if (tid < RR * (BC / 4)) *reinterpret_cast<float4*>(UT + (tid >> 3) * LDB + 4 * (tid & 7)) = pu;
        if (tid < 8)
            reinterpret_cast<float4*>(gam)[tid] = pgr;
        else if (tid < 16)
            reinterpret_cast<float4*>(rr)[tid - 8] = pgr;
    };
    auto copy_state = [&](float* dst) {  // Ms -> global rows [row0, row0 + nr)
        for (int idx = tid; idx < nr * (D / 4); idx += CT) {
            const int j = idx / (D / 4), i4 = idx - j * (D / 4);
            reinterpret_cast<float4*>(dst + (long long)j * D)[i4] =
                *reinterpret_cast<const float4*>(Ms + j * ld + 4 * i4);
        }
    };

    {  // entry state
        const float* src = FWD ? A.state0 + (head * D + row0) * D
                               : A.ckpt + ((head * A.n_ck + blockIdx.y) * D + row0) * D;
        for (int idx = tid; idx < RR * (D / 4); idx += CT) {
            const int j = idx / (D / 4), i4 = idx - j * (D / 4);
            *reinterpret_cast<float4*>(Ms + j * ld + 4 * i4) =
                j < nr ? __ldg(reinterpret_cast<const float4*>(src + (long long)j * D) + i4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    issue(c_begin);
    int y_t0 = 0, y_nb = 0;  // the chunk whose Y^T is staged in YT
    auto write_y = [&]() {
        for (int idx = tid; idx < y_nb * nr; idx += CT) {
            const int t = idx / nr, j = idx - t * nr;
            A.y[(((long long)n * A.T + y_t0 + t) * A.H_v + h) * D + row0 + j] = YT[j * LDB + t];
        }
    };
    for (int c = c_begin; c < c_end; ++c) {
        const ChunkPos cp = chunk_pos(A, c);
        __syncthreads();
        if (FWD && y_nb > 0) write_y();
        if (!FWD && c > c_begin) copy_state(A.ws + A.o_Mc + (head * A.n_chunks + c) * (long long)(D * D) + (long long)row0 * D);
        commit();
        if (c + 1 < c_end) issue(c + 1);
        if (FWD && cp.loc == 0) copy_state(A.ckpt_out + ((head * A.n_ck + cp.seg) * D + row0) * D);
        __syncthreads();
        {  // [W M^T; Q M^T]^T  (RR x 2BC, or RR x BC)
            constexpr int NN = FWD ? 2 * BC : BC;
            constexpr int TN = NN / 32;
            using Map = GemmMap<RR, NN, TM1, TN, true>;
            float acc[TM1][TN];
            zero_acc(acc);
            block_gemm<RR, NN, TM1, TN, false, true>(acc, Ms, ld, WQs, ld, D, tid);
#pragma unroll
            for (int i = 0; i < TM1; ++i) {
                const int j = Map::row(tid, i);
#pragma unroll
                for (int jj = 0; jj < TN; ++jj) {
                    const int t = Map::col(tid, jj);
                    if (t < BC) {
                        const float d = __fsub_rn(UT[j * LDB + t], acc[i][jj]);
                        DT[j * LDB + t] = d;
                        DrT[j * LDB + t] = __fmul_rn(rr[t], d);
                    } else {
                        YT[j * LDB + t - BC] = __fmul_rn(gam[t - BC], acc[i][jj]);
                    }
                }
            }
        }
        __syncthreads();
        if (FWD) {  // Y^T += (QD Delta)^T,  then scale
            using Map = GemmMap<RR, BC, TM1, 1, true>;
            float acc[TM1][1];
            zero_acc(acc);
            block_gemm<RR, BC, TM1, 1, false, true>(acc, DT, LDB, QD, LDB, BC, tid);
#pragma unroll
            for (int i = 0; i < TM1; ++i)
#pragma unroll
                for (int jj = 0; jj < 1; ++jj) {
                    const int j = Map::row(tid, i), t = Map::col(tid, jj);
                    YT[j * LDB + t] = __fmul_rn(A.scale, __fadd_rn(YT[j * LDB + t], acc[i][jj]));
                }
            y_t0 = cp.t0;
            y_nb = cp.nb;
        }
        {  // M <- gamma_last M + (r (.) Delta)^T K
            const float gl = gam[BC - 1];
            using Map = GemmMap<RR, D, TM3, 4, false>;
            float acc[TM3][4];
            zero_acc(acc);
            block_gemm<RR, D, TM3, 4, false, false>(acc, DrT, LDB, Ks, ld, BC, tid);
#pragma unroll
            for (int i = 0; i < TM3; ++i) {
                float4* mp = reinterpret_cast<float4*>(Ms + Map::row(tid, i) * ld + Map::col(tid, 0));
                float4 m = *mp;
                m.x = __fmaf_rn(gl, m.x, acc[i][0]);
                m.y = __fmaf_rn(gl, m.y, acc[i][1]);
                m.z = __fmaf_rn(gl, m.z, acc[i][2]);
                m.w = __fmaf_rn(gl, m.w, acc[i][3]);
                *mp = m;
            }
        }
    }
    __syncthreads();
    if (FWD) {
        write_y();
        copy_state(A.state_T + (head * D + row0) * D);
    } else {
        copy_state(A.ws + A.o_Mc + (head * A.n_chunks + c_end) * (long long)(D * D) + (long long)row0 * D);
    }
}

// ---------------------------------------------------------------------------------
// The dM chain in reverse, rows [p RR, p RR + RR) of one head.  Per chunk (dDelta^T and
// dX^T kept transposed, rows j):
//   dDelta^T = (r (.) (K dM^T))^T + scale (QD^T dY)^T
//   dX^T     = (T^T dDelta)^T
//   dM      <- gamma_last dM + [scale gamma (.) dY ; -gamma (.) dX]^T [Q; K]
// Parks dM (as it enters the chunk from the right), dDelta^T and dX^T for the gradient
// kernel.  The next chunk's operands are loaded into registers while the current one
// computes.
template <int D>
__global__ void __launch_bounds__(CT) gdn_chunk_dstate_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    constexpr int NF = D / 32;
    constexpr int RR = Rows<D>::RR;
    constexpr int TM1 = RR / 8;
    constexpr int TM4 = RR * D / 1024;
    constexpr int LDA = 2 * BC + 4;
    const int tid = threadIdx.x, p = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h % A.H_k;
    const long long head = (long long)n * A.H_v + h;
    const int row0 = p * RR;
    const int nr = min(RR, D - row0);  // real rows of this CTA
    extern __shared__ __align__(16) float sm[];
    float* dMs = sm;                   // RR x ld
    float* QKs = dMs + RR * ld;        // [Q; K]  2BC x ld
    float* dYT = QKs + 2 * BC * ld;    // RR x LDB each:
    float* QDT = dYT + RR * LDB;
    float* TT = QDT + BC * LDB;
    float* dDT = TT + BC * LDB;
    float* Ap = dDT + RR * LDB;        // RR x LDA
    float* vec = Ap + RR * LDA;
    float *gam = vec, *rr = vec + BC;

    float4 pq[NF], pk[NF], pdy, pqt, ptt, pgr;
    auto issue = [&](int c) {
        const ChunkPos cp = chunk_pos(A, c);
        const long long ch = head * A.n_chunks + c;
        const long long tk = (long long)(n / A.rep) * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
        const long long tq = (long long)(n / A.rep) * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
        pf_rows<D>(pk, A.k + tk, A.ks1, cp.nb, A.vec_k, tid);
        pf_rows<D>(pq, A.q + tq, A.qs1, cp.nb, A.vec_q, tid);
        {  // dY rows t, own columns: float4 index tid -> (t, j4), RR/4 float4 per row
            const int t = tid / (RR / 4), j4 = tid - t * (RR / 4);
            pdy = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tid < BC * (RR / 4) && t < cp.nb && 4 * j4 < nr) {
                const float* g = A.gy + (long long)n * A.gys0 + (long long)(cp.t0 + t) * A.gys1 +
                                 (long long)h * A.gys2 + row0 + 4 * j4;
                pdy = A.vec_gy ? __ldg(reinterpret_cast<const float4*>(g))
                               : make_float4(__ldg(g), __ldg(g + 1), __ldg(g + 2), __ldg(g + 3));
            }
        }
        pqt = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_QDT + ch * (BC * BC)) + tid);
        ptt = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_T + ch * (BC * BC)) + tid);
        if (tid < 8)
            pgr = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_gam + ch * BC) + tid);
        else if (tid < 16)
            pgr = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_r + ch * BC) + tid - 8);
    };
    auto commit = [&]() {
        put_rows<D>(QKs, ld, pq, tid);
        put_rows<D>(QKs + BC * ld, ld, pk, tid);
        if (tid < BC * (RR / 4)) {
            const int t = tid / (RR / 4), j = 4 * (tid - t * (RR / 4));
            dYT[(j + 0) * LDB + t] = pdy.x;
            dYT[(j + 1) * LDB + t] = pdy.y;
            dYT[(j + 2) * LDB + t] = pdy.z;
            dYT[(j + 3) * LDB + t] = pdy.w;
        }
        *reinterpret_cast<float4*>(QDT + (tid >> 3) * LDB + 4 * (tid & 7)) = pqt;
        *reinterpret_cast<float4*>(TT + (tid >> 3) * LDB + 4 * (tid & 7)) = ptt;
        if (tid < 8)
            reinterpret_cast<float4*>(gam)[tid] = pgr;
        else if (tid < 16)
            reinterpret_cast<float4*>(rr)[tid - 8] = pgr;
    };

    for (int idx = tid; idx < RR * (D / 4); idx += CT) {
        const int j = idx / (D / 4), i4 = idx - j * (D / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (A.dstate_T && j < nr)
            x = __ldg(reinterpret_cast<const float4*>(A.dstate_T + (head * D + row0 + j) * D) + i4);
        *reinterpret_cast<float4*>(dMs + j * ld + 4 * i4) = x;
    }
    issue(A.n_chunks - 1);
    using MapS = GemmMap<RR, BC, TM1, 1, true>;
    for (int c = A.n_chunks - 1; c >= 0; --c) {
        const long long ch = head * A.n_chunks + c;
        __syncthreads();
        commit();
        if (c > 0) issue(c - 1);
        {  // park dM (the gradient of this chunk's end state)
            float* dst = A.ws + A.o_dM + ch * (long long)(D * D) + (long long)row0 * D;
            for (int idx = tid; idx < nr * (D / 4); idx += CT) {
                const int j = idx / (D / 4), i4 = idx - j * (D / 4);
                reinterpret_cast<float4*>(dst + (long long)j * D)[i4] =
                    *reinterpret_cast<const float4*>(dMs + j * ld + 4 * i4);
            }
        }
        __syncthreads();
        {  // dDelta^T = r (.) (dM K^T) + scale dY^T QD
            float acc[TM1][1], acc2[TM1][1];
            zero_acc(acc);
            zero_acc(acc2);
            block_gemm<RR, BC, TM1, 1, false, true>(acc, dMs, ld, QKs + BC * ld, ld, D, tid);
            block_gemm<RR, BC, TM1, 1, false, true>(acc2, dYT, LDB, QDT, LDB, BC, tid);
            float* dst = A.ws + A.o_dDel + ch * (BC * D) + (long long)row0 * BC;
#pragma unroll
            for (int i = 0; i < TM1; ++i) {
                const int j = MapS::row(tid, i), t = MapS::col(tid, 0);
                const float val = __fmaf_rn(A.scale, acc2[i][0], __fmul_rn(rr[t], acc[i][0]));
                dDT[j * LDB + t] = val;
                if (j < nr) dst[j * BC + t] = val;
            }
        }
        __syncthreads();
        {  // dX^T = dDelta^T T;  Ap = [scale gamma (.) dY^T | -gamma (.) dX^T]
            float acc[TM1][1];
            zero_acc(acc);
            block_gemm<RR, BC, TM1, 1, false, true>(acc, dDT, LDB, TT, LDB, BC, tid);
            float* dst = A.ws + A.o_dX + ch * (BC * D) + (long long)row0 * BC;
#pragma unroll
            for (int i = 0; i < TM1; ++i) {
                const int j = MapS::row(tid, i), t = MapS::col(tid, 0);
                if (j < nr) dst[j * BC + t] = acc[i][0];
                Ap[j * LDA + BC + t] = -__fmul_rn(gam[t], acc[i][0]);
                Ap[j * LDA + t] = __fmul_rn(__fmul_rn(A.scale, gam[t]), dYT[j * LDB + t]);
            }
        }
        __syncthreads();
        {  // dM <- gamma_last dM + Ap [Q; K]
            const float gl = gam[BC - 1];
            using Map = GemmMap<RR, D, TM4, 4, false>;
            float acc[TM4][4];
            zero_acc(acc);
            block_gemm<RR, D, TM4, 4, false, false>(acc, Ap, LDA, QKs, ld, 2 * BC, tid);
#pragma unroll
            for (int i = 0; i < TM4; ++i) {
                float4* mp = reinterpret_cast<float4*>(dMs + Map::row(tid, i) * ld + Map::col(tid, 0));
                float4 m = *mp;
                m.x = __fmaf_rn(gl, m.x, acc[i][0]);
                m.y = __fmaf_rn(gl, m.y, acc[i][1]);
                m.z = __fmaf_rn(gl, m.z, acc[i][2]);
                m.w = __fmaf_rn(gl, m.w, acc[i][3]);
                *mp = m;
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < nr * D; idx += CT) {
        const int j = idx / D, i = idx - j * D;
        A.dstate0[(head * D + row0 + j) * D + i] = dMs[j * ld + i];
    }
}

// ---------------------------------------------------------------------------------
// Gradients of one chunk for one key head and the value heads it serves.
template <int D>
__global__ void __launch_bounds__(CT, 1) gdn_chunk_grad_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    constexpr int TM = D / 32;  // (BC x D) tiles
    using MapQ = GemmMap<BC, D, TM, 4, false>;
    const int c = blockIdx.x, hk = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
    const int lane = tid & 31;
    const ChunkPos cp = chunk_pos(A, c);
    const int r = A.H_v / A.H_k;

    extern __shared__ __align__(16) float sm[];
    float* QKs = sm;                  // [Q; K]  2BC x ld
    float* Ks = QKs + BC * ld;
    float* MB = QKs + 2 * BC * ld;    // D x ld: M_c, then dM_end
    float* Xs = MB + D * ld;          // V, then X
    float* Dls = Xs + BC * ld;        // Delta
    float* dYs = Dls + BC * ld;       // dY
    float* dXT = dYs + BC * ld;       // dX^T   D x LDB
    float* dDT = dXT + D * LDB;       // dDelta^T  D x LDB
    float* Dm = dDT + D * LDB;        // BC x LDB each:
    float* KKm = Dm + BC * LDB;
    float* QKm = KKm + BC * LDB;
    float* Zs = QKm + BC * LDB;
    float* Ts = Zs + BC * LDB;
    float* Ps = Ts + BC * LDB;        // dQKD (lower incl), then its Dm-weighted form
    float* Ss = Ps + BC * LDB;        // stacked under Ps: symmetric dKK
    float* dTs = Ss + BC * LDB;       // dT, then P1, then dD (.) Dm
    float* W1 = dTs + BC * LDB;       // dZ, then dA
    float* W2 = dTs;                  // P1 = dZ Z^T (dT is dead by then)
    float* vec = W1 + BC * LDB;
    float *gs = vec, *bs = vec + BC, *gam = vec + 3 * BC;
    float *dgam = vec + 4 * BC, *dr = vec + 5 * BC, *dG = vec + 6 * BC, *dbs = vec + 7 * BC;
    float* red = vec + 8 * BC;        // CT/32 partials

    {
        const long long tq = (long long)(n / A.rep) * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
        const long long tk = (long long)(n / A.rep) * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
        load_rows_pad(QKs, ld, A.q + tq, A.qs1, cp.nb, D, A.vec_q, tid);
        load_rows_pad(Ks, ld, A.k + tk, A.ks1, cp.nb, D, A.vec_k, tid);
    }
    float aq[TM][4], ak[TM][4];
    zero_acc(aq);
    zero_acc(ak);

    for (int rho = 0; rho < r; ++rho) {
        const int h = hk + rho * A.H_k;
        const long long head = (long long)n * A.H_v + h;
        const long long ch = head * A.n_chunks + c;
        __syncthreads();
        if (rho + 1 < r) {  // the next value head's rows and tiles into L2 while this one computes
            const int h1 = h + A.H_k;
            const long long head1 = (long long)n * A.H_v + h1, ch1 = head1 * A.n_chunks + c;
            if (tid < cp.nb * (D / 32)) {
                const int t = tid / (D / 32), q = tid - t * (D / 32);
                tc::prefetch_l2(A.v + (long long)n * A.vs0 + (long long)(cp.t0 + t) * A.vs1 + (long long)h1 * A.vs2 + 32 * q);
                tc::prefetch_l2(A.gy + (long long)n * A.gys0 + (long long)(cp.t0 + t) * A.gys1 + (long long)h1 * A.gys2 + 32 * q);
            }
            prefetch_span(A.ws + A.o_dX + ch1 * (BC * D), BC * D, tid);
            prefetch_span(A.ws + A.o_dDel + ch1 * (BC * D), BC * D, tid);
            prefetch_span(cp.loc == 0 ? A.ckpt + (head1 * A.n_ck + cp.seg) * (long long)(D * D)
                                      : A.ws + A.o_Mc + ch1 * (long long)(D * D),
                          D * D, tid);
            prefetch_span(A.ws + A.o_Tr + ch1 * (BC * BC), BC * BC, tid);
            prefetch_span(A.ws + A.o_Z + ch1 * (BC * BC), BC * BC, tid);
            prefetch_span(A.ws + A.o_KK + ch1 * (BC * BC), BC * BC, tid);
            prefetch_span(A.ws + A.o_QK + ch1 * (BC * BC), BC * BC, tid);
            prefetch_span(A.ws + A.o_Dm + ch1 * (BC * BC), BC * BC, tid);
        }
        load_gate_beta(A, n, h, cp, gs, bs, tid);
        {
            const long long tv = (long long)n * A.vs0 + (long long)cp.t0 * A.vs1 + (long long)h * A.vs2;
            load_rows_pad(Xs, ld, A.v + tv, A.vs1, cp.nb, D, A.vec_v, tid);
            const long long tg = (long long)n * A.gys0 + (long long)cp.t0 * A.gys1 + (long long)h * A.gys2;
            load_rows_pad(dYs, ld, A.gy + tg, A.gys1, cp.nb, D, A.vec_gy, tid);
            const float* msrc = (cp.loc == 0)
                                    ? A.ckpt + (head * A.n_ck + cp.seg) * (long long)(D * D)
                                    : A.ws + A.o_Mc + ch * (long long)(D * D);
            if (A.want_tc) {  // the tensor-core chains park in the unit layout
                load_units(dXT, LDB, A.ws + A.o_dX + ch * (BC * D), D, BC, tid);
                load_units(dDT, LDB, A.ws + A.o_dDel + ch * (BC * D), D, BC, tid);
                if (cp.loc == 0)
                    load_ws(MB, ld, msrc, D, D, tid);
                else
                    load_units(MB, ld, msrc, D, D, tid);
            } else {
                load_ws(dXT, LDB, A.ws + A.o_dX + ch * (BC * D), D, BC, tid);
                load_ws(dDT, LDB, A.ws + A.o_dDel + ch * (BC * D), D, BC, tid);
                load_ws(MB, ld, msrc, D, D, tid);
            }
        }
        load_ws(Ts, LDB, A.ws + A.o_Tr + ch * (BC * BC), BC, BC, tid);
        load_ws(Zs, LDB, A.ws + A.o_Z + ch * (BC * BC), BC, BC, tid);
        load_ws(KKm, LDB, A.ws + A.o_KK + ch * (BC * BC), BC, BC, tid);
        load_ws(QKm, LDB, A.ws + A.o_QK + ch * (BC * BC), BC, BC, tid);
        load_ws(Dm, LDB, A.ws + A.o_Dm + ch * (BC * BC), BC, BC, tid);
        if (tid < BC) gam[tid] = __ldg(A.ws + A.o_gam + ch * BC + tid);
        __syncthreads();

        float hq[TM][4], hkk[TM][4];
        {  // X = V - gamma (.) K M^T
            using Map = GemmMap<BC, D, TM, 4, true>;
            float acc[TM][4];
            zero_acc(acc);
            block_gemm<BC, D, TM, 4, false, true>(acc, Ks, ld, MB, ld, D, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int t = Map::row(tid, i);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int jj = Map::col(tid, j);
                    Xs[t * ld + jj] = __fsub_rn(Xs[t * ld + jj], __fmul_rn(gam[t], acc[i][j]));
                }
            }
        }
        {  // dY M and dX M: dq = scale gamma (dY M), dk = -gamma (dX M); dgam partials
            float acc[TM][4], acc2[TM][4];
            zero_acc(acc);
            zero_acc(acc2);
            block_gemm_dual<BC, D, TM, 4, false, true, false>(acc, dYs, ld, acc2, dXT, LDB, MB, ld,
                                                              D, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int t = MapQ::row(tid, i);
                const int c0 = MapQ::col(tid, 0);
                const float4 qv = *reinterpret_cast<const float4*>(QKs + t * ld + c0);
                const float4 kv = *reinterpret_cast<const float4*>(Ks + t * ld + c0);
                const float sg = __fmul_rn(A.scale, gam[t]);
                hq[i][0] = __fmul_rn(sg, acc[i][0]);
                hq[i][1] = __fmul_rn(sg, acc[i][1]);
                hq[i][2] = __fmul_rn(sg, acc[i][2]);
                hq[i][3] = __fmul_rn(sg, acc[i][3]);
                hkk[i][0] = -__fmul_rn(gam[t], acc2[i][0]);
                hkk[i][1] = -__fmul_rn(gam[t], acc2[i][1]);
                hkk[i][2] = -__fmul_rn(gam[t], acc2[i][2]);
                hkk[i][3] = -__fmul_rn(gam[t], acc2[i][3]);
                float part = 0.f;
                part = __fmaf_rn(__fmul_rn(A.scale, qv.x), acc[i][0], part);
                part = __fmaf_rn(-kv.x, acc2[i][0], part);
                part = __fmaf_rn(__fmul_rn(A.scale, qv.y), acc[i][1], part);
                part = __fmaf_rn(-kv.y, acc2[i][1], part);
                part = __fmaf_rn(__fmul_rn(A.scale, qv.z), acc[i][2], part);
                part = __fmaf_rn(-kv.z, acc2[i][2], part);
                part = __fmaf_rn(__fmul_rn(A.scale, qv.w), acc[i][3], part);
                part = __fmaf_rn(-kv.w, acc2[i][3], part);
                // row t: 4 lanes of the warp (lane bits 0-1), then the warp columns
                part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, 1));
                part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, 2));
                if ((tid & 3) == 0) Ss[MapQ::wc(tid) * LDB + t] = part;
            }
        }
        __syncthreads();
        {  // Delta = T X
            using Map = GemmMap<BC, D, TM, 4, false>;
            float acc[TM][4];
            zero_acc(acc);
            block_gemm<BC, D, TM, 4, false, false>(acc, Ts, LDB, Xs, ld, BC, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i)
                *reinterpret_cast<float4*>(Dls + Map::row(tid, i) * ld + Map::col(tid, 0)) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        {  // MB <- dM_end, with <dM_end, M_c> on the way
            float part = 0.f;
            const float* src = A.ws + A.o_dM + ch * (long long)(D * D);
            for (int idx = tid; idx < D * (D / 4); idx += CT) {
                int j, i4;
                if (A.want_tc) {  // unit layout
                    j = idx % D;
                    i4 = idx / D;
                } else {
                    j = idx / (D / 4);
                    i4 = idx - j * (D / 4);
                }
                const float4 dm = __ldg(reinterpret_cast<const float4*>(src) + (A.want_tc ? idx : j * (D / 4) + i4));
                float4* mp = reinterpret_cast<float4*>(MB + j * ld + 4 * i4);
                const float4 m = *mp;
                part = __fmaf_rn(dm.x, m.x, part);
                part = __fmaf_rn(dm.y, m.y, part);
                part = __fmaf_rn(dm.z, m.z, part);
                part = __fmaf_rn(dm.w, m.w, part);
                *mp = dm;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, o));
            if (lane == 0) red[tid >> 5] = part;
        }
        __syncthreads();
        {  // Delta dM_end: dk += r (.) (Delta dM); dr = rowsum(K (.) Delta dM)
            float acc[TM][4];
            zero_acc(acc);
            block_gemm<BC, D, TM, 4, false, false>(acc, Dls, ld, MB, ld, D, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int t = MapQ::row(tid, i);
                const float rt = Dm[(BC - 1) * LDB + t];
                const float4 kv = *reinterpret_cast<const float4*>(Ks + t * ld + MapQ::col(tid, 0));
                float part = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) hkk[i][j] = __fmaf_rn(rt, acc[i][j], hkk[i][j]);
                part = __fmaf_rn(kv.x, acc[i][0], part);
                part = __fmaf_rn(kv.y, acc[i][1], part);
                part = __fmaf_rn(kv.z, acc[i][2], part);
                part = __fmaf_rn(kv.w, acc[i][3], part);
                part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, 1));
                part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, 2));
                if ((tid & 3) == 0) Ss[(8 + MapQ::wc(tid)) * LDB + t] = part;
            }
        }
        {  // dQKD = lower(scale dY Delta^T);  dT = dDelta X^T
            using Map = GemmMap<BC, BC, 2, 2, true>;
            float acc[2][2], acc2[2][2];
            zero_acc(acc);
            zero_acc(acc2);
            block_gemm<BC, BC, 2, 2, false, true>(acc, dYs, ld, Dls, ld, D, tid);
            block_gemm<BC, BC, 2, 2, true, true>(acc2, dDT, LDB, Xs, ld, D, tid);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int t = Map::row(tid, i);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int tau = Map::col(tid, j);
                    Ps[t * LDB + tau] = (tau <= t) ? __fmul_rn(A.scale, acc[i][j]) : 0.f;
                    dTs[t * LDB + tau] = (tau <= t) ? acc2[i][j] : 0.f;
                }
            }
        }
        __syncthreads();
        // dZ = dT diag(beta); dbeta_a[tau] = sum_t Z[t][tau] dT[t][tau]
        for (int idx = tid; idx < BC * BC; idx += CT) {
            const int t = idx / BC, tau = idx - t * BC;
            W1[t * LDB + tau] = __fmul_rn(dTs[t * LDB + tau], bs[tau]);
        }
        if (tid < BC) {
            float s = 0.f;
            for (int t = tid; t < BC; ++t) s = __fmaf_rn(Zs[t * LDB + tid], dTs[t * LDB + tid], s);
            dbs[tid] = s;
            // gather the per-warp-column partials of dgam and dr
            float g = 0.f, rsum = 0.f;
            for (int w = 0; w < MapQ::WGC; ++w) {
                g = __fadd_rn(g, Ss[w * LDB + tid]);
                rsum = __fadd_rn(rsum, Ss[(8 + w) * LDB + tid]);
            }
            dgam[tid] = g;
            dr[tid] = rsum;
        }
        __syncthreads();
        {  // P1 = dZ Z^T
            using Map = GemmMap<BC, BC, 2, 2, true>;
            float acc[2][2];
            zero_acc(acc);
            block_gemm<BC, BC, 2, 2, false, true>(acc, W1, LDB, Zs, LDB, BC, tid);
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) W2[Map::row(tid, i) * LDB + Map::col(tid, j)] = acc[i][j];
        }
        __syncthreads();
        {  // dA = strict_lower(-Z^T P1)
            using Map = GemmMap<BC, BC, 1, 4, false>;
            float acc[1][4];
            zero_acc(acc);
            block_gemm<BC, BC, 1, 4, true, false>(acc, Zs, LDB, W2, LDB, BC, tid);
            const int t = Map::row(tid, 0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tau = Map::col(tid, j);
                W1[t * LDB + tau] = (tau < t) ? -acc[0][j] : 0.f;
            }
        }
        __syncthreads();
        // dbeta_b[t] = sum_tau dA L; dL = beta_t dA; dKK = dL Dm; dD; E = dD Dm
        // Ss <- dKK (strict lower), Ps <- dQKD (.) Dm, dTs <- E
        for (int idx = tid; idx < BC * BC; idx += CT) {
            const int t = idx / BC, tau = idx - t * BC;
            const float dm = Dm[t * LDB + tau];
            const float dA = W1[t * LDB + tau];
            const float dL = __fmul_rn(bs[t], dA);
            float dD = __fmul_rn(Ps[t * LDB + tau], QKm[t * LDB + tau]);
            dD = __fmaf_rn(dL, KKm[t * LDB + tau], dD);
            if (t == BC - 1) dD = __fadd_rn(dD, dr[tau]);
            Ss[t * LDB + tau] = __fmul_rn(dL, dm);
            Ps[t * LDB + tau] = __fmul_rn(Ps[t * LDB + tau], dm);
            dTs[t * LDB + tau] = __fmul_rn(dD, dm);
        }
        __syncthreads();
        if (tid < BC) {  // row/column sums, dbeta_b, dgam of the last token
            const int t = tid;
            float rs = 0.f, cs = 0.f, bb = 0.f;
            for (int tau = 0; tau < BC; ++tau) {
                rs = __fadd_rn(rs, dTs[t * LDB + tau]);
                cs = __fadd_rn(cs, dTs[tau * LDB + t]);
                bb = __fmaf_rn(W1[t * LDB + tau],
                               __fmul_rn(Dm[t * LDB + tau], KKm[t * LDB + tau]), bb);
            }
            float dgt = dgam[t];
            if (t == BC - 1) {
                float dot = 0.f;
                for (int w = 0; w < CT / 32; ++w) dot = __fadd_rn(dot, red[w]);
                dgt = __fadd_rn(dgt, dot);
            }
            dG[t] = __fadd_rn(__fmaf_rn(gam[t], dgt, rs), -cs);
            dbs[t] = __fadd_rn(dbs[t], bb);
        }
        // symmetric dKK into Ss (after the sums above read W1/Dm/KKm only)
        __syncthreads();
        for (int idx = tid; idx < BC * BC; idx += CT) {
            const int t = idx / BC, tau = idx - t * BC;
            if (tau > t) Ss[t * LDB + tau] = Ss[tau * LDB + t];
        }
        __syncthreads();
        {  // dq += (dQKD (.) Dm) K
            float acc[TM][4];
            zero_acc(acc);
            block_gemm<BC, D, TM, 4, false, false>(acc, Ps, LDB, Ks, ld, BC, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) hq[i][j] = __fadd_rn(hq[i][j], acc[i][j]);
        }
        {  // dk += [dQKD (.) Dm ; dKK + dKK^T]^T [Q; K]
            float acc[TM][4];
            zero_acc(acc);
            block_gemm<BC, D, TM, 4, true, false>(acc, Ps, LDB, QKs, ld, 2 * BC, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) hkk[i][j] = __fadd_rn(hkk[i][j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                aq[i][j] = __fadd_rn(aq[i][j], hq[i][j]);
                ak[i][j] = __fadd_rn(ak[i][j], hkk[i][j]);
            }
        // dg = reverse cumsum of dG; dbeta; dv = dX
        if (tid < 32) {
            float x = dG[BC - 1 - tid];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(kFullMask, x, o);
                if (tid >= o) x = __fadd_rn(x, y);
            }
            const int t = BC - 1 - tid;
            if (t < cp.nb) {
                const long long tok = (long long)n * A.T + cp.t0 + t;
                A.dg[tok * A.H_v + h] = x;
                A.dbeta[tok * A.H_v + h] = dbs[t];
            }
        }
        for (int idx = tid; idx < BC * (D / 4); idx += CT) {
            const int i4 = idx / BC, t = idx - i4 * BC;
            if (t >= cp.nb) continue;
            float4* dst = reinterpret_cast<float4*>(
                A.dv + (((long long)n * A.T + cp.t0 + t) * A.H_v + h) * D);
            dst[i4] = make_float4(dXT[(4 * i4 + 0) * LDB + t], dXT[(4 * i4 + 1) * LDB + t],
                                  dXT[(4 * i4 + 2) * LDB + t], dXT[(4 * i4 + 3) * LDB + t]);
        }
    }
    // dq, dk of the key head (value heads summed in ascending order)
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int t = MapQ::row(tid, i);
        if (t >= cp.nb) continue;
        const long long row = (((long long)n * A.T + cp.t0 + t) * A.H_k + hk) * D;
        const int c0 = MapQ::col(tid, 0);
        *reinterpret_cast<float4*>(A.dq + row + c0) = make_float4(aq[i][0], aq[i][1], aq[i][2], aq[i][3]);
        *reinterpret_cast<float4*>(A.dk + row + c0) = make_float4(ak[i][0], ak[i][1], ak[i][2], ak[i][3]);
    }
}

// ---------------------------------------------------------------------------------
// Shared-memory sizes (bytes) and launchers.
template <int D>
size_t prep_smem()
{
    return sizeof(float) * (3 * BC * Ld<D>::v + 5 * BC * LDB + 4 * BC);
}
size_t kda_prep_smem()
{
    return sizeof(float) * (5 * BC * Ld<128>::v + 4 * BC * LDB + BC);
}
template <int D>
size_t state_smem()
{
    constexpr int RR = Rows<D>::RR;
    return sizeof(float) * (RR * Ld<D>::v + 3 * BC * Ld<D>::v + 5 * BC * LDB + 2 * BC);
}
template <int D>
size_t dstate_smem()
{
    return sizeof(float) *
           (Rows<D>::RR * Ld<D>::v + 2 * BC * Ld<D>::v + 4 * BC * LDB + Rows<D>::RR * (2 * BC + 4) +
            2 * BC);
}
template <int D>
size_t grad_smem()
{
    return sizeof(float) * (2 * BC * Ld<D>::v + D * Ld<D>::v + 3 * BC * Ld<D>::v +
                            2 * D * LDB + 9 * BC * LDB + 8 * BC + CT / 32);
}

template <typename K>
static int set_smem(K kern, size_t bytes)
{
    return (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

#define GDN_LAUNCH(kern, grid, smem)                                                   \
    do {                                                                               \
        int e_ = set_smem(kern, smem);                                                 \
        if (e_) return e_;                                                             \
        kern<<<grid, CT, smem, s>>>(a);                                                \
        e_ = (int)cudaGetLastError();                                                  \
        if (e_) return e_;                                                             \
        tap.mark(s);                                                                   \
    } while (0)

// Chunk range r of R: whole checkpoint segments (range_segments), [c_lo, c_hi).
static void range_of(const ChunkArgs& a, int R, bool backward, int r, ChunkArgs& out)
{
    int s_lo = 0, s_hi = 0;
    range_segments(a.n_ck, R, backward, r, &s_lo, &s_hi);
    out = a;
    out.c_lo = min(a.n_chunks, s_lo * a.cps);
    out.c_hi = min(a.n_chunks, s_hi * a.cps);
}

static int launch_prep_range(const ChunkArgs& a, int R, bool backward, int r, cudaStream_t st)
{
    ChunkArgs ar;
    range_of(a, R, backward, r, ar);
    if (a.kda) {
        int err = set_smem(gdn_kda_prep_kernel, kda_prep_smem());
        if (err) return err;
        gdn_kda_prep_kernel<<<dim3((ar.c_hi - ar.c_lo) * a.H_v, a.N), CT, kda_prep_smem(), st>>>(ar);
        return (int)cudaGetLastError();
    }
    int err = set_smem(gdn_chunk_prep_kernel<128>, prep_smem<128>());
    if (err) return err;
    gdn_chunk_prep_kernel<128><<<dim3((ar.c_hi - ar.c_lo) * a.H_v, a.N), CT, prep_smem<128>(), st>>>(ar);
    return (int)cudaGetLastError();
}

// The pipelined tensor-core path at head size 128.  The chunks are cut into R
// segment-aligned ranges (range_of); only events order the library streams, and the call
// forks from and joins back to the caller's stream.
//
// Forward, ranges first to last: prep(r) on the middle-priority stream, then the state
// chain of range r on the high-priority one (the chain's 48 CTAs leave most SMs free);
// prep(r + 1) is enqueued once chain(r) has been, so that the chain's whole-SM CTAs are
// placed before the prep fills the GPU.
//
// Backward, ranges last to first, four streams (most urgent first):
//   chains:    dM chain of range r (after prep(r)), carrying dM to range r - 1
//   preps:     prep(r), then prep(r - 1) once the dM chain of r has been enqueued
//   gradients: after the dM chain of r, the gradient launches of range r, one per place (a
//              launch for place k > 0 may start in the tail of the one for place k - 1)
//   sums:      the sum over value heads of the range's chunks once its gradient launches are
//              done (or of each place's, kSumByPlace), at the least urgent level: its CTAs
//              take what the gradient CTAs leave free
// so that the gradient work of one range runs while the chain walks the next.  With timing
// events set, the backward instead runs its stages one after another as a single range
// (prep and dM chain, gradient step, sum), each between two events.
// The gradient launches of a chunk range: one per place in a segment, in order, each
// parking the entry states of the next place's chunks (launch_tc_grad).
static int launch_grads(const ChunkArgs& ar, cudaStream_t st)
{
    ChunkArgs g = ar;
    int e = 0;
    for (int k = 0; k < ar.cps && !e; ++k) {
        g.grad_loc = k;
        e = launch_tc_grad(g, st);
    }
    return e;
}

// The gradient launches of range r on the gradient stream and the sums over value heads on
// the sum stream: one sum per place once that place's launch is done, or one for the range
// after its last launch (kSumByPlace).
static int grads_and_sums(const ChunkArgs& ar, int r, Pipeline* P)
{
    const cudaStream_t bg = (cudaStream_t)P->bg, su = (cudaStream_t)P->sum;
    const bool by_place = kSumByPlace && ar.cps <= kMaxPlaces;
    ChunkArgs g = ar;
    int e = 0;
    for (int k = 0; k < ar.cps && !e; ++k) {
        g.grad_loc = k;
        if (tc_grad_units(g) <= 0) continue;
        e = launch_tc_grad(g, bg);
        if (!e && by_place) {
            e = (int)cudaEventRecord((cudaEvent_t)P->place_done[r][k], bg);
            if (!e) e = (int)cudaStreamWaitEvent(su, (cudaEvent_t)P->place_done[r][k], 0);
            if (!e) e = launch_tc_dqdk_sum(g, su);
        }
    }
    if (!e && !by_place) {
        e = (int)cudaEventRecord((cudaEvent_t)P->grad_done[r], bg);
        if (!e) e = (int)cudaStreamWaitEvent(su, (cudaEvent_t)P->grad_done[r], 0);
        if (!e) e = launch_tc_dqdk_sum(ar, su);
    }
    return e;
}

static int tc_pipelined(const ChunkArgs& a, cudaStream_t user, bool backward, EventTap& tap)
{
    Pipeline* P = nullptr;
    int e = acquire_pipeline(&P);
    if (e) return e;
    const cudaStream_t hi = (cudaStream_t)P->hi, lo = (cudaStream_t)P->lo, bg = (cudaStream_t)P->bg;
    const cudaStream_t su = (cudaStream_t)P->sum;
    const bool staged = backward && tap.ev != nullptr;
    const int R = staged ? 1 : pipeline_ranges(a.n_ck, backward);
    tap.mark(user);
    e = (int)cudaEventRecord((cudaEvent_t)P->fork, user);
    if (!e) e = (int)cudaStreamWaitEvent(lo, (cudaEvent_t)P->fork, 0);
    if (!e) e = (int)cudaStreamWaitEvent(hi, (cudaEvent_t)P->fork, 0);
    if (!e && backward && !staged) e = (int)cudaStreamWaitEvent(bg, (cudaEvent_t)P->fork, 0);
    if (!e && backward && !staged) e = (int)cudaStreamWaitEvent(su, (cudaEvent_t)P->fork, 0);
    int order[kMaxRanges], nr = 0;
    for (int i = 0; i < R; ++i) {
        const int r = backward ? R - 1 - i : i;
        ChunkArgs ar;
        range_of(a, R, backward, r, ar);
        if (ar.c_hi > ar.c_lo) order[nr++] = r;
    }
    auto prep = [&](int r) -> int {
        int err = launch_prep_range(a, R, backward, r, lo);
        if (!err) err = (int)cudaEventRecord((cudaEvent_t)P->prep_done[r], lo);
        return err;
    };
    if (!e && nr > 0) e = prep(order[0]);
    for (int i = 0; i < nr && !e; ++i) {
        const int r = order[i];
        ChunkArgs ar;
        range_of(a, R, backward, r, ar);
        e = (int)cudaStreamWaitEvent(hi, (cudaEvent_t)P->prep_done[r], 0);
        if (!e) e = (int)cudaEventRecord((cudaEvent_t)P->chain_go[r], hi);
        if (!e) {
            if (!backward) e = launch_tc_state(ar, hi);
            else e = launch_tc_dstate(ar, hi);
        }
        if (!e && backward && !staged) {
            e = (int)cudaEventRecord((cudaEvent_t)P->ds_done[r], hi);
            if (!e) e = (int)cudaStreamWaitEvent(bg, (cudaEvent_t)P->ds_done[r], 0);
            if (!e) e = grads_and_sums(ar, r, P);
        }
        if (!e && i + 1 < nr) {
            e = (int)cudaStreamWaitEvent(lo, (cudaEvent_t)P->chain_go[r], 0);
            if (!e) e = prep(order[i + 1]);
        }
    }
    if (!e) e = (int)cudaEventRecord((cudaEvent_t)P->join_hi, hi);
    if (!e) e = (int)cudaEventRecord((cudaEvent_t)P->join_lo, lo);
    if (!e) e = (int)cudaStreamWaitEvent(user, (cudaEvent_t)P->join_hi, 0);
    if (!e) e = (int)cudaStreamWaitEvent(user, (cudaEvent_t)P->join_lo, 0);
    if (!e && backward && !staged) {
        e = (int)cudaEventRecord((cudaEvent_t)P->join_bg, bg);
        if (!e) e = (int)cudaStreamWaitEvent(user, (cudaEvent_t)P->join_bg, 0);
        if (!e) e = (int)cudaEventRecord((cudaEvent_t)P->join_sum, su);
        if (!e) e = (int)cudaStreamWaitEvent(user, (cudaEvent_t)P->join_sum, 0);
    }
    release_pipeline();
    if (e) return e;
    tap.mark(user);
    if (!staged) return 0;
    e = launch_grads(a, user);
    if (e) return e;
    tap.mark(user);
    e = launch_tc_dqdk_sum(a, user);
    if (e) return e;
    tap.mark(user);
    return 0;
}

template <int D>
static int chunk_forward_t(const ChunkArgs& a, cudaStream_t s, EventTap& tap)
{
    if constexpr (D == 128) {
        if (a.want_tc) return tc_pipelined(a, s, false, tap);
    }
    tap.mark(s);
    GDN_LAUNCH(gdn_chunk_prep_kernel<D>, dim3(a.n_chunks * a.H_v, a.N), prep_smem<D>());
    GDN_LAUNCH((gdn_chunk_state_kernel<D, true>), dim3(Rows<D>::P, a.H_v, a.N), state_smem<D>());
    return 0;
}

// The sequence broadcast at head sizes 32, 64: dq, dk of q/k sequence nq are the sums of the
// gradient kernel's per-value-sequence parts over sequences nq rep .. nq rep + rep - 1, in
// ascending order.  per = T H_k D floats per sequence.
__global__ void __launch_bounds__(256) gdn_seq_sum_kernel(const float* dqS, const float* dkS, float* dq, float* dk,
                                                          long long per, int nq_count, int rep)
{
    const long long total = 2LL * nq_count * per;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int which = idx >= total / 2;
        const long long e = idx - which * (total / 2);
        const long long nq = e / per, o = e - nq * per;
        const float* src = (which ? dkS : dqS) + nq * rep * per + o;
        float acc = 0.f;
        for (int j = 0; j < rep; ++j) acc = __fadd_rn(acc, src[(long long)j * per]);
        (which ? dk : dq)[e] = acc;
    }
}

template <int D>
static int chunk_backward_t(const ChunkArgs& a, cudaStream_t s, EventTap& tap)
{
    if constexpr (D == 128) {
        if (a.want_tc) return tc_pipelined(a, s, true, tap);
    }
    tap.mark(s);
    GDN_LAUNCH(gdn_chunk_prep_kernel<D>, dim3(a.n_chunks * a.H_v, a.N), prep_smem<D>());
    if (a.cps > 1)
        GDN_LAUNCH((gdn_chunk_state_kernel<D, false>), dim3(Rows<D>::P, a.n_ck, a.N * a.H_v),
                   state_smem<D>());
    GDN_LAUNCH(gdn_chunk_dstate_kernel<D>, dim3(Rows<D>::P, a.H_v, a.N), dstate_smem<D>());
    if (a.rep <= 1) {
        GDN_LAUNCH(gdn_chunk_grad_kernel<D>, dim3(a.n_chunks, a.H_k, a.N), grad_smem<D>());
        return 0;
    }
    {  // sequence broadcast: each value sequence's dq, dk into the workspace, then their sums
        ChunkArgs g = a;
        g.dq = a.ws + a.o_dqS;
        g.dk = a.ws + a.o_dkS;
        int e = set_smem(gdn_chunk_grad_kernel<D>, grad_smem<D>());
        if (e) return e;
        gdn_chunk_grad_kernel<D><<<dim3(a.n_chunks, a.H_k, a.N), CT, grad_smem<D>(), s>>>(g);
        e = (int)cudaGetLastError();
        if (e) return e;
        tap.mark(s);
        const long long per = (long long)a.T * a.H_k * D;
        const int nq = a.N / a.rep;
        long long blocks = (2LL * nq * per + 255) / 256;
        if (blocks > 152LL * 16) blocks = 152LL * 16;
        if (blocks > 0)
            gdn_seq_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>(g.dq, g.dk, a.dq, a.dk, per, nq, a.rep);
        e = (int)cudaGetLastError();
        if (e) return e;
        tap.mark(s);
    }
    return 0;
}
#undef GDN_LAUNCH

int launch_chunk_forward(const ChunkArgs& a, int D, void* stream, EventTap& tap)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (D == 32) return chunk_forward_t<32>(a, s, tap);
    if (D == 64) return chunk_forward_t<64>(a, s, tap);
    if (D == 128) return chunk_forward_t<128>(a, s, tap);
    return (int)cudaErrorInvalidValue;
}

int launch_chunk_backward(const ChunkArgs& a, int D, void* stream, EventTap& tap)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (D == 32) return chunk_backward_t<32>(a, s, tap);
    if (D == 64) return chunk_backward_t<64>(a, s, tap);
    if (D == 128) return chunk_backward_t<128>(a, s, tap);
    return (int)cudaErrorInvalidValue;
}

}  // namespace gdn
