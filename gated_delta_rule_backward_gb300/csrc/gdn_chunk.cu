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

namespace gdn {

constexpr int CT = 256;        // threads per CTA (all chunk kernels)
constexpr int LDB = BC + 4;    // leading dimension of BC-wide shared rows
constexpr int RR = 32;         // rows of M per CTA in the state kernels
constexpr int LDR = RR + 4;
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

// ---------------------------------------------------------------------------------
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
    {  // [QK; KK] = [Q; K] K^T
        using Map = GemmMap<2 * BC, BC, 4, 2, true>;
        float acc[4][2];
        zero_acc(acc);
        block_gemm<2 * BC, BC, 4, 2, false, true>(acc, QKs, ld, Ks, ld, D, tid);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = Map::row(tid, i);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = Map::col(tid, j);
                if (m < BC)
                    QKm[m * LDB + n] = (n <= m) ? acc[i][j] : 0.f;
                else
                    KKm[(m - BC) * LDB + n] = (n < m - BC) ? acc[i][j] : 0.f;
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Dm[t * LDB + tau] = (tau <= t) ? expf(__fsub_rn(Gs[t], Gs[tau])) : 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // forward substitution, lane j owns column j of Z
        const int j = tid;
        for (int t = 0; t < BC; ++t) {
            float z;
            if (t < j) {
                z = 0.f;
            } else if (t == j) {
                z = 1.f;
            } else {
                float a0 = 0.f, a1 = 0.f;
                int tau = j;
                for (; tau + 1 < t; tau += 2) {
                    a0 = __fmaf_rn(__fmul_rn(Dm[t * LDB + tau], KKm[t * LDB + tau]),
                                   Zs[tau * LDB + j], a0);
                    a1 = __fmaf_rn(__fmul_rn(Dm[t * LDB + tau + 1], KKm[t * LDB + tau + 1]),
                                   Zs[(tau + 1) * LDB + j], a1);
                }
                if (tau < t)
                    a0 = __fmaf_rn(__fmul_rn(Dm[t * LDB + tau], KKm[t * LDB + tau]),
                                   Zs[tau * LDB + j], a0);
                z = -__fmul_rn(bs[t], __fadd_rn(a0, a1));
            }
            Zs[t * LDB + j] = z;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Ts[t * LDB + tau] = __fmul_rn(Zs[t * LDB + tau], bs[tau]);
    }
    __syncthreads();
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

// ---------------------------------------------------------------------------------
// Prep: one CTA per (chunk, value head, sequence).
template <int D>
__global__ void __launch_bounds__(CT) gdn_chunk_prep_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    const int c = blockIdx.x, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
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
    float* TG = Ts + BC * LDB;
    float* vec = TG + BC * LDB;       // gs, bs, Gs, gam
    float *gs = vec, *bs = vec + BC, *Gs = vec + 2 * BC, *gam = vec + 3 * BC;

    const long long tq = (long long)n * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
    const long long tk = (long long)n * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
    load_rows_pad(QKs, ld, A.q + tq, A.qs1, cp.nb, D, A.vec_q, tid);
    load_rows_pad(QKs + BC * ld, ld, A.k + tk, A.ks1, cp.nb, D, A.vec_k, tid);
    if (A.want_wu) {
        const long long tv = (long long)n * A.vs0 + (long long)cp.t0 * A.vs1 + (long long)h * A.vs2;
        load_rows_pad(Vs, ld, A.v + tv, A.vs1, cp.nb, D, A.vec_v, tid);
    }
    load_gate_beta(A, n, h, cp, gs, bs, tid);
    __syncthreads();
    chunk_prep<D>(QKs, gs, bs, Gs, gam, Dm, KKm, QKm, Zs, Ts, tid);

    float* wsT = A.ws + A.o_T + ch * (BC * BC);
    float* wsQ = A.ws + A.o_QKD + ch * (BC * BC);
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        wsT[idx] = Ts[t * LDB + tau];
        wsQ[idx] = __fmul_rn(QKm[t * LDB + tau], Dm[t * LDB + tau]);
        TG[t * LDB + tau] = __fmul_rn(Ts[t * LDB + tau], gam[tau]);
    }
    if (tid < BC) {
        A.ws[A.o_gam + ch * BC + tid] = gam[tid];
        A.ws[A.o_r + ch * BC + tid] = Dm[(BC - 1) * LDB + tid];
    }
    if (!A.want_wu) return;
    __syncthreads();
    // W = T diag(gamma) K,  U = T V   (BC x D each)
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
        for (int j = 0; j < 4; ++j) wsU[Map::row(tid, i) * D + Map::col(tid, j)] = acc[i][j];
}

// ---------------------------------------------------------------------------------
// State chain, rows [p RR, p RR + RR) of M for one head.
//   forward  (blockIdx.y = head, blockIdx.x = p): every chunk in order; writes
//            ckpt at segment starts, y, and state_T.
//   recompute(blockIdx.y = segment, blockIdx.x = p, blockIdx.z = head): from ckpt[s]
//            through the segment's chunks but its last, parking each chunk-entry state.
template <int D, bool FWD>
__global__ void __launch_bounds__(CT) gdn_chunk_state_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    constexpr int TM3 = D / 32;  // M_end tile: RR x D
    const int tid = threadIdx.x, p = blockIdx.x;
    int n, h, c_begin, c_end;
    if (FWD) {
        h = blockIdx.y;
        n = blockIdx.z;
        c_begin = 0;
        c_end = A.n_chunks;
    } else {
        const int head = blockIdx.z;
        n = head / A.H_v;
        h = head - n * A.H_v;
        const int s = blockIdx.y;
        c_begin = s * A.cps;
        const int seg_len = min(A.T, s * A.C + A.C) - s * A.C;
        c_end = c_begin + (seg_len + BC - 1) / BC - 1;  // chunks whose end state is needed
        if (c_end <= c_begin) return;
    }
    const int hk = h % A.H_k;
    const long long head = (long long)n * A.H_v + h;
    const int row0 = p * RR;

    extern __shared__ __align__(16) float sm[];
    float* Ms = sm;                   // RR x ld   (rows of M)
    float* WQ = Ms + RR * ld;         // [W; gamma Q]  2BC x ld
    float* RK = WQ + 2 * BC * ld;     // r (.) K   BC x ld
    float* Us = RK + BC * ld;         // BC x LDR
    float* Dls = Us + BC * LDR;       // Delta  BC x LDR
    float* Y1 = Dls + BC * LDR;       // BC x LDR
    float* QD = Y1 + BC * LDR;        // BC x LDB
    float* vec = QD + BC * LDB;       // gam, r
    float *gam = vec, *rr = vec + BC;

    // entry state
    {
        const float* src;
        if (FWD) {
            src = A.state0 + (head * D + row0) * D;
        } else {
            src = A.ckpt + ((head * A.n_ck + blockIdx.y) * D + row0) * D;
        }
        for (int idx = tid; idx < RR * (D / 4); idx += CT) {
            const int j = idx / (D / 4), i4 = idx - j * (D / 4);
            *reinterpret_cast<float4*>(Ms + j * ld + 4 * i4) =
                __ldg(reinterpret_cast<const float4*>(src + (long long)j * D) + i4);
        }
    }
    for (int c = c_begin; c < c_end; ++c) {
        const ChunkPos cp = chunk_pos(A, c);
        const long long ch = head * A.n_chunks + c;
        __syncthreads();
        if (FWD && cp.loc == 0) {  // checkpoint: the state entering segment cp.seg
            float* dst = A.ckpt_out + ((head * A.n_ck + cp.seg) * D + row0) * D;
            for (int idx = tid; idx < RR * (D / 4); idx += CT) {
                const int j = idx / (D / 4), i4 = idx - j * (D / 4);
                reinterpret_cast<float4*>(dst + (long long)j * D)[i4] =
                    *reinterpret_cast<const float4*>(Ms + j * ld + 4 * i4);
            }
        }
        if (tid < BC) {
            gam[tid] = A.ws[A.o_gam + ch * BC + tid];
            rr[tid] = A.ws[A.o_r + ch * BC + tid];
        }
        load_ws(WQ, ld, A.ws + A.o_W + ch * (BC * D), BC, D, tid);
        for (int idx = tid; idx < BC * (RR / 4); idx += CT) {  // U[:, own rows]
            const int t = idx / (RR / 4), j4 = idx - t * (RR / 4);
            *reinterpret_cast<float4*>(Us + t * LDR + 4 * j4) = __ldg(
                reinterpret_cast<const float4*>(A.ws + A.o_U + ch * (BC * D) + t * D + row0) + j4);
        }
        __syncthreads();
        const long long tk = (long long)n * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
        load_rows_pad(RK, ld, A.k + tk, A.ks1, cp.nb, D, A.vec_k, tid, rr);
        if (FWD) {
            const long long tq =
                (long long)n * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
            load_rows_pad(WQ + BC * ld, ld, A.q + tq, A.qs1, cp.nb, D, A.vec_q, tid, gam);
            load_ws(QD, LDB, A.ws + A.o_QKD + ch * (BC * BC), BC, BC, tid);
        }
        __syncthreads();
        const float gl = gam[BC - 1];
        // [W M^T ; gamma Q M^T]  (2BC x RR)  -> Delta = U - W M^T,  Y1
        {
            constexpr int MR = FWD ? 2 * BC : BC;
            using Map = GemmMap<MR, RR, MR / 16, 2, true>;
            float acc[MR / 16][2];
            zero_acc(acc);
            block_gemm<MR, RR, MR / 16, 2, false, true>(acc, WQ, ld, Ms, ld, D, tid);
#pragma unroll
            for (int i = 0; i < MR / 16; ++i) {
                const int m = Map::row(tid, i);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int nn = Map::col(tid, j);
                    if (m < BC)
                        Dls[m * LDR + nn] = __fsub_rn(Us[m * LDR + nn], acc[i][j]);
                    else
                        Y1[(m - BC) * LDR + nn] = acc[i][j];
                }
            }
        }
        __syncthreads();
        if (FWD) {  // Y = scale (Y1 + lower(QK^T (.) Dm) Delta)
            using Map = GemmMap<BC, RR, 1, 4, false>;
            float acc[1][4];
            zero_acc(acc);
            block_gemm<BC, RR, 1, 4, false, false>(acc, QD, LDB, Dls, LDR, BC, tid);
            const int t = Map::row(tid, 0);
            if (t < cp.nb) {
                float* yrow = A.y + (((long long)n * A.T + cp.t0 + t) * A.H_v + h) * D + row0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int nn = Map::col(tid, j);
                    yrow[nn] = __fmul_rn(A.scale, __fadd_rn(Y1[t * LDR + nn], acc[0][j]));
                }
            }
        }
        {  // M_end = gamma_last M + Delta^T (r (.) K)   (RR x D)
            using Map = GemmMap<RR, D, TM3, 4, false>;
            float acc[TM3][4];
            zero_acc(acc);
            block_gemm<RR, D, TM3, 4, true, false>(acc, Dls, LDR, RK, ld, BC, tid);
#pragma unroll
            for (int i = 0; i < TM3; ++i) {
                const int j = Map::row(tid, i);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int ii = Map::col(tid, jj);
                    Ms[j * ld + ii] = __fmaf_rn(gl, Ms[j * ld + ii], acc[i][jj]);
                }
            }
        }
        if (!FWD) {  // park the entry state of chunk c + 1
            __syncthreads();
            float* dst = A.ws + A.o_Mc + (ch + 1) * (long long)(D * D) + (long long)row0 * D;
            for (int idx = tid; idx < RR * (D / 4); idx += CT) {
                const int j = idx / (D / 4), i4 = idx - j * (D / 4);
                reinterpret_cast<float4*>(dst + (long long)j * D)[i4] =
                    *reinterpret_cast<const float4*>(Ms + j * ld + 4 * i4);
            }
        }
    }
    if (FWD) {
        __syncthreads();
        float* dst = A.state_T + (head * D + row0) * D;
        for (int idx = tid; idx < RR * (D / 4); idx += CT) {
            const int j = idx / (D / 4), i4 = idx - j * (D / 4);
            reinterpret_cast<float4*>(dst + (long long)j * D)[i4] =
                *reinterpret_cast<const float4*>(Ms + j * ld + 4 * i4);
        }
    }
}

// ---------------------------------------------------------------------------------
// The dM chain in reverse, rows [p RR, p RR + RR) of one head.  Per chunk:
//   dDelta = r (.) (K dM^T) + scale QKD^T dY
//   dX     = T^T dDelta
//   dM    <- gamma_last dM + dY^T (scale gamma Q) - dX^T (gamma K)
// Parks dM (as it enters the chunk from the right), dDelta and dX in the workspace.
template <int D>
__global__ void __launch_bounds__(CT) gdn_chunk_dstate_kernel(const ChunkArgs A)
{
    constexpr int ld = Ld<D>::v;
    constexpr int TM4 = D / 32;
    const int tid = threadIdx.x, p = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h % A.H_k;
    const long long head = (long long)n * A.H_v + h;
    const int row0 = p * RR;

    extern __shared__ __align__(16) float sm[];
    float* dMs = sm;                   // RR x ld
    float* Ks = dMs + RR * ld;         // BC x ld (raw k)
    float* Bst = Ks + BC * ld;         // [scale gamma Q; gamma K]  2BC x ld
    float* DYX = Bst + 2 * BC * ld;    // [dY; -dX]  2BC x LDR (own rows)
    float* dDs = DYX + 2 * BC * LDR;   // BC x LDR
    float* Ts = dDs + BC * LDR;        // BC x LDB
    float* QD = Ts + BC * LDB;         // BC x LDB
    float* vec = QD + BC * LDB;
    float *gam = vec, *rr = vec + BC, *sgam = vec + 2 * BC;

    for (int idx = tid; idx < RR * (D / 4); idx += CT) {
        const int j = idx / (D / 4), i4 = idx - j * (D / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (A.dstate_T)
            x = __ldg(reinterpret_cast<const float4*>(A.dstate_T + (head * D + row0 + j) * D) + i4);
        *reinterpret_cast<float4*>(dMs + j * ld + 4 * i4) = x;
    }
    for (int c = A.n_chunks - 1; c >= 0; --c) {
        const ChunkPos cp = chunk_pos(A, c);
        const long long ch = head * A.n_chunks + c;
        __syncthreads();
        if (tid < BC) {
            const float gm = A.ws[A.o_gam + ch * BC + tid];
            gam[tid] = gm;
            sgam[tid] = __fmul_rn(A.scale, gm);
            rr[tid] = A.ws[A.o_r + ch * BC + tid];
        }
        {  // park dM (the gradient of this chunk's end state)
            float* dst = A.ws + A.o_dM + ch * (long long)(D * D) + (long long)row0 * D;
            for (int idx = tid; idx < RR * (D / 4); idx += CT) {
                const int j = idx / (D / 4), i4 = idx - j * (D / 4);
                reinterpret_cast<float4*>(dst + (long long)j * D)[i4] =
                    *reinterpret_cast<const float4*>(dMs + j * ld + 4 * i4);
            }
        }
        load_ws(Ts, LDB, A.ws + A.o_T + ch * (BC * BC), BC, BC, tid);
        load_ws(QD, LDB, A.ws + A.o_QKD + ch * (BC * BC), BC, BC, tid);
        const long long tgy =
            (long long)n * A.gys0 + (long long)cp.t0 * A.gys1 + (long long)h * A.gys2 + row0;
        load_rows_pad(DYX, LDR, A.gy + tgy, A.gys1, cp.nb, RR, A.vec_gy, tid);
        __syncthreads();
        const long long tk = (long long)n * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
        const long long tq = (long long)n * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
        load_rows_pad(Ks, ld, A.k + tk, A.ks1, cp.nb, D, A.vec_k, tid);
        load_rows_pad(Bst, ld, A.q + tq, A.qs1, cp.nb, D, A.vec_q, tid, sgam);
        load_rows_pad(Bst + BC * ld, ld, A.k + tk, A.ks1, cp.nb, D, A.vec_k, tid, gam);
        __syncthreads();
        {  // dDelta = r (.) (K dM^T)
            using Map = GemmMap<BC, RR, 2, 2, true>;
            float acc[2][2];
            zero_acc(acc);
            block_gemm<BC, RR, 2, 2, false, true>(acc, Ks, ld, dMs, ld, D, tid);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int t = Map::row(tid, i);
#pragma unroll
                for (int j = 0; j < 2; ++j) dDs[t * LDR + Map::col(tid, j)] = __fmul_rn(rr[t], acc[i][j]);
            }
        }
        __syncthreads();
        {  // dDelta += scale QKD^T dY
            using Map = GemmMap<BC, RR, 1, 4, false>;
            float acc[1][4];
            zero_acc(acc);
            block_gemm<BC, RR, 1, 4, true, false>(acc, QD, LDB, DYX, LDR, BC, tid);
            const int t = Map::row(tid, 0);
            float* dst = A.ws + A.o_dDel + ch * (BC * D) + t * D + row0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nn = Map::col(tid, j);
                const float val = __fmaf_rn(A.scale, acc[0][j], dDs[t * LDR + nn]);
                dDs[t * LDR + nn] = val;
                dst[nn] = val;
            }
        }
        __syncthreads();
        {  // dX = T^T dDelta
            using Map = GemmMap<BC, RR, 1, 4, false>;
            float acc[1][4];
            zero_acc(acc);
            block_gemm<BC, RR, 1, 4, true, false>(acc, Ts, LDB, dDs, LDR, BC, tid);
            const int t = Map::row(tid, 0);
            float* dst = A.ws + A.o_dX + ch * (BC * D) + t * D + row0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nn = Map::col(tid, j);
                DYX[(BC + t) * LDR + nn] = -acc[0][j];
                dst[nn] = acc[0][j];
            }
        }
        __syncthreads();
        {  // dM <- gamma_last dM + [dY; -dX]^T [scale gamma Q; gamma K]
            const float gl = gam[BC - 1];
            using Map = GemmMap<RR, D, TM4, 4, false>;
            float acc[TM4][4];
            zero_acc(acc);
            block_gemm<RR, D, TM4, 4, true, false>(acc, DYX, LDR, Bst, ld, 2 * BC, tid);
#pragma unroll
            for (int i = 0; i < TM4; ++i) {
                const int j = Map::row(tid, i);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int ii = Map::col(tid, jj);
                    dMs[j * ld + ii] = __fmaf_rn(gl, dMs[j * ld + ii], acc[i][jj]);
                }
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < RR * D; idx += CT) {
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
    float* dXs = dYs + BC * ld;       // dX
    float* dDs = dXs + BC * ld;       // dDelta
    float* Dm = dDs + BC * ld;        // BC x LDB each:
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
    float *gs = vec, *bs = vec + BC, *Gs = vec + 2 * BC, *gam = vec + 3 * BC;
    float *dgam = vec + 4 * BC, *dr = vec + 5 * BC, *dG = vec + 6 * BC, *dbs = vec + 7 * BC;
    float* red = vec + 8 * BC;        // CT/32 partials

    {
        const long long tq = (long long)n * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
        const long long tk = (long long)n * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
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
        load_gate_beta(A, n, h, cp, gs, bs, tid);
        {
            const long long tv = (long long)n * A.vs0 + (long long)cp.t0 * A.vs1 + (long long)h * A.vs2;
            load_rows_pad(Xs, ld, A.v + tv, A.vs1, cp.nb, D, A.vec_v, tid);
            const long long tg = (long long)n * A.gys0 + (long long)cp.t0 * A.gys1 + (long long)h * A.gys2;
            load_rows_pad(dYs, ld, A.gy + tg, A.gys1, cp.nb, D, A.vec_gy, tid);
            load_ws(dXs, ld, A.ws + A.o_dX + ch * (BC * D), BC, D, tid);
            load_ws(dDs, ld, A.ws + A.o_dDel + ch * (BC * D), BC, D, tid);
            const float* msrc = (cp.loc == 0)
                                    ? A.ckpt + (head * A.n_ck + cp.seg) * (long long)(D * D)
                                    : A.ws + A.o_Mc + ch * (long long)(D * D);
            load_ws(MB, ld, msrc, D, D, tid);
        }
        __syncthreads();
        chunk_prep<D>(QKs, gs, bs, Gs, gam, Dm, KKm, QKm, Zs, Ts, tid);

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
            block_gemm<BC, D, TM, 4, false, false>(acc, dYs, ld, MB, ld, D, tid);
            block_gemm<BC, D, TM, 4, false, false>(acc2, dXs, ld, MB, ld, D, tid);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int t = MapQ::row(tid, i);
                float part = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ii = MapQ::col(tid, j);
                    hq[i][j] = __fmul_rn(__fmul_rn(A.scale, gam[t]), acc[i][j]);
                    hkk[i][j] = -__fmul_rn(gam[t], acc2[i][j]);
                    part = __fmaf_rn(__fmul_rn(A.scale, QKs[t * ld + ii]), acc[i][j], part);
                    part = __fmaf_rn(-Ks[t * ld + ii], acc2[i][j], part);
                }
                // row t is spread over the MapQ::NX lanes of one warp segment
#pragma unroll
                for (int o = MapQ::NX / 2; o > 0; o >>= 1)
                    part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, o));
                if ((tid % MapQ::NX) == 0) dgam[t] = part;
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
#pragma unroll
                for (int j = 0; j < 4; ++j) Dls[Map::row(tid, i) * ld + Map::col(tid, j)] = acc[i][j];
        }
        {  // MB <- dM_end, with <dM_end, M_c> on the way
            float part = 0.f;
            const float* src = A.ws + A.o_dM + ch * (long long)(D * D);
            for (int idx = tid; idx < D * (D / 4); idx += CT) {
                const int j = idx / (D / 4), i4 = idx - j * (D / 4);
                const float4 dm = __ldg(reinterpret_cast<const float4*>(src + (long long)j * D) + i4);
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
                float part = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ii = MapQ::col(tid, j);
                    hkk[i][j] = __fmaf_rn(rt, acc[i][j], hkk[i][j]);
                    part = __fmaf_rn(Ks[t * ld + ii], acc[i][j], part);
                }
#pragma unroll
                for (int o = MapQ::NX / 2; o > 0; o >>= 1)
                    part = __fadd_rn(part, __shfl_xor_sync(kFullMask, part, o));
                if ((tid % MapQ::NX) == 0) dr[t] = part;
            }
        }
        {  // dQKD = lower(scale dY Delta^T);  dT = dDelta X^T
            using Map = GemmMap<BC, BC, 2, 2, true>;
            float acc[2][2], acc2[2][2];
            zero_acc(acc);
            zero_acc(acc2);
            block_gemm<BC, BC, 2, 2, false, true>(acc, dYs, ld, Dls, ld, D, tid);
            block_gemm<BC, BC, 2, 2, false, true>(acc2, dDs, ld, Xs, ld, D, tid);
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
        for (int idx = tid; idx < cp.nb * (D / 4); idx += CT) {
            const int t = idx / (D / 4), i4 = idx - t * (D / 4);
            float4* dst = reinterpret_cast<float4*>(
                A.dv + (((long long)n * A.T + cp.t0 + t) * A.H_v + h) * D);
            dst[i4] = *reinterpret_cast<const float4*>(dXs + t * ld + 4 * i4);
        }
    }
    // dq, dk of the key head (value heads summed in ascending order)
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int t = MapQ::row(tid, i);
        if (t >= cp.nb) continue;
        const long long row = (((long long)n * A.T + cp.t0 + t) * A.H_k + hk) * D;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int ii = MapQ::col(tid, j);
            A.dq[row + ii] = aq[i][j];
            A.dk[row + ii] = ak[i][j];
        }
    }
}

// ---------------------------------------------------------------------------------
// Shared-memory sizes (bytes) and launchers.
template <int D>
size_t prep_smem()
{
    return sizeof(float) * (3 * BC * Ld<D>::v + 6 * BC * LDB + 4 * BC);
}
template <int D>
size_t state_smem()
{
    return sizeof(float) * (RR * Ld<D>::v + 3 * BC * Ld<D>::v + 3 * BC * LDR + BC * LDB + 2 * BC);
}
template <int D>
size_t dstate_smem()
{
    return sizeof(float) *
           (RR * Ld<D>::v + 3 * BC * Ld<D>::v + 3 * BC * LDR + 2 * BC * LDB + 3 * BC);
}
template <int D>
size_t grad_smem()
{
    return sizeof(float) * (2 * BC * Ld<D>::v + D * Ld<D>::v + 5 * BC * Ld<D>::v +
                            9 * BC * LDB + 8 * BC + CT / 32);
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

template <int D>
static int chunk_forward_t(const ChunkArgs& a, cudaStream_t s, EventTap& tap)
{
    tap.mark(s);
    GDN_LAUNCH(gdn_chunk_prep_kernel<D>, dim3(a.n_chunks, a.H_v, a.N), prep_smem<D>());
    GDN_LAUNCH((gdn_chunk_state_kernel<D, true>), dim3(D / RR, a.H_v, a.N), state_smem<D>());
    return 0;
}

template <int D>
static int chunk_backward_t(const ChunkArgs& a, cudaStream_t s, EventTap& tap)
{
    tap.mark(s);
    GDN_LAUNCH(gdn_chunk_prep_kernel<D>, dim3(a.n_chunks, a.H_v, a.N), prep_smem<D>());
    if (a.cps > 1)
        GDN_LAUNCH((gdn_chunk_state_kernel<D, false>), dim3(D / RR, a.n_ck, a.N * a.H_v),
                   state_smem<D>());
    GDN_LAUNCH(gdn_chunk_dstate_kernel<D>, dim3(D / RR, a.H_v, a.N), dstate_smem<D>());
    GDN_LAUNCH(gdn_chunk_grad_kernel<D>, dim3(a.n_chunks, a.H_k, a.N), grad_smem<D>());
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
