// ssm_diag.cu -- the selective scan with one decay per state (Mamba-1: one channel a head,
// 16 states) split by checkpoint segments, so that segments run side by side.
//
// Source: "dillon-blake llama.cpp PR #26", the SSM_SCAN_BACK section (the reverse walk, the
// final-state seed, the group fold; the token-serial form is in ssm_scan.cu).  With a decay
// per state, every (channel h, state j) is a scalar linear recurrence
//   s_t = a_t s_{t-1} + b_t,   a_t = exp(dt_t A[h][j]),   b_t = B_t[j] x_t dt_t,
// so a segment [t0, t1) maps its entry state s to G s + dS, with G the product of its a_t
// and dS its scan from a zero state.  The reverse walk regroups the same way: the gradient
// reaching s_t is g_t = a_{t+1} g_{t+1} + dy_t C_t[j], so a block of tokens [t0, t1) maps the
// gradient arriving from its right, c (already carried through a_{t1}), to U + G c, with
// U = a_{t0} gl_{t0}, gl its reverse scan from zero and G the product of its a_t; d_s is the
// last such carry.  The rest is the walk's per-token algebra:
//   dx_t = dt_t sum_j g_t B_t[j],   ddt_t = sum_j g_t (B_t[j] x_t + A[h][j] a_t s_{t-1}),
//   dB_t[j] += g_t x_t dt_t,        dC_t[j] += dy_t s_t          (dB, dC summed over a group).
//
// Kernels (a CTA holds 16 channels x 16 states, thread = (channel, state)):
//   forward   diag_fwd_local_kernel (segment, channel block): dS and G of the segment
//             diag_chain_kernel     (channel, state): s_{k+1} = G_k s_k + dS_k: the checkpoints
//                                   and s_T
//             diag_fwd_out_kernel   (segment, channel block): y from the segment's checkpoint
//   backward  diag_bwd_prep_kernel  (segment, channel block): the entry state, U and G of each
//                                   32-token sub-block of the segment
//             diag_dchain_kernel    (channel, state): the carry arriving at every sub-block,
//                                   last first; d_s
//             diag_bwd_grad_kernel  (sub-block, channel block): the sub-block's states from its
//                                   entry state, then its tokens in reverse: dx, ddt, and the
//                                   block's dB, dC partials
//             diag_reduce_kernel    (token): dB, dC summed over a group's channel blocks
// Every sum runs in a fixed order (no atomics): results do not change from run to run.
#include "ssm_diag.h"

#include <algorithm>
#include <cmath>

namespace ssm {
namespace diag {

constexpr int S = kS;
constexpr int SB = kSB;
constexpr int TB = 256;        // threads of the per-block kernels
constexpr int CHB = TB / S;    // channels a CTA
constexpr int NW = TB / 32;    // warps a CTA
constexpr int TC = 64;         // threads of the chain kernels (a Mamba-1 layer's 1536 x 16
                               // chains then spread over all SMs)

struct Pos {
    long long h, g;
    int j, cb;
};
// Channel h and state j of thread tid in channel block blk; g its group, cb the block's index
// within the group.
__device__ __forceinline__ Pos pos_of(const Args& a, long long blk, int tid)
{
    Pos p;
    p.h = blk * CHB + (tid >> 4);
    p.j = tid & (S - 1);
    p.g = blk * CHB / (a.H / a.G);
    p.cb = (int)(blk - p.g * a.nbg);
    return p;
}

// A tile of up to SB tokens [t0, t0 + nt) of the CTA's 16 channels in shared memory, one
// coalesced load a value: dt, x, dy [SB][16 channels] and B, C [SB][16 states] (the arrays
// passed as null are skipped).  Ends with a barrier.
struct Tile {
    float *dt, *x, *dy, *B, *C;
};
__device__ __forceinline__ void stage(const Args& a, long long n, long long blk, long long g, long long t0, int nt,
                                      const Tile& s, int tid)
{
    for (int i = tid; i < nt * CHB; i += TB) {
        const int tt = i / CHB, c = i - tt * CHB;
        const long long row = n * a.T + t0 + tt;
        const long long hx = row * a.H + blk * CHB + c, bx = (row * a.G + g) * S + c;
        if (s.dt) s.dt[i] = a.dt[hx];
        if (s.x) s.x[i] = a.x[hx];
        if (s.dy) s.dy[i] = a.dy[hx];
        if (s.B) s.B[i] = a.B[bx];
        if (s.C) s.C[i] = a.C[bx];
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------------
// Forward 1: the segment's scan from a zero state (dS, into the slot the chain turns into the
// next checkpoint, s_T for the last) and its decay G (in the y region of the output, which the
// output kernel overwrites afterwards).  Grid (n_ck, H / 16, N).
__global__ void __launch_bounds__(TB) diag_fwd_local_kernel(const Args a)
{
    __shared__ float sdt[SB * CHB], sx[SB * CHB], sB[SB * S];
    const int tid = threadIdx.x;
    const int k = blockIdx.x;
    const long long n = blockIdx.z;
    const Pos p = pos_of(a, blockIdx.y, tid);
    const int c = tid >> 4;
    const float Aj = a.A[p.h * S + p.j];
    const long long t0 = (long long)k * a.K, t1 = std::min(a.T, t0 + a.K);
    float s = 0.f, G = 1.f;
    for (long long tb = t0; tb < t1; tb += SB) {
        const int nt = (int)std::min((long long)SB, t1 - tb);
        if (tb > t0) __syncthreads();
        stage(a, n, blockIdx.y, p.g, tb, nt, Tile{sdt, sx, nullptr, sB, nullptr}, tid);
#pragma unroll 4
        for (int tt = 0; tt < nt; ++tt) {
            const float d = sdt[tt * CHB + c];
            const float av = expf(__fmul_rn(d, Aj));
            s = __fmaf_rn(av, s, __fmul_rn(sB[tt * S + p.j], __fmul_rn(sx[tt * CHB + c], d)));
            G = __fmul_rn(G, av);
        }
    }
    const long long head = n * a.H + p.h;
    float* dst = k + 1 < a.n_ck ? a.ckpt + (head * a.n_ck + k + 1) * S : a.sT + head * S;
    dst[p.j] = s;
    a.y[((n * a.n_ck + k) * a.H + p.h) * S + p.j] = G;
}

// Forward 2: the chain over segments, one (channel, state) a thread.  Grid (ceil(16 H / TC), N).
// Checkpoint 0 is s0; slot k + 1 (or s_T) holds dS_k and becomes s_{k+1}.
__global__ void __launch_bounds__(TC) diag_chain_kernel(const Args a)
{
    const long long i = (long long)blockIdx.x * TC + threadIdx.x;
    const long long n = blockIdx.y;
    if (i >= a.H * S) return;
    const long long h = i / S;
    const int j = (int)(i - h * S);
    const long long head = n * a.H + h;
    float* ck = a.ckpt + head * a.n_ck * S + j;
    float* sTp = a.sT + head * S + j;
    const float* Gp = a.y + n * a.n_ck * a.H * S + i;
    const long long gs = a.H * S;
    auto slot = [&](int k) { return k + 1 < a.n_ck ? ck + (long long)(k + 1) * S : sTp; };
    float s = a.s0[head * S + j];
    ck[0] = s;
    float gb[4], db[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        gb[r] = r < a.n_ck ? Gp[r * gs] : 1.f;
        db[r] = r < a.n_ck ? *slot(r) : 0.f;
    }
    for (int k0 = 0; k0 < a.n_ck; k0 += 4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int k = k0 + r;
            if (k < a.n_ck) {
                s = __fmaf_rn(gb[r], s, db[r]);
                if (k + 4 < a.n_ck) {
                    gb[r] = Gp[(k + 4) * gs];
                    db[r] = *slot(k + 4);
                }
                *slot(k) = s;
            }
        }
    }
}

// Forward 3: y of the segment's tokens from its checkpoint.  Grid (n_ck, H / 16, N).
__global__ void __launch_bounds__(TB) diag_fwd_out_kernel(const Args a)
{
    __shared__ float sdt[SB * CHB], sx[SB * CHB], sB[SB * S], sC[SB * S];
    __shared__ float ysum[SB * TB];  // s_t C_t[j] per token and thread, summed over j after the tile
    const int tid = threadIdx.x;
    const int c = tid >> 4;
    const int k = blockIdx.x;
    const long long n = blockIdx.z;
    const Pos p = pos_of(a, blockIdx.y, tid);
    const float Aj = a.A[p.h * S + p.j];
    const long long t0 = (long long)k * a.K, t1 = std::min(a.T, t0 + a.K);
    float s = a.ckpt[((n * a.H + p.h) * a.n_ck + k) * S + p.j];
    for (long long tb = t0; tb < t1; tb += SB) {
        const int nt = (int)std::min((long long)SB, t1 - tb);
        if (tb > t0) __syncthreads();
        stage(a, n, blockIdx.y, p.g, tb, nt, Tile{sdt, sx, nullptr, sB, sC}, tid);
#pragma unroll 4
        for (int tt = 0; tt < nt; ++tt) {
            const float d = sdt[tt * CHB + c];
            const float av = expf(__fmul_rn(d, Aj));
            s = __fmaf_rn(av, s, __fmul_rn(sB[tt * S + p.j], __fmul_rn(sx[tt * CHB + c], d)));
            ysum[tt * TB + tid] = __fmul_rn(s, sC[tt * S + p.j]);
        }
        __syncthreads();
        for (int i = tid; i < nt * CHB; i += TB) {  // (token, channel) pairs
            const int tt = i / CHB, ch = i - tt * CHB;
            const float* v = ysum + tt * TB + ch * S;
            float y = 0.f;
#pragma unroll
            for (int e = 0; e < S; ++e) y = __fadd_rn(y, v[(e + ch) & (S - 1)]);  // rotated: no bank conflicts
            a.y[(n * a.T + tb + tt) * a.H + blockIdx.y * CHB + ch] = y;
        }
    }
}

// ---------------------------------------------------------------------------------
// Backward 1: per 32-token sub-block of the segment, its entry state (replayed from the
// checkpoint by the forward's own step) and its U, G.  Sub-blocks past the sequence's end get
// U = 0, G = 1.  Grid (n_ck, H / 16, N).
__global__ void __launch_bounds__(TB) diag_bwd_prep_kernel(const Args a)
{
    __shared__ float sdt[SB * CHB], sx[SB * CHB], sdy[SB * CHB], sB[SB * S], sC[SB * S];
    __shared__ float aring[SB * TB];  // the forward pass's decays, for the reverse pass
    const int tid = threadIdx.x;
    const int c = tid >> 4;
    const int k = blockIdx.x;
    const long long n = blockIdx.z;
    const Pos p = pos_of(a, blockIdx.y, tid);
    const float Aj = a.A[p.h * S + p.j];
    const long long t0 = (long long)k * a.K, t1 = std::min(a.T, t0 + a.K);
    float s = a.ckpt_in[((n * a.H + p.h) * a.n_ck + k) * S + p.j];
    for (int i = 0; i < a.spk; ++i) {
        const long long ts0 = t0 + (long long)i * SB, ts1 = std::min(t1, ts0 + SB);
        const long long o = ((n * a.nsb + (long long)k * a.spk + i) * a.H + p.h) * S + p.j;
        a.sin_sb[o] = s;
        if (ts0 >= ts1) {
            a.U[o] = 0.f;
            a.Gb[o] = 1.f;
            continue;
        }
        const int nt = (int)(ts1 - ts0);
        if (i > 0) __syncthreads();
        stage(a, n, blockIdx.y, p.g, ts0, nt, Tile{sdt, sx, sdy, sB, sC}, tid);
#pragma unroll 4
        for (int tt = 0; tt < nt; ++tt) {
            const float d = sdt[tt * CHB + c];
            const float av = expf(__fmul_rn(d, Aj));
            aring[tt * TB + tid] = av;
            s = __fmaf_rn(av, s, __fmul_rn(sB[tt * S + p.j], __fmul_rn(sx[tt * CHB + c], d)));
        }
        float gl = 0.f, G = 1.f, a_next = 1.f;
#pragma unroll 4
        for (int tt = nt - 1; tt >= 0; --tt) {
            const float av = aring[tt * TB + tid];
            if (tt < nt - 1) gl = __fmul_rn(a_next, gl);
            gl = __fmaf_rn(sdy[tt * CHB + c], sC[tt * S + p.j], gl);
            G = __fmul_rn(G, av);
            a_next = av;
        }
        a.U[o] = __fmul_rn(a_next, gl);
        a.Gb[o] = G;
    }
}

// Backward 2: the carry arriving at every sub-block from its right, last first, one (channel,
// state) a thread; d_s the carry past token 0.  Grid (ceil(16 H / TC), N).
__global__ void __launch_bounds__(TC) diag_dchain_kernel(const Args a)
{
    const long long i = (long long)blockIdx.x * TC + threadIdx.x;
    const long long n = blockIdx.y;
    if (i >= a.H * S) return;
    const long long gs = a.H * S;
    const long long base = n * a.nsb * gs + i;
    float c = a.dsT[n * gs + i];
    float ub[4], gb[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long long sb = a.nsb - 1 - r;
        ub[r] = sb >= 0 ? a.U[base + sb * gs] : 0.f;
        gb[r] = sb >= 0 ? a.Gb[base + sb * gs] : 1.f;
    }
    for (int r0 = 0; r0 < a.nsb; r0 += 4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int rr = r0 + r;
            if (rr < a.nsb) {
                const long long sb = a.nsb - 1 - rr;
                a.carry[base + sb * gs] = c;
                c = __fmaf_rn(gb[r], c, ub[r]);
                if (rr + 4 < a.nsb) {
                    ub[r] = a.U[base + (sb - 4) * gs];
                    gb[r] = a.Gb[base + (sb - 4) * gs];
                }
            }
        }
    }
    a.ds0[n * gs + i] = c;
}

// Backward 3: every gradient of one 32-token sub-block for 16 channels.  Grid (nsb, H / 16, N).
__global__ void __launch_bounds__(TB) diag_bwd_grad_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* ring = sm;              // [SB][TB]: the state entering each token
    float* aring = ring + SB * TB; // [SB][TB]: its decay
    float* red = aring + SB * TB;  // [SB][NW][2 S]: warp sums of the dB, dC terms
    float* sdt = red + SB * NW * 2 * S;  // the sub-block's inputs
    float* sx = sdt + SB * CHB;
    float* sdy = sx + SB * CHB;
    float* sB = sdy + SB * CHB;
    float* sC = sB + SB * S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, c = tid >> 4;
    const int sb = blockIdx.x;
    const long long n = blockIdx.z;
    const Pos p = pos_of(a, blockIdx.y, tid);
    const int k = sb / a.spk, i = sb - k * a.spk;
    const long long t0 = (long long)k * a.K, t1 = std::min(a.T, t0 + a.K);
    const long long ts0 = t0 + (long long)i * SB, ts1 = std::min(t1, ts0 + SB);
    const int nt = (int)(ts1 - ts0);
    if (nt <= 0) return;  // a sub-block past the sequence's end (the whole CTA)
    const float Aj = a.A[p.h * S + p.j];
    const long long o = ((n * a.nsb + sb) * a.H + p.h) * S + p.j;
    float s = a.sin_sb[o];
    float g = a.carry[o], a_next = 1.f;
    stage(a, n, blockIdx.y, p.g, ts0, nt, Tile{sdt, sx, sdy, sB, sC}, tid);
#pragma unroll 4
    for (int tt = 0; tt < nt; ++tt) {
        ring[tt * TB + tid] = s;
        const float d = sdt[tt * CHB + c];
        const float av = expf(__fmul_rn(d, Aj));
        aring[tt * TB + tid] = av;
        s = __fmaf_rn(av, s, __fmul_rn(sB[tt * S + p.j], __fmul_rn(sx[tt * CHB + c], d)));
    }
#pragma unroll 4
    for (int tt = nt - 1; tt >= 0; --tt) {
        const float d = sdt[tt * CHB + c], xv = sx[tt * CHB + c], dyv = sdy[tt * CHB + c];
        const float Bt = sB[tt * S + p.j], C = sC[tt * S + p.j];
        const float av = aring[tt * TB + tid];
        if (tt < nt - 1) g = __fmul_rn(a_next, g);
        g = __fmaf_rn(dyv, C, g);  // the gradient reaching s_t
        const float sp = ring[tt * TB + tid];
        const float xdt = __fmul_rn(xv, d);
        const float st = __fmaf_rn(av, sp, __fmul_rn(Bt, xdt));  // s_t, the forward's own step
        float vB = __fmul_rn(g, xdt), vC = __fmul_rn(dyv, st);
        // this token's dx and ddt terms over the slots just read (summed over states below)
        ring[tt * TB + tid] = __fmul_rn(g, Bt);
        aring[tt * TB + tid] = __fmul_rn(g, __fmaf_rn(__fmul_rn(Aj, av), sp, __fmul_rn(Bt, xv)));
        // the warp's two channels, then the warps in ascending order below
        vB = __fadd_rn(vB, __shfl_xor_sync(0xffffffffu, vB, 16));
        vC = __fadd_rn(vC, __shfl_xor_sync(0xffffffffu, vC, 16));
        if (lane < S) {
            red[(tt * NW + warp) * 2 * S + lane] = vB;
            red[(tt * NW + warp) * 2 * S + S + lane] = vC;
        }
        a_next = av;
    }
    __syncthreads();
    for (int i2 = tid; i2 < nt * CHB; i2 += TB) {  // (token, channel) pairs
        const int tt = i2 / CHB, ch = i2 - tt * CHB;
        const float* vx = ring + tt * TB + ch * S;
        const float* vd = aring + tt * TB + ch * S;
        float dxs = 0.f, dds = 0.f;
#pragma unroll
        for (int e = 0; e < S; ++e) {  // states from j = ch on, rotated: no bank conflicts
            const int j = (e + ch) & (S - 1);
            dxs = __fadd_rn(dxs, vx[j]);
            dds = __fadd_rn(dds, vd[j]);
        }
        const long long o2 = (n * a.T + ts0 + tt) * a.H + blockIdx.y * CHB + ch;
        a.dx[o2] = __fmul_rn(dxs, sdt[tt * CHB + ch]);
        a.ddt[o2] = dds;
    }
    float* part = a.partBC + (long long)p.cb * 2 * S;
    for (int idx = tid; idx < nt * 2 * S; idx += TB) {
        const int tt = idx / (2 * S), c = idx - tt * 2 * S;
        float acc = 0.f;
        for (int w = 0; w < NW; ++w) acc = __fadd_rn(acc, red[(tt * NW + w) * 2 * S + c]);
        part[(((n * a.T + ts0 + tt) * a.G + p.g) * a.nbg) * 2 * S + c] = acc;
    }
}

// Backward 4: dB, dC of each token: its group's channel-block partials summed in ascending order.
__global__ void __launch_bounds__(256) diag_reduce_kernel(const Args a)
{
    const long long tok = blockIdx.x;  // n T + t
    for (long long i = threadIdx.x; i < a.G * 2 * S; i += blockDim.x) {
        const long long g = i / (2 * S), c = i - g * 2 * S;
        const float* src = a.partBC + (tok * a.G + g) * (long long)a.nbg * 2 * S + c;
        float acc = 0.f;
        for (int b = 0; b < a.nbg; ++b) acc = __fadd_rn(acc, src[(long long)b * 2 * S]);
        if (c < S)
            a.dB[(tok * a.G + g) * S + c] = acc;
        else
            a.dC[(tok * a.G + g) * S + c - S] = acc;
    }
}

// ---------------------------------------------------------------------------------
// Host side.

constexpr size_t kSmemGrad = sizeof(float) * (2 * SB * TB + SB * NW * 2 * S + 3 * SB * CHB + 2 * SB * S);

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

Workspace workspace_layout(long long N, long long T, long long H, long long G, int K)
{
    Workspace w{};
    const long long n_ck = (T + K - 1) / K, spk = (K + SB - 1) / SB;
    const size_t per = sizeof(float) * (size_t)(N * n_ck * spk * H) * S;
    size_t o = 0;
    w.sin_sb = o;
    o += align256(per);
    w.U = o;
    o += align256(per);
    w.Gb = o;
    o += align256(per);
    w.carry = o;
    o += align256(per);
    w.partBC = o;
    o += align256(sizeof(float) * (size_t)(N * T * G * ((H / G) / CHB)) * 2 * S);
    w.total = o;
    return w;
}

int forward(const Args& a, cudaStream_t st)
{
    const dim3 seg((unsigned)a.n_ck, (unsigned)(a.H / CHB), (unsigned)a.N);
    const dim3 chain((unsigned)((a.H * S + TC - 1) / TC), (unsigned)a.N);
    diag_fwd_local_kernel<<<seg, TB, 0, st>>>(a);
    diag_chain_kernel<<<chain, TC, 0, st>>>(a);
    diag_fwd_out_kernel<<<seg, TB, 0, st>>>(a);
    return (int)cudaGetLastError();
}

int backward(const Args& a, cudaStream_t st)
{
    const dim3 seg((unsigned)a.n_ck, (unsigned)(a.H / CHB), (unsigned)a.N);
    const dim3 chain((unsigned)((a.H * S + TC - 1) / TC), (unsigned)a.N);
    const dim3 sub((unsigned)a.nsb, (unsigned)(a.H / CHB), (unsigned)a.N);
    cudaError_t e = cudaFuncSetAttribute(diag_bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemGrad);
    if (e != cudaSuccess) return (int)e;
    diag_bwd_prep_kernel<<<seg, TB, 0, st>>>(a);
    diag_dchain_kernel<<<chain, TC, 0, st>>>(a);
    diag_bwd_grad_kernel<<<sub, TB, kSmemGrad, st>>>(a);
    diag_reduce_kernel<<<(unsigned)(a.N * a.T), 256, 0, st>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace diag
}  // namespace ssm
