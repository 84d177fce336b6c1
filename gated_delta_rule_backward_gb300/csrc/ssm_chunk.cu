// ssm_chunk.cu -- the selective scan with one decay per head (Mamba-2) in chunked form: the
// products of a chunk as CTA-level tensor-pipe products (warp-level tf32 MMAs, three-pass
// split for fp32 accuracy; gdn_mma.cuh) that run for every chunk at once, and only an
// elementwise chain over chunk states left serial.
//
// Source: "dillon-blake llama.cpp PR #26", the SSM_SCAN_BACK section (the reverse walk, the
// final-state seed, the group fold; the token-serial form is in ssm_scan.cu).  The chunked form
// is the same recurrence regrouped.  For a chunk of L tokens of one head, with l_t = dt_t A,
// c_t = sum_{tau <= t} l_tau (within the chunk), e_t = exp(c_t), w_t = exp(c_{L-1} - c_t),
// g = exp(c_{L-1}), Xd = diag(dt) X (L x P), Q = C B^T (L x L) and the decay mask
// Lm[t][tau] = exp(c_t - c_tau) for tau <= t (0 above), s_in the state entering the chunk:
//   s_t   = e_t s_in + sum_{tau <= t} exp(c_t - c_tau) Xd_tau (x) B_tau
//   Y     = (Lm (.) Q) Xd + diag(e) C s_in^T
//   s_out = g s_in + dS,   dS = (diag(w) Xd)^T B
// and, with dY and dS_out (the gradient reaching s_out), M = Lm (.) Q, dM = dY Xd^T,
// dQ = Lm (.) dM, u = B dS_out^T:
//   dS_in = g dS_out + (diag(e) dY)^T C
//   dXd   = M^T dY + diag(w) u,          dx = dt (.) dXd
//   dC    = dQ B + diag(e) dY s_in,      dB = dQ^T C + diag(w) Xd dS_out
//   dc_t  = rowsum(M (.) dM)_t - colsum(M (.) dM)_t + e_t sum_p dY[t][p] (C s_in^T)[t][p] - v_t,
//           v_t = w_t sum_p Xd[t][p] u[t][p], and at t = L - 1 also + g <dS_out, s_in> + sum_t v_t
//   ddt_t = sum_p x[t][p] dXd[t][p] + A sum_{t' >= t} dc_t'
// (the chain rule through each factor: exp(c_t - c_tau) depends on c_t and c_tau, e_t on c_t,
// w_tau on c_{L-1} and c_tau, g on c_{L-1}; c is the running sum of l = dt A).  Tokens past
// the end of the sequence enter as dt = 0 and x = B = C = dy = 0, which changes nothing.
//
// Kernels (L = 64 tokens, P = 64 channels, S = 128 states; a segment is the m = K / L chunks
// between two checkpoints).  With one chunk a segment (m = 1) the chunk kernels take a block of
// HB heads of one group, whose B, C and Q they load or compute once; with several, one head
// and walk the segment's chunks:
//   forward   ssd_state_hb_kernel / ssd_seg_state_kernel
//                                   dS of the segment from a zero state, and its decay G
//             ssd_chain_kernel      (state slice, head): s_{k+1} = G_k s_k + dS_k over the
//                                   segments: the checkpoints, s_T
//             ssd_output_hb_kernel / ssd_output_kernel
//                                   y of each chunk from its entry state (m > 1: the state
//                                   carried across the segment's chunks)
//   backward  ssd_dprep_hb_kernel / ssd_dprep_kernel
//                                   (diag(e) dY)^T C of each chunk, g, and the entry states of
//                                   the segment's inner chunks (m > 1)
//             ssd_dchain_kernel     (state slice, head): dS_out of every chunk, last first; d_s
//             ssd_grad_kernel       (chunk, block of HB heads of a group): every gradient of
//                                   the chunk; dB, dC summed over the block's heads in registers
//             ssd_reduce_kernel     (token): dB, dC summed over a group's blocks
// Every sum runs in a fixed order (no atomics): results do not change from run to run.
#include "ssm_chunk.h"

#include <algorithm>
#include <cmath>

#include "gdn_mma.cuh"

namespace ssm {
namespace ssd {

using gdn::block_mma;
using gdn::MmaAcc;
using gdn::zero_mma;

constexpr int L = kChunk;
constexpr int P = kP;
constexpr int S = kS;
constexpr int PS = P * S;
constexpr int CT = 256;     // threads of every kernel but the reduction
constexpr int LD64 = 68;    // leading dimension of 64-wide tiles (4 mod 32)
constexpr int LD128 = 132;  // of 128-wide tiles
constexpr int T64 = L * LD64;
constexpr int T128 = L * LD128;
constexpr int NSCAL = 4 * L + 4;  // dt, c, e, w, then g and a spare
constexpr int SLICES = PS / (4 * CT);  // state slices of the chain kernels (a float4 a thread)

// Output maps of the 64 x 64 and 64 x 128 products (the same for every operand layout).
using Map64 = gdn::MmaMap<64, 64>;
using Map128 = gdn::MmaMap<64, 128>;
using Acc64 = MmaAcc<64, 64>;
using Acc128 = MmaAcc<64, 128>;
// The gradient kernel's: 16 warps on a 4 x 4 grid.
constexpr int GT = 512;
using G64 = gdn::MmaMap<64, 64, 4, 4>;
using G128 = gdn::MmaMap<64, 128, 4, 4>;
using GAcc64 = MmaAcc<64, 64, 4, 4>;
using GAcc128 = MmaAcc<64, 128, 4, 4>;

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 fma4(float g, float4 s, float4 d)
{
    return make_float4(__fmaf_rn(g, s.x, d.x), __fmaf_rn(g, s.y, d.y), __fmaf_rn(g, s.z, d.z), __fmaf_rn(g, s.w, d.w));
}
__device__ __forceinline__ float4 mul4(float4 v, float s)
{
    return make_float4(__fmul_rn(v.x, s), __fmul_rn(v.y, s), __fmul_rn(v.z, s), __fmul_rn(v.w, s));
}
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc)
{
    return __fmaf_rn(a.w, b.w, __fmaf_rn(a.z, b.z, __fmaf_rn(a.y, b.y, __fmaf_rn(a.x, b.x, acc))));
}
__device__ __forceinline__ void st2(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }

// Sum over the 4 lanes sharing a row of a product (lane bits 0, 1), and over the 8 lanes
// sharing a column (lane bits 2 .. 4).  Butterflies: every lane ends with the same bits.
__device__ __forceinline__ float row_lanes(float v)
{
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float col_lanes(float v)
{
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
    return __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
}

// Per-chunk scalars of one head in shared memory.
struct Scal {
    float* p;
    __device__ float* dt() const { return p; }
    __device__ float* c() const { return p + L; }
    __device__ float* e() const { return p + 2 * L; }
    __device__ float* w() const { return p + 3 * L; }
    __device__ float& g() const { return p[4 * L]; }
};

// dt, c, e, w, g of chunk [t0, t0 + L) of head h.  Ends without a barrier.
__device__ __forceinline__ void load_scalars(const Args& a, long long n, long long h, long long t0, int nt,
                                             Scal s, int tid)
{
    if (tid < L) s.dt()[tid] = tid < nt ? a.dt[(n * a.T + t0 + tid) * a.H + h] : 0.f;
    __syncthreads();
    if (tid == 0) {
        const float A = a.A[h];
        float c = 0.f;
        for (int t = 0; t < L; ++t) {
            c = __fadd_rn(c, __fmul_rn(s.dt()[t], A));
            s.c()[t] = c;
        }
        s.g() = expf(c);
    }
    __syncthreads();
    if (tid < L) {
        s.e()[tid] = expf(s.c()[tid]);
        s.w()[tid] = expf(__fsub_rn(s.c()[L - 1], s.c()[tid]));
    }
}

// Rows [t0, t0 + L) of B or C (one group's [.., S] slab) into a tile, zero past the end.
template <int NTH = CT>
__device__ __forceinline__ void load_bc(float* tile, const float* src, const Args& a, long long n, long long g,
                                        long long t0, int nt, int tid)
{
    for (int i = tid; i < L * S / 4; i += NTH) {
        const int t = i / (S / 4), q = i - t * (S / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nt) v = ld4(src + ((n * a.T + t0 + t) * a.G + g) * S + 4 * q);
        st4(tile + t * LD128 + 4 * q, v);
    }
}

// Row t, float4 q of head h's [.., P] slab of x or dy (zero past the end).
__device__ __forceinline__ float4 head_row4(const float* src, const Args& a, long long n, long long h, long long t0,
                                            int t, int q, int nt)
{
    if (t >= nt) return make_float4(0.f, 0.f, 0.f, 0.f);
    return ld4(src + ((n * a.T + t0 + t) * a.H + h) * P + 4 * q);
}

// Xd = diag(dt) X into xd (if not null) and diag(w) Xd into xw (if not null).
__device__ __forceinline__ void load_xd(float* xd, float* xw, const Args& a, long long n, long long h, long long t0,
                                        int nt, Scal s, int tid)
{
    for (int i = tid; i < L * P / 4; i += CT) {
        const int t = i / (P / 4), q = i - t * (P / 4);
        const float4 v = mul4(head_row4(a.x, a, n, h, t0, t, q, nt), s.dt()[t]);
        if (xd) st4(xd + t * LD64 + 4 * q, v);
        if (xw) st4(xw + t * LD64 + 4 * q, mul4(v, s.w()[t]));
    }
}

// L2 prefetches ahead of a head's loads, one 128-byte line a call and thread: the chunk's rows
// of head h in a [.., P] slab (2 lines a row, threads < 2 nt), and a dense state (threads
// < 256).
__device__ __forceinline__ void prefetch_rows(const float* src, const Args& a, long long n, long long h,
                                              long long t0, int nt, int tid)
{
    if (tid < 2 * nt) gdn::tc::prefetch_l2(src + ((n * a.T + t0 + (tid >> 1)) * a.H + h) * P + 32 * (tid & 1));
}
__device__ __forceinline__ void prefetch_state(const float* src, int tid)
{
    if (tid < PS / 32) gdn::tc::prefetch_l2(src + 32 * tid);
}

// A dense [P][S] state into a tile (ld LD128) and back.
template <int NTH = CT>
__device__ __forceinline__ void load_state(float* tile, const float* src, int tid)
{
    for (int i = tid; i < PS / 4; i += NTH) {
        const int p = i / (S / 4), q = i - p * (S / 4);
        st4(tile + p * LD128 + 4 * q, ld4(src + p * S + 4 * q));
    }
}
__device__ __forceinline__ void store_state(float* dst, const float* tile, int tid)
{
    for (int i = tid; i < PS / 4; i += CT) {
        const int p = i / (S / 4), q = i - p * (S / 4);
        st4(dst + p * S + 4 * q, ld4(tile + p * LD128 + 4 * q));
    }
}

// A 64 x 128 accumulator (rows p, columns j) to a dense [P][S] state.
__device__ __forceinline__ void store_acc128(float* dst, const Acc128& acc, int tid)
{
#pragma unroll
    for (int i = 0; i < Map128::MT; ++i)
#pragma unroll
        for (int j = 0; j < Map128::NT; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                st2(dst + Map128::row(tid, i, 2 * h) * S + Map128::col(tid, j, 0), acc[i][j][2 * h],
                    acc[i][j][2 * h + 1]);
}

// s <- g s + (diag(w) Xd)^T B across one chunk (sXw: diag(w) Xd, rows tau; sB: the chunk's B
// rows; sS: the state, rows p).  The forward's walk and the backward's replay both use it, so
// the replayed entry states are the forward's bit for bit.  Barriers on both sides.
__device__ __forceinline__ void state_step(float* sS, const float* sXw, const float* sB, float g, int tid)
{
    Acc128 acc;
    zero_mma<64, 128>(acc);
    block_mma<64, 128, true, false>(acc, sXw, LD64, sB, LD128, L, tid);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < Map128::MT; ++i)
#pragma unroll
        for (int j = 0; j < Map128::NT; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float* x = sS + Map128::row(tid, i, r) * LD128 + Map128::col(tid, j, r);
                *x = __fmaf_rn(g, *x, acc[i][j][r]);
            }
    __syncthreads();
}

struct Seg {
    long long n, h, g, head;
    int seg, ch0, ch1;
};
__device__ __forceinline__ Seg seg_of(const Args& a)
{
    Seg s;
    s.seg = blockIdx.x;
    s.h = blockIdx.y;
    s.n = blockIdx.z;
    s.g = s.h / (a.H / a.G);
    s.head = s.n * a.H + s.h;
    s.ch0 = s.seg * a.m;
    s.ch1 = min(a.nch, s.ch0 + a.m);
    return s;
}

// A block of HB heads of one group at one chunk: grid (nch, G nhb, N).
struct Blk {
    long long n, g, h0, t0;
    int ch, hb, nt;
};
__device__ __forceinline__ Blk blk_of(const Args& a)
{
    Blk b;
    b.ch = blockIdx.x;
    b.n = blockIdx.z;
    b.g = blockIdx.y / a.nhb;
    b.hb = (int)(blockIdx.y - b.g * a.nhb);
    b.h0 = b.g * (a.H / a.G) + (long long)b.hb * a.HB;
    b.t0 = (long long)b.ch * L;
    b.nt = (int)min((long long)L, a.T - b.t0);
    return b;
}

// The forward's segment decays G_k wait for the chain in the y region of the output, which the
// output kernels overwrite afterwards: float (n n_ck + k) H + h (n_ck <= T, so it fits).
__device__ __forceinline__ float* decay_slot(const Args& a, long long n, long long k, long long h)
{
    return a.y + (n * a.n_ck + k) * a.H + h;
}

// ---------------------------------------------------------------------------------
// Forward 1, one chunk a segment: dS of chunk ch for HB heads into the slot the chain turns
// into checkpoint ch + 1 (the last chunk's into s_T), and g.  Grid (nch, G nhb, N).
__global__ void __launch_bounds__(CT, 3) ssd_state_hb_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sB = sm;
    float* sXw = sB + T128;
    const Scal sc{sXw + T64};
    const int tid = threadIdx.x;
    const Blk b = blk_of(a);
    prefetch_rows(a.x, a, b.n, b.h0, b.t0, b.nt, tid);
    load_bc(sB, a.B, a, b.n, b.g, b.t0, b.nt, tid);
    for (int hh = 0; hh < a.HB; ++hh) {
        const long long h = b.h0 + hh, head = b.n * a.H + h;
        __syncthreads();
        if (hh + 1 < a.HB) prefetch_rows(a.x, a, b.n, h + 1, b.t0, b.nt, tid);
        load_scalars(a, b.n, h, b.t0, b.nt, sc, tid);
        __syncthreads();
        load_xd(nullptr, sXw, a, b.n, h, b.t0, b.nt, sc, tid);
        __syncthreads();
        Acc128 acc;
        zero_mma<64, 128>(acc);
        block_mma<64, 128, true, false>(acc, sXw, LD64, sB, LD128, L, tid);
        float* dst = b.ch + 1 < a.n_ck ? a.ckpt + (head * a.n_ck + b.ch + 1) * PS : a.sT + head * PS;
        store_acc128(dst, acc, tid);
        if (tid == 0) *decay_slot(a, b.n, b.ch, h) = sc.g();
    }
}

// ---------------------------------------------------------------------------------
// Forward 1, several chunks a segment: dS of each segment (its state change from a zero entry state), into the slot
// the chain turns into the next checkpoint (the last segment's into s_T).  Grid (n_ck, H, N).
__global__ void __launch_bounds__(CT, 2) ssd_seg_state_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sB = sm;
    float* sXw = sB + T128;
    const Scal sc{sXw + T64};
    const int tid = threadIdx.x;
    const Seg z = seg_of(a);
    Acc128 acc;
    zero_mma<64, 128>(acc);
    float G = 1.f;  // the segment's decay, the product of its chunks' g in order
    for (int ch = z.ch0; ch < z.ch1; ++ch) {
        const long long t0 = (long long)ch * L;
        const int nt = (int)min((long long)L, a.T - t0);
        __syncthreads();
        load_scalars(a, z.n, z.h, t0, nt, sc, tid);
        __syncthreads();
        load_bc(sB, a.B, a, z.n, z.g, t0, nt, tid);
        load_xd(nullptr, sXw, a, z.n, z.h, t0, nt, sc, tid);
        __syncthreads();
        Acc128 tmp;
        zero_mma<64, 128>(tmp);
        block_mma<64, 128, true, false>(tmp, sXw, LD64, sB, LD128, L, tid);
        const float g = sc.g();
        G = __fmul_rn(G, g);
#pragma unroll
        for (int i = 0; i < Map128::MT; ++i)
#pragma unroll
            for (int j = 0; j < Map128::NT; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[i][j][r] = __fmaf_rn(g, acc[i][j][r], tmp[i][j][r]);
    }
    float* dst = z.seg + 1 < a.n_ck ? a.ckpt + (z.head * a.n_ck + z.seg + 1) * PS : a.sT + z.head * PS;
    store_acc128(dst, acc, tid);
    if (tid == 0) *decay_slot(a, z.n, z.seg, z.h) = G;
}

// Forward 2: the chain over segments, one float4 of one head's state a thread.  Grid
// (SLICES, H, N).  Checkpoint 0 is s0; slot k + 1 (or s_T) holds dS_k and becomes s_{k+1}.
__global__ void __launch_bounds__(CT) ssd_chain_kernel(const Args a)
{
    __shared__ float gs[CT];
    const int tid = threadIdx.x;
    const long long h = blockIdx.y, n = blockIdx.z, head = n * a.H + h;
    const long long off = 4LL * (blockIdx.x * CT + tid);
    float* ck = a.ckpt + head * a.n_ck * PS + off;
    float* sTp = a.sT + head * PS + off;
    auto slot = [&](int k) { return k + 1 < a.n_ck ? ck + (long long)(k + 1) * PS : sTp; };
    float4 s = ld4(a.s0 + head * PS + off);
    st4(ck, s);
    float4 buf[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) buf[k] = k < a.n_ck ? ld4(slot(k)) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < a.n_ck; base += CT) {
        __syncthreads();
        if (base + tid < a.n_ck) gs[tid] = *decay_slot(a, n, base + tid, h);
        __syncthreads();
        const int nb = min(CT, a.n_ck - base);
        for (int k0 = 0; k0 < nb; k0 += 4) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (k0 + r < nb) {
                    const int kk = base + k0 + r;
                    s = fma4(gs[k0 + r], s, buf[r]);
                    if (kk + 4 < a.n_ck) buf[r] = ld4(slot(kk + 4));
                    st4(slot(kk), s);
                }
            }
        }
    }
}

// Forward 3, one chunk a segment: y of chunk ch for HB heads from checkpoint ch, Q = C B^T
// computed once and kept in registers (each thread masks the elements it owns), the state
// tile over B's once Q is done: two CTAs an SM.  Grid (nch, G nhb, N).
__global__ void __launch_bounds__(CT, 2) ssd_output_hb_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sB = sm;
    float* sS = sB;          // the state entering the chunk, rows p (after Q)
    float* sC = sB + T128;
    float* sXd = sC + T128;
    float* sM = sXd + T64;   // Lm (.) Q
    const Scal sc{sM + T64};
    const int tid = threadIdx.x;
    const Blk b = blk_of(a);
    auto prefetch_head = [&](long long h) {
        prefetch_rows(a.x, a, b.n, h, b.t0, b.nt, tid);
        prefetch_state(a.ckpt + ((b.n * a.H + h) * a.n_ck + b.ch) * PS, tid);
    };
    prefetch_head(b.h0);
    load_bc(sB, a.B, a, b.n, b.g, b.t0, b.nt, tid);
    load_bc(sC, a.C, a, b.n, b.g, b.t0, b.nt, tid);
    __syncthreads();
    Acc64 q;  // C B^T, rows t, columns tau
    zero_mma<64, 64>(q);
    block_mma<64, 64, false, true>(q, sC, LD128, sB, LD128, S, tid);
    for (int hh = 0; hh < a.HB; ++hh) {
        const long long h = b.h0 + hh, head = b.n * a.H + h;
        __syncthreads();  // B (first head) or the previous head's tiles are no longer read
        if (hh + 1 < a.HB) prefetch_head(h + 1);
        load_scalars(a, b.n, h, b.t0, b.nt, sc, tid);
        __syncthreads();
        load_xd(sXd, nullptr, a, b.n, h, b.t0, b.nt, sc, tid);
        load_state(sS, a.ckpt + (head * a.n_ck + b.ch) * PS, tid);
        __syncthreads();
        Acc64 yi;  // C s_in^T, rows t, columns p
        zero_mma<64, 64>(yi);
        block_mma<64, 64, false, true>(yi, sC, LD128, sS, LD128, S, tid);
        {
            const float* c = sc.c();
#pragma unroll
            for (int i = 0; i < Map64::MT; ++i)
#pragma unroll
                for (int j = 0; j < Map64::NT; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int t = Map64::row(tid, i, r), tau = Map64::col(tid, j, r);
                        sM[t * LD64 + tau] = tau <= t ? __fmul_rn(expf(__fsub_rn(c[t], c[tau])), q[i][j][r]) : 0.f;
                    }
        }
        __syncthreads();
        Acc64 yy;
        zero_mma<64, 64>(yy);
        block_mma<64, 64, false, false>(yy, sM, LD64, sXd, LD64, L, tid);
#pragma unroll
        for (int i = 0; i < Map64::MT; ++i)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int t = Map64::row(tid, i, 2 * hr);
                if (t >= b.nt) continue;
                const float e = sc.e()[t];
                float* yrow = a.y + ((b.n * a.T + b.t0 + t) * a.H + h) * P;
#pragma unroll
                for (int j = 0; j < Map64::NT; ++j)
                    st2(yrow + Map64::col(tid, j, 0), __fmaf_rn(e, yi[i][j][2 * hr], yy[i][j][2 * hr]),
                        __fmaf_rn(e, yi[i][j][2 * hr + 1], yy[i][j][2 * hr + 1]));
            }
    }
}

// Forward 3, several chunks a segment: y of every chunk of a segment from the segment's
// checkpoint.  Grid (n_ck, H, N).
__global__ void __launch_bounds__(CT, 1) ssd_output_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sB = sm;
    float* sC = sB + T128;
    float* sS = sC + T128;   // the state entering the chunk, rows p
    float* sXd = sS + T128;
    float* sM = sXd + T64;   // Lm (.) Q, then diag(w) Xd
    const Scal sc{sM + T64};
    const int tid = threadIdx.x;
    const Seg z = seg_of(a);
    load_state(sS, a.ckpt + (z.head * a.n_ck + z.seg) * PS, tid);
    for (int ch = z.ch0; ch < z.ch1; ++ch) {
        const long long t0 = (long long)ch * L;
        const int nt = (int)min((long long)L, a.T - t0);
        __syncthreads();
        load_scalars(a, z.n, z.h, t0, nt, sc, tid);
        __syncthreads();
        load_bc(sB, a.B, a, z.n, z.g, t0, nt, tid);
        load_bc(sC, a.C, a, z.n, z.g, t0, nt, tid);
        load_xd(sXd, nullptr, a, z.n, z.h, t0, nt, sc, tid);
        __syncthreads();
        Acc64 yi;  // C s_in^T, rows t, columns p
        {  // M = Lm (.) C B^T
            Acc64 q;
            zero_mma<64, 64>(q);
            zero_mma<64, 64>(yi);
            block_mma<64, 64, false, true>(q, sC, LD128, sB, LD128, S, tid);
            block_mma<64, 64, false, true>(yi, sC, LD128, sS, LD128, S, tid);
            const float* c = sc.c();
#pragma unroll
            for (int i = 0; i < Map64::MT; ++i)
#pragma unroll
                for (int j = 0; j < Map64::NT; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int t = Map64::row(tid, i, r), tau = Map64::col(tid, j, r);
                        sM[t * LD64 + tau] =
                            tau <= t ? __fmul_rn(expf(__fsub_rn(c[t], c[tau])), q[i][j][r]) : 0.f;
                    }
        }
        __syncthreads();
        {  // y = M Xd + diag(e) C s_in^T
            Acc64 yy;
            zero_mma<64, 64>(yy);
            block_mma<64, 64, false, false>(yy, sM, LD64, sXd, LD64, L, tid);
#pragma unroll
            for (int i = 0; i < Map64::MT; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = Map64::row(tid, i, 2 * h);
                    if (t >= nt) continue;
                    const float e = sc.e()[t];
                    float* yrow = a.y + ((z.n * a.T + t0 + t) * a.H + z.h) * P;
#pragma unroll
                    for (int j = 0; j < Map64::NT; ++j)
                        st2(yrow + Map64::col(tid, j, 0), __fmaf_rn(e, yi[i][j][2 * h], yy[i][j][2 * h]),
                            __fmaf_rn(e, yi[i][j][2 * h + 1], yy[i][j][2 * h + 1]));
                }
        }
        if (ch + 1 < z.ch1) {  // carry the state to the next chunk of the segment
            __syncthreads();
            for (int i = tid; i < L * P / 4; i += CT) {
                const int t = i / (P / 4), q = i - t * (P / 4);
                st4(sM + t * LD64 + 4 * q, mul4(ld4(sXd + t * LD64 + 4 * q), sc.w()[t]));
            }
            __syncthreads();
            state_step(sS, sM, sB, sc.g(), tid);
        }
    }
}

// ---------------------------------------------------------------------------------
// Backward 1, one chunk a segment: (diag(e) dY)^T C of chunk ch for HB heads into their dd
// slots, g into gvec.  Grid (nch, G nhb, N).
__global__ void __launch_bounds__(CT, 3) ssd_dprep_hb_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sC = sm;
    float* sYe = sC + T128;  // diag(e) dY
    const Scal sc{sYe + T64};
    const int tid = threadIdx.x;
    const Blk b = blk_of(a);
    prefetch_rows(a.dy, a, b.n, b.h0, b.t0, b.nt, tid);
    load_bc(sC, a.C, a, b.n, b.g, b.t0, b.nt, tid);
    for (int hh = 0; hh < a.HB; ++hh) {
        const long long h = b.h0 + hh;
        const long long slot = ((b.n * a.nch + b.ch) * a.H + h) * PS;
        __syncthreads();
        if (hh + 1 < a.HB) prefetch_rows(a.dy, a, b.n, h + 1, b.t0, b.nt, tid);
        load_scalars(a, b.n, h, b.t0, b.nt, sc, tid);
        __syncthreads();
        if (tid == 0) a.gvec[(b.n * a.nch + b.ch) * a.H + h] = sc.g();
        for (int i = tid; i < L * P / 4; i += CT) {
            const int t = i / (P / 4), q = i - t * (P / 4);
            st4(sYe + t * LD64 + 4 * q, mul4(head_row4(a.dy, a, b.n, h, b.t0, t, q, b.nt), sc.e()[t]));
        }
        __syncthreads();
        Acc128 acc;
        zero_mma<64, 128>(acc);
        block_mma<64, 128, true, false>(acc, sYe, LD64, sC, LD128, L, tid);
        store_acc128(a.dd + slot, acc, tid);
    }
}

// Backward 1, several chunks a segment: per chunk of a segment, (diag(e) dY)^T C into its dd
// slot and g into gvec, and the entry states of the segment's inner chunks (sin_all),
// replayed from the checkpoint by the forward's own step.  Grid (n_ck, H, N).
__global__ void __launch_bounds__(CT, 2) ssd_dprep_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sC = sm;
    float* sYe = sC + T128;  // diag(e) dY, then diag(w) Xd
    const Scal sc{sYe + T64};
    float* sB = sYe + T64 + NSCAL;  // m > 1 only
    float* sS = sB + T128;
    const int tid = threadIdx.x;
    const Seg z = seg_of(a);
    const bool replay = a.m > 1;
    if (replay) load_state(sS, a.ckpt_in + (z.head * a.n_ck + z.seg) * PS, tid);
    for (int ch = z.ch0; ch < z.ch1; ++ch) {
        const long long t0 = (long long)ch * L;
        const int nt = (int)min((long long)L, a.T - t0);
        const long long slot = ((z.n * a.nch + ch) * a.H + z.h) * PS;
        __syncthreads();
        if (replay && ch > z.ch0) store_state(a.sin_all + slot, sS, tid);
        load_scalars(a, z.n, z.h, t0, nt, sc, tid);
        __syncthreads();
        if (tid == 0) a.gvec[(z.n * a.nch + ch) * a.H + z.h] = sc.g();
        load_bc(sC, a.C, a, z.n, z.g, t0, nt, tid);
        for (int i = tid; i < L * P / 4; i += CT) {
            const int t = i / (P / 4), q = i - t * (P / 4);
            st4(sYe + t * LD64 + 4 * q, mul4(head_row4(a.dy, a, z.n, z.h, t0, t, q, nt), sc.e()[t]));
        }
        __syncthreads();
        Acc128 acc;
        zero_mma<64, 128>(acc);
        block_mma<64, 128, true, false>(acc, sYe, LD64, sC, LD128, L, tid);
        store_acc128(a.dd + slot, acc, tid);
        if (replay && ch + 1 < z.ch1) {
            __syncthreads();
            load_bc(sB, a.B, a, z.n, z.g, t0, nt, tid);
            load_xd(nullptr, sYe, a, z.n, z.h, t0, nt, sc, tid);
            __syncthreads();
            state_step(sS, sYe, sB, sc.g(), tid);
        }
    }
}

// Backward 2: dS_out of every chunk, last first, one float4 of one head's state a thread:
// dd's slot of chunk c holds (diag(e) dY)^T C and becomes dS_out(c); d_s = dS_in(0).  Grid
// (SLICES, H, N).
__global__ void __launch_bounds__(CT) ssd_dchain_kernel(const Args a)
{
    __shared__ float gs[CT];
    const int tid = threadIdx.x;
    const long long h = blockIdx.y, n = blockIdx.z, head = n * a.H + h;
    const long long off = 4LL * (blockIdx.x * CT + tid);
    auto slot = [&](int r) {  // r-th chunk from the end
        return a.dd + ((n * a.nch + (a.nch - 1 - r)) * a.H + h) * PS + off;
    };
    float4 d = ld4(a.dsT + head * PS + off);
    float4 buf[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) buf[k] = k < a.nch ? ld4(slot(k)) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < a.nch; base += CT) {
        __syncthreads();
        if (base + tid < a.nch) gs[tid] = a.gvec[(n * a.nch + (a.nch - 1 - base - tid)) * a.H + h];
        __syncthreads();
        const int nb = min(CT, a.nch - base);
        for (int k0 = 0; k0 < nb; k0 += 4) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (k0 + r < nb) {
                    const int rr = base + k0 + r;
                    const float4 x = buf[r];
                    if (rr + 4 < a.nch) buf[r] = ld4(slot(rr + 4));
                    st4(slot(rr), d);
                    d = fma4(gs[k0 + r], d, x);
                }
            }
        }
    }
    st4(a.ds0 + head * PS + off, d);
}

// Backward 3: every gradient of one chunk for HB heads of one group.  Grid (nch, G nhb, N),
// 16 warps (the products on a 4 x 4 warp grid: one CTA fits an SM, and twice the warps of the
// other kernels hide the latencies of its phases).  dx and ddt are complete per (chunk, head)
// and go straight out; dB and dC are summed over the block's heads in registers (ascending)
// and written as the block's partial.
__global__ void __launch_bounds__(GT, 1) ssd_grad_kernel(const Args a)
{
    extern __shared__ __align__(16) float sm[];
    float* sB = sm;
    float* sC = sB + T128;
    float* sSt = sC + T128;  // s_in, then dS_out (rows p)
    float* sQ = sSt + T128;  // C B^T
    float* sXd = sQ + T64;
    float* sXw = sXd + T64;  // diag(w) Xd
    float* sdY = sXw + T64;
    float* sM = sdY + T64;   // Lm (.) Q
    float* sdQ = sM + T64;   // Lm (.) dM
    float* sYe = sdQ + T64;  // diag(e) dY
    float* pRow = sYe + T64;      // [L][4] row sums of M (.) dM
    float* pCol = pRow + 4 * L;   // [L][4] column sums of M (.) dM
    float* pInt = pCol + 4 * L;   // [L][4] sum_p diag(e) dY (C s_in^T)
    float* pV = pInt + 4 * L;     // [L][4] sum_p Xd u
    float* pX = pV + 4 * L;       // [L][4] sum_p x dXd
    float* dc = pX + 4 * L;       // [L]
    float* red = dc + L;          // [16]
    const Scal sc{red + 16};
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ch = blockIdx.x;
    const long long n = blockIdx.z;
    const long long hpg = a.H / a.G;
    const long long g = blockIdx.y / a.nhb;
    const int hb = (int)(blockIdx.y - g * a.nhb);
    const long long h0 = g * hpg + (long long)hb * a.HB;
    const long long t0 = (long long)ch * L;
    const int nt = (int)min((long long)L, a.T - t0);
    const int gq = lane >> 2, tq = lane & 3;
    const int wr = G64::wr(tid), wc = G64::wc(tid);  // the same for both output shapes
    const int seg = ch / a.m;
    const bool at_ck = ch == seg * a.m;
    // A head's x, dy rows, s_in and dS_out into L2 ahead of their loads (the first head's now,
    // each next one's while the current one computes): 3 lines of 128 bytes a thread.
    auto prefetch_head = [&](long long h) {
        const long long slot = ((n * a.nch + ch) * a.H + h) * PS;
        prefetch_state(at_ck ? a.ckpt_in + ((n * a.H + h) * a.n_ck + seg) * PS : a.sin_all + slot, tid);
        prefetch_state(a.dd + slot, tid);
        prefetch_rows(a.x, a, n, h, t0, nt, tid);
        prefetch_rows(a.dy, a, n, h, t0, nt, tid);
    };
    prefetch_head(h0);

    load_bc<GT>(sB, a.B, a, n, g, t0, nt, tid);
    load_bc<GT>(sC, a.C, a, n, g, t0, nt, tid);
    __syncthreads();
    {  // Q = C B^T, shared by the block's heads
        GAcc64 q;
        zero_mma<64, 64, 4, 4>(q);
        block_mma<64, 64, false, true, 4, 4>(q, sC, LD128, sB, LD128, S, tid);
#pragma unroll
        for (int i = 0; i < G64::MT; ++i)
#pragma unroll
            for (int j = 0; j < G64::NT; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r) sQ[G64::row(tid, i, r) * LD64 + G64::col(tid, j, r)] = q[i][j][r];
    }
    GAcc128 accB, accC;
    zero_mma<64, 128, 4, 4>(accB);
    zero_mma<64, 128, 4, 4>(accC);

    for (int hh = 0; hh < a.HB; ++hh) {
        const long long h = h0 + hh;
        const long long head = n * a.H + h;
        const long long slot = ((n * a.nch + ch) * a.H + h) * PS;
        __syncthreads();  // the previous head's reads (tiles, scalars, partials) are done
        if (hh + 1 < a.HB) prefetch_head(h + 1);
        load_scalars(a, n, h, t0, nt, sc, tid);
        __syncthreads();
        for (int i = tid; i < L * P / 4; i += GT) {
            const int t = i / (P / 4), q = i - t * (P / 4);
            const float4 xd = mul4(head_row4(a.x, a, n, h, t0, t, q, nt), sc.dt()[t]);
            const float4 dy = head_row4(a.dy, a, n, h, t0, t, q, nt);
            st4(sXd + t * LD64 + 4 * q, xd);
            st4(sXw + t * LD64 + 4 * q, mul4(xd, sc.w()[t]));
            st4(sdY + t * LD64 + 4 * q, dy);
            st4(sYe + t * LD64 + 4 * q, mul4(dy, sc.e()[t]));
        }
        load_state<GT>(sSt, at_ck ? a.ckpt_in + (head * a.n_ck + seg) * PS : a.sin_all + slot, tid);
        __syncthreads();
        {  // with s_in: E = diag(e) dY s_in; dC += E, and sum_p diag(e) dY (C s_in^T) per row,
           // which is sum_j C (.) E
            GAcc128 E;
            zero_mma<64, 128, 4, 4>(E);
            block_mma<64, 128, false, false, 4, 4>(E, sYe, LD64, sSt, LD128, P, tid);
#pragma unroll
            for (int i = 0; i < G128::MT; ++i)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int t = G128::row(tid, i, 2 * hr);
                    float v = 0.f;
#pragma unroll
                    for (int j = 0; j < G128::NT; ++j)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = 2 * hr + e;
                            v = __fmaf_rn(sC[t * LD128 + G128::col(tid, j, r)], E[i][j][r], v);
                            accC[i][j][r] = __fadd_rn(accC[i][j][r], E[i][j][r]);
                        }
                    v = row_lanes(v);
                    if (tq == 0) pInt[t * 4 + wc] = v;
                }
        }
        __syncthreads();
        {  // dS_out over s_in, and <dS_out, s_in>
            const float* dso = a.dd + slot;
            float v = 0.f;
            for (int i = tid; i < PS / 4; i += GT) {
                const int p = i / (S / 4), q = i - p * (S / 4);
                float* x = sSt + p * LD128 + 4 * q;
                const float4 d = ld4(dso + p * S + 4 * q);
                v = dot4(d, ld4(x), v);
                st4(x, d);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red[warp] = v;
        }
        __syncthreads();
        GAcc64 u;  // B dS_out^T: rows tokens, columns channels
        {  // dM = dY Xd^T; M, dQ; the rows and columns of M (.) dM; u; sum_p Xd u
            GAcc64 dm;
            zero_mma<64, 64, 4, 4>(dm);
            zero_mma<64, 64, 4, 4>(u);
            block_mma<64, 64, false, true, 4, 4>(dm, sdY, LD64, sXd, LD64, P, tid);
            block_mma<64, 64, false, true, 4, 4>(u, sB, LD128, sSt, LD128, S, tid);
            const float* c = sc.c();
            float cs[G64::NT][2];
#pragma unroll
            for (int j = 0; j < G64::NT; ++j) cs[j][0] = cs[j][1] = 0.f;
#pragma unroll
            for (int i = 0; i < G64::MT; ++i)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int t = G64::row(tid, i, 2 * hr);
                    float rs = 0.f, vs = 0.f;
#pragma unroll
                    for (int j = 0; j < G64::NT; ++j)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = 2 * hr + e;
                            const int tau = G64::col(tid, j, r);
                            const float lm = tau <= t ? expf(__fsub_rn(c[t], c[tau])) : 0.f;
                            const float m = __fmul_rn(lm, sQ[t * LD64 + tau]);
                            sM[t * LD64 + tau] = m;
                            sdQ[t * LD64 + tau] = __fmul_rn(lm, dm[i][j][r]);
                            const float R = __fmul_rn(m, dm[i][j][r]);
                            rs = __fadd_rn(rs, R);
                            cs[j][e] = __fadd_rn(cs[j][e], R);
                            // u's row is token t here, its column channel tau
                            vs = __fmaf_rn(sXd[t * LD64 + tau], u[i][j][r], vs);
                        }
                    rs = row_lanes(rs);
                    vs = row_lanes(vs);
                    if (tq == 0) {
                        pRow[t * 4 + wc] = rs;
                        pV[t * 4 + wc] = vs;
                    }
                }
#pragma unroll
            for (int j = 0; j < G64::NT; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float v = col_lanes(cs[j][e]);
                    if (gq == 0) pCol[G64::col(tid, j, e) * 4 + wr] = v;
                }
        }
        __syncthreads();
        {  // dXd = M^T dY + diag(w) u; dx; sum_p x dXd
            GAcc64 dxd;
            zero_mma<64, 64, 4, 4>(dxd);
            block_mma<64, 64, true, false, 4, 4>(dxd, sM, LD64, sdY, LD64, L, tid);
#pragma unroll
            for (int i = 0; i < G64::MT; ++i)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int tau = G64::row(tid, i, 2 * hr);
                    const float w = sc.w()[tau], d = sc.dt()[tau];
                    float xs = 0.f;
                    const long long o = ((n * a.T + t0 + tau) * a.H + h) * P;
#pragma unroll
                    for (int j = 0; j < G64::NT; ++j) {
                        const int p = G64::col(tid, j, 0);
                        const float g0 = __fmaf_rn(w, u[i][j][2 * hr], dxd[i][j][2 * hr]);
                        const float g1 = __fmaf_rn(w, u[i][j][2 * hr + 1], dxd[i][j][2 * hr + 1]);
                        if (tau < nt) {
                            const float2 xv = *reinterpret_cast<const float2*>(a.x + o + p);
                            xs = __fmaf_rn(xv.y, g1, __fmaf_rn(xv.x, g0, xs));
                            st2(a.dx + o + p, __fmul_rn(d, g0), __fmul_rn(d, g1));
                        }
                    }
                    xs = row_lanes(xs);
                    if (tq == 0) pX[tau * 4 + wc] = xs;
                }
        }
        // dC += dQ B;  dB += dQ^T C + diag(w) Xd dS_out
        block_mma<64, 128, false, false, 4, 4>(accC, sdQ, LD64, sB, LD128, L, tid);
        block_mma<64, 128, true, false, 4, 4>(accB, sdQ, LD64, sC, LD128, L, tid);
        block_mma<64, 128, false, false, 4, 4>(accB, sXw, LD64, sSt, LD128, P, tid);
        __syncthreads();
        if (warp == 0) {  // dc, its reverse running sum, ddt
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int t = lane + 32 * k;
                const float* r4 = pRow + 4 * t;
                const float* i4 = pInt + 4 * t;
                const float* v4 = pV + 4 * t;
                const float* x4 = pX + 4 * t;
                const float rs = __fadd_rn(__fadd_rn(r4[0], r4[1]), __fadd_rn(r4[2], r4[3]));
                const float* c4 = pCol + 4 * t;
                const float cs = __fadd_rn(__fadd_rn(c4[0], c4[1]), __fadd_rn(c4[2], c4[3]));
                const float it = __fadd_rn(__fadd_rn(i4[0], i4[1]), __fadd_rn(i4[2], i4[3]));
                const float v = __fmul_rn(sc.w()[t], __fadd_rn(__fadd_rn(v4[0], v4[1]), __fadd_rn(v4[2], v4[3])));
                const float xs = __fadd_rn(__fadd_rn(x4[0], x4[1]), __fadd_rn(x4[2], x4[3]));
                dc[t] = __fsub_rn(__fadd_rn(__fsub_rn(rs, cs), it), v);
                pV[4 * t] = v;
                pX[4 * t] = xs;
            }
            __syncwarp();
            if (lane == 0) {
                float dot = 0.f, vt = 0.f;
                for (int k = 0; k < GT / 32; ++k) dot = __fadd_rn(dot, red[k]);
                for (int t = 0; t < L; ++t) vt = __fadd_rn(vt, pV[4 * t]);
                dc[L - 1] = __fadd_rn(dc[L - 1], __fmaf_rn(sc.g(), dot, vt));
                float run = 0.f;
                for (int t = L - 1; t >= 0; --t) {
                    run = __fadd_rn(run, dc[t]);
                    dc[t] = run;
                }
            }
            __syncwarp();
            const float A = a.A[h];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int t = lane + 32 * k;
                if (t < nt) a.ddt[(n * a.T + t0 + t) * a.H + h] = __fmaf_rn(A, dc[t], pX[4 * t]);
            }
        }
    }
    // this block's dB, dC partial: rows t < nt
    float* part = a.partBC + (long long)hb * 2 * S;
#pragma unroll
    for (int i = 0; i < G128::MT; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int t = G128::row(tid, i, 2 * hr);
            if (t >= nt) continue;
            float* row = part + ((n * a.T + t0 + t) * a.G + g) * (long long)a.nhb * 2 * S;
#pragma unroll
            for (int j = 0; j < G128::NT; ++j) {
                const int c = G128::col(tid, j, 0);
                st2(row + c, accB[i][j][2 * hr], accB[i][j][2 * hr + 1]);
                st2(row + S + c, accC[i][j][2 * hr], accC[i][j][2 * hr + 1]);
            }
        }
}

// Backward 4: dB, dC of each token: its group's block partials summed in ascending order.
__global__ void __launch_bounds__(256) ssd_reduce_kernel(const Args a)
{
    const long long tok = blockIdx.x;  // n T + t
    for (long long i = threadIdx.x; i < a.G * 2 * S; i += blockDim.x) {
        const long long g = i / (2 * S), c = i - g * 2 * S;
        const float* src = a.partBC + (tok * a.G + g) * (long long)a.nhb * 2 * S + c;
        float acc = 0.f;
        for (int b = 0; b < a.nhb; ++b) acc = __fadd_rn(acc, src[(long long)b * 2 * S]);
        if (c < S)
            a.dB[(tok * a.G + g) * S + c] = acc;
        else
            a.dC[(tok * a.G + g) * S + c - S] = acc;
    }
}

// ---------------------------------------------------------------------------------
// Host side.

constexpr size_t kSmemSegState = sizeof(float) * (T128 + T64 + NSCAL);
constexpr size_t kSmemOutput = sizeof(float) * (3 * T128 + 2 * T64 + NSCAL);
constexpr size_t kSmemOutputHb = sizeof(float) * (2 * T128 + 2 * T64 + NSCAL);
constexpr size_t kSmemDprep1 = sizeof(float) * (T128 + T64 + NSCAL);
constexpr size_t kSmemDprepR = sizeof(float) * (3 * T128 + T64 + NSCAL);
constexpr size_t kSmemGrad = sizeof(float) * (3 * T128 + 7 * T64 + 20 * L + L + 16 + NSCAL);
static_assert(kSmemGrad <= 232448, "the gradient kernel's shared memory");
static_assert(PS % (4 * CT) == 0, "state slices");

int heads_per_block(long long N, long long nch, long long H, long long G)
{
    const long long hpg = H / G;
    for (int hb = 4; hb >= 1; hb >>= 1)
        if (hpg % hb == 0 && N * nch * G * (hpg / hb) >= 3 * 152) return hb;
    return 1;
}

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

Workspace workspace_layout(long long N, long long T, long long H, long long G, int K, int HB)
{
    Workspace w{};
    const long long nch = (T + L - 1) / L;
    const long long nhb = (H / G) / HB;
    const size_t states = sizeof(float) * (size_t)(N * nch * H) * PS;
    size_t o = 0;
    w.dd = o;
    o += align256(states);
    w.sin_all = o;
    o += K > L ? align256(states) : 0;
    w.gvec = o;
    o += align256(sizeof(float) * (size_t)(N * nch * H));
    w.partBC = o;
    o += align256(sizeof(float) * (size_t)(N * T * G * nhb) * 2 * S);
    w.total = o;
    return w;
}

template <typename Kern>
static int launch(Kern kern, dim3 grid, size_t smem, const Args& a, cudaStream_t st, int threads = CT)
{
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
    }
    kern<<<grid, threads, smem, st>>>(a);
    return (int)cudaGetLastError();
}

int forward(const Args& a, cudaStream_t st)
{
    const unsigned H = (unsigned)a.H, N = (unsigned)a.N, nck = (unsigned)a.n_ck;
    const dim3 blk((unsigned)a.nch, (unsigned)(a.G * a.nhb), N);
    int e = a.m == 1 ? launch(ssd_state_hb_kernel, blk, kSmemSegState, a, st)
                     : launch(ssd_seg_state_kernel, dim3(nck, H, N), kSmemSegState, a, st);
    if (!e) e = launch(ssd_chain_kernel, dim3(SLICES, H, N), 0, a, st);
    if (!e)
        e = a.m == 1 ? launch(ssd_output_hb_kernel, blk, kSmemOutputHb, a, st)
                     : launch(ssd_output_kernel, dim3(nck, H, N), kSmemOutput, a, st);
    return e;
}

int backward(const Args& a, cudaStream_t st)
{
    const unsigned H = (unsigned)a.H, N = (unsigned)a.N, nck = (unsigned)a.n_ck;
    const dim3 blk((unsigned)a.nch, (unsigned)(a.G * a.nhb), N);
    int e = a.m == 1 ? launch(ssd_dprep_hb_kernel, blk, kSmemDprep1, a, st)
                     : launch(ssd_dprep_kernel, dim3(nck, H, N), kSmemDprepR, a, st);
    if (!e) e = launch(ssd_dchain_kernel, dim3(SLICES, H, N), 0, a, st);
    if (!e) e = launch(ssd_grad_kernel, blk, kSmemGrad, a, st, GT);
    if (!e) {
        ssd_reduce_kernel<<<(unsigned)(a.N * a.T), 256, 0, st>>>(a);
        e = (int)cudaGetLastError();
    }
    return e;
}

}  // namespace ssd
}  // namespace ssm
