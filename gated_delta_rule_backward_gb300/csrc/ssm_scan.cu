// ssm_scan.cu -- the selective scan (Mamba-1 / Mamba-2) and its reverse walk on sm_103a.
//
// "dillon-blake llama.cpp PR #26", SSM_SCAN_BACK section: a reverse recurrence carrying the
// state gradient from the last token to the first, five gradients packed like the forward's
// output, one decay per head (Mamba-2) or per state (Mamba-1), the final-state cotangent
// seeding the walk, states recomputed from checkpoints, heads folded into groups.
//
// Rows and columns.  The state of one sequence is a matrix with a row per (head, channel)
// pair, row = h P + p, and a column per state index j.  Every term of the recurrence is
// row-local except the outputs dB, dC (sums over the rows of a group) and ddt (a sum over
// the rows of a head), so a thread owns SL columns of one row (SL = 4 for up to 32 states,
// else 16), the NSL = S / SL threads of a row sit in adjacent lanes, a warp holds
// RPW = 32 / NSL rows and a CTA of W warps RPC = W RPW rows, all in one group.  The columns of
// lane ns are runs of four, j = 4 (ns + NSL q) + r (q < SL / 4, r < 4): the lanes of a row read
// a token's B and C, and a state row, as consecutive 16-byte units (no shared-memory bank
// conflicts, coalesced global accesses).  Row sums run over lanes with shuffles, over warps in shared
// memory (fixed order), and over a group's CTAs in ssm_reduce_kernel (fixed order); nothing
// uses atomics.
//
// The walk (one CTA per row block) takes the checkpoint segments of K tokens last first.
// Level 1 walks a segment forward from its checkpoint and drops a sub-checkpoint every kC2
// tokens into the workspace; level 2 recomputes each sub-segment's states into a shared-memory
// ring (last sub-segment first) and walks them in reverse.  The recompute runs the forward's
// own step, so every state is the forward's bit for bit and the results do not depend on K.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <string>

#include "../../include/ssm.h"
#include "ssm_chunk.h"
#include "ssm_diag.h"

namespace gdn {
void set_last_error(const char* msg);
}

namespace ssm {

constexpr int kC2 = 4;    // tokens per level-2 sub-segment (the ring)
constexpr int kTT = 32;   // tokens per tile of the forward

struct Args {
    const float *x, *dt, *A, *B, *C, *s0, *ckpt_in, *dy, *dsT;
    float *y, *sT, *ckpt, *ds0, *dx, *ddt, *dB, *dC;
    float *sub, *partBC, *partDt;
    long long N, T, H, P, S, G;
    int K, n_ck, per_state, RPC, nb_g, nb_h, nsub;
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Column of a thread's value e (e < SL) for lane slot ns: runs of four.
template <int NSL>
__device__ __forceinline__ int col_of(int ns, int e) { return 4 * (ns + NSL * (e >> 2)) + (e & 3); }

// A thread's SL values of a state row (row base `r`, 16-byte aligned) as float4 loads.
template <int NSL, int SL>
__device__ __forceinline__ void load_row16(float (&v)[SL], const float* r, int ns)
{
#pragma unroll
    for (int q = 0; q < SL / 4; ++q) {
        const float4 x = ld4(r + 4 * (ns + NSL * q));
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
}
template <int NSL, int SL>
__device__ __forceinline__ void store_row16(float* r, const float (&v)[SL], int ns)
{
#pragma unroll
    for (int q = 0; q < SL / 4; ++q) st4(r + 4 * (ns + NSL * q), make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
}
// A token's SL values of a row vector in shared memory (B or C), the same columns.
template <int NSL, int SL>
__device__ __forceinline__ void load_vec16(float (&v)[SL], const float* r, int ns)
{
    load_row16<NSL, SL>(v, r, ns);
}

// Sum of v over the NSL lanes of a row (lanes differ in their low bits).
template <int NSL>
__device__ __forceinline__ float row_sum(float v)
{
#pragma unroll
    for (int o = 1; o < NSL; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One token of the scan on a thread's SL columns: s = a s + B (x dt).
template <bool PS, int SL>
__device__ __forceinline__ void scan_step(float (&s)[SL], const float (&Bt)[SL], float xdt, float dtv,
                                          const float (&Av)[SL], float a_head)
{
#pragma unroll
    for (int e = 0; e < SL; ++e) {
        const float a = PS ? expf(__fmul_rn(dtv, Av[e])) : a_head;
        s[e] = __fmaf_rn(a, s[e], __fmul_rn(Bt[e], xdt));
    }
}

// ---------------------------------------------------------------------------------
// Forward: grid (row blocks, N), W warps.  Tiles of kTT tokens of B, C (the CTA's group), x
// (its rows), dt and (Mamba-2) a = exp(dt A) per head go to shared memory; y is staged and
// stored row-contiguously.
template <int NSL, int SL, bool PS>
__global__ void __launch_bounds__(256) ssm_fwd_kernel(const Args a)
{
    constexpr int RPW = 32 / NSL;
    const int W = blockDim.x >> 5, NT = blockDim.x, RPC = W * RPW;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ns = lane % NSL, lrow = warp * RPW + lane / NSL;
    const long long n = blockIdx.y, row0 = (long long)blockIdx.x * RPC, row = row0 + lrow;
    const long long P = a.P, S = a.S, H = a.H, T = a.T, G = a.G;
    const long long h = row / P, p = row % P;
    const long long h_lo = row0 / P;
    const int nh = (int)((row0 + RPC - 1) / P - h_lo + 1);
    const long long g = h_lo / (H / G);
    extern __shared__ __align__(16) float sm[];
    float* sB = sm;                          // [kTT][S]
    float* sC = sB + kTT * S;                // [kTT][S]
    float* sx = sC + kTT * S;                // [kTT][RPC]
    float* sy = sx + kTT * RPC;              // [kTT][RPC]
    float* sdt = sy + kTT * RPC;             // [kTT][nh]
    float* sa = sdt + kTT * nh;              // [kTT][nh]   (Mamba-2)

    float Av[SL];
#pragma unroll
    for (int e = 0; e < SL; ++e) Av[e] = PS ? a.A[h * S + col_of<NSL>(ns, e)] : a.A[h];
    float s[SL];
    load_row16<NSL, SL>(s, a.s0 + ((n * H + h) * P + p) * S, ns);
    float* ckr = a.ckpt + (((n * H + h) * a.n_ck) * P + p) * S;  // + k P S per checkpoint
    if (T == 0) store_row16<NSL, SL>(ckr, s, ns);
    int ck_next = 0;   // tokens to the next checkpoint
    int ck_i = 0;      // its index

    for (long long t0 = 0; t0 < T; t0 += kTT) {
        const int nt = (int)std::min<long long>(kTT, T - t0);
        __syncthreads();
        for (int i = tid; i < nt * (int)S / 4; i += NT) {
            const int tt = i / ((int)S / 4), c4 = i % ((int)S / 4);
            const long long base = ((n * T + t0 + tt) * G + g) * S + 4 * c4;
            st4(sB + tt * S + 4 * c4, ld4(a.B + base));
            st4(sC + tt * S + 4 * c4, ld4(a.C + base));
        }
        for (int i = tid; i < nt * RPC; i += NT) {
            const int tt = i / RPC, r = i % RPC;
            sx[i] = a.x[(n * T + t0 + tt) * H * P + row0 + r];
        }
        for (int i = tid; i < nt * nh; i += NT) {
            const int tt = i / nh, k = i % nh;
            const float dv = a.dt[(n * T + t0 + tt) * H + h_lo + k];
            sdt[i] = dv;
            if (!PS) sa[i] = expf(__fmul_rn(dv, a.A[h_lo + k]));
        }
        __syncthreads();
        const int hk = (int)(h - h_lo);
        const int Si = (int)S;
        for (int tt = 0; tt < nt; ++tt) {
            if (ck_next == 0) {
                store_row16<NSL, SL>(ckr + (long long)ck_i * P * S, s, ns);
                ck_next = a.K;
                ++ck_i;
            }
            --ck_next;
            const float dtv = sdt[tt * nh + hk];
            const float xdt = __fmul_rn(sx[tt * RPC + lrow], dtv);
            float Bt[SL], Ct[SL];
            load_vec16<NSL, SL>(Bt, sB + tt * Si, ns);
            load_vec16<NSL, SL>(Ct, sC + tt * Si, ns);
            scan_step<PS, SL>(s, Bt, xdt, dtv, Av, PS ? 0.f : sa[tt * nh + hk]);
            float y4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < SL; ++e) y4[e & 3] = __fmaf_rn(s[e], Ct[e], y4[e & 3]);
            float yp = __fadd_rn(__fadd_rn(y4[0], y4[1]), __fadd_rn(y4[2], y4[3]));
            yp = row_sum<NSL>(yp);
            if (ns == 0) sy[tt * RPC + lrow] = yp;
        }
        __syncthreads();
        for (int i = tid; i < nt * RPC; i += NT) {
            const int tt = i / RPC, r = i % RPC;
            a.y[(n * T + t0 + tt) * H * P + row0 + r] = sy[i];
        }
    }
    float* sTr = a.sT + ((n * H + h) * P + p) * S;  // (packed: 4-byte alignment only)
#pragma unroll
    for (int e = 0; e < SL; ++e) sTr[col_of<NSL>(ns, e)] = s[e];
}

// ---------------------------------------------------------------------------------
// The reverse walk: grid (row blocks, N), W warps.
//
// Its stages (a sub-segment's tokens of B, x, dt, and for level 2 also C and dy) run in a
// fixed order: for each segment, last first, level 1's sub-segments 0 .. nsub - 2, then level
// 2's nsub - 1 .. 0.  Each stage's inputs are copied into one of two shared-memory buffers by
// cp.async while the previous stage computes from the other.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem)
{
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Position in the walk's stage sequence.
struct Cursor {
    int seg, lvl, k;  // lvl 1: level 1 (k ascending); lvl 2: level 2 (k descending); seg < 0: done
};

template <int NSL, int SL, bool PS>
__global__ void __launch_bounds__(256) ssm_bwd_kernel(const Args a)
{
    constexpr int RPW = 32 / NSL;
    constexpr int NV = 2 * SL;            // dB and dC terms of a thread per token
    constexpr int NH = NV / RPW;          // of them, held per lane after the row reduce-scatter
    static_assert(NV >= RPW, "one term per lane at least");
    const int W = blockDim.x >> 5, NT = blockDim.x, RPC = W * RPW;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ns = lane % NSL, lrow = warp * RPW + lane / NSL;
    const long long n = blockIdx.y, row0 = (long long)blockIdx.x * RPC, row = row0 + lrow;
    const long long P = a.P, S = a.S, H = a.H, T = a.T, G = a.G, K = a.K;
    const long long h = row / P, p = row % P;
    const long long h_lo = row0 / P;
    const int nh = (int)((row0 + RPC - 1) / P - h_lo + 1);
    const long long g = h_lo / (H / G);
    const int hk = (int)(h - h_lo);
    const long long rows_g = (H / G) * P;
    const int bg = (int)((row0 % rows_g) / RPC);              // this CTA among its group's
    const int bh = P >= RPC ? (int)((row0 % P) / RPC) : 0;    // this CTA among its head's
    const int Si = (int)S;

    extern __shared__ __align__(16) float sm[];
    float* ring = sm;                                  // [kC2][SL / 4][NT] float4
    // warp partials of dB, dC: [kC2][W][2S + 2S / 64], column c at c + c / 64, so that the row
    // groups of a warp (whose terms sit 64 columns apart after the reduce-scatter) store to
    // distinct banks
    const int LB = 2 * Si + 2 * Si / 64;
    float* sbc = ring + kC2 * NT * SL;
    float* sdx = sbc + kC2 * W * LB;                   // [kC2][RPC]
    float* sdr = sdx + kC2 * RPC;                      // [kC2][RPC]  ddt row partials
    float* stg = sdr + kC2 * RPC;                      // two stage buffers, each:
    const int stage_floats = 2 * kC2 * Si + 2 * kC2 * RPC + ((kC2 * nh + 3) & ~3);
    //   [kC2][S] B, [kC2][S] C, [kC2][RPC] x, [kC2][RPC] dy, [kC2][nh] dt

    float Av[SL];
#pragma unroll
    for (int e = 0; e < SL; ++e) Av[e] = PS ? a.A[h * S + col_of<NSL>(ns, e)] : a.A[h];
    const float A_head = PS ? 0.f : a.A[h];
    float ds[SL];
    {
        const float* d = a.dsT + ((n * H + h) * P + p) * S;  // (packed: scalar loads)
#pragma unroll
        for (int e = 0; e < SL; ++e) ds[e] = d[col_of<NSL>(ns, e)];
    }
    // sub-checkpoint k of this thread: float4 q at subr + 4 ((SL / 4 k + q) NT)
    constexpr int Q = SL / 4;
    float* subr = a.sub + ((long long)blockIdx.y * gridDim.x + blockIdx.x) * a.nsub * NT * SL + 4 * tid;
    auto put4 = [&](float* base, int k, const float (&v)[SL]) {
#pragma unroll
        for (int q = 0; q < Q; ++q)
            st4(base + 4 * ((Q * k + q) * NT), make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
    };
    auto get4 = [&](float (&v)[SL], const float* base, int k) {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const float4 x = ld4(base + 4 * ((Q * k + q) * NT));
            v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
        }
    };
    float* ringr = ring + 4 * tid;

    auto seg_t0 = [&](int seg) { return (long long)seg * K; };
    auto seg_t1 = [&](int seg) { return std::min<long long>(T, (long long)seg * K + K); };
    auto seg_nsub = [&](int seg) { return (int)((seg_t1(seg) - seg_t0(seg) + kC2 - 1) / kC2); };
    auto seg_start = [&](int seg) {  // the first stage of segment seg (or of an earlier one)
        for (; seg >= 0; --seg) {
            if (seg_t1(seg) <= seg_t0(seg)) continue;
            const int ns_ = seg_nsub(seg);
            return ns_ > 1 ? Cursor{seg, 1, 0} : Cursor{seg, 2, 0};
        }
        return Cursor{-1, 0, 0};
    };
    auto advance = [&](Cursor c) {
        const int ns_ = seg_nsub(c.seg);
        if (c.lvl == 1) return c.k + 1 < ns_ - 1 ? Cursor{c.seg, 1, c.k + 1} : Cursor{c.seg, 2, ns_ - 1};
        if (c.k > 0) return Cursor{c.seg, 2, c.k - 1};
        return seg_start(c.seg - 1);
    };
    // copies of stage c's inputs into buffer `buf`
    auto issue = [&](Cursor c, int buf) {
        float* b = stg + buf * stage_floats;
        const long long ts = seg_t0(c.seg) + (long long)c.k * kC2;
        const int nt = (int)std::min<long long>(kC2, seg_t1(c.seg) - ts);
        const bool all = c.lvl == 2;
        const float* Bb = a.B + ((n * T + ts) * G + g) * S;
        const float* Cb = a.C + ((n * T + ts) * G + g) * S;
        const int S4 = Si / 4, GS = (int)(G * S);
        for (int i = tid; i < nt * S4; i += NT) {
            const int tt = i / S4, c4 = i - tt * S4;
            cp_async16(b + tt * Si + 4 * c4, Bb + tt * GS + 4 * c4);
            if (all) cp_async16(b + kC2 * Si + tt * Si + 4 * c4, Cb + tt * GS + 4 * c4);
        }
        const float* xb = a.x + (n * T + ts) * H * P + row0;
        const float* yb = a.dy + (n * T + ts) * H * P + row0;
        const int HP = (int)(H * P);
        float* bx = b + 2 * kC2 * Si;
        for (int i = tid; i < nt * RPC; i += NT) {
            const int tt = i / RPC, r = i - tt * RPC;
            cp_async4(bx + i, xb + tt * HP + r);
            if (all) cp_async4(bx + kC2 * RPC + i, yb + tt * HP + r);
        }
        const float* db = a.dt + (n * T + ts) * H + h_lo;
        float* bd = bx + 2 * kC2 * RPC;
        for (int i = tid; i < nt * nh; i += NT) {
            const int tt = i / nh, k = i - tt * nh;
            cp_async4(bd + i, db + tt * (int)H + k);
        }
        cp_async_commit();
    };

    Cursor c = seg_start(a.n_ck - 1);
    if (c.seg >= 0) issue(c, 0);
    int buf = 0;
    float s[SL];
    while (c.seg >= 0) {
        const Cursor nx = advance(c);
        cp_async_wait_all();
        __syncthreads();                   // stage c has landed; every thread is done with buf ^ 1
        if (nx.seg >= 0) issue(nx, buf ^ 1);
        const float* b = stg + buf * stage_floats;
        const float* sB = b;
        const float* sC = b + kC2 * Si;
        const float* sx = b + 2 * kC2 * Si;
        const float* sdy = sx + kC2 * RPC;
        const float* sdt = sdy + kC2 * RPC;
        const long long t0 = seg_t0(c.seg), t1 = seg_t1(c.seg);
        const int nsub = seg_nsub(c.seg);
        const long long ts = t0 + (long long)c.k * kC2;
        const int nt = (int)std::min<long long>(kC2, t1 - ts);
        if (c.lvl == 1) {
            // level 1: the segment forward from its checkpoint; a sub-checkpoint every kC2 tokens
            if (c.k == 0) load_row16<NSL, SL>(s, a.ckpt_in + (((n * H + h) * a.n_ck + c.seg) * P + p) * S, ns);
            put4(subr, c.k, s);
            for (int tt = 0; tt < nt; ++tt) {
                const float dtv = sdt[tt * nh + hk];
                float Bt[SL];
                load_vec16<NSL, SL>(Bt, sB + tt * Si, ns);
                scan_step<PS, SL>(s, Bt, __fmul_rn(sx[tt * RPC + lrow], dtv), dtv, Av,
                                  PS ? 0.f : expf(__fmul_rn(dtv, A_head)));
            }
            if (c.k + 1 == nsub - 1) put4(subr, c.k + 1, s);
        } else {
            // level 2: the sub-segment's states into the ring, then its tokens in reverse
            if (nsub == 1)
                load_row16<NSL, SL>(s, a.ckpt_in + (((n * H + h) * a.n_ck + c.seg) * P + p) * S, ns);
            else
                get4(s, subr, c.k);
            for (int tt = 0; tt < nt; ++tt) {  // ring slot tt: the state entering token ts + tt
                put4(ringr, tt, s);
                const float dtv = sdt[tt * nh + hk];
                float Bt[SL];
                load_vec16<NSL, SL>(Bt, sB + tt * Si, ns);
                scan_step<PS, SL>(s, Bt, __fmul_rn(sx[tt * RPC + lrow], dtv), dtv, Av,
                                  PS ? 0.f : expf(__fmul_rn(dtv, A_head)));
            }
            // s is now the state after the sub-segment's last token
            for (int tt = nt - 1; tt >= 0; --tt) {
                float sp[SL];  // the state entering the token
                get4(sp, ringr, tt);
                const float dtv = sdt[tt * nh + hk];
                const float a_head = PS ? 0.f : expf(__fmul_rn(dtv, A_head));
                const float xv = sx[tt * RPC + lrow], dyv = sdy[tt * RPC + lrow];
                const float xdt = __fmul_rn(xv, dtv);
                float Bt[SL], Ct[SL];
                load_vec16<NSL, SL>(Bt, sB + tt * Si, ns);
                load_vec16<NSL, SL>(Ct, sC + tt * Si, ns);
                float v[NV];
                float dxp = 0.f, ddtp = 0.f;
#pragma unroll
                for (int e = 0; e < SL; ++e) {
                    const float av = PS ? expf(__fmul_rn(dtv, Av[e])) : a_head;
                    ds[e] = __fmaf_rn(dyv, Ct[e], ds[e]);             // the output term
                    v[SL + e] = __fmul_rn(dyv, s[e]);                 // dC term (s = s_t)
                    v[e] = __fmul_rn(ds[e], xdt);                     // dB term
                    dxp = __fmaf_rn(ds[e], Bt[e], dxp);
                    // d(dt): the write B x and the decay A a s_{t-1}
                    ddtp = __fmaf_rn(ds[e], __fmaf_rn(__fmul_rn(Av[e], av), sp[e], __fmul_rn(Bt[e], xv)), ddtp);
                    ds[e] = __fmul_rn(av, ds[e]);                     // carried to s_{t-1}
                    s[e] = sp[e];
                }
                dxp = row_sum<NSL>(dxp);
                ddtp = row_sum<NSL>(ddtp);
                if (ns == 0) {
                    sdx[tt * RPC + lrow] = __fmul_rn(dxp, dtv);
                    sdr[tt * RPC + lrow] = ddtp;
                }
                // dB, dC terms summed over the warp's rows (lanes differing in their high bits):
                // recursive halving leaves each lane NH of them, starting at index `base`
                int base = 0;
#pragma unroll
                for (int o = 16, m = NV / 2; o >= NSL; o >>= 1, m >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < m; ++i) {
                        const float send = up ? v[i] : v[i + m];
                        const float keep = up ? v[i + m] : v[i];
                        v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
                    }
                    base += up ? m : 0;
                }
                float* wp = sbc + (tt * W + warp) * LB;
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                    const int idx = base + i;
                    const int cc = idx < SL ? col_of<NSL>(ns, idx) : Si + col_of<NSL>(ns, idx - SL);
                    wp[cc + (cc >> 6)] = v[i];
                }
            }
            __syncthreads();
            // this sub-segment's per-token sums: dB, dC over the warps, ddt over rows, dx
            float* pbc = a.partBC + (((n * T + ts) * G + g) * a.nb_g + bg) * 2 * S;
            const long long pstride = G * a.nb_g * 2 * S;  // one token further
            for (int i = tid; i < nt * 2 * Si; i += NT) {
                const int tt = i / (2 * Si), cc = i - tt * 2 * Si;
                float acc = 0.f;
                for (int w = 0; w < W; ++w) acc = __fadd_rn(acc, sbc[(tt * W + w) * LB + cc + (cc >> 6)]);
                pbc[tt * pstride + cc] = acc;
            }
            if (P >= RPC) {
                for (int tt = tid; tt < nt; tt += NT) {
                    float acc = 0.f;
                    for (int r = 0; r < RPC; ++r) acc = __fadd_rn(acc, sdr[tt * RPC + r]);
                    a.partDt[((n * T + ts + tt) * H + h_lo) * a.nb_h + bh] = acc;
                }
            } else {
                for (int i = tid; i < nt * nh; i += NT) {
                    const int tt = i / nh, k2 = i % nh;
                    float acc = 0.f;
                    for (int r = 0; r < (int)P; ++r) acc = __fadd_rn(acc, sdr[tt * RPC + k2 * (int)P + r]);
                    a.partDt[((n * T + ts + tt) * H + h_lo + k2) * a.nb_h] = acc;
                }
            }
            const long long dxo = (n * T + ts) * H * P + row0;
            for (int i = tid; i < nt * RPC; i += NT) {
                const int tt = i / RPC, r = i % RPC;
                a.dx[dxo + (long long)tt * H * P + r] = sdx[i];
            }
        }
        c = nx;
        buf ^= 1;
    }
    cp_async_wait_all();
    store_row16<NSL, SL>(a.ds0 + ((n * H + h) * P + p) * S, ds, ns);
}

// dB, dC: each group's CTA partials summed in ascending order; ddt: each head's.
__global__ void __launch_bounds__(256) ssm_reduce_kernel(const Args a)
{
    const long long G = a.G, S = a.S, H = a.H;
    const long long tok = blockIdx.x;  // n T + t
    for (long long i = threadIdx.x; i < G * 2 * S; i += blockDim.x) {
        const long long g = i / (2 * S), c = i % (2 * S);
        float acc = 0.f;
        const float* src = a.partBC + ((tok * G + g) * a.nb_g) * 2 * S + c;
        for (int b = 0; b < a.nb_g; ++b) acc = __fadd_rn(acc, src[(long long)b * 2 * S]);
        if (c < S)
            a.dB[(tok * G + g) * S + c] = acc;
        else
            a.dC[(tok * G + g) * S + c - S] = acc;
    }
    for (long long hh = threadIdx.x; hh < H; hh += blockDim.x) {
        float acc = 0.f;
        for (int b = 0; b < a.nb_h; ++b) acc = __fadd_rn(acc, a.partDt[(tok * H + hh) * a.nb_h + b]);
        a.ddt[tok * H + hh] = acc;
    }
}

// ---------------------------------------------------------------------------------
// Host side.

struct Plan {
    long long N, T, H, P, S, G, K, n_ck;
    int per_state, SL, NSL, RPW, W, RPC, nb_g, nb_h, nsub, ctas;
    bool chunked;  // the chunked form (ssm_chunk.cu) runs
    int HB, nch;   // its heads per gradient CTA and chunks per sequence
    bool diag;     // the segmented form for a decay per state (ssm_diag.cu) runs
};

// The chunked form takes one decay per head, 64 channels and 128 states (the Mamba-2 layer's
// head), at least one token and checkpoints on chunk boundaries.
static bool chunked_shape(const ssm_params_t* p)
{
    return p->a_per_state == 0 && p->P == ssd::kP && p->S == ssd::kS && p->T >= 1;
}

// States per thread: 4 up to 32 states (a Mamba-1 layer has 16: four times the threads, the
// rows being few), else 16.
static int states_per_thread(long long S) { return S <= 32 ? 4 : 16; }

static int plan_of(const ssm_params_t* p, Plan& pl, std::string& why)
{
    if (!p) {
        why = "NULL params";
        return GDN_ERR_INVALID_ARG;
    }
    if (p->N < 0 || p->T < 0 || p->H < 1 || p->P < 1 || p->S < 1 || p->G < 1 || p->K < 0 ||
        p->reserved0 != 0 || p->reserved1 != 0 || (p->a_per_state != 0 && p->a_per_state != 1)) {
        why = "sizes: N, T >= 0; H, P, S, G >= 1; K >= 0; a_per_state 0 or 1; reserved fields 0";
        return GDN_ERR_INVALID_ARG;
    }
    if (p->H % p->G) {
        why = "H must be a multiple of G";
        return GDN_ERR_INVALID_ARG;
    }
    pl.N = p->N; pl.T = p->T; pl.H = p->H; pl.P = p->P; pl.S = p->S; pl.G = p->G;
    pl.per_state = p->a_per_state;
    pl.K = p->K > 0 ? p->K : (p->T > 1 ? (long long)std::ceil(std::sqrt((double)p->T)) : 1);
    if (p->K == 0 && chunked_shape(p)) pl.K = (pl.K + ssd::kChunk - 1) / ssd::kChunk * ssd::kChunk;
    pl.chunked = chunked_shape(p) && pl.K % ssd::kChunk == 0;
    pl.nch = (int)((pl.T + ssd::kChunk - 1) / ssd::kChunk);
    pl.HB = pl.chunked ? ssd::heads_per_block(pl.N, pl.nch, pl.H, pl.G) : 1;
    pl.n_ck = p->T <= 0 ? 1 : (p->T + pl.K - 1) / pl.K;
    // a decay per state, one channel a head, 16 states, whole blocks of 16 channels in a group,
    // and the segment decays' scratch (16 floats a segment and channel) inside y
    pl.diag = p->a_per_state == 1 && p->P == 1 && p->S == diag::kS && p->T >= 1 && (p->H / p->G) % 16 == 0 &&
              p->H % p->G == 0 && pl.n_ck * diag::kS <= p->T;
    if (pl.S != 16 && pl.S != 32 && pl.S != 64 && pl.S != 128 && pl.S != 256) {
        why = "S (d_state) must be 16, 32, 64, 128 or 256";
        return GDN_ERR_UNSUPPORTED;
    }
    pl.SL = states_per_thread(pl.S);
    pl.NSL = (int)(pl.S / pl.SL);
    pl.RPW = 32 / pl.NSL;
    const long long rows = pl.H * pl.P, rows_g = (pl.H / pl.G) * pl.P;
    // the largest CTA (up to 8 warps) whose rows lie in one group and cover whole heads or
    // part of one, among those that still give every SM two blocks; else the smallest such
    // CTA.  (Two blocks an SM rather than one: the Mamba-2 layer's walk 8.06 -> 7.54 ms at twice
    // the dB/dC partials in the workspace, 0.72 -> 1.39 GB.)
    pl.W = 0;
    for (int W = 8; W >= 1; W >>= 1) {
        const long long R = (long long)W * pl.RPW;
        if (rows_g % R != 0 || !(pl.P % R == 0 || R % pl.P == 0)) continue;
        pl.W = W;
        if (rows / R >= 2 * 152) break;
    }
    if (pl.W == 0) {
        why = "the channels of a group (H / G * P) must be a multiple of " + std::to_string(pl.RPW) +
              " and P a multiple or a divisor of the rows of a block";
        return GDN_ERR_UNSUPPORTED;
    }
    pl.RPC = pl.W * pl.RPW;
    pl.nb_g = (int)(rows_g / pl.RPC);
    pl.nb_h = pl.P >= pl.RPC ? (int)(pl.P / pl.RPC) : 1;
    pl.nsub = (int)((pl.K + kC2 - 1) / kC2);
    pl.ctas = (int)(rows / pl.RPC);
    return GDN_OK;
}

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

struct WsLayout {
    size_t sub, partBC, partDt, total;
};

static WsLayout ws_layout(const Plan& pl)
{
    WsLayout w{};
    if (pl.chunked) {
        w.total = ssd::workspace_layout(pl.N, pl.T, pl.H, pl.G, (int)pl.K, pl.HB).total;
        return w;
    }
    if (pl.diag) {
        w.total = diag::workspace_layout(pl.N, pl.T, pl.H, pl.G, (int)pl.K).total;
        return w;
    }
    size_t o = 0;
    w.sub = o;
    o += align256(sizeof(float) * (size_t)pl.N * pl.ctas * pl.nsub * (32 * pl.W) * pl.SL);
    w.partBC = o;
    o += align256(sizeof(float) * (size_t)pl.N * pl.T * pl.G * pl.nb_g * 2 * pl.S);
    w.partDt = o;
    o += align256(sizeof(float) * (size_t)pl.N * pl.T * pl.H * pl.nb_h);
    w.total = o;
    return w;
}

static size_t fwd_smem(const Plan& pl)
{
    const long long nh = pl.P >= pl.RPC ? 1 : pl.RPC / pl.P;
    return sizeof(float) * (size_t)(2 * kTT * pl.S + 2 * kTT * pl.RPC + 2 * kTT * nh);
}

static size_t bwd_smem(const Plan& pl)
{
    const long long nh = pl.P >= pl.RPC ? 1 : pl.RPC / pl.P;
    const long long NT = 32LL * pl.W;
    const long long stage = 2 * kC2 * pl.S + 2 * kC2 * pl.RPC + ((kC2 * nh + 3) & ~3LL);
    const long long LB = 2 * pl.S + 2 * pl.S / 64;
    return sizeof(float) * (size_t)(kC2 * NT * pl.SL + (long long)kC2 * pl.W * LB + 2 * kC2 * pl.RPC + 2 * stage);
}

static bool aligned16(const void* q) { return ((uintptr_t)q & 15) == 0; }

static bool overlap(const void* a, size_t an, const void* b, size_t bn)
{
    const char *x = (const char*)a, *y = (const char*)b;
    return an && bn && x < y + bn && y < x + an;
}

template <bool FWD, int NSL, int SL, bool PS>
static int launch_t(const Args& a, const Plan& pl, cudaStream_t st)
{
    const size_t smem = FWD ? fwd_smem(pl) : bwd_smem(pl);
    auto kern = FWD ? ssm_fwd_kernel<NSL, SL, PS> : ssm_bwd_kernel<NSL, SL, PS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    kern<<<dim3(pl.ctas, (unsigned)pl.N), 32 * pl.W, smem, st>>>(a);
    return (int)cudaGetLastError();
}

template <bool FWD>
static int launch(const Args& a, const Plan& pl, cudaStream_t st)
{
#define SSM_CASE(NN, LL)                                                                      \
    if (pl.NSL == NN && pl.SL == LL)                                                          \
        return pl.per_state ? launch_t<FWD, NN, LL, true>(a, pl, st) : launch_t<FWD, NN, LL, false>(a, pl, st);
    SSM_CASE(4, 4)    // 16 states
    SSM_CASE(8, 4)    // 32
    SSM_CASE(4, 16)   // 64
    SSM_CASE(8, 16)   // 128
    SSM_CASE(16, 16)  // 256
    SSM_CASE(8, 8)    // 64 at 8 states a thread
    SSM_CASE(16, 8)   // 128 at 8 states a thread
#undef SSM_CASE
    return (int)cudaErrorInvalidValue;
}

static ssd::Args chunk_args(const Plan& pl)
{
    ssd::Args c{};
    c.N = pl.N; c.T = pl.T; c.H = pl.H; c.G = pl.G;
    c.K = (int)pl.K; c.n_ck = (int)pl.n_ck; c.nch = pl.nch; c.m = (int)(pl.K / ssd::kChunk);
    c.HB = pl.HB; c.nhb = (int)(pl.H / pl.G / pl.HB);
    return c;
}

static diag::Args diag_args(const Plan& pl)
{
    diag::Args c{};
    c.N = pl.N; c.T = pl.T; c.H = pl.H; c.G = pl.G;
    c.K = (int)pl.K; c.n_ck = (int)pl.n_ck; c.spk = (int)((pl.K + diag::kSB - 1) / diag::kSB);
    c.nsb = c.n_ck * c.spk; c.nbg = (int)(pl.H / pl.G / 16);
    return c;
}

static int fail(int code, const std::string& msg)
{
    gdn::set_last_error(msg.c_str());
    return code;
}

}  // namespace ssm

using namespace ssm;

extern "C" int64_t ssm_checkpoint_interval(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    if (!p || p->T < 0) return 1;
    if (plan_of(p, pl, why) != GDN_OK) return p->K > 0 ? p->K : (p->T > 1 ? (int64_t)std::ceil(std::sqrt((double)p->T)) : 1);
    return pl.K;
}

extern "C" int64_t ssm_num_checkpoints(const ssm_params_t* p)
{
    const int64_t K = ssm_checkpoint_interval(p);
    return (!p || p->T <= 0) ? 1 : (p->T + K - 1) / K;
}

extern "C" size_t ssm_packed_out_elems(const ssm_params_t* p)
{
    if (!p) return 0;
    return (size_t)(p->N * p->T * p->H * p->P + p->N * p->H * p->P * p->S);
}

extern "C" size_t ssm_packed_grad_elems(const ssm_params_t* p)
{
    if (!p) return 0;
    return (size_t)(p->N * p->H * p->P * p->S + p->N * p->T * p->H * p->P + p->N * p->T * p->H +
                    2 * p->N * p->T * p->G * p->S);
}

extern "C" size_t ssm_backward_workspace_bytes(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    if (plan_of(p, pl, why) != GDN_OK) return 0;
    return ws_layout(pl).total;
}

extern "C" int ssm_supported(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    const int e = plan_of(p, pl, why);
    if (e) gdn::set_last_error(why.c_str());
    return e;
}

extern "C" int ssm_chunked(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    return plan_of(p, pl, why) == GDN_OK && pl.chunked ? 1 : 0;
}

extern "C" int ssm_form(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    if (plan_of(p, pl, why) != GDN_OK) return -1;
    return pl.chunked ? 1 : pl.diag ? 2 : 0;
}

extern "C" int ssm_forward_launches(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    if (plan_of(p, pl, why) != GDN_OK || pl.N == 0) return 0;
    return pl.chunked || pl.diag ? 3 : 1;
}

extern "C" int ssm_backward_launches(const ssm_params_t* p)
{
    Plan pl{};
    std::string why;
    if (plan_of(p, pl, why) != GDN_OK || pl.N == 0 || pl.T == 0) return 0;
    return pl.chunked || pl.diag ? 4 : 2;
}

extern "C" int ssm_forward(const ssm_params_t* p, const float* s0, const float* x, const float* dt, const float* A,
                           const float* B, const float* C, float* out_packed, float* ckpt, void* stream)
{
    Plan pl{};
    std::string why;
    int e = plan_of(p, pl, why);
    if (e) return fail(e, why);
    if (pl.N == 0) return GDN_OK;
    const size_t fl = sizeof(float);
    const size_t n_s = (size_t)(pl.N * pl.H * pl.P * pl.S), n_x = (size_t)(pl.N * pl.T * pl.H * pl.P);
    const size_t n_dt = (size_t)(pl.N * pl.T * pl.H), n_bc = (size_t)(pl.N * pl.T * pl.G * pl.S);
    const size_t n_a = (size_t)(pl.per_state ? pl.H * pl.S : pl.H), n_ck = (size_t)(pl.N * pl.H * pl.n_ck * pl.P * pl.S);
    const bool need_t = pl.T > 0;
    if (!s0 || !A || !out_packed || !ckpt || (need_t && (!x || !dt || !B || !C)))
        return fail(GDN_ERR_INVALID_ARG, "ssm_forward: NULL pointer");
    const void* ins[] = {s0, x, dt, A, B, C, out_packed, ckpt};
    for (const void* q : ins)
        if (q && !aligned16(q)) return fail(GDN_ERR_INVALID_ARG, "ssm_forward: pointers must be 16-byte aligned");
    const std::pair<const void*, size_t> in[] = {{s0, n_s}, {x, n_x}, {dt, n_dt}, {A, n_a}, {B, n_bc}, {C, n_bc}};
    const std::pair<const void*, size_t> out[] = {{out_packed, n_x + n_s}, {ckpt, n_ck}};
    for (auto& o : out) {
        for (auto& i : in)
            if (i.first && overlap(o.first, o.second * fl, i.first, i.second * fl))
                return fail(GDN_ERR_ALIAS, "ssm_forward: an output overlaps an input");
    }
    if (overlap(out_packed, (n_x + n_s) * fl, ckpt, n_ck * fl)) return fail(GDN_ERR_ALIAS, "ssm_forward: outputs overlap");
    Args a{};
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.s0 = s0;
    a.y = out_packed;
    a.sT = out_packed + n_x;
    a.ckpt = ckpt;
    a.N = pl.N; a.T = pl.T; a.H = pl.H; a.P = pl.P; a.S = pl.S; a.G = pl.G;
    a.K = (int)pl.K; a.n_ck = (int)pl.n_ck; a.per_state = pl.per_state; a.RPC = pl.RPC;
    if (pl.chunked) {
        ssd::Args c = chunk_args(pl);
        c.x = x; c.dt = dt; c.A = A; c.B = B; c.C = C; c.s0 = s0;
        c.y = a.y; c.sT = a.sT; c.ckpt = ckpt;
        e = ssd::forward(c, (cudaStream_t)stream);
    } else if (pl.diag) {
        diag::Args c = diag_args(pl);
        c.x = x; c.dt = dt; c.A = A; c.B = B; c.C = C; c.s0 = s0;
        c.y = a.y; c.sT = a.sT; c.ckpt = ckpt;
        e = diag::forward(c, (cudaStream_t)stream);
    } else {
        e = launch<true>(a, pl, (cudaStream_t)stream);
    }
    if (e) return fail(GDN_ERR_CUDA, std::string("ssm_forward: ") + cudaGetErrorString((cudaError_t)e));
    return GDN_OK;
}

extern "C" int ssm_backward(const ssm_params_t* p, const float* x, const float* dt, const float* A, const float* B,
                            const float* C, const float* ckpt, const float* grad_in, float* grad_out, void* workspace,
                            size_t workspace_bytes, void* stream)
{
    Plan pl{};
    std::string why;
    int e = plan_of(p, pl, why);
    if (e) return fail(e, why);
    if (pl.N == 0) return GDN_OK;
    const size_t fl = sizeof(float);
    const size_t n_s = (size_t)(pl.N * pl.H * pl.P * pl.S), n_x = (size_t)(pl.N * pl.T * pl.H * pl.P);
    const size_t n_dt = (size_t)(pl.N * pl.T * pl.H), n_bc = (size_t)(pl.N * pl.T * pl.G * pl.S);
    const size_t n_a = (size_t)(pl.per_state ? pl.H * pl.S : pl.H), n_ck = (size_t)(pl.N * pl.H * pl.n_ck * pl.P * pl.S);
    const WsLayout w = ws_layout(pl);
    const bool need_t = pl.T > 0;
    if (!A || !ckpt || !grad_in || !grad_out || (need_t && (!x || !dt || !B || !C || !workspace)))
        return fail(GDN_ERR_INVALID_ARG, "ssm_backward: NULL pointer");
    const void* ptrs[] = {x, dt, A, B, C, ckpt, grad_in, grad_out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return fail(GDN_ERR_INVALID_ARG, "ssm_backward: pointers must be 16-byte aligned");
    if (need_t && workspace_bytes < w.total)
        return fail(GDN_ERR_WORKSPACE, "ssm_backward: workspace smaller than ssm_backward_workspace_bytes()");
    const size_t n_go = n_s + n_x + n_dt + 2 * n_bc;
    const std::pair<const void*, size_t> in[] = {{x, n_x}, {dt, n_dt}, {A, n_a}, {B, n_bc}, {C, n_bc},
                                                 {ckpt, n_ck}, {grad_in, n_x + n_s}};
    for (auto& i : in) {
        if (i.first && overlap(grad_out, n_go * fl, i.first, i.second * fl))
            return fail(GDN_ERR_ALIAS, "ssm_backward: the output overlaps an input");
        if (need_t && i.first && overlap(workspace, w.total, i.first, i.second * fl))
            return fail(GDN_ERR_ALIAS, "ssm_backward: the workspace overlaps an input");
    }
    if (need_t && overlap(workspace, w.total, grad_out, n_go * fl))
        return fail(GDN_ERR_ALIAS, "ssm_backward: the workspace overlaps the output");
    cudaStream_t st = (cudaStream_t)stream;
    float* go = grad_out;
    Args a{};
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.ckpt_in = ckpt;
    a.dy = grad_in;
    a.dsT = grad_in + n_x;
    a.ds0 = go;
    a.dx = go + n_s;
    a.ddt = go + n_s + n_x;
    a.dB = go + n_s + n_x + n_dt;
    a.dC = go + n_s + n_x + n_dt + n_bc;
    a.N = pl.N; a.T = pl.T; a.H = pl.H; a.P = pl.P; a.S = pl.S; a.G = pl.G;
    a.K = (int)pl.K; a.n_ck = (int)pl.n_ck; a.per_state = pl.per_state; a.RPC = pl.RPC;
    a.nb_g = pl.nb_g; a.nb_h = pl.nb_h; a.nsub = pl.nsub;
    if (!need_t) {  // no tokens: d_s is the final-state cotangent
        e = (int)cudaMemcpyAsync(go, a.dsT, n_s * fl, cudaMemcpyDeviceToDevice, st);
        if (e) return fail(GDN_ERR_CUDA, std::string("ssm_backward: ") + cudaGetErrorString((cudaError_t)e));
        return GDN_OK;
    }
    char* ws = (char*)workspace;
    if (pl.chunked) {
        const ssd::Workspace cw = ssd::workspace_layout(pl.N, pl.T, pl.H, pl.G, (int)pl.K, pl.HB);
        ssd::Args c = chunk_args(pl);
        c.x = x; c.dt = dt; c.A = A; c.B = B; c.C = C; c.ckpt_in = ckpt; c.dy = a.dy; c.dsT = a.dsT;
        c.ds0 = a.ds0; c.dx = a.dx; c.ddt = a.ddt; c.dB = a.dB; c.dC = a.dC;
        c.dd = (float*)(ws + cw.dd);
        c.sin_all = (float*)(ws + cw.sin_all);
        c.gvec = (float*)(ws + cw.gvec);
        c.partBC = (float*)(ws + cw.partBC);
        e = ssd::backward(c, st);
        if (e) return fail(GDN_ERR_CUDA, std::string("ssm_backward: ") + cudaGetErrorString((cudaError_t)e));
        return GDN_OK;
    }
    if (pl.diag) {
        const diag::Workspace dw = diag::workspace_layout(pl.N, pl.T, pl.H, pl.G, (int)pl.K);
        diag::Args c = diag_args(pl);
        c.x = x; c.dt = dt; c.A = A; c.B = B; c.C = C; c.ckpt_in = ckpt; c.dy = a.dy; c.dsT = a.dsT;
        c.ds0 = a.ds0; c.dx = a.dx; c.ddt = a.ddt; c.dB = a.dB; c.dC = a.dC;
        c.sin_sb = (float*)(ws + dw.sin_sb);
        c.U = (float*)(ws + dw.U);
        c.Gb = (float*)(ws + dw.Gb);
        c.carry = (float*)(ws + dw.carry);
        c.partBC = (float*)(ws + dw.partBC);
        e = diag::backward(c, st);
        if (e) return fail(GDN_ERR_CUDA, std::string("ssm_backward: ") + cudaGetErrorString((cudaError_t)e));
        return GDN_OK;
    }
    a.sub = (float*)(ws + w.sub);
    a.partBC = (float*)(ws + w.partBC);
    a.partDt = (float*)(ws + w.partDt);
    e = launch<false>(a, pl, st);
    if (!e) {
        ssm_reduce_kernel<<<(unsigned)(pl.N * pl.T), 256, 0, st>>>(a);
        e = (int)cudaGetLastError();
    }
    if (e) return fail(GDN_ERR_CUDA, std::string("ssm_backward: ") + cudaGetErrorString((cudaError_t)e));
    return GDN_OK;
}
