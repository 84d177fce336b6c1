// gdn_tc_grad.cu -- the gradient step of the chunked backward (scalar gate, head size
// 128) on the 5th-generation tensor cores: one CTA per (chunk, value head) computes every
// gradient of the chunk for that value head, and a small kernel sums the value heads of
// each key head.
//
// With M = M_c the chunk-entry state, dM = dM_end the gradient of the chunk's end state
// (128 x 128, rows j = value index, columns i = key index) and the chunk's rows t, the
// chunked form of the recurrence of "metal: GATED_DELTA_NET_BACK" (derived in
// gdn_chunk.cu) gives, through the chain rule:
//   X      = V - diag(gamma) K M^T          D_X = M K^T             (A = M,     rows j)
//   Delta  = T X                            CUDA cores, rows j in registers
//   D2     = M^T [s gamma dY ; -gamma dX]^T                           (A = M^T,   rows i)
//   D3     = dM^T Delta^T                                             (A = dM^T,  rows i)
//   D4     = [dY ; dDelta ; 0] [Delta ; X]^T   its blocks dY Delta^T and dDelta X^T
//   the 32 x 32 algebra of T, Z, the decay matrix and the gate (CUDA cores), giving P
//   (the Dm-weighted lower(s dY Delta^T)) and S (the symmetrised key-key gradient)
//   D2    += [K^T P^T | Q^T P + K^T S]      (A = [Q^T | K^T] from the prep kernel, rows i)
//   dq_h = D2[:, 0:32]^T,   dk_h = (D2[:, 32:64] + D3 diag(r))^T,   dv = dX,
//   dg (reverse scan of the gate gradient), dbeta.
// Every product is a three-pass split with an fp32 accumulator in TMEM (gdn_tc.cuh): bf16
// hi/lo (kind::f16) for all but D2's first part, which keeps tf32 hi/lo because the exact
// tf32 split of M^T also gives <dM, M>.  The A operands built here go to TMEM, the B
// operands to padded shared-memory tiles.
#include <cuda_runtime.h>

#include "gdn_gemm.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

// Status word of this file's kernel: 0, or GDN_ERR_TIMEOUT (6) after a bounded wait gave up.
__device__ int g_tcg_status;

namespace {

constexpr int TD = 128;
constexpr int GT = 288;           // 8 compute warps + the issuer warp
constexpr int kIss = 256;
constexpr uint32_t kCA = 0;       // TMEM: A operand, hi in 0..127, lo in 128..255
constexpr uint32_t kCX = 256;     //       D_X (32)
constexpr uint32_t kC2 = 288;     //       D2  (64: dq part, dk part)
constexpr uint32_t kC3 = 352;     //       D3  (32)
constexpr uint32_t kC4 = 384;     //       D4  (64)
constexpr uint32_t kCN = 128;     //       D_N = (r Delta)^T K (128, once M^T is dead)
constexpr uint32_t kCNA = 448;    //       its bf16 A operand (r Delta)^T: hi 448.., lo 464..
constexpr uint32_t kCols = 512;
constexpr int kStatusTimeout = 6;
constexpr int LDF = BC + 4;       // leading dimension of the 32 x 32 fp32 tiles

// B tiles built here: k-chunk-major with a 16-byte pad between k-chunks, so that 32
// threads writing one row (32 consecutive k) hit 32 distinct banks.
__device__ __forceinline__ int padoff(int r, int k, int lbo_floats)
{
    return (k >> 2) * lbo_floats + ((r >> 3) << 5) + ((r & 7) << 2) + (k & 3);
}
constexpr int kLbo64 = 8 * 128 + 16;        // bytes between k-chunks, 64-row tile
constexpr int kT64 = 32 * kLbo64 / 4;       // floats per 64-row, K = 128 tile (hi or lo)
// The bf16 tiles built here ([Delta ; X]) keep the layout with 8 elements (16 bytes) per
// core-matrix row: a 64-row, K = 128 tile has 16 k-chunks, kLbo64 bytes apart.
constexpr int kT64h = 16 * kLbo64 / 4;      // floats per 64-row, K = 128 bf16 tile (hi or lo)
__device__ __forceinline__ int padoff16(int r, int k, int lbo = kLbo64)  // byte offset of (r, k)
{
    return (k >> 3) * lbo + ((r >> 3) << 7) + ((r & 7) << 4) + ((k & 7) << 1);
}
constexpr int kLbo32 = 4 * 128 + 16;        // 32-row tile
constexpr int kTP = 4 * kLbo32 / 4;         // 32 rows, K = 32 (bf16: 4 k-chunks of 8)
constexpr int kTPS = 8 * kLbo32 / 4;        // 32 rows, K = 64 (bf16)
constexpr int kLdM = TD + 4;                // fp32 staging, row-major rows of TD floats
constexpr int kLdU = 4 * TD + 4;            // fp32 staging of a unit-layout park: one row of
                                            // 128 float4 per 4 columns, 16 bytes of pad between

// shared memory (floats): three big regions reused phase by phase, then small arrays
constexpr int kR0 = 0;                      // K tile (prep's layout) | [Delta ; X] tile hi, lo
constexpr int kR1 = kR0 + 2 * kT64;         // [s gamma dY ; -gamma dX] hi, lo | dDelta, dY |
                                            // 32 x 32 algebra tiles and the P, [P ; S] tiles
constexpr int kR2 = kR1 + 2 * kT64;         // M, then dM, fp32 staging | [Q^T | K^T] tile
static_assert(BC * kLdU <= TD * kLdM, "unit-layout staging of M fits the region");
constexpr int kR3 = kR2 + TD * kLdM;
constexpr int kSTr = kR3;                   // T, Z, KK^T, QK^T, Dm: row-major 32 x 32 each
constexpr int kSZ = kSTr + BC * BC;
constexpr int kSKK = kSZ + BC * BC;
constexpr int kSQK = kSKK + BC * BC;
constexpr int kSDm = kSQK + BC * BC;
constexpr int kSGam = kSDm + BC * BC;       // gamma, r (bulk copied), beta
constexpr int kSR = kSGam + BC;
constexpr int kSB = kSR + BC;
constexpr int kSRed = kSB + BC;             // 4 lane quarters x 96 partial sums
constexpr int kSVec = kSRed + 4 * 96;       // gdg, dr, dG, dbeta, dot
// KDA gate: gamma_last (128), <dM, M> per column from the two column halves (2 x 128), and
// the chunk-end gate partials of the two token halves (2 x 128)
constexpr int kSGl = kSVec + 4 * BC + 4;
constexpr int kSColS = kSGl + TD;
constexpr int kSLast = kSColS + 2 * TD;
constexpr int kGFloats = kSLast + 2 * TD;
constexpr size_t kGSmemBytes = sizeof(float) * kGFloats + 64;
static_assert(kGSmemBytes <= 227 * 1024, "shared memory");
// 32 x 32 tiles in R1 after D2 is done: Ps, Ss, dTs, W1, W2, Zs (LDF), then the B tiles
constexpr int kAPs = kR1;
constexpr int kASs = kAPs + BC * LDF;
constexpr int kAdT = kASs + BC * LDF;
constexpr int kAW1 = kAdT + BC * LDF;
constexpr int kAW2 = kAW1 + BC * LDF;
constexpr int kAZ = kAW2 + BC * LDF;
constexpr int kABP = kAZ + BC * LDF;        // P (rows t, K = 32) hi, lo
constexpr int kABPS = kABP + 2 * kTP;       // [P ; S]^T (rows t, K = 64) hi, lo
constexpr int kAZb = kABP;                 // Z diag(beta) (LDF): dead before the B tiles are built
static_assert(kAZb + BC * LDF <= kR2, "R1 overflow");
constexpr int kKcol = kR1 + 6 * BC * LDF;   // KDA, step (9): the column-side exchange and dG
constexpr int kKdg = kKcol + BC * TD;
static_assert(kKdg + BC * TD <= kR2, "KDA tiles overflow R1");
static_assert(kABPS + 2 * kTPS <= kR2, "R1 overflow");
constexpr int kDdStage = kR1 + 6 * BC * LDF;   // dDelta (unit layout, 8 x kLdU), then
constexpr int kDyStage = kDdStage + BC * kLdM; // dY rows t (32 x kLdM), before the algebra
static_assert((BC / 4) * kLdU <= BC * kLdM && kDyStage + BC * kLdM <= kR2, "R1 overflow");

constexpr uint32_t kBytesKb = sizeof(float) * (kDkQKT - kDkKb);
constexpr uint32_t kBytesFac = sizeof(float) * 5 * BC * BC;
constexpr uint32_t kBytesFacKda = sizeof(float) * 4 * BC * BC;  // no decay matrix
constexpr uint32_t kBytesKrt = sizeof(float) * kTcKdaTile;      // (K (.) R)^T, bf16 hi/lo
// KDA tiles of step (9), dense rows of TD floats: q, k, a = exp(g), gamma in R0; the
// (K (.) R)^T tile, R and the row-side exchange in R2; the column-side exchange and the gate
// gradient in R1 after the 32 x 32 algebra tiles.
constexpr int kKq = kR0, kKk = kR0 + BC * TD, kKa = kR0 + 2 * BC * TD, kKg = kR0 + 3 * BC * TD;
constexpr int kKrt = kR2, kKr = kR2 + kTcKdaTile, kKrowQ = kKr + BC * TD, kKrowK = kKrowQ + BC * TD;
static_assert(kKg + BC * TD <= kR1 && kKrowK + BC * TD <= kR3, "KDA tiles overflow R0 / R2");
constexpr uint32_t kBytesGR = sizeof(float) * 2 * BC;
constexpr uint32_t kBytesQKT = sizeof(float) * (kTcDkElems - kDkQKT);
constexpr uint32_t kBytesState = sizeof(float) * TD * TD;
constexpr uint32_t kBytesDd = sizeof(float) * BC * TD;

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The warp sums of N values per lane (N = 32 or 16) by recursive halving: lane l ends with
// the sum of value l (N = 32) or l / 2 (N = 16) in v[0].  Each partial sum pairs the same
// lanes in the same order as warp_sum, so the sums are warp_sum's bit for bit, in
// N - 1 + (32 / N - 1) shuffles instead of 5 N.
template <int N>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N], int lane)
{
    static_assert(N == 32 || N == 16, "32 or 16 values");
#pragma unroll
    for (int m = N / 2, o = 16; m >= 1; m >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;  // keeps the upper half of the live values
#pragma unroll
        for (int i = 0; i < m; ++i) {
            const float send = up ? v[i] : v[i + m];
            const float keep = up ? v[i + m] : v[i];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
    if (N == 16) v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

__device__ __forceinline__ void put_split(float* tile, int half, int off, float x)
{
    uint32_t hi, lo;
    tc::split_tf32(x, hi, lo);
    tile[off] = __uint_as_float(hi);
    tile[half + off] = __uint_as_float(lo);
}

// x as bf16 hi (at byte offset off of the tile) and lo (`half` floats further).
__device__ __forceinline__ void put_split16(float* tile, int off, float x, int half = kT64h)
{
    const uint32_t h = tc::pack_bf16x2(x, 0.f);
    const uint32_t l = tc::pack_bf16x2(__fsub_rn(x, __uint_as_float(h << 16)), 0.f);
    unsigned char* b = reinterpret_cast<unsigned char*>(tile);
    *reinterpret_cast<uint16_t*>(b + off) = (uint16_t)h;
    *reinterpret_cast<uint16_t*>(b + 4 * half + off) = (uint16_t)l;
}

// x0, x1 at consecutive K (x0 even) as one 4-byte word of bf16 hi at byte offset off and one of lo.
__device__ __forceinline__ void put_split16x2(float* tile, int off, float x0, float x1, int half)
{
    uint32_t h, l;
    tc::split_bf16x2(x0, x1, h, l);
    unsigned char* b = reinterpret_cast<unsigned char*>(tile);
    *reinterpret_cast<uint32_t*>(b + off) = h;
    *reinterpret_cast<uint32_t*>(b + 4 * half + off) = l;
}

// The same in kind::f16 with bf16 operands: K = 16 slices, A in TMEM two K elements per column.
__device__ __forceinline__ void mma3_t16(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b_hi, uint64_t b_lo,
                                         uint32_t lbo, int s0, int s1, uint32_t idesc, bool acc)
{
    for (int s = s0; s < s1; ++s) {
        const uint64_t off = (uint64_t)((2 * lbo * s) >> 4);
        tc::mma_ts16(d, a_hi + 8 * s, b_hi + off, idesc, (acc || s > s0) ? 1u : 0u);
        tc::mma_ts16(d, a_hi + 8 * s, b_lo + off, idesc, 1);
        tc::mma_ts16(d, a_lo + 8 * s, b_hi + off, idesc, 1);
    }
}

// Issues a K-slices [s0, s1) three-pass product D (+)= A B^T, A in TMEM (column base a).
__device__ __forceinline__ void mma3_t(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b_hi, uint64_t b_lo,
                                       uint32_t lbo, int s0, int s1, uint32_t idesc, bool acc)
{
    for (int s = s0; s < s1; ++s) {
        const uint64_t off = (uint64_t)((2 * lbo * s) >> 4);
        tc::mma_ts(d, a_hi + 8 * s, b_hi + off, idesc, (acc || s > s0) ? 1u : 0u);
        tc::mma_ts(d, a_hi + 8 * s, b_lo + off, idesc, 1);
        tc::mma_ts(d, a_lo + 8 * s, b_hi + off, idesc, 1);
    }
}

// Step (9) of the KDA gradient on the CUDA cores (compute warps; thread = key column i = row,
// half hc).  With P = dAqk (lower, diagonal included), S = dAkk (strictly lower) from the 32 x 32
// algebra and E[t][tau] = a[tau + 1] ... a[t] per column (running products of a = exp(g), in
// the prep's order):
//   row side (hc = 0): dqA[t] = sum_tau P[t][tau] k[tau] E,   dkA+[t] = sum_tau S[t][tau] k[tau] E
//   column side (hc = 1): dkA-[tau] = sum_t (P[t][tau] q[t] + S[t][tau] k[t]) E
// Then, for this thread's tokens, with D2 = [d(Q (.) gamma) | d(K (.) gamma)] and
// d3 = d(K (.) R) from the tensor cores:
//   dq = gamma d(Q (.) gamma) + dqA,  dk+ = gamma d(K (.) gamma) + dkA+,
//   dk- = R d(K (.) R) + dkA-,        dk = dk+ + dk-
// and the gradient of the cumulative gate G (every factor exp(+G_t) or exp(-G_tau) of a
// product gives q dq, k dk+ or -k dk-):
//   dG[t] = q dq + k (dk+ - dk-),  dG[last] += sum_tau k R d(K (.) R) + gamma_last <dM, M>_i
// dg is the reverse running sum of dG over the chunk.  Writes this value head's dq, dk parts
// and dg; returns false if the wait for the tiles gave up.
__device__ __forceinline__ bool kda_tail(const ChunkArgs& A, float* sm, uint32_t tmem, uint64_t* bar_kda, int tid,
                                         int warp, int row, int hc, int tb, int nb, int t0, int n, int hk, int h,
                                         long long ch, long long tok0, const float (&d3)[16])
{
    float* sQ = sm + kKq;
    float* sK = sm + kKk;
    float* sA = sm + kKa;
    const float* sG = sm + kKg;
    const float* sR = sm + kKr;
    float* rowQ = sm + kKrowQ;
    float* rowK = sm + kKrowK;
    float* col = sm + kKcol;
    float* dGs = sm + kKdg;
    const float* Ps = sm + kAPs;
    const float* Ss = sm + kASs;
    const int i = row;
    const bool rows_bulk = A.vec_q && A.vec_k && A.vec_g;
    // the rows the copies leave out: the padding (q = k = 0, g = 0), and every row without them
    for (int idx = tid; idx < BC * TD; idx += 256) {
        const int t = idx / TD, c = idx - t * TD;
        if (t >= nb) {
            sQ[idx] = 0.f;
            sK[idx] = 0.f;
            sA[idx] = 0.f;
        } else if (!rows_bulk) {
            sQ[idx] = __ldg(A.q + (long long)(n / A.rep) * A.qs0 + (long long)(t0 + t) * A.qs1 + (long long)hk * A.qs2 + c);
            sK[idx] = __ldg(A.k + (long long)(n / A.rep) * A.ks0 + (long long)(t0 + t) * A.ks1 + (long long)hk * A.ks2 + c);
            sA[idx] = __ldg(A.g + ((tok0 + t) * A.H_v + h) * TD + c);
        }
    }
    const bool ok = tc::mbar_wait(bar_kda, 0);
    tc::bar_sync_first(256);
    for (int idx = tid; idx < BC * TD; idx += 256) sA[idx] = expf(sA[idx]);
    tc::bar_sync_first(256);
    // E[tau] = E[t][tau] is carried in registers and multiplied by a_t for tau < t (by 1
    // otherwise: exact).  The token loop stays rolled and tau runs in blocks of 8, skipped
    // above the diagonal: the whole triangle unrolled would be tens of KB of straight-line
    // code, which each warp runs once.  P[t][tau] = 0 for tau > t and S[t][tau] = 0 for
    // tau >= t, so the diagonal block's extra slots add zeros.
    if (hc == 0) {
        float kc[BC], E[BC];
#pragma unroll
        for (int tau = 0; tau < BC; ++tau) {
            kc[tau] = sK[tau * TD + i];
            E[tau] = 1.f;
        }
#pragma unroll 1
        for (int t = 0; t < BC; ++t) {
            const float at = sA[t * TD + i];
            float dq = 0.f, dk = 0.f;
#pragma unroll
            for (int b = 0; b < BC / 8; ++b) {
                if (8 * b <= t) {
                    float pr[8], sr[8];
                    *reinterpret_cast<float4*>(pr) = *reinterpret_cast<const float4*>(Ps + t * LDF + 8 * b);
                    *reinterpret_cast<float4*>(pr + 4) = *reinterpret_cast<const float4*>(Ps + t * LDF + 8 * b + 4);
                    *reinterpret_cast<float4*>(sr) = *reinterpret_cast<const float4*>(Ss + t * LDF + 8 * b);
                    *reinterpret_cast<float4*>(sr + 4) = *reinterpret_cast<const float4*>(Ss + t * LDF + 8 * b + 4);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int tau = 8 * b + u;
                        E[tau] = __fmul_rn(E[tau], tau < t ? at : 1.f);
                        const float w = __fmul_rn(kc[tau], E[tau]);
                        dq = __fmaf_rn(pr[u], w, dq);
                        dk = __fmaf_rn(sr[u], w, dk);
                    }
                }
            }
            rowQ[t * TD + i] = dq;
            rowK[t * TD + i] = dk;
        }
    } else {
        float E[BC], acc[BC];
#pragma unroll
        for (int tau = 0; tau < BC; ++tau) {
            E[tau] = 1.f;
            acc[tau] = 0.f;
        }
#pragma unroll 1
        for (int t = 0; t < BC; ++t) {
            const float at = sA[t * TD + i], qt = sQ[t * TD + i], kt = sK[t * TD + i];
#pragma unroll
            for (int b = 0; b < BC / 8; ++b) {
                if (8 * b <= t) {
                    float pr[8], sr[8];
                    *reinterpret_cast<float4*>(pr) = *reinterpret_cast<const float4*>(Ps + t * LDF + 8 * b);
                    *reinterpret_cast<float4*>(pr + 4) = *reinterpret_cast<const float4*>(Ps + t * LDF + 8 * b + 4);
                    *reinterpret_cast<float4*>(sr) = *reinterpret_cast<const float4*>(Ss + t * LDF + 8 * b);
                    *reinterpret_cast<float4*>(sr + 4) = *reinterpret_cast<const float4*>(Ss + t * LDF + 8 * b + 4);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int tau = 8 * b + u;
                        E[tau] = __fmul_rn(E[tau], tau < t ? at : 1.f);
                        const float pe = __fmaf_rn(sr[u], kt, __fmul_rn(pr[u], qt));
                        acc[tau] = __fmaf_rn(pe, E[tau], acc[tau]);
                    }
                }
            }
        }
#pragma unroll
        for (int tau = 0; tau < BC; ++tau) col[tau * TD + i] = acc[tau];
    }
    tc::bar_sync_first(256);
    {
        float dQG[16], dKG[16];
        tc::ld16(tc::taddr(tmem, warp, kC2 + tb), dQG);
        tc::ld16(tc::taddr(tmem, warp, kC2 + BC + tb), dKG);
        tc::wait_ld();
        float* dqo = A.ws + A.o_dqM + ch * (BC * TD) + i;
        float* dko = A.ws + A.o_dkM + ch * (BC * TD) + i;
        float last = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int t = tb + e, o = t * TD + i;
            const float gt = sG[o], qt = sQ[o], kt = sK[o];
            const float dq = __fmaf_rn(gt, dQG[e], rowQ[o]);
            const float dkp = __fmaf_rn(gt, dKG[e], rowK[o]);
            const float dkr = __fmul_rn(sR[o], d3[e]);
            const float dkm = __fadd_rn(dkr, col[o]);
            dqo[t * TD] = dq;
            dko[t * TD] = __fadd_rn(dkp, dkm);
            dGs[o] = __fmaf_rn(qt, dq, __fmul_rn(kt, __fsub_rn(dkp, dkm)));
            last = __fmaf_rn(kt, dkr, last);
        }
        sm[kSLast + hc * TD + i] = last;
    }
    tc::bar_sync_first(256);
    if (hc == 0) {  // dg: reverse running sum of dG down column i, the chunk-end terms on the last row
        const float colsum = __fadd_rn(sm[kSColS + i], sm[kSColS + TD + i]);
        const float extra = __fmaf_rn(sm[kSGl + i], colsum, __fadd_rn(sm[kSLast + i], sm[kSLast + TD + i]));
        float x = 0.f;
        for (int t = BC - 1; t >= 0; --t) {
            float v = dGs[t * TD + i];
            if (t == BC - 1) v = __fadd_rn(v, extra);
            x = __fadd_rn(x, v);
            if (t < nb) A.dg[((tok0 + t) * A.H_v + h) * TD + i] = x;
        }
    }
    return ok;
}

}  // namespace

// KDA: the per-key-column gate.  Every tensor-core product keeps its form (the decay is
// inside the operands the prep built: K (.) gamma for D_X, (K (.) R)^T for the successor
// state, gamma = r = 1); the decay-weighted 32 x 32 products of step (9) and the per-column
// gate gradient run on the CUDA cores.
template <bool KDA>
__global__ void __launch_bounds__(GT, 1) gdn_tc_grad_kernel(const ChunkArgs A)
{
    extern __shared__ __align__(1024) float sm[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kGFloats);
    uint64_t* bar_ld = bars;       // K tile, chunk factors, gamma, r
    uint64_t* bar_qkt = bars + 1;  // [Q^T | K^T]
    uint64_t* bar_mma = bars + 2;
    uint64_t* bar_m = bars + 3;    // M
    uint64_t* bar_dm = bars + 4;   // dM
    uint64_t* bar_dd = bars + 5;   // dDelta, dY rows
    uint64_t* bar_kda = bars + 6;  // KDA: q, k, g rows, gamma and R tiles for step (9)
    uint64_t* bar_park = bars + 7; // the successor state's product (scalar gate)
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ int s_armed;        // bit b: bars[b] waits for bulk copies

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool compute = warp < 8;
    const bool issuer = tid == kIss;
    const int row = 32 * (warp & 3) + lane;  // this thread's TMEM lane
    const int hc = (warp >> 2) & 1;          // half: 64 of the K columns, 16 of the 32 tokens
    const int tb = 16 * hc;                  // this thread's tokens [tb, tb + 16)
    const int c = A.grad_loc < 0 ? A.c_lo + blockIdx.x : (A.c_lo / A.cps + blockIdx.x) * A.cps + A.grad_loc;
    const int h = blockIdx.y, n = blockIdx.z;
    const int hk = h % A.H_k;
    const long long head = (long long)n * A.H_v + h;
    const long long ch = head * A.n_chunks + c;
    const long long ck = ((long long)n * A.H_k + hk) * A.n_chunks + c;  // key head's blocks
    const int seg = c / A.cps, loc = c - seg * A.cps;
    const int t0 = seg * A.C + loc * BC;
    const int nb = min(BC, min(A.T, seg * A.C + A.C) - t0);
    const long long tok0 = (long long)n * A.T + t0;
    // the next chunk of this segment takes its entry state from this CTA (M_N below)
    const bool park_next = A.grad_loc >= 0 && t0 + BC < min(A.T, seg * A.C + A.C);
    // the next place's launch may place its CTAs as soon as every CTA of this one has started:
    // they run their independent loads in this launch's tail and wait for its parks.  (M is
    // copied first: issuing the K tile and factors ahead of it made the backward 3 % slower.)
    tc::grid_dep_launch();

    if (tid == 0) {
        tc::mbar_init(bar_ld, 1);
        tc::mbar_init(bar_qkt, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init(bar_m, 1);
        tc::mbar_init(bar_dm, 1);
        tc::mbar_init(bar_dd, 1);
        tc::mbar_init(bar_kda, 1);
        tc::mbar_init(bar_park, 1);
        tc::mbar_fence_init();
        s_err = 0;
        s_armed = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, kCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t aHi = tmem + kCA, aLo = tmem + kCA + 128;
    float* sM = sm + kR2;
    const bool m_unit = loc > 0;  // M: a parked state (unit layout) or the row-major checkpoint
    if (issuer)  // see tc::prefetch_l2 (measured 0.95 vs 1.08 ms per launch at the bench size)
        tc::prefetch_l2(A.q + (long long)(n / A.rep) * A.qs0 + (long long)t0 * A.qs1 + (long long)hk * A.qs2);
    if (warp == 8) {  // M into R2 by the bulk-copy engine: 32 padded runs, or 128 padded rows
        if (lane == 0) {
            s_armed = (1 << 0) | (1 << 3);
            tc::mbar_expect_tx(bar_m, kBytesState);
        }
        __syncwarp();
        if (m_unit) {
            tc::grid_dep_wait();  // the park is written by the preceding launch
            tc::bulk_g2s(sM + lane * kLdU, A.ws + A.o_Mc + ch * (long long)(TD * TD) + lane * 4 * TD,
                         sizeof(float) * 4 * TD, bar_m);
        } else {
            const float* ck0 = A.ckpt + (head * A.n_ck + seg) * (long long)(TD * TD);
            for (int r = lane; r < TD; r += 32) tc::bulk_g2s(sM + r * kLdM, ck0 + r * TD, sizeof(float) * TD, bar_m);
        }
    }
    if (issuer) {
        tc::mbar_expect_tx(bar_ld, kBytesKb + (KDA ? kBytesFacKda + (uint32_t)sizeof(float) * TD : kBytesFac) + kBytesGR);
        if (KDA)  // D_X = M (K (.) gamma)^T
            tc::bulk_g2s(sm + kR0, A.ws + A.o_KG + ch * kTcKdaTile, kBytesKb, bar_ld);
        else
            tc::bulk_g2s(sm + kR0, A.ws + A.o_DK + ck * kTcDkElems + kDkKb, kBytesKb, bar_ld);
        const long long f = ch * (BC * BC);
        tc::bulk_g2s(sm + kSTr, A.ws + A.o_Tr + f, sizeof(float) * BC * BC, bar_ld);
        tc::bulk_g2s(sm + kSZ, A.ws + A.o_Z + f, sizeof(float) * BC * BC, bar_ld);
        tc::bulk_g2s(sm + kSKK, A.ws + A.o_KK + f, sizeof(float) * BC * BC, bar_ld);
        tc::bulk_g2s(sm + kSQK, A.ws + A.o_QK + f, sizeof(float) * BC * BC, bar_ld);
        if (KDA)
            tc::bulk_g2s(sm + kSGl, A.ws + A.o_gL + ch * TD, sizeof(float) * TD, bar_ld);
        else
            tc::bulk_g2s(sm + kSDm, A.ws + A.o_Dm + f, sizeof(float) * BC * BC, bar_ld);
        tc::bulk_g2s(sm + kSGam, A.ws + A.o_gam + ch * BC, sizeof(float) * BC, bar_ld);
        tc::bulk_g2s(sm + kSR, A.ws + A.o_r + ch * BC, sizeof(float) * BC, bar_ld);
    }
    const float* sGam = sm + kSGam;
    const float* sR = sm + kSR;
    float* sB = sm + kSB;
    float* red = sm + kSRed;
    float* vec = sm + kSVec;  // gdg, dr, dG, dbeta, dot

    // (0) build A = M (rows j) from the staged M.  The loads of step (1), which do not depend
    //     on M, go out while the copy is in flight.
    uint32_t ph = 0;
    bool mma_out = false;  // issuer: a committed MMA group not yet seen complete, phase ph_out
    bool park_out = false; // issuer: the successor state's product committed to bar_park
    uint32_t ph_out = 0;
    bool ok = true;
    float vx[32], dy[16];
    float4 dx[4];
    if (compute) {
        const float* gy = A.gy + (long long)n * A.gys0 + (long long)t0 * A.gys1 + (long long)h * A.gys2 + row;
        const float4* dx4 = reinterpret_cast<const float4*>(A.ws + A.o_dX + ch * (BC * TD));
        const float* vp = A.v + (long long)n * A.vs0 + (long long)t0 * A.vs1 + (long long)h * A.vs2 + row;
#pragma unroll
        for (int e = 0; e < 16; ++e) dy[e] = (tb + e < nb) ? __ldg(gy + (long long)(tb + e) * A.gys1) : 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) dx[b] = __ldg(dx4 + (4 * hc + b) * TD + row);
#pragma unroll
        for (int t = 0; t < BC; ++t) vx[t] = (t < nb) ? __ldg(vp + (long long)t * A.vs1) : 0.f;
        if (tid < BC) {
            const bool real = tid < nb;
            sB[tid] = real ? __ldg(A.beta + (tok0 + tid) * A.H_v + h) : 0.f;
        }
        // a park is written by the preceding launch: this thread reads it (here through shared
        // memory, in (10) from global memory) only after that launch has completed
        if (m_unit) tc::grid_dep_wait();
        if (!tc::mbar_wait(bar_m, 0)) s_err = 1;
#pragma unroll 1
        for (int q = 0; q < 8; ++q) {
            float4 a, b;
            if (m_unit) {
                a = *reinterpret_cast<const float4*>(sM + (16 * hc + 2 * q) * kLdU + 4 * row);
                b = *reinterpret_cast<const float4*>(sM + (16 * hc + 2 * q + 1) * kLdU + 4 * row);
            } else {
                a = *reinterpret_cast<const float4*>(sM + row * kLdM + 64 * hc + 8 * q);
                b = *reinterpret_cast<const float4*>(sM + row * kLdM + 64 * hc + 8 * q + 4);
            }
            uint32_t hi[4], lo[4];  // bf16, two columns per TMEM column
            tc::split_bf16x2(a.x, a.y, hi[0], lo[0]);
            tc::split_bf16x2(a.z, a.w, hi[1], lo[1]);
            tc::split_bf16x2(b.x, b.y, hi[2], lo[2]);
            tc::split_bf16x2(b.z, b.w, hi[3], lo[3]);
            tc::st4(tc::taddr(tmem, warp, kCA + 32 * hc + 4 * q), hi);
            tc::st4(tc::taddr(tmem, warp, kCA + 64 + 32 * hc + 4 * q), lo);
        }
        tc::wait_st();
    }
    tc::fence_before();
    __syncthreads();
    if (s_err) goto done;

    // (1) D_X = M K^T.  Meanwhile: the B tile [s gamma dY ; -gamma dX] and dv.
    if (issuer) {
        tc::fence_after();
        if (!tc::mbar_wait(bar_ld, 0)) s_err = 1;
        if (!s_err) {
            mma3_t16(tmem + kCX, aHi, aHi + 64, tc::tile_desc(sm + kR0, 32), tc::tile_desc(sm + kR0 + 32 * TD / 2, 32),
                     (32 / 8) * 128, 0, TD / 16, tc::idesc_bf16(32), false);
            tc::commit(bar_mma);
            mma_out = true;
            ph_out = ph;
        }
    } else if (compute) {
        if (!tc::mbar_wait(bar_ld, 0)) s_err = 1;
        float* b2 = sm + kR1;
        float* dvp = A.dv + (tok0 * A.H_v + h) * TD + row;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float dxv[4] = {dx[b].x, dx[b].y, dx[b].z, dx[b].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = tb + 4 * b + e;
                put_split(b2, kT64, padoff(t, row, kLbo64 / 4), __fmul_rn(__fmul_rn(A.scale, sGam[t]), dy[4 * b + e]));
                put_split(b2, kT64, padoff(BC + t, row, kLbo64 / 4), -__fmul_rn(sGam[t], dxv[e]));
                if (t < nb) dvp[(long long)t * A.H_v * TD] = dxv[e];
            }
        }
    }
    ok = tc::mbar_wait(bar_mma, ph);
    if (issuer && ok) mma_out = false;
    ph ^= 1;
    tc::fence_after();
    // (2) A = M^T (rows i); D_X goes to registers first (A = M is dead: D_X is done)
    float x[32];
    if (compute) {
        tc::ld32(tc::taddr(tmem, warp, kCX), x);
        tc::wait_ld();
        {  // M[j][row] for this thread's 64 j
            const float* mc = sM + (m_unit ? (row >> 2) * kLdU + (row & 3) : row);
            const int js = m_unit ? 4 : kLdM;
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) tc::split_tf32(mc[(64 * hc + 8 * q + e) * js], hi[e], lo[e]);
                tc::st8(tc::taddr(tmem, warp, kCA + 64 * hc + 8 * q), hi);
                tc::st8(tc::taddr(tmem, warp, kCA + 128 + 64 * hc + 8 * q), lo);
            }
        }
        tc::wait_st();
    }
    if (!ok) s_err = 1;
    tc::fence_before();
    __syncthreads();
    if (s_err) goto done;
    // (3) D2 = M^T [s gamma dY ; -gamma dX]^T on the tensor cores.  Meanwhile dM replaces M
    //     in R2 (bulk copy) and X^T, Delta^T (rows j) go into the [Delta ; X] tile.
    if (warp == 8) {
        if (lane == 0) {
            tc::fence_async_smem();
            s_armed |= 1 << 4;
            tc::mbar_expect_tx(bar_dm, kBytesState);
        }
        __syncwarp();
        tc::bulk_g2s(sM + lane * kLdU, A.ws + A.o_dM + ch * (long long)(TD * TD) + lane * 4 * TD,
                     sizeof(float) * 4 * TD, bar_dm);
        __syncwarp();
    }
    if (issuer) {
        tc::fence_after();
        mma3_t(tmem + kC2, aHi, aLo, tc::make_desc(tc::smem_addr(sm + kR1), kLbo64, 128),
               tc::make_desc(tc::smem_addr(sm + kR1 + kT64), kLbo64, 128), kLbo64, 0, TD / 8,
               tc::idesc_tf32(64), false);
        tc::commit(bar_mma);
            mma_out = true;
            ph_out = ph;
    } else if (compute) {
        const float* sT = sm + kSTr;
#pragma unroll
        for (int t = 0; t < BC; ++t) x[t] = __fsub_rn(vx[t], __fmul_rn(sGam[t], x[t]));
        float* b34 = sm + kR0;  // the K tile is dead: D_X is done
        float rd[16];           // r (.) Delta, row `row`, this thread's tokens
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int t = tb + e;
            float acc = 0.f;
            const float4* tr = reinterpret_cast<const float4*>(sT + t * BC);  // T row t, broadcast
#pragma unroll
            for (int k4 = 0; k4 < BC / 4; ++k4) {
                const float4 w = tr[k4];
                acc = __fmaf_rn(w.x, x[4 * k4], acc);
                acc = __fmaf_rn(w.y, x[4 * k4 + 1], acc);
                acc = __fmaf_rn(w.z, x[4 * k4 + 2], acc);
                acc = __fmaf_rn(w.w, x[4 * k4 + 3], acc);
            }
            put_split16(b34, padoff16(t, row), acc);
            put_split16(b34, padoff16(BC + t, row), hc ? x[16 + e] : x[e]);
            rd[e] = __fmul_rn(sR[t], acc);
        }
        tc::fence_async_smem();  // the tile is read by the tensor cores from (5) on
        if (park_next) {  // (r Delta)^T, rows j, K = t: the bf16 A operand of M_N
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) tc::split_bf16x2(rd[2 * e], rd[2 * e + 1], hi[e], lo[e]);
            tc::st8(tc::taddr(tmem, warp, kCNA + 8 * hc), hi);
            tc::st8(tc::taddr(tmem, warp, kCNA + 16 + 8 * hc), lo);
        }
    }
    ok = tc::mbar_wait(bar_mma, ph);
    if (issuer && ok) mma_out = false;
    ph ^= 1;
    tc::fence_after();
    // (4) A = dM^T (rows i) and <dM, M> (M^T still in TMEM).  R1's B tile is dead: dDelta and
    //     the dY rows come into it.
    if (warp == 8) {
        const bool dy_bulk = A.vec_gy != 0;
        if (lane == 0) {
            s_armed |= 1 << 5;
            tc::mbar_expect_tx(bar_dd, kBytesDd + (dy_bulk ? nb * (uint32_t)sizeof(float) * TD : 0u));
        }
        __syncwarp();
        if (lane < BC / 4)
            tc::bulk_g2s(sm + kDdStage + lane * kLdU, A.ws + A.o_dDel + ch * (BC * TD) + lane * 4 * TD,
                         sizeof(float) * 4 * TD, bar_dd);
        if (dy_bulk && lane < nb)
            tc::bulk_g2s(sm + kDyStage + lane * kLdM,
                         A.gy + (long long)n * A.gys0 + (long long)(t0 + lane) * A.gys1 + (long long)h * A.gys2,
                         sizeof(float) * TD, bar_dd);
    }
    if (compute) {
        if (!tc::mbar_wait(bar_dm, 0)) s_err = 1;
        const float* dmc = sM + (row >> 2) * kLdU + (row & 3);  // dM[j][row] at dmc[4 j]
        {
            float dot = 0.f;
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                const int j0 = 64 * hc + 8 * q;
                float mh[8], ml[8];
                tc::ld8(tc::taddr(tmem, warp, kCA + j0), mh);
                tc::ld8(tc::taddr(tmem, warp, kCA + 128 + j0), ml);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dot = __fmaf_rn(dmc[4 * (j0 + e)], __fadd_rn(mh[e], ml[e]), dot);  // hi + lo = M exactly
            }
            if (KDA) {  // per key column i = row: this half's 64 j
                sm[kSColS + hc * TD + row] = dot;
            } else {
                dot = warp_sum(dot);
                if (lane == 0) red[(warp & 3) * 96 + 64 + hc] = dot;
            }
        }
        // every compute thread has read M^T before dM^T (bf16, two j per column) overwrites it
        tc::fence_before();
        tc::bar_sync_first(256);
        tc::fence_after();
#pragma unroll 1
        for (int q = 0; q < 8; ++q) {
            const int j0 = 64 * hc + 8 * q;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) tc::split_bf16x2(dmc[4 * (j0 + 2 * e)], dmc[4 * (j0 + 2 * e + 1)], hi[e], lo[e]);
            tc::st4(tc::taddr(tmem, warp, kCA + j0 / 2), hi);
            tc::st4(tc::taddr(tmem, warp, kCA + 64 + j0 / 2), lo);
        }
        tc::wait_st();
    }
    if (!ok) s_err = 1;
    tc::fence_before();
    __syncthreads();
    if (s_err) goto done;
    // (5) [Q^T | K^T] into the staging region (dM is in TMEM now), then D3 = dM^T Delta^T.
    if (issuer) {
        tc::fence_after();
        tc::fence_async_smem();
        s_armed |= 1 << 1;
        if (KDA) {  // (K (.) R)^T, the B operand of the successor state
            tc::mbar_expect_tx(bar_qkt, kBytesKrt);
            tc::bulk_g2s(sm + kKrt, A.ws + A.o_KRT + ch * kTcKdaTile, kBytesKrt, bar_qkt);
        } else {
            tc::mbar_expect_tx(bar_qkt, kBytesQKT);
            tc::bulk_g2s(sm + kR2, A.ws + A.o_DK + ck * kTcDkElems + kDkQKT, kBytesQKT, bar_qkt);
        }
        mma3_t16(tmem + kC3, aHi, aHi + 64, tc::make_desc(tc::smem_addr(sm + kR0), kLbo64, 128),
                 tc::make_desc(tc::smem_addr(sm + kR0 + kT64h), kLbo64, 128), kLbo64, 0, TD / 16,
                 tc::idesc_bf16(32), false);
        tc::commit(bar_mma);
            mma_out = true;
            ph_out = ph;
    }
    ok = tc::mbar_wait(bar_mma, ph);
    if (issuer && ok) mma_out = false;
    ph ^= 1;
    tc::fence_after();
    // (6) the gamma dgamma partials (from D2, which holds M^T [s gamma dY ; -gamma dX]^T until
    //     step (9)) and the dr partials (from D3, kept for dk), with q_t, k_t of this
    //     thread's tokens read from the [Q^T | K^T] tile (bf16 hi + lo: 16 significant bits); then
    //     A = [dY ; dDelta ; 0] (rows t)
    float d3[16];
    if (!KDA && issuer && park_next) {
        // the next chunk's entry state: D_N = (r Delta)^T K (A = (r Delta)^T from (3), K from the
        // k-slices 2, 3 of [Q^T | K^T]), beside the sums below and the 32 x 32 algebra (columns
        // 128.. have been free since (4))
        if (!tc::mbar_wait(bar_qkt, 0)) {
            s_err = 1;
        } else {
            const uint64_t qhi = tc::tile_desc(sm + kR2, TD), qlo = tc::tile_desc(sm + kR2 + BC * TD, TD);
            const uint32_t id128 = tc::idesc_bf16(128);
#pragma unroll
            for (int s = 0; s < BC / 16; ++s) {
                const uint64_t b_h = tc::desc_kslice(qhi, TD, s + BC / 16), b_l = tc::desc_kslice(qlo, TD, s + BC / 16);
                tc::mma_ts16(tmem + kCN, tmem + kCNA + 8 * s, b_h, id128, s > 0);
                tc::mma_ts16(tmem + kCN, tmem + kCNA + 8 * s, b_l, id128, 1);
                tc::mma_ts16(tmem + kCN, tmem + kCNA + 16 + 8 * s, b_h, id128, 1);
            }
            tc::commit(bar_park);
            park_out = true;
        }
    }
    if (compute) {
        if (!tc::mbar_wait(bar_dd, 0) || !tc::mbar_wait(bar_qkt, 0)) s_err = 1;
        if (KDA) {  // d3 = (K (.) R)'s gradient, kept for step (9); the gate sums come there
            tc::ld16(tc::taddr(tmem, warp, kC3 + tb), d3);
            tc::wait_ld();
        } else {
            float dq[16], dk[16];
            tc::ld16(tc::taddr(tmem, warp, kC2 + tb), dq);
            tc::ld16(tc::taddr(tmem, warp, kC2 + BC + tb), dk);
            tc::ld16(tc::taddr(tmem, warp, kC3 + tb), d3);
            tc::wait_ld();
            // the bf16 [Q^T | K^T] tile: 16-byte unit kc * 128 + row holds t' = 8 kc .. 8 kc + 7
            const uint4* qkt = reinterpret_cast<const uint4*>(sm + kR2) + row;
            constexpr int kLo = BC * TD / 4;  // lo half of the tile, in 16-byte units
            auto lo16 = [](uint32_t w) { return __uint_as_float(w << 16); };
            auto hi16 = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
            float gs[32];  // this thread's terms of the 16 + 16 sums over rows i
#pragma unroll
            for (int cq = 0; cq < 2; ++cq) {
                const int kq = (tb >> 3) + cq, kk = BC / 8 + kq;
                const uint4 qh = qkt[kq * TD], ql = qkt[kLo + kq * TD];
                const uint4 kh = qkt[kk * TD], kl = qkt[kLo + kk * TD];
                const uint32_t qhw[4] = {qh.x, qh.y, qh.z, qh.w}, qlw[4] = {ql.x, ql.y, ql.z, ql.w};
                const uint32_t khw[4] = {kh.x, kh.y, kh.z, kh.w}, klw[4] = {kl.x, kl.y, kl.z, kl.w};
                float qv[8], kv[8];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    qv[2 * w] = __fadd_rn(lo16(qhw[w]), lo16(qlw[w]));
                    qv[2 * w + 1] = __fadd_rn(hi16(qhw[w]), hi16(qlw[w]));
                    kv[2 * w] = __fadd_rn(lo16(khw[w]), lo16(klw[w]));
                    kv[2 * w + 1] = __fadd_rn(hi16(khw[w]), hi16(klw[w]));
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int x = 8 * cq + e;
                    gs[x] = __fmaf_rn(kv[e], dk[x], __fmul_rn(qv[e], dq[x]));
                    gs[16 + x] = __fmul_rn(kv[e], d3[x]);
                }
            }
            warp_reduce_scatter<32>(gs, lane);  // lane l: sum l (l < 16: g1 of token tb + l, else g2)
            red[(warp & 3) * 96 + (lane < 16 ? tb + lane : BC + tb + lane - 16)] = gs[0];
        }
        const int quarter = warp & 3;
        const float* gyr = A.gy + (long long)n * A.gys0 + (long long)(t0 + lane) * A.gys1 + (long long)h * A.gys2 + 64 * hc;
        const float* sdd = sm + kDdStage + (lane >> 2) * kLdU + (lane & 3) + 4 * 64 * hc;  // dDelta[lane][j]
        const float* sdy = sm + kDyStage + lane * kLdM + 64 * hc;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {  // 32 of this thread's 64 columns at a time
            float v[32];
            if (quarter == 0) {  // rows 0..31: dY row t = lane
                if (lane < nb && A.vec_gy) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 x = *reinterpret_cast<const float4*>(sdy + 32 * half + 4 * u);
                        v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = (lane < nb) ? __ldg(gyr + 32 * half + e) : 0.f;
                }
            } else if (quarter == 1) {  // rows 32..63: dDelta row t = lane
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = sdd[4 * (32 * half + e)];
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {  // bf16, two j per column
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) tc::split_bf16x2(v[16 * q + 2 * e], v[16 * q + 2 * e + 1], hi[e], lo[e]);
                const int c0 = 32 * hc + 16 * half + 8 * q;
                tc::st8(tc::taddr(tmem, warp, kCA + c0), hi);
                tc::st8(tc::taddr(tmem, warp, kCA + 64 + c0), lo);
            }
        }
        tc::wait_st();
    }
    if (!ok) s_err = 1;
    tc::fence_before();
    __syncthreads();
    if (s_err) goto done;
    // (7) D4 = [dY ; dDelta ; 0] [Delta ; X]^T.  Meanwhile the scalars.
    if (issuer) {
        tc::fence_after();
        mma3_t16(tmem + kC4, aHi, aHi + 64, tc::make_desc(tc::smem_addr(sm + kR0), kLbo64, 128),
                 tc::make_desc(tc::smem_addr(sm + kR0 + kT64h), kLbo64, 128), kLbo64, 0, TD / 16,
                 tc::idesc_bf16(64), false);
        tc::commit(bar_mma);
            mma_out = true;
            ph_out = ph;
    } else if (compute) {
        if (KDA) {
        } else if (tid < 2 * BC) {
            vec[tid] = __fadd_rn(__fadd_rn(red[tid], red[96 + tid]), __fadd_rn(red[192 + tid], red[288 + tid]));
        } else if (tid == 2 * BC) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) v = __fadd_rn(v, __fadd_rn(red[w * 96 + 64], red[w * 96 + 65]));
            vec[4 * BC] = v;
        }
        // Z and Z diag(beta) into LDF tiles (operands of the two small products)
        float* Zs = sm + kAZ;
        float* Zb = sm + kAZb;
        for (int idx = tid; idx < BC * BC; idx += 256) {
            const float z = sm[kSZ + idx];
            Zs[(idx >> 5) * LDF + (idx & 31)] = z;
            Zb[(idx >> 5) * LDF + (idx & 31)] = __fmul_rn(z, sB[idx & 31]);
        }
    }
    ok = tc::mbar_wait(bar_mma, ph);
    if (issuer && ok) mma_out = false;
    ph ^= 1;
    tc::fence_after();
    if (KDA && warp == 8) {
        // step (9)'s tiles: gamma, R from the prep; q, k, g rows from the inputs (R0 is free: D4
        // is done; R2 past the (K (.) R)^T tile has been free since (5))
        const bool rows_bulk = A.vec_q && A.vec_k && A.vec_g;
        if (lane == 0) {
            s_armed |= 1 << 6;
            tc::mbar_expect_tx(bar_kda, 2u * (uint32_t)sizeof(float) * BC * TD +
                                            (rows_bulk ? 3u * (uint32_t)nb * (uint32_t)sizeof(float) * TD : 0u));
            tc::bulk_g2s(sm + kKg, A.ws + A.o_kGam + ch * (BC * TD), sizeof(float) * BC * TD, bar_kda);
            tc::bulk_g2s(sm + kKr, A.ws + A.o_kR + ch * (BC * TD), sizeof(float) * BC * TD, bar_kda);
        }
        __syncwarp();
        if (rows_bulk && lane < nb) {
            const long long t = t0 + lane;
            tc::bulk_g2s(sm + kKq + lane * TD, A.q + (long long)(n / A.rep) * A.qs0 + t * A.qs1 + (long long)hk * A.qs2,
                         sizeof(float) * TD, bar_kda);
            tc::bulk_g2s(sm + kKk + lane * TD, A.k + (long long)(n / A.rep) * A.ks0 + t * A.ks1 + (long long)hk * A.ks2,
                         sizeof(float) * TD, bar_kda);
            tc::bulk_g2s(sm + kKa + lane * TD, A.g + ((tok0 + lane) * A.H_v + h) * TD, sizeof(float) * TD, bar_kda);
        }
    }
    if (compute) {
        // (8) the 32 x 32 algebra.  D4 blocks: rows 0..31 cols 0..31 = dY Delta^T,
        //     rows 32..63 cols 32..63 = dDelta X^T.
        float* Ps = sm + kAPs;
        float* Ss = sm + kASs;
        float* dTs = sm + kAdT;
        float* W1 = sm + kAW1;
        float* W2 = sm + kAW2;
        const float* Zs = sm + kAZ;
        const float* Dm = sm + kSDm;
        const float* KKm = sm + kSKK;
        const float* QKm = sm + kSQK;
        const float* bs = sB;
        float* gdg = vec;
        float* dr = vec + BC;
        float* dG = vec + 2 * BC;
        float* dbs = vec + 3 * BC;
        const float dot = vec[4 * BC];
        const float* Zb = sm + kAZb;
        if ((warp & 3) < 2) {  // warps 0, 1, 4, 5: TMEM lanes 0..63, 16 of the 32 columns each
            const int blk = warp & 1, c0 = 16 * (warp >> 2);
            float v[16];
            tc::ld16(tc::taddr(tmem, warp, kC4 + BC * blk + c0), v);
            tc::wait_ld();
            const int t = lane;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int tau = c0 + e;
                if (blk == 0)
                    Ps[t * LDF + tau] = (tau <= t) ? __fmul_rn(A.scale, v[e]) : 0.f;
                else
                    dTs[t * LDF + tau] = (tau <= t) ? v[e] : 0.f;
            }
        }
        tc::bar_sync_first(256);
        {  // P1 = dZ Z^T with dZ = dT diag(beta): the rows of dT against those of Z diag(beta)
            using Map = GemmMap<BC, BC, 2, 2, true>;
            float acc[2][2];
            zero_acc(acc);
            block_gemm<BC, BC, 2, 2, false, true>(acc, dTs, LDF, Zb, LDF, BC, tid);
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) W2[Map::row(tid, i) * LDF + Map::col(tid, j)] = acc[i][j];
        }
        tc::bar_sync_first(256);
        {  // dA = strict_lower(-Z^T P1)
            using Map = GemmMap<BC, BC, 1, 4, false>;
            float acc[1][4];
            zero_acc(acc);
            block_gemm<BC, BC, 1, 4, true, false>(acc, Zs, LDF, W2, LDF, BC, tid);
            const int t = Map::row(tid, 0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tau = Map::col(tid, j);
                W1[t * LDF + tau] = (tau < t) ? -acc[0][j] : 0.f;
            }
        }
        tc::bar_sync_first(256);
        // dL = beta_t dA; dKK = dL (.) Dm; dD = dQKD (.) QK + dL (.) KK (+ dr on the last row);
        // the E = dD (.) Dm sums give the gate gradient (E into W2: P1 is dead)
        for (int idx = tid; idx < BC * BC; idx += 256) {
            const int t = idx >> 5, tau = idx & 31;
            const float dA = W1[t * LDF + tau];
            const float dL = __fmul_rn(bs[t], dA);
            if (KDA) {  // the decay is inside Akk, Aqk: their gradients are dL and P themselves
                Ss[t * LDF + tau] = dL;
                continue;
            }
            const float dm = Dm[idx];
            float dD = __fmul_rn(Ps[t * LDF + tau], QKm[idx]);
            dD = __fmaf_rn(dL, KKm[idx], dD);
            if (t == BC - 1) dD = __fadd_rn(dD, dr[tau]);
            Ss[t * LDF + tau] = __fmul_rn(dL, dm);
            Ps[t * LDF + tau] = __fmul_rn(Ps[t * LDF + tau], dm);
            W2[t * LDF + tau] = __fmul_rn(dD, dm);
        }
        tc::bar_sync_first(256);
        {  // warp w, t = 4 w + q: dbeta_a[t] = sum_t' Z[t'][t] dT[t'][t] and dbeta_b[t] = sum_tau
           // dA (KK, or Dm (.) KK); the scalar gate also the row and column sums of E
            float sv[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int t = 4 * warp + q, tau = lane;
                const float dA = W1[t * LDF + tau];
                sv[4 * q] = __fmul_rn(Zs[tau * LDF + t], dTs[tau * LDF + t]);
                sv[4 * q + 1] = KDA ? __fmul_rn(dA, KKm[t * BC + tau])
                                    : __fmul_rn(dA, __fmul_rn(Dm[t * BC + tau], KKm[t * BC + tau]));
                sv[4 * q + 2] = KDA ? 0.f : W2[t * LDF + tau];
                sv[4 * q + 3] = KDA ? 0.f : W2[tau * LDF + t];
            }
            warp_reduce_scatter<16>(sv, lane);  // lane l: sum l / 2, i.e. lane 8 q + 2 k: sum k of t = 4 w + q
            const float bb = __shfl_down_sync(0xffffffffu, sv[0], 2);
            const float rs = __shfl_down_sync(0xffffffffu, sv[0], 4);
            const float cs = __shfl_down_sync(0xffffffffu, sv[0], 6);
            if ((lane & 7) == 0) {
                const int t = 4 * warp + (lane >> 3);
                dbs[t] = __fadd_rn(sv[0], bb);
                if (!KDA) {
                    float g = gdg[t];
                    if (t == BC - 1) g = __fmaf_rn(sGam[t], dot, g);
                    dG[t] = __fadd_rn(__fadd_rn(g, rs), -cs);
                }
            }
        }
        tc::bar_sync_first(256);
        if (KDA && warp == 0) {  // dbeta (dg comes in step (9))
            if (lane < nb) A.dbeta[(tok0 + lane) * A.H_v + h] = dbs[lane];
        } else if (warp == 0) {  // dg = reverse cumsum of dG; dbeta
            float x = dG[BC - 1 - lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x = __fadd_rn(x, y);
            }
            const int t = BC - 1 - lane;
            if (t < nb) {
                A.dg[(tok0 + t) * A.H_v + h] = x;
                A.dbeta[(tok0 + t) * A.H_v + h] = dbs[t];
            }
        }
        // B tiles of the last products: P (rows t, K = t'), [P ; S]^T (rows t, K = t' < 64);
        // S is the symmetric dKK + dKK^T of its strict lower part
        float* bp = sm + kABP;
        float* bps = sm + kABPS;
        auto S_at = [&](int a, int b) {  // S[a][b] from the strict lower part
            return (b > a) ? Ss[b * LDF + a] : (b < a ? Ss[a * LDF + b] : 0.f);
        };
        for (int idx = tid; idx < BC * BC / 2 && !KDA; idx += 256) {
            const int t = idx & 31, tau = 2 * (idx >> 5);  // consecutive threads: consecutive rows t
            const float2 p = *reinterpret_cast<const float2*>(Ps + t * LDF + tau);
            put_split16x2(bp, padoff16(t, tau, kLbo32), p.x, p.y, kTP);
            put_split16x2(bps, padoff16(t, tau, kLbo32), Ps[tau * LDF + t], Ps[(tau + 1) * LDF + t], kTPS);
            put_split16x2(bps, padoff16(t, BC + tau, kLbo32), S_at(t, tau), S_at(t, tau + 1), kTPS);
        }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    // (9) D2 += [K^T P^T | Q^T P + K^T S]  (KDA: the successor state only; the decay-weighted
    //     products run on the CUDA cores meanwhile)
    if (issuer && KDA) {
        tc::fence_after();
        if (!tc::mbar_wait(bar_qkt, 0)) s_err = 1;
        if (!s_err) {
            if (park_next) {  // M_N = Delta^T (K (.) R): B = (K (.) R)^T, rows i, K = t
                const uint64_t khi = tc::tile_desc(sm + kKrt, TD), klo = tc::tile_desc(sm + kKrt + kTcKdaTile / 2, TD);
                const uint32_t id128 = tc::idesc_bf16(128);
#pragma unroll
                for (int s = 0; s < BC / 16; ++s) {
                    const uint64_t b_h = tc::desc_kslice(khi, TD, s), b_l = tc::desc_kslice(klo, TD, s);
                    tc::mma_ts16(tmem + kCN, tmem + kCNA + 8 * s, b_h, id128, s > 0);
                    tc::mma_ts16(tmem + kCN, tmem + kCNA + 8 * s, b_l, id128, 1);
                    tc::mma_ts16(tmem + kCN, tmem + kCNA + 16 + 8 * s, b_h, id128, 1);
                }
            }
            tc::commit(bar_mma);
            mma_out = true;
            ph_out = ph;
        }
    } else if (KDA && compute) {
        if (!kda_tail(A, sm, tmem, bar_kda, tid, warp, row, hc, tb, nb, t0, n, hk, h, ch, tok0, d3)) s_err = 1;
    } else if (issuer) {
        tc::fence_after();
        if (!tc::mbar_wait(bar_qkt, 0)) s_err = 1;
        if (!s_err) {
            const uint64_t qhi = tc::tile_desc(sm + kR2, TD), qlo = tc::tile_desc(sm + kR2 + BC * TD, TD);
            const uint32_t id32 = tc::idesc_bf16(32);
            // dq part: A = K^T (k-slices 2, 3 of the bf16 [Q^T | K^T]), B = P
            const uint64_t phi = tc::make_desc(tc::smem_addr(sm + kABP), kLbo32, 128);
            const uint64_t plo = tc::make_desc(tc::smem_addr(sm + kABP + kTP), kLbo32, 128);
#pragma unroll
            for (int s = 0; s < BC / 16; ++s) {
                const uint64_t a_h = tc::desc_kslice(qhi, TD, s + BC / 16), a_l = tc::desc_kslice(qlo, TD, s + BC / 16);
                const uint64_t off = (uint64_t)((2 * kLbo32 * s) >> 4);
                tc::mma_ss16(tmem + kC2, a_h, phi + off, id32, 1);
                tc::mma_ss16(tmem + kC2, a_h, plo + off, id32, 1);
                tc::mma_ss16(tmem + kC2, a_l, phi + off, id32, 1);
            }
            // dk part: A = [Q^T | K^T], B = [P ; S]^T
            const uint64_t shi = tc::make_desc(tc::smem_addr(sm + kABPS), kLbo32, 128);
            const uint64_t slo = tc::make_desc(tc::smem_addr(sm + kABPS + kTPS), kLbo32, 128);
#pragma unroll
            for (int s = 0; s < 2 * BC / 16; ++s) {
                const uint64_t a_h = tc::desc_kslice(qhi, TD, s), a_l = tc::desc_kslice(qlo, TD, s);
                const uint64_t off = (uint64_t)((2 * kLbo32 * s) >> 4);
                tc::mma_ss16(tmem + kC2 + BC, a_h, shi + off, id32, 1);
                tc::mma_ss16(tmem + kC2 + BC, a_h, slo + off, id32, 1);
                tc::mma_ss16(tmem + kC2 + BC, a_l, shi + off, id32, 1);
            }
            tc::commit(bar_mma);  // (and the successor state's product, issued in (6))
            mma_out = true;
            ph_out = ph;
        }
    }
    // the park's gamma_last M term: M is read again from where (0) got it (L2 still holds it),
    // into registers while the products of (9) run
    const float4* msrc;  // (no initialisers here: the error exits jump past this point)
    int sstride;
    float4 mpre[KDA ? 1 : 16];
    msrc = m_unit
        ? reinterpret_cast<const float4*>(A.ws + A.o_Mc + ch * (long long)(TD * TD)) + 16 * hc * TD + row
        : reinterpret_cast<const float4*>(A.ckpt + (head * A.n_ck + seg) * (long long)(TD * TD) + row * TD + 64 * hc);
    sstride = m_unit ? TD : 1;
    if (!KDA && compute && park_next) {
#pragma unroll
        for (int u = 0; u < (KDA ? 1 : 16); ++u) mpre[u] = __ldg(msrc + u * sstride);
    }
    ok = tc::mbar_wait(bar_mma, ph);
    if (issuer && ok) mma_out = false;
    tc::fence_after();
    // (10) this value head's dq and dk (rows i = row, tokens [tb, tb + 16)) -> workspace
    if (compute && ok) {
        if (!KDA) {  // (KDA: written in step (9))
            float dq[16], dk[16];
            tc::ld16(tc::taddr(tmem, warp, kC2 + tb), dq);
            tc::ld16(tc::taddr(tmem, warp, kC2 + BC + tb), dk);
            tc::wait_ld();
            float* dqo = A.ws + A.o_dqM + ch * (BC * TD) + row;
            float* dko = A.ws + A.o_dkM + ch * (BC * TD) + row;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int t = tb + e;
                dqo[t * TD] = dq[e];
                dko[t * TD] = __fmaf_rn(sR[t], d3[e], dk[e]);
            }
        }
        if (park_next) {
            // the next chunk's entry state M_N = gamma_last M + (r Delta)^T K, row `row`, this
            // thread's 64 columns, parked in the unit layout (a warp writes 512-byte runs).
            const float gl = sGam[BC - 1];
            float4* dst = reinterpret_cast<float4*>(A.ws + A.o_Mc + (ch + 1) * (long long)(TD * TD)) + 16 * hc * TD + row;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float v[32];
                tc::ld32(tc::taddr(tmem, warp, kCN + 64 * hc + 32 * h2), v);
                tc::wait_ld();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int u = 8 * h2 + q;
                    const float4 mo = KDA ? __ldg(msrc + u * sstride) : mpre[KDA ? 0 : u];
                    float4 gq = make_float4(gl, gl, gl, gl);
                    if (KDA)  // columns 4 u .. 4 u + 3 of this half decay by their own gamma_last
                        gq = *reinterpret_cast<const float4*>(sm + kSGl + 64 * hc + 4 * u);
                    dst[u * TD] = make_float4(__fmaf_rn(gq.x, mo.x, v[4 * q]), __fmaf_rn(gq.y, mo.y, v[4 * q + 1]),
                                              __fmaf_rn(gq.z, mo.z, v[4 * q + 2]), __fmaf_rn(gq.w, mo.w, v[4 * q + 3]));
                }
            }
        }
    }
    if (!ok) s_err = 1;
done:
    __syncthreads();
    if (s_err && issuer) {
        atomicExch(&g_tcg_status, kStatusTimeout);
        // the products in flight must be done before the tensor memory is released; if they
        // are not, say so (bit 8: the tensor memory may be written after its release)
        if (mma_out && !tc::mbar_wait(bar_mma, ph_out)) atomicOr(&g_tcg_status, 1 << 8);
        if (park_out && !tc::mbar_wait(bar_park, 0)) atomicOr(&g_tcg_status, 1 << 8);
        for (int b = 0; b < 7; ++b)  // let this CTA's bulk copies land before it exits
            if (s_armed & (1 << b)) tc::mbar_wait(bars + b, 0);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_free(tmem, kCols);
}

// dq, dk of each key head: the value heads' parts summed in ascending order (and, with the
// sequence broadcast, the value sequences of each q/k sequence nq, ascending); the chunks of
// [c_lo, c_hi), or with grad_loc = k >= 0 those at place k of their segment.
__global__ void __launch_bounds__(256) gdn_tc_dqdk_sum_kernel(const ChunkArgs A)
{
    const int c = A.grad_loc < 0 ? A.c_lo + blockIdx.x : (A.c_lo / A.cps + blockIdx.x) * A.cps + A.grad_loc;
    const int hk = blockIdx.y, nq = blockIdx.z;
    const int seg = c / A.cps, loc = c - seg * A.cps;
    const int t0 = seg * A.C + loc * BC;
    const int nb = min(BC, min(A.T, seg * A.C + A.C) - t0);
    const int r = A.H_v / A.H_k;
    for (int idx = threadIdx.x; idx < nb * (TD / 4); idx += 256) {
        const int t = idx / (TD / 4), i4 = idx - t * (TD / 4);
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f), k = q;
        for (int j = 0; j < A.rep; ++j) {
            const int n = nq * A.rep + j;
            for (int rho = 0; rho < r; ++rho) {
                const long long ch = ((long long)n * A.H_v + hk + rho * A.H_k) * A.n_chunks + c;
                const float4 a = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_dqM + ch * (BC * TD) + t * TD) + i4);
                const float4 b = __ldg(reinterpret_cast<const float4*>(A.ws + A.o_dkM + ch * (BC * TD) + t * TD) + i4);
                q = make_float4(__fadd_rn(q.x, a.x), __fadd_rn(q.y, a.y), __fadd_rn(q.z, a.z), __fadd_rn(q.w, a.w));
                k = make_float4(__fadd_rn(k.x, b.x), __fadd_rn(k.y, b.y), __fadd_rn(k.z, b.z), __fadd_rn(k.w, b.w));
            }
        }
        const long long o = (((long long)nq * A.T + t0 + t) * A.H_k + hk) * TD;
        reinterpret_cast<float4*>(A.dq + o)[i4] = q;
        reinterpret_cast<float4*>(A.dk + o)[i4] = k;
    }
}

template <bool KDA>
static int launch_tc_grad_t(const ChunkArgs& a, cudaStream_t s)
{
    int e = (int)cudaFuncSetAttribute(gdn_tc_grad_kernel<KDA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kGSmemBytes);
    if (e) return e;
    const int units = tc_grad_units(a);
    if (units <= 0) return 0;
    // A launch for place k > 0 follows the one for place k - 1 on the same stream and reads
    // its parks only after griddepcontrol.wait: it may start in that launch's tail.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units, a.H_v, a.N);
    cfg.blockDim = dim3(GT);
    cfg.dynamicSmemBytes = kGSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = a.grad_loc > 0 ? 1 : 0;
    e = (int)cudaLaunchKernelEx(&cfg, gdn_tc_grad_kernel<KDA>, a);
    if (e) return e;
    return (int)cudaGetLastError();
}

int launch_tc_grad(const ChunkArgs& a, void* stream)
{
    return a.kda ? launch_tc_grad_t<true>(a, (cudaStream_t)stream) : launch_tc_grad_t<false>(a, (cudaStream_t)stream);
}

int tc_grad_units(const ChunkArgs& a)
{
    if (a.c_hi <= a.c_lo) return 0;
    if (a.grad_loc < 0) return a.c_hi - a.c_lo;
    // segments of [c_lo, c_hi) (segment-aligned) with a chunk at place grad_loc: all but
    // possibly the last, which may be short
    const int s_lo = a.c_lo / a.cps, s_hi = (a.c_hi + a.cps - 1) / a.cps;
    const int last = a.c_hi - (s_hi - 1) * a.cps;  // chunks of the range's last segment
    return (s_hi - s_lo) - (a.grad_loc >= last ? 1 : 0);
}

int launch_tc_dqdk_sum(const ChunkArgs& a, void* stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    const int units = tc_grad_units(a);  // every chunk of [c_lo, c_hi), or those at place grad_loc
    if (units <= 0) return 0;
    gdn_tc_dqdk_sum_kernel<<<dim3(units, a.H_k, a.N / a.rep), 256, 0, s>>>(a);
    return (int)cudaGetLastError();
}

int tc_grad_take_status(void* stream, int* status)
{
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    int e = (int)cudaMemcpyFromSymbolAsync(&v, g_tcg_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (!e) e = (int)cudaStreamSynchronize(s);
    if (e) return e;
    if (v) {
        const int zero = 0;
        e = (int)cudaMemcpyToSymbolAsync(g_tcg_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (!e) e = (int)cudaStreamSynchronize(s);
    }
    *status = v;
    return e;
}

}  // namespace gdn
