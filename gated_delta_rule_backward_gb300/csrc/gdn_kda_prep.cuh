// gdn_kda_prep.cuh -- the chunk-parallel prep of the per-key-column (KDA) gate in chunked
// form at head size 128, for the tensor-core chains and gradient step.  Included by
// gdn_chunk.cu (it uses that file's row loaders, warp-level products and triangular
// inverse).
//
// The gate of Kimi Delta Attention (meTile "Training kernels and gradients", section
// "Recurrent delta attention": a per-key-channel log-decay) decays column i of the state
// by a_i = exp(g_i) per token.  Regrouped by chunks of BC tokens with entering state M_c,
// and with, per key column i,
//   gamma[t]    = a[0] ... a[t]                    (the decay from the chunk start)
//   E[t][tau]   = a[tau + 1] ... a[t]   (tau <= t) (the decay between two tokens)
//   R[tau]      = E[BC - 1][tau]                   (the decay to the chunk end)
// the recurrence is, exactly:
//   Aqk[t][tau] = sum_i q[t][i] k[tau][i] E[t][tau][i]   (tau <= t, else 0)
//   Akk[t][tau] = sum_i k[t][i] k[tau][i] E[t][tau][i]   (tau <  t, else 0)
//   Z = (I + diag(beta) Akk)^-1,  T = Z diag(beta)
//   X = V - (K (.) gamma) M_c^T,  Delta = T X                  (row t = delta_t)
//   Y = scale ((Q (.) gamma) M_c^T + Aqk Delta)
//   M_end = M_c diag(gamma[BC - 1]) + Delta^T (K (.) R)
// (by induction on t: the decayed state before token t is M_c diag(gamma[t]) +
// sum_{tau < t} delta_tau (k_tau (.) E[t][tau])^T).  The decay products are formed by
// running products of a along t, never as exp(G_t) / exp(G_tau): no quotient of two small
// numbers appears, so nothing overflows however strong the decay.
//
// The scalar gate's kernels then run unchanged in form: the state chain takes Q (.) gamma
// (per value head) where it took Q, [scale Aqk; (K (.) R)^T] where it took
// [scale QD; (r K)^T], gamma = 1 and decays M column by column with gamma[BC - 1]; the dM
// chain takes K (.) R, [Q (.) gamma; K (.) gamma] and r = gamma = 1.

namespace gdn {

// Reduces 16 values across the warp: afterwards lane l holds the warp-wide sum of v[l / 2]
// (bits 4..1 of the lane index).  15 + 1 shuffles instead of 16 x 5.
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const bool up = lane & 16;
        const float send = up ? v[j] : v[j + 8], keep = up ? v[j + 8] : v[j];
        v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const bool up = lane & 8;
        const float send = up ? v[j] : v[j + 4], keep = up ? v[j + 4] : v[j];
        v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const bool up = lane & 4;
        const float send = up ? v[j] : v[j + 2], keep = up ? v[j + 2] : v[j];
        v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    {
        const bool up = lane & 2;
        const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
        v[0] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
    return __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

// The decay-weighted products of one chunk: Aqk (lower, diagonal included) and Akk (strictly
// lower) into row-major BC x LDB tiles that are zero on entry, and R (the decay of each token
// to the chunk end, per column) into Rs.  As holds a = exp(g) (rows t, padded rows 1).  Warp
// w takes the columns tau of {w, 15 - w, 16 + w, 31 - w} (66 (t, tau) pairs each); its lanes
// hold 4 key columns each and walk t upwards from tau, carrying E[t][tau] as a running
// product, 8 tokens per warp reduction.
__device__ __forceinline__ void kda_decay_products(const float* Qs, const float* Ks, const float* As,
                                                   float* Aqk, float* Akk, float* Rs, int ld, int tid)
{
    const int warp = tid >> 5, lane = tid & 31, i0 = 4 * lane;
    const int taus[4] = {warp, 15 - warp, 16 + warp, 31 - warp};
#pragma unroll 1
    for (int s = 0; s < 4; ++s) {
        const int tau = taus[s];
        const float4 kt = *reinterpret_cast<const float4*>(Ks + tau * ld + i0);
        float4 e = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll 1
        for (int t0 = tau; t0 < BC; t0 += 8) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = t0 + j;
                float qk = 0.f, kk = 0.f;
                if (t < BC) {
                    if (t > tau) {
                        const float4 a = *reinterpret_cast<const float4*>(As + t * ld + i0);
                        e = make_float4(__fmul_rn(e.x, a.x), __fmul_rn(e.y, a.y), __fmul_rn(e.z, a.z),
                                        __fmul_rn(e.w, a.w));
                    }
                    const float4 q = *reinterpret_cast<const float4*>(Qs + t * ld + i0);
                    const float4 k = *reinterpret_cast<const float4*>(Ks + t * ld + i0);
                    const float4 w = make_float4(__fmul_rn(kt.x, e.x), __fmul_rn(kt.y, e.y), __fmul_rn(kt.z, e.z),
                                                 __fmul_rn(kt.w, e.w));
                    qk = __fmaf_rn(q.w, w.w, __fmaf_rn(q.z, w.z, __fmaf_rn(q.y, w.y, __fmul_rn(q.x, w.x))));
                    if (t > tau)
                        kk = __fmaf_rn(k.w, w.w, __fmaf_rn(k.z, w.z, __fmaf_rn(k.y, w.y, __fmul_rn(k.x, w.x))));
                    if (t == BC - 1) *reinterpret_cast<float4*>(Rs + tau * ld + i0) = e;
                }
                v[j] = qk;
                v[8 + j] = kk;
            }
            const float sum = warp_sum16(v, lane);
            const int idx = lane >> 1, t = t0 + (idx & 7);
            if ((lane & 1) == 0 && t < BC) {
                if (idx < 8)
                    Aqk[t * LDB + tau] = sum;
                else
                    Akk[t * LDB + tau] = sum;
            }
        }
    }
}

// Prep of the KDA gate, head size 128: one CTA per (chunk, value head, sequence), the value
// heads of one key head in adjacent CTAs.  Forward (want_wu): the state chain's operands.
// Backward (want_factors): the gradient step's factors and tiles, and the dM chain's operands.
__global__ void __launch_bounds__(CT, 2) gdn_kda_prep_kernel(const ChunkArgs A)
{
    constexpr int D = 128;
    constexpr int ld = Ld<D>::v;
    const int slot = blockIdx.x % A.H_v, c = A.c_lo + blockIdx.x / A.H_v, n = blockIdx.y, tid = threadIdx.x;
    const int h = (slot % (A.H_v / A.H_k)) * A.H_k + slot / (A.H_v / A.H_k);
    const int hk = h % A.H_k;
    const ChunkPos cp = chunk_pos(A, c);
    const long long ch = ((long long)n * A.H_v + h) * A.n_chunks + c;

    extern __shared__ __align__(16) float sm[];
    float* Qs = sm;                 // q rows
    float* Ks = Qs + BC * ld;       // k rows (forward: K (.) gamma at the end)
    float* Vs = Ks + BC * ld;       // v rows, then U (forward); dY rows (backward)
    float* Gs = Vs + BC * ld;       // a = exp(g), then gamma
    float* Rs = Gs + BC * ld;       // R
    float* Aqk = Rs + BC * ld;      // BC x LDB each
    float* Akk = Aqk + BC * LDB;
    float* Zs = Akk + BC * LDB;
    float* Ts = Zs + BC * LDB;
    float* bs = Ts + BC * LDB;      // beta (BC)

    const long long tq = (long long)(n / A.rep) * A.qs0 + (long long)cp.t0 * A.qs1 + (long long)hk * A.qs2;
    const long long tk = (long long)(n / A.rep) * A.ks0 + (long long)cp.t0 * A.ks1 + (long long)hk * A.ks2;
    const long long tok0 = (long long)n * A.T + cp.t0;
    {  // every load in flight before the first store; g rows are [token][value head][d]
        float4 rq[D / 32], rk[D / 32], rv[D / 32], rg[D / 32];
        pf_rows<D>(rq, A.q + tq, A.qs1, cp.nb, A.vec_q, tid);
        pf_rows<D>(rk, A.k + tk, A.ks1, cp.nb, A.vec_k, tid);
        if (A.want_wu) {
            const long long tv = (long long)n * A.vs0 + (long long)cp.t0 * A.vs1 + (long long)h * A.vs2;
            pf_rows<D>(rv, A.v + tv, A.vs1, cp.nb, A.vec_v, tid);
        } else {
            const long long tg = (long long)n * A.gys0 + (long long)cp.t0 * A.gys1 + (long long)h * A.gys2;
            pf_rows<D>(rv, A.gy + tg, A.gys1, cp.nb, A.vec_gy, tid);
        }
        pf_rows<D>(rg, A.g + (tok0 * A.H_v + h) * D, (long long)A.H_v * D, cp.nb, A.vec_g, tid);
        if (tid < BC) bs[tid] = tid < cp.nb ? __ldg(A.beta + (tok0 + tid) * A.H_v + h) : 0.f;
        put_rows<D>(Qs, ld, rq, tid);
        put_rows<D>(Ks, ld, rk, tid);
        put_rows<D>(Vs, ld, rv, tid);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)  // a = exp(g); padded rows have g = 0, a = 1
            rg[kk] = make_float4(expf(rg[kk].x), expf(rg[kk].y), expf(rg[kk].z), expf(rg[kk].w));
        put_rows<D>(Gs, ld, rg, tid);
        for (int idx = tid; idx < 2 * BC * LDB; idx += CT) Aqk[idx] = 0.f;  // Aqk, Akk
    }
    __syncthreads();
    kda_decay_products(Qs, Ks, Gs, Aqk, Akk, Rs, ld, tid);
    __syncthreads();
    if (tid < D) {  // gamma: running product of a down column tid
        float gm = 1.f;
        for (int t = 0; t < BC; ++t) {
            gm = __fmul_rn(gm, Gs[t * ld + tid]);
            Gs[t * ld + tid] = gm;
        }
        A.ws[A.o_gL + ch * D + tid] = gm;
    }
    for (int idx = tid; idx < BC * BC; idx += CT) {
        const int t = idx / BC, tau = idx - t * BC;
        Ts[t * LDB + tau] = (tau < t) ? __fmul_rn(bs[t], Akk[t * LDB + tau]) : 0.f;
        Zs[t * LDB + tau] = 0.f;
    }
    if (tid < BC) {  // the scalar gate's gamma and r slots: ones (the decay is in the operands)
        A.ws[A.o_gam + ch * BC + tid] = 1.f;
        A.ws[A.o_r + ch * BC + tid] = 1.f;
    }
    __syncthreads();
    unit_lower_inverse(Ts, Zs, Aqk, bs, tid);  // Aqk's strict upper half is zero

    if (A.want_wu) {
        // ---- forward: the state chain's operands
        float* w1 = A.ws + A.o_W1 + ch * kTcWElems;
        float* q1 = A.ws + A.o_Q1 + ch * kTcQElems;
        float* b23 = A.ws + A.o_B23 + ch * kTcB23Elems;
        float* u = A.ws + A.o_U + ch * (BC * D);
        int fm, fn;
        mma_32x128_origin(tid, fm, fn);
        float c4[4][4];
        mma_32x128x32<false>(c4, Ts, LDB, Vs, ld, tid);  // U = T V
        for (int uu = tid; uu < BC * (D / 8); uu += CT) {  // Q (.) gamma, row-group-major units
            const int t = ((uu >> 7) << 3) + (uu & 7), kc = (uu >> 3) & 15;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(Qs[t * ld + 8 * kc + e], Gs[t * ld + 8 * kc + e]);
            tc::put_bf16x8(q1, kTcQElems / 2, uu, x);
        }
        for (int idx = tid; idx < 160 * (BC / 8); idx += CT) {  // [scale Aqk; (K (.) R)^T]
            const int r = idx % 160, kc = idx / 160;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int tau = 8 * kc + e;
                x[e] = (r < BC) ? __fmul_rn(A.scale, Aqk[r * LDB + tau])
                                : __fmul_rn(Ks[tau * ld + r - BC], Rs[tau * ld + r - BC]);
            }
            tc::put_bf16x8(b23, kTcB23Elems / 2, idx, x);
        }
        __syncthreads();  // Vs, Ks are read above: U and K (.) gamma replace them
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                *reinterpret_cast<float2*>(Vs + (fm + 8 * hf) * ld + fn + 8 * nt) =
                    make_float2(c4[nt][2 * hf], c4[nt][2 * hf + 1]);
        for (int idx = tid; idx < BC * D; idx += CT) {
            const int t = idx / D, i = idx - t * D;
            Ks[t * ld + i] = __fmul_rn(Ks[t * ld + i], Gs[t * ld + i]);
        }
        __syncthreads();
        mma_32x128x32<false>(c4, Ts, LDB, Ks, ld, tid);  // W = T (K (.) gamma)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int off = tc::kmaj16_rg(fm + 8 * hf, fn + 8 * nt, D);
                uint32_t hi, lo;
                tc::split_bf16x2(c4[nt][2 * hf], c4[nt][2 * hf + 1], hi, lo);
                reinterpret_cast<uint32_t*>(w1)[off] = hi;
                reinterpret_cast<uint32_t*>(w1 + kTcWElems / 2)[off] = lo;
            }
        for (int idx = tid; idx < (BC / 4) * D; idx += CT) {  // U^T, unit = b * 128 + j
            const int j = idx % D, b = idx / D;
            *reinterpret_cast<float4*>(u + 4 * idx) =
                make_float4(Vs[(4 * b) * ld + j], Vs[(4 * b + 1) * ld + j], Vs[(4 * b + 2) * ld + j],
                            Vs[(4 * b + 3) * ld + j]);
        }
    }
    if (!A.want_factors) return;

    // ---- backward: the gradient step's factors and tiles, the dM chain's operands
    {
        float* fT = A.ws + A.o_Tr + ch * (BC * BC);
        float* fZ = A.ws + A.o_Z + ch * (BC * BC);
        float* fK = A.ws + A.o_KK + ch * (BC * BC);
        float* fQ = A.ws + A.o_QK + ch * (BC * BC);
        for (int idx = tid; idx < BC * BC; idx += CT) {
            const int t = idx / BC, tau = idx - t * BC;
            fT[idx] = Ts[t * LDB + tau];
            fZ[idx] = Zs[t * LDB + tau];
            fK[idx] = Akk[t * LDB + tau];
            fQ[idx] = Aqk[t * LDB + tau];
        }
        float4* gg = reinterpret_cast<float4*>(A.ws + A.o_kGam + ch * (BC * D));
        float4* rr = reinterpret_cast<float4*>(A.ws + A.o_kR + ch * (BC * D));
        for (int idx = tid; idx < BC * (D / 4); idx += CT) {  // gamma, R: fp32 rows t
            const int t = idx / (D / 4), i4 = idx - t * (D / 4);
            gg[idx] = *reinterpret_cast<const float4*>(Gs + t * ld + 4 * i4);
            rr[idx] = *reinterpret_cast<const float4*>(Rs + t * ld + 4 * i4);
        }
    }
    float* blk = A.ws + A.o_DS + ch * kTcDsElems;
    float* kblk = A.ws + A.o_DK + ch * kTcDkElems;
    {  // E^T = scale Aqk^T dY (rows t), stored as E (rows j), fp32
        float c4[4][4];
        mma_32x128x32<true>(c4, Aqk, LDB, Vs, ld, tid);
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
                    e[4 * ((t >> 2) * D + j) + (t & 3)] = __fmul_rn(A.scale, c4[nt][2 * hf + x]);
                }
    }
    // bf16 tiles, k-chunk-major: 16-byte unit kc * R + row holds 8 consecutive K elements
    for (int idx = tid; idx < (BC / 8) * D; idx += CT) {  // scale dY^T, unit kc * 128 + j
        const int j = idx % D, kc = idx / D;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(A.scale, Vs[(8 * kc + e) * ld + j]);
        tc::put_bf16x8(blk + kDsG, 128 * 32 / 2, idx, x);
    }
    for (int idx = tid; idx < (D / 8) * BC; idx += CT) {  // K (.) R and K (.) gamma, rows t
        const int t = idx % BC, kc = idx / BC;
        float x[8], y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float kv = Ks[t * ld + 8 * kc + e];
            x[e] = __fmul_rn(kv, Rs[t * ld + 8 * kc + e]);
            y[e] = __fmul_rn(kv, Gs[t * ld + 8 * kc + e]);
        }
        tc::put_bf16x8(kblk + kDkKb, 32 * 128 / 2, idx, x);
        tc::put_bf16x8(A.ws + A.o_KG + ch * kTcKdaTile, 32 * 128 / 2, idx, y);
    }
    for (int idx = tid; idx < (2 * BC / 8) * D; idx += CT) {  // [(Q (.) gamma)^T | (K (.) gamma)^T] rows i
        const int i = idx % D, kc = idx / D;
        const float* src = kc < BC / 8 ? Qs : Ks;
        const int t0 = 8 * (kc % (BC / 8));
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(src[(t0 + e) * ld + i], Gs[(t0 + e) * ld + i]);
        tc::put_bf16x8(kblk + kDkQKT, 128 * 64 / 2, idx, x);
    }
    for (int idx = tid; idx < (BC / 8) * D; idx += CT) {  // (K (.) R)^T rows i, unit kc * 128 + i
        const int i = idx % D, kc = idx / D;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(Ks[(8 * kc + e) * ld + i], Rs[(8 * kc + e) * ld + i]);
        tc::put_bf16x8(A.ws + A.o_KRT + ch * kTcKdaTile, 128 * 32 / 2, idx, x);
    }
    for (int idx = tid; idx < (BC / 8) * BC; idx += CT) {  // T^T rows t: T[t'][t], unit kc * 32 + t
        const int t = idx % BC, kc = idx / BC;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = Ts[(8 * kc + e) * LDB + t];
        tc::put_bf16x8(blk + kDsTT, 32 * 32 / 2, idx, x);
    }
    if (tid < BC) {
        blk[kDsR + tid] = 1.f;
        blk[kDsGam + tid] = 1.f;
    }
}

}  // namespace gdn
