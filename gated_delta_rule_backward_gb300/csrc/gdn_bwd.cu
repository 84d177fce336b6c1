// gdn_bwd.cu -- backward of the gated delta rule (GATED_DELTA_NET_BACK) for sm_103a.
//
// Grid (P, H_v, N): CTA p owns rows [p R, p R + R) of M = S^T and of its cotangent dM
// for one (sequence, value head).  The dM chain is row-local ("metal:
// GATED_DELTA_NET_BACK", PR #16 review: "Each row pass writes only its own row"), so
// the only cross-row quantities are outputs -- the column sums dq, dk, (KDA) dg and the
// scalars dbeta, (scalar-gate) dg -- and they never feed back.  They are summed over a
// warp's row groups with shuffles, over the CTA's warps in shared memory (fixed order),
// and over the P row blocks and the r value heads sharing a key head by
// gdn_reduce_kernel (fixed order, no atomics).
//
// Checkpointed recompute, two levels (PR #16 body: "checkpointed recompute
// (C ~ sqrt(T))"): the segment of C tokens that starts at checkpoint s is first walked
// forward to drop a sub-checkpoint every c2 tokens (level 1, into the workspace); then
// for each sub-segment, last first, its c2 decayed states S'_t = a_t (.) M_{t-1} are
// recomputed into a shared-memory ring (level 2) and walked in reverse.  The recompute
// runs the forward's own step function, so every state is bit-identical to the
// forward's and the result does not depend on C or c2.
//
// Reverse step for token t, per element of a row j (PR #16 review, term by term):
//   M_t = S' + k delta^T                  (recomputed from the ring)
//   dq_i   += scale gy_j M_t[j][i]         dM += scale gy_j q_i
//   dd_j    = sum_i dM[j][i] k_i           dk_i += dM[j][i] delta_j   (dM before du)
//   du_j    = -beta dd_j                   dk_i += S'[j][i] du_j
//   dS'     = dM + k du^T                  dg   += dS' (.) S'
//   dM      = a (.) dS'
//   dv_j = beta dd_j, dbeta += dd_j (v_j - u_j)
//
// D is the column width the kernel computes in (S_k, or 32 for S_k = 16 with zero padding
// columns); the S_v rows are the grid's row blocks, independent of S_k.
#include <cuda_runtime.h>

#include "gdn_device.cuh"

namespace gdn {

__device__ __forceinline__ float4 fmav4(float4 a, float4 b, float4 acc)
{
    return make_float4(__fmaf_rn(a.x, b.x, acc.x), __fmaf_rn(a.y, b.y, acc.y),
                       __fmaf_rn(a.z, b.z, acc.z), __fmaf_rn(a.w, b.w, acc.w));
}

template <int D, int RT, bool KDA>
__global__ void __launch_bounds__(256, 1) gdn_bwd_kernel(const BwdArgs A)
{
    constexpr int NV = D / 32;
    constexpr int NQ = KDA ? 3 : 2;  // column quantities: dq, dk (, dg)
    constexpr int NX = 4 * NV * NQ;  // column partials per lane per token
    constexpr int NY = NX / 4;       // after the reduce-scatter over row groups
    const int NT = blockDim.x, W = NT >> 5;
    const int R = 4 * RT * W;
    const int P = gridDim.x;
    const int p = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h % A.H_k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, cl = lane & 7;
    const int lrow0 = warp * 4 * RT + grp * RT;
    const int row0 = p * R + lrow0;
    const int c2 = A.c2;
    const int ncol = NQ * D;

    extern __shared__ __align__(16) float sm[];
    const BwdSmem L = bwd_smem_layout(D, RT, W, c2, KDA);
    float4* ring = reinterpret_cast<float4*>(sm + L.ring);  // [c2][RT*NV][NT]
    float* sk = sm + L.sk;
    float* sq = sm + L.sq;
    float* sa = sm + L.sa;
    float* sb = sm + L.sb;
    float* sv = sm + L.sv;
    float* sgy = sm + L.sgy;
    float* sdel = sm + L.sdel;
    float* svmu = sm + L.svmu;
    float* sdd = sm + L.sdd;
    float* scol = sm + L.scol;
    float* sdg = sm + L.sdg;

    const long long head = (long long)n * A.H_v + h;
    const long long cta = head * P + p;
    const int SK = A.SK, DV = A.DV;
    float4* sub = reinterpret_cast<float4*>(A.sub) +
                  cta * (long long)(A.nsub_max > 1 ? A.nsub_max - 1 : 0) * (RT * NV * NT);

    float4 dm[RT][NV];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int v = 0; v < NV; ++v)
            dm[r][v] = A.dstate_T ? ld_state4(A.dstate_T + (head * DV + row0 + r) * SK, v, cl, SK)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    zero_pad_cols(sk, c2, SK, D, tid, NT);
    zero_pad_cols(sq, c2, SK, D, tid, NT);
    if (KDA) zero_pad_cols(sa, c2, SK, D, tid, NT);

    // Stage the inputs of tokens [ta, ta + nt) in shared memory.
    auto load_tile = [&](int ta, int nt, bool for_walk) {
        const long long tok0 = (long long)n * A.T + ta;
        load_rows(sk, A.k + (long long)(n / A.rep) * A.ks0 + (long long)ta * A.ks1 + hk * A.ks2, A.ks1, nt, SK,
                  A.vec_k, tid, NT, D);
        if (KDA) {
            load_rows_exp(sa, A.g + (tok0 * A.H_v + h) * SK, (long long)A.H_v * SK, nt, SK,
                          A.vec_g, tid, NT, D);
        } else {
            for (int tt = tid; tt < nt; tt += NT) sa[tt] = expf(__ldg(A.g + (tok0 + tt) * A.H_v + h));
        }
        for (int tt = tid; tt < nt; tt += NT) sb[tt] = __ldg(A.beta + (tok0 + tt) * A.H_v + h);
        load_rows(sv, A.v + n * A.vs0 + (long long)ta * A.vs1 + h * A.vs2 + p * R, A.vs1, nt, R,
                  A.vec_v, tid, NT);
        if (for_walk) {
            load_rows(sq, A.q + (long long)(n / A.rep) * A.qs0 + (long long)ta * A.qs1 + hk * A.qs2, A.qs1, nt, SK,
                      A.vec_q, tid, NT, D);
            load_rows(sgy, A.gy + n * A.gys0 + (long long)ta * A.gys1 + h * A.gys2 + p * R,
                      A.gys1, nt, R, A.vec_gy, tid, NT);
        }
    };

    auto load_state = [&](float4 (&m)[RT][NV], const float* src) {  // rows of SK floats
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int v = 0; v < NV; ++v) m[r][v] = ld_state4(src + (lrow0 + r) * SK, v, cl, SK);
    };

    for (int s = A.n_ck - 1; s >= 0; --s) {
        const int t0 = s * A.C, t1 = min(A.T, t0 + A.C);
        const int nsub = (t1 - t0 + c2 - 1) / c2;
        // ckpt[n][h][s], this CTA's rows
        const float* cks = A.ckpt + ((head * A.n_ck + s) * DV + p * R) * SK;

        // ---- level 1: sub-checkpoints at tokens t0 + b c2, b = 1 .. nsub-1 ----
        if (nsub > 1) {
            float4 m[RT][NV];
            load_state(m, cks);
            for (int b = 0; b < nsub - 1; ++b) {
                const int ta = t0 + b * c2;
                __syncthreads();
                load_tile(ta, c2, false);
                __syncthreads();
                for (int tt = 0; tt < c2; ++tt) {
                    float4 kv[NV], av[NV], sp[RT][NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        kv[v] = lds_cols<D>(sk + tt * D, v, cl);
                        if (KDA) av[v] = lds_cols<D>(sa + tt * D, v, cl);
                    }
                    float vj[RT], u[RT], delta[RT];
#pragma unroll
                    for (int r = 0; r < RT; ++r) vj[r] = sv[tt * R + lrow0 + r];
                    recurrence_step<NV, RT, KDA>(m, sp, kv, av, KDA ? 0.f : sa[tt], sb[tt], vj, u,
                                                 delta);
                }
                float4* dst = sub + (long long)b * (RT * NV * NT);
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int v = 0; v < NV; ++v) dst[(r * NV + v) * NT + tid] = m[r][v];
            }
        }

        // ---- level 2 + reverse walk, one sub-segment at a time, last first ----
        for (int b = nsub - 1; b >= 0; --b) {
            const int ta = t0 + b * c2, tb = min(t1, ta + c2), nt = tb - ta;
            __syncthreads();
            load_tile(ta, nt, true);
            __syncthreads();

            {  // recompute the sub-segment's states into the ring
                float4 m[RT][NV];
                if (b == 0) {
                    load_state(m, cks);
                } else {
                    const float4* src = sub + (long long)(b - 1) * (RT * NV * NT);
#pragma unroll
                    for (int r = 0; r < RT; ++r)
#pragma unroll
                        for (int v = 0; v < NV; ++v) m[r][v] = src[(r * NV + v) * NT + tid];
                }
                for (int tt = 0; tt < nt; ++tt) {
                    float4 kv[NV], av[NV], sp[RT][NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        kv[v] = lds_cols<D>(sk + tt * D, v, cl);
                        if (KDA) av[v] = lds_cols<D>(sa + tt * D, v, cl);
                    }
                    float vj[RT], u[RT], delta[RT];
#pragma unroll
                    for (int r = 0; r < RT; ++r) vj[r] = sv[tt * R + lrow0 + r];
                    recurrence_step<NV, RT, KDA>(m, sp, kv, av, KDA ? 0.f : sa[tt], sb[tt], vj, u,
                                                 delta);
                    float4* slot = ring + tt * (RT * NV * NT);
#pragma unroll
                    for (int r = 0; r < RT; ++r)
#pragma unroll
                        for (int v = 0; v < NV; ++v) slot[(r * NV + v) * NT + tid] = sp[r][v];
                    if (cl == 0) {
#pragma unroll
                        for (int r = 0; r < RT; ++r) {
                            sdel[tt * R + lrow0 + r] = delta[r];
                            svmu[tt * R + lrow0 + r] = __fsub_rn(vj[r], u[r]);
                        }
                    }
                }
            }
            __syncwarp();

            for (int tt = nt - 1; tt >= 0; --tt) {
                float4 kv[NV], qv[NV], av[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    kv[v] = lds_cols<D>(sk + tt * D, v, cl);
                    qv[v] = lds_cols<D>(sq + tt * D, v, cl);
                    if (KDA) av[v] = lds_cols<D>(sa + tt * D, v, cl);
                }
                const float as = KDA ? 0.f : sa[tt];
                const float beta = sb[tt];
                float sg[RT], del[RT];
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    sg[r] = __fmul_rn(A.scale, sgy[tt * R + lrow0 + r]);
                    del[r] = sdel[tt * R + lrow0 + r];
                }
                float4 spv[RT][NV];
                const float4* slot = ring + tt * (RT * NV * NT);
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int v = 0; v < NV; ++v) spv[r][v] = slot[(r * NV + v) * NT + tid];

                const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
                float4 Xq[NV], Xk[NV], Xg[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v) Xq[v] = Xk[v] = Xg[v] = z4;
                float dd[RT];
#pragma unroll
                for (int r = 0; r < RT; ++r) {
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const float4 mt = fma4(kv[v], del[r], spv[r][v]);  // M_t (forward's bits)
                        Xq[v] = axpy4(mt, sg[r], Xq[v]);                    // dq: M_t^T (scale gy)
                        dm[r][v] = fma4(qv[v], sg[r], dm[r][v]);            // dM += scale gy q^T
                        Xk[v] = axpy4(dm[r][v], del[r], Xk[v]);             // dk: dM^T delta
                    }
                    dd[r] = dot_part<NV>(dm[r], kv);                        // dd = dM k
                }
#pragma unroll
                for (int r = 0; r < RT; ++r) dd[r] = rowsum8(dd[r]);
                float4 G4 = z4;
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    const float du = -__fmul_rn(beta, dd[r]);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        Xk[v] = axpy4(spv[r][v], du, Xk[v]);                // dk: S'^T du
                        dm[r][v] = fma4(kv[v], du, dm[r][v]);               // dS' = dM + k du^T
                        if (KDA)
                            Xg[v] = fmav4(dm[r][v], spv[r][v], Xg[v]);      // dg_i: dS' (.) S'
                        else
                            G4 = fmav4(dm[r][v], spv[r][v], G4);
                        dm[r][v] = KDA ? mul4(av[v], dm[r][v]) : mul4(as, dm[r][v]);  // a (.) dS'
                    }
                }
                if (cl == 0) {
#pragma unroll
                    for (int r = 0; r < RT; ++r) sdd[tt * R + lrow0 + r] = dd[r];
                }
                // column partials: reduce over the warp's row groups, park per warp in smem
                float X[NX];
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    X[4 * v + 0] = Xq[v].x; X[4 * v + 1] = Xq[v].y;
                    X[4 * v + 2] = Xq[v].z; X[4 * v + 3] = Xq[v].w;
                    X[4 * NV + 4 * v + 0] = Xk[v].x; X[4 * NV + 4 * v + 1] = Xk[v].y;
                    X[4 * NV + 4 * v + 2] = Xk[v].z; X[4 * NV + 4 * v + 3] = Xk[v].w;
                    if (KDA) {
                        X[8 * NV + 4 * v + 0] = Xg[v].x; X[8 * NV + 4 * v + 1] = Xg[v].y;
                        X[8 * NV + 4 * v + 2] = Xg[v].z; X[8 * NV + 4 * v + 3] = Xg[v].w;
                    }
                }
                float Y[NY];
                reduce_scatter_groups<NX>(X, Y, grp);
                float* cdst = scol + (warp * c2 + tt) * ncol;
                if constexpr (NY % 4 == 0) {
#pragma unroll
                    for (int i = 0; i < NY; i += 4) {
                        const int idx = grp * NY + i;
                        const int q = idx / (4 * NV), v = (idx % (4 * NV)) / 4;
                        reinterpret_cast<float4*>(cdst + q * D + 32 * v + 4 * cl)[0] =
                            make_float4(Y[i], Y[i + 1], Y[i + 2], Y[i + 3]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NY; ++i) {
                        const int idx = grp * NY + i;
                        const int q = idx / (4 * NV), rem = idx % (4 * NV);
                        cdst[q * D + 32 * (rem / 4) + 4 * cl + (rem % 4)] = Y[i];
                    }
                }
                if (!KDA)
                    sdg[(warp * c2 + tt) * 32 + lane] =
                        __fadd_rn(__fadd_rn(G4.x, G4.y), __fadd_rn(G4.z, G4.w));
            }
            __syncthreads();

            // ---- end of sub-segment: CTA partials out, dv out ----
            const long long tok0 = (long long)n * A.T + ta;
            for (int idx = tid; idx < nt * ncol; idx += NT) {
                const int tt = idx / ncol, col = idx - tt * ncol;
                float acc = scol[tt * ncol + col];
                for (int w = 1; w < W; ++w) acc = __fadd_rn(acc, scol[(w * c2 + tt) * ncol + col]);
                A.ws_col[(((tok0 + tt) * A.H_v + h) * P + p) * ncol + col] = acc;
            }
            for (int tt = warp; tt < nt; tt += W) {
                // dbeta partial: sum over this CTA's rows of dd_j (v_j - u_j)
                float db = 0.f;
                for (int j = lane; j < R; j += 32)
                    db = __fmaf_rn(sdd[tt * R + j], svmu[tt * R + j], db);
                float dg = 0.f;
                if (!KDA)
                    for (int w = 0; w < W; ++w) dg = __fadd_rn(dg, sdg[(w * c2 + tt) * 32 + lane]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    db = __fadd_rn(db, __shfl_xor_sync(kFull, db, o));
                    dg = __fadd_rn(dg, __shfl_xor_sync(kFull, dg, o));
                }
                if (lane == 0) {
                    float* sc = A.ws_sc + (((tok0 + tt) * A.H_v + h) * P + p) * 2;
                    sc[0] = db;
                    sc[1] = dg;
                }
            }
            for (int idx = tid; idx < nt * R; idx += NT) {
                const int tt = idx / R, j = idx - tt * R;
                A.dv[((tok0 + tt) * A.H_v + h) * DV + p * R + j] = __fmul_rn(sb[tt], sdd[idx]);
            }
        }
    }

    // dstate0 = dM after the last reverse step (the gradient of the initial state)
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        float* dst = A.dstate0 + (head * DV + row0 + r) * SK;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            if (32 * v + 4 * cl >= SK) continue;  // padding columns (S_k = 16)
            if (A.vec_ds0) {
                reinterpret_cast<float4*>(dst)[8 * v + cl] = dm[r][v];
            } else {
                float* e = dst + 32 * v + 4 * cl;
                e[0] = dm[r][v].x; e[1] = dm[r][v].y; e[2] = dm[r][v].z; e[3] = dm[r][v].w;
            }
        }
    }
}

// Fixed-order sums of the per-CTA partials: dq/dk over the value heads h_k, h_k + H_k,
// ... (ascending) and, inside each, over the P row blocks; dg (KDA), dbeta and dg
// (scalar gate) over the row blocks.
// The partials are D wide (the kernels' column width); the outputs SK wide (S_k).  With the
// sequence broadcast, dq/dk of q/k sequence nq sum the value sequences nq rep .. nq rep +
// rep - 1 in ascending order, each as above.
__global__ void __launch_bounds__(256) gdn_reduce_kernel(const ReduceArgs A)
{
    const long long nqk = (long long)(A.N / A.rep) * A.T * A.H_k * A.SK;
    const long long nhv = (long long)A.N * A.T * A.H_v;
    const long long ndg = A.kda ? nhv * A.SK : 0;
    const long long total = 2 * nqk + ndg + nhv;
    const int ncol = A.NQ * A.D;
    const int r = A.H_v / A.H_k;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        if (idx < 2 * nqk) {
            const int which = idx >= nqk;  // 0: dq, 1: dk
            const long long e = idx - which * nqk;
            const int i = (int)(e % A.SK);
            const long long tokhk = e / A.SK;  // (n*T + t)*H_k + hk
            const int hkk = (int)(tokhk % A.H_k);
            const long long tokq = tokhk / A.H_k;  // nq*T + t
            const long long nq = tokq / A.T, t = tokq - nq * A.T;
            // per value head: the sum over its P row blocks; then the value heads in
            // ascending order (equal, bit for bit, to summing explicitly replicated heads),
            // and the value sequences of the q/k sequence in ascending order
            float acc = 0.f;
            for (int j = 0; j < A.rep; ++j) {
                const long long tok = (nq * A.rep + j) * A.T + t;
                for (int rho = 0; rho < r; ++rho) {
                    const float* src = A.ws_col + ((tok * A.H_v + hkk + rho * A.H_k) * A.P) * ncol +
                                       which * A.D + i;
                    float part = 0.f;
                    for (int pp = 0; pp < A.P; ++pp) part = __fadd_rn(part, src[(long long)pp * ncol]);
                    acc = __fadd_rn(acc, part);
                }
            }
            (which ? A.dk : A.dq)[e] = acc;
        } else if (idx < 2 * nqk + ndg) {
            const long long e = idx - 2 * nqk;
            const int i = (int)(e % A.SK);
            const long long tokh = e / A.SK;
            const float* src = A.ws_col + tokh * A.P * ncol + 2 * A.D + i;
            float acc = 0.f;
            for (int pp = 0; pp < A.P; ++pp) acc = __fadd_rn(acc, src[(long long)pp * ncol]);
            A.dg[e] = acc;
        } else {
            const long long e = idx - 2 * nqk - ndg;
            const float* src = A.ws_sc + e * A.P * 2;
            float db = 0.f, dg = 0.f;
            for (int pp = 0; pp < A.P; ++pp) {
                db = __fadd_rn(db, src[2 * pp]);
                dg = __fadd_rn(dg, src[2 * pp + 1]);
            }
            A.dbeta[e] = db;
            if (!A.kda) A.dg[e] = dg;
        }
    }
}

template <int D, int RT, bool KDA>
static int launch_bwd_t(const BwdArgs& a, int W, void* stream)
{
    const int R = 4 * RT * W;
    const BwdSmem L = bwd_smem_layout(D, RT, W, a.c2, KDA);
    const size_t smem = (size_t)L.total * sizeof(float);
    auto kern = gdn_bwd_kernel<D, RT, KDA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(a.DV / R, a.H_v, a.N);
    kern<<<grid, 32 * W, smem, (cudaStream_t)stream>>>(a);
    return (int)cudaGetLastError();
}

int launch_backward(const BwdArgs& a, int D, int RT, int W, bool kda, void* stream)
{
#define GDN_BWD_CASE(DD, RR)                                                          \
    if (D == DD && RT == RR)                                                          \
        return kda ? launch_bwd_t<DD, RR, true>(a, W, stream)                         \
                   : launch_bwd_t<DD, RR, false>(a, W, stream);
    GDN_BWD_CASE(32, 1)
    GDN_BWD_CASE(64, 1)
    GDN_BWD_CASE(128, 1)
    GDN_BWD_CASE(32, 2)
    GDN_BWD_CASE(64, 2)
    GDN_BWD_CASE(128, 2)
    GDN_BWD_CASE(256, 1)
#undef GDN_BWD_CASE
    return (int)cudaErrorInvalidValue;
}

int launch_reduce(const ReduceArgs& a, void* stream)
{
    const long long nqk = (long long)(a.N / a.rep) * a.T * a.H_k * a.SK;
    const long long nhv = (long long)a.N * a.T * a.H_v;
    const long long total = 2 * nqk + (a.kda ? nhv * a.SK : 0) + nhv;
    if (total == 0) return 0;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    gdn_reduce_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace gdn
