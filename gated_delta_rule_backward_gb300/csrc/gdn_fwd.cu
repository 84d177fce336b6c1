// gdn_fwd.cu -- forward of the gated delta rule (sm_103a).
//
// Grid (P, H_v, N): CTA p owns rows [p R, p R + R) of M = S^T for one (sequence, value
// head).  Rows are independent in the forward (every term of the step is row-local:
// "metal: GATED_DELTA_NET_BACK", PR #16 review "APPROVED at 739b9bf", "Thread j owns
// row j of M"), so CTAs never communicate and warps never wait on one another inside
// a tile: each warp runs its own chain of tokens over its rows.
//
// Per tile of tc tokens the CTA stages k, q, a = exp(g), beta and its own rows of v in
// shared memory; the state lives in registers (RT rows x D/8 columns per lane).  The
// state entering token c*C is written to ckpt[c] (PR #16 body: checkpointed recompute).
//
// D is the column width the kernel computes in (the key head size S_k, or 32 for S_k = 16,
// whose padding columns hold zeros throughout); the S_v rows of M are the grid's
// S_v / R row blocks, so S_k and S_v are independent.
#include <cuda_runtime.h>

#include "gdn_device.cuh"

namespace gdn {

template <int D, int RT, bool KDA>
__global__ void __launch_bounds__(128, D <= 128 ? 3 : 1) gdn_fwd_kernel(const FwdArgs A)
{
    constexpr int NV = D / 32;
    const int NT = blockDim.x, W = NT >> 5;
    const int R = 4 * RT * W;
    const int p = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h % A.H_k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, cl = lane & 7;
    const int lrow0 = warp * 4 * RT + grp * RT;
    const int row0 = p * R + lrow0;
    const int tc = A.tc;

    extern __shared__ __align__(16) float sm[];
    const FwdSmem L = fwd_smem_layout(D, RT, W, tc, KDA);
    float* sk = sm + L.sk;
    float* sq = sm + L.sq;
    float* sa = sm + L.sa;
    float* sb = sm + L.sb;
    float* sv = sm + L.sv;
    float* sy = sm + L.sy;

    const long long head = (long long)n * A.H_v + h;
    const int SK = A.SK, DV = A.DV;
    float4 m[RT][NV];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int v = 0; v < NV; ++v) m[r][v] = ld_state4(A.state0 + (head * DV + row0 + r) * SK, v, cl, SK);
    zero_pad_cols(sk, A.tc, SK, D, tid, NT);
    zero_pad_cols(sq, A.tc, SK, D, tid, NT);
    if (KDA) zero_pad_cols(sa, A.tc, SK, D, tid, NT);

    for (int t0 = 0; t0 < A.T; t0 += tc) {
        const int nt = min(tc, A.T - t0);
        __syncthreads();
        load_rows<4>(sk, A.k + (long long)(n / A.rep) * A.ks0 + (long long)t0 * A.ks1 + hk * A.ks2, A.ks1, nt, SK,
                  A.vec_k, tid, NT, D);
        load_rows<4>(sq, A.q + (long long)(n / A.rep) * A.qs0 + (long long)t0 * A.qs1 + hk * A.qs2, A.qs1, nt, SK,
                  A.vec_q, tid, NT, D);
        const long long tok0 = (long long)n * A.T + t0;
        if (KDA) {
            load_rows_exp<4>(sa, A.g + (tok0 * A.H_v + h) * SK, (long long)A.H_v * SK, nt, SK,
                          A.vec_g, tid, NT, D);
        } else {
            for (int tt = tid; tt < nt; tt += NT) sa[tt] = expf(__ldg(A.g + (tok0 + tt) * A.H_v + h));
        }
        for (int tt = tid; tt < nt; tt += NT) sb[tt] = __ldg(A.beta + (tok0 + tt) * A.H_v + h);
        load_rows<4>(sv, A.v + n * A.vs0 + (long long)t0 * A.vs1 + h * A.vs2 + p * R, A.vs1, nt, R,
                  A.vec_v, tid, NT);
        __syncthreads();

        for (int tt = 0; tt < nt; ++tt) {
            const int t = t0 + tt;
            if (t % A.C == 0) {
                float* ck = A.ckpt + ((head * A.n_ck + t / A.C) * DV + row0) * SK;
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int v = 0; v < NV; ++v) st_state4(ck + r * SK, v, cl, SK, m[r][v]);
            }
            float4 kv[NV], qv[NV], av[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                kv[v] = lds_cols<D>(sk + tt * D, v, cl);
                qv[v] = lds_cols<D>(sq + tt * D, v, cl);
                if (KDA) av[v] = lds_cols<D>(sa + tt * D, v, cl);
            }
            const float as = KDA ? 0.f : sa[tt];
            float vj[RT], u[RT], delta[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r) vj[r] = sv[tt * R + lrow0 + r];
            float4 sp[RT][NV];
            recurrence_step<NV, RT, KDA>(m, sp, kv, av, as, sb[tt], vj, u, delta);
            // y_j = scale * sum_i M_t[j][i] q_i  (meTile: output = scale * state^T query)
            float w[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r) w[r] = dot_part<NV>(m[r], qv);
#pragma unroll
            for (int r = 0; r < RT; ++r) w[r] = rowsum8(w[r]);
            if (cl == 0) {
#pragma unroll
                for (int r = 0; r < RT; ++r) sy[tt * R + lrow0 + r] = __fmul_rn(A.scale, w[r]);
            }
        }
        __syncthreads();
        // y rows of this CTA for the tile: R contiguous floats per token
        float* ydst = A.y + (tok0 * A.H_v + h) * DV + p * R;
        const long long ystride = (long long)A.H_v * DV;
        for (int idx = tid; idx < nt * R; idx += NT) {
            const int tt = idx / R, j = idx - tt * R;
            ydst[tt * ystride + j] = sy[tt * R + j];
        }
    }

#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int v = 0; v < NV; ++v) st_state4(A.state_T + (head * DV + row0 + r) * SK, v, cl, SK, m[r][v]);
}

template <int D, int RT, bool KDA>
static int launch_fwd_t(const FwdArgs& a, int W, void* stream)
{
    const int R = 4 * RT * W;
    const FwdSmem L = fwd_smem_layout(D, RT, W, a.tc, KDA);
    const size_t smem = (size_t)L.total * sizeof(float);
    auto kern = gdn_fwd_kernel<D, RT, KDA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(a.DV / R, a.H_v, a.N);
    kern<<<grid, 32 * W, smem, (cudaStream_t)stream>>>(a);
    return (int)cudaGetLastError();
}

int launch_forward(const FwdArgs& a, int D, int RT, int W, bool kda, void* stream)
{
#define GDN_FWD_CASE(DD, RR)                                                          \
    if (D == DD && RT == RR)                                                          \
        return kda ? launch_fwd_t<DD, RR, true>(a, W, stream)                         \
                   : launch_fwd_t<DD, RR, false>(a, W, stream);
    GDN_FWD_CASE(32, 1)
    GDN_FWD_CASE(64, 1)
    GDN_FWD_CASE(128, 1)
    GDN_FWD_CASE(32, 2)
    GDN_FWD_CASE(64, 2)
    GDN_FWD_CASE(128, 2)
    GDN_FWD_CASE(256, 1)
#undef GDN_FWD_CASE
    return (int)cudaErrorInvalidValue;
}

}  // namespace gdn
