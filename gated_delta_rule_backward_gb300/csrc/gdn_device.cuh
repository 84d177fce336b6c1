// gdn_device.cuh -- device helpers shared by the forward and backward kernels.
//
// Bit-exactness contract: the backward recomputes the forward's states, and results
// must not depend on the checkpoint interval.  Every step that produces a state
// element (the decay S' = a (.) M, the dot u = S' k, delta, the update M = S' + k delta)
// is written here once, with explicit round-to-nearest intrinsics so the compiler
// cannot contract or reorder it differently in the two kernels.
#pragma once

#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float4 mul4(float a, float4 x)
{
    return make_float4(__fmul_rn(a, x.x), __fmul_rn(a, x.y), __fmul_rn(a, x.z),
                       __fmul_rn(a, x.w));
}

__device__ __forceinline__ float4 mul4(float4 a, float4 x)
{
    return make_float4(__fmul_rn(a.x, x.x), __fmul_rn(a.y, x.y), __fmul_rn(a.z, x.z),
                       __fmul_rn(a.w, x.w));
}

// x + k * d, element-wise (the rank-one write M = S' + k delta^T for one row)
__device__ __forceinline__ float4 fma4(float4 k, float d, float4 x)
{
    return make_float4(__fmaf_rn(k.x, d, x.x), __fmaf_rn(k.y, d, x.y),
                       __fmaf_rn(k.z, d, x.z), __fmaf_rn(k.w, d, x.w));
}

// acc + x * s, element-wise
__device__ __forceinline__ float4 axpy4(float4 x, float s, float4 acc)
{
    return make_float4(__fmaf_rn(x.x, s, acc.x), __fmaf_rn(x.y, s, acc.y),
                       __fmaf_rn(x.z, s, acc.z), __fmaf_rn(x.w, s, acc.w));
}

// Partial dot of one row slice held by a lane: four independent accumulators (one per
// float4 component) over the lane's NV float4 blocks, combined in a fixed order.
template <int NV>
__device__ __forceinline__ float dot_part(const float4 (&x)[NV], const float4 (&y)[NV])
{
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        a0 = __fmaf_rn(x[v].x, y[v].x, a0);
        a1 = __fmaf_rn(x[v].y, y[v].y, a1);
        a2 = __fmaf_rn(x[v].z, y[v].z, a2);
        a3 = __fmaf_rn(x[v].w, y[v].w, a3);
    }
    return __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
}

// Sum over the 8 column lanes of a row group (xor butterfly; every lane of the group
// ends with the same value because IEEE addition is commutative).
__device__ __forceinline__ float rowsum8(float x)
{
    x = __fadd_rn(x, __shfl_xor_sync(kFull, x, 1));
    x = __fadd_rn(x, __shfl_xor_sync(kFull, x, 2));
    x = __fadd_rn(x, __shfl_xor_sync(kFull, x, 4));
    return x;
}

// Sum across the 4 row groups of a warp (lane bits 3 and 4) by reduce-scatter: on
// return, the lanes of row group g hold Y[i] = sum over groups of X[g*(n/4) + i].
template <int n>
__device__ __forceinline__ void reduce_scatter_groups(const float (&X)[n], float (&Y)[n / 4],
                                                      int grp)
{
    static_assert(n % 4 == 0, "n must be a multiple of 4");
    float Z[n / 2];
    const bool hi = (grp & 2) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
        const float send = hi ? X[i] : X[n / 2 + i];
        const float keep = hi ? X[n / 2 + i] : X[i];
        Z[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 16));
    }
    const bool odd = (grp & 1) != 0;
#pragma unroll
    for (int i = 0; i < n / 4; ++i) {
        const float send = odd ? Z[i] : Z[n / 4 + i];
        const float keep = odd ? Z[n / 4 + i] : Z[i];
        Y[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 8));
    }
}

// One recurrence step for the RT rows a lane holds (meTile "Recurrent delta attention":
// decay before correction; PR #16 row form).  In: m = M_{t-1}.  Out: m = M_t,
// sp = S' = a (.) M_{t-1}, u (row dots, identical on the 8 lanes of a row), and delta.
template <int NV, int RT, bool KDA>
__device__ __forceinline__ void recurrence_step(float4 (&m)[RT][NV], float4 (&sp)[RT][NV],
                                                const float4 (&kv)[NV], const float4 (&av)[NV],
                                                float as, float beta, const float (&vj)[RT],
                                                float (&u)[RT], float (&delta)[RT])
{
#pragma unroll
    for (int r = 0; r < RT; ++r) {
#pragma unroll
        for (int v = 0; v < NV; ++v) sp[r][v] = KDA ? mul4(av[v], m[r][v]) : mul4(as, m[r][v]);
        u[r] = dot_part<NV>(sp[r], kv);
    }
#pragma unroll
    for (int r = 0; r < RT; ++r) u[r] = rowsum8(u[r]);
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        delta[r] = __fmul_rn(beta, __fsub_rn(vj[r], u[r]));
#pragma unroll
        for (int v = 0; v < NV; ++v) m[r][v] = fma4(kv[v], delta[r], sp[r][v]);
    }
}

// The 16-byte path of load_rows: up to B loads per thread are in flight before the first
// of their shared-memory stores, so a tile costs one global round trip per batch instead
// of one per load.  f maps each loaded float4 to the stored one.  Shared rows are ld
// floats apart (ld >= width).
template <int B, typename F>
__device__ __forceinline__ void load_rows_vec(float* dst, const float* src, long long stride,
                                              int nt, int width, int tid, int nthr, F f, int ld)
{
    const int per = width >> 2, total = nt * per;
    for (int base = tid; base < total; base += B * nthr) {
        float4 x[B];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int idx = base + b * nthr;
            if (idx < total) {
                const int tt = idx / per, i4 = idx - tt * per;
                x[b] = __ldg(reinterpret_cast<const float4*>(src + tt * stride) + i4);
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int idx = base + b * nthr;
            if (idx < total) {
                const int tt = idx / per, i4 = idx - tt * per;
                reinterpret_cast<float4*>(dst + tt * ld)[i4] = f(x[b]);
            }
        }
    }
}

// Cooperative copy of nt rows of `width` floats (row stride `stride` in global memory)
// into a shared tile whose rows are ld floats apart (ld = width unless given; the columns
// [width, ld) are left as they are).  vec: every row start is 16-byte aligned and
// width % 4 == 0.  B: loads per thread in flight at once on the 16-byte path.
template <int B = 1>
__device__ __forceinline__ void load_rows(float* dst, const float* src, long long stride,
                                          int nt, int width, bool vec, int tid, int nthr, int ld = 0)
{
    if (ld == 0) ld = width;
    if (vec) {
        load_rows_vec<B>(dst, src, stride, nt, width, tid, nthr, [](float4 x) { return x; }, ld);
    } else {
        for (int idx = tid; idx < nt * width; idx += nthr) {
            const int tt = idx / width, i = idx - tt * width;
            dst[tt * ld + i] = __ldg(src + tt * stride + i);
        }
    }
}

// As load_rows, storing exp(x) (the gate a = exp(g), accurate expf).
template <int B = 1>
__device__ __forceinline__ void load_rows_exp(float* dst, const float* src, long long stride,
                                              int nt, int width, bool vec, int tid, int nthr, int ld = 0)
{
    if (ld == 0) ld = width;
    if (vec) {
        load_rows_vec<B>(dst, src, stride, nt, width, tid, nthr,
                      [](float4 x) { return make_float4(expf(x.x), expf(x.y), expf(x.z), expf(x.w)); }, ld);
    } else {
        for (int idx = tid; idx < nt * width; idx += nthr) {
            const int tt = idx / width, i = idx - tt * width;
            dst[tt * ld + i] = expf(__ldg(src + tt * stride + i));
        }
    }
}

// One lane's float4 block v of a state row of SK floats in global memory (SK may be below
// the kernel's column width: the blocks past SK read as zero and are never written).
__device__ __forceinline__ float4 ld_state4(const float* row, int v, int cl, int SK)
{
    return (32 * v + 4 * cl < SK) ? __ldg(reinterpret_cast<const float4*>(row) + 8 * v + cl)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ void st_state4(float* row, int v, int cl, int SK, float4 x)
{
    if (32 * v + 4 * cl < SK) reinterpret_cast<float4*>(row)[8 * v + cl] = x;
}

// Zero the columns [sk, ld) of the first `rows` rows of a shared tile (head size 16 runs
// at column width 32: its padding columns stay zero, so k = q = 0 and M = 0 there).
__device__ __forceinline__ void zero_pad_cols(float* dst, int rows, int sk, int ld, int tid, int nthr)
{
    if (sk >= ld) return;
    for (int idx = tid; idx < rows * (ld - sk); idx += nthr) {
        const int t = idx / (ld - sk), i = sk + idx - t * (ld - sk);
        dst[t * ld + i] = 0.f;
    }
}

// Shared-memory float4 view of column block v of the lane's row slice in a D-wide row.
template <int D>
__device__ __forceinline__ float4 lds_cols(const float* row, int v, int cl)
{
    return reinterpret_cast<const float4*>(row)[8 * v + cl];
}

}  // namespace gdn
