// gdn_tc.cuh -- 5th-generation tensor-core (tcgen05) building blocks for sm_103a, in inline PTX.
//
// Every product here is D[128][N] (+)= A[128][K] B[N][K]^T with an fp32 accumulator in
// tensor memory (TMEM), issued by one thread of the CTA:
//   * A is read from TMEM (lane = row) or from shared memory; B is read from shared memory;
//   * fp32-level accuracy comes from a three-pass split x = hi + lo, a b ~= hi_a hi_b +
//     hi_a lo_b + lo_a hi_b, in one of two kinds:
//       - kind::tf32 (K = 8 per instruction): hi, lo tf32 values (split_tf32), one TMEM column
//         per K element;
//       - kind::f16 with bf16 operands (K = 16 per instruction, half the instructions): hi, lo
//         bf16 values rounded to nearest (split_bf16x2), two K elements per TMEM column, the
//         even one in the low half.  hi + lo carries 16 significant bits and the exponent
//         range of fp32.
//
// Shared-memory operand layout (no swizzle, K-major): an R x K tile of 4-byte elements is
// stored as core matrices of 8 rows x 4 elements (128 contiguous bytes, row-major inside;
// for 2-byte elements 8 rows x 8 elements, with the same byte strides below);
// core matrix (k-chunk kc, row group g) starts at float offset (kc * (R / 8) + g) * 32.
// Its descriptor has leading-dimension byte offset LBO = R / 8 * 128 (the step between
// k-chunks) and stride byte offset SBO = 128 (the step between row groups); the K = 8
// slice s of the tile starts 2 s LBO bytes in.
//
// Every wait on an mbarrier is bounded: it gives up after kWaitLimitNs and reports the
// failure, so a kernel can record an error status and return instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace tc {

constexpr uint64_t kWaitLimitNs = 200000000ull;  // 0.2 s

// Float offset of element (r, k) of an R-row operand tile in the layout above.
GDN_HD inline int kmaj(int r, int k, int R)
{
    return (((k >> 2) * (R >> 3) + (r >> 3)) << 5) + ((r & 7) << 2) + (k & 3);
}
// The row-group-major variant of a tile with K elements per row: core matrix (row group g,
// k-chunk kc) at float offset (g * (K / 4) + kc) * 32, so each group of 8 rows is one
// contiguous block and tiles of whole row groups stack by concatenation.  LBO = 128 bytes,
// SBO = K * 32 bytes; the K = 8 slice s starts 256 s bytes in.
GDN_HD inline int kmaj_rg(int r, int k, int K)
{
    return (((r >> 3) * (K >> 2) + (k >> 2)) << 5) + ((r & 7) << 2) + (k & 3);
}
// The same layout for 2-byte (bf16) elements: the 32-bit word holding elements (r, k) and
// (r, k + 1) of a row-group-major tile, k even (core matrices of 8 rows x 8 elements; LBO =
// 128 bytes, SBO = K * 16 bytes; the K = 16 slice s starts 256 s bytes in).
GDN_HD inline int kmaj16_rg(int r, int k, int K)
{
    return (((r >> 3) * (K >> 3) + (k >> 3)) << 5) + ((r & 7) << 2) + ((k & 7) >> 1);
}

#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor (no swizzle; version bits 46-47 = 1).
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Descriptor of an R-row tile at `base` (layout above), advanced to its K = 8 slice s.
__device__ __forceinline__ uint64_t tile_desc(const float* base, int R)
{
    return make_desc(smem_addr(base), (uint32_t)(R / 8) * 128u, 128u);
}
__device__ __forceinline__ uint64_t desc_kslice(uint64_t d, int R, int s)
{
    return d + (uint64_t)((2 * (R / 8) * 128 * s) >> 4);
}
__device__ __forceinline__ uint64_t tile_desc_rg(const float* base, int K)
{
    return make_desc(smem_addr(base), 128u, (uint32_t)K * 32u);
}
__device__ __forceinline__ uint64_t desc_kslice_rg(uint64_t d, int s)
{
    return d + (uint64_t)(16 * s);
}
// Row-group-major tile of bf16 elements with K per row (kmaj16_rg); its K = 16 slice s is
// desc_kslice_rg(d, s), and a k-chunk-major bf16 tile takes tile_desc / desc_kslice as they are.
__device__ __forceinline__ uint64_t tile_desc16_rg(const void* base, int K)
{
    return make_desc(smem_addr(base), 128u, (uint32_t)K * 16u);
}

// Instruction descriptor, kind::tf32: fp32 accumulator, tf32 A and B, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_tf32(int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Instruction descriptor, kind::f16 with bf16 A and B: fp32 accumulator, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
// D (+)= A B^T, kind::f16 (bf16 operands), A in TMEM (two K elements per column).
__device__ __forceinline__ void mma_ts16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D (+)= A B^T, kind::f16 (bf16 operands), A and B in shared memory.
__device__ __forceinline__ void mma_ss16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrives on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
        smem_addr(bar)));
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes made visible to the async proxy (MMA, bulk copies).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch.  launch_dependents lets the next kernel on the stream (when it
// is launched with programmatic stream serialisation) start its CTAs once every CTA of this grid
// has issued it or exited; wait blocks the calling thread until the preceding grid has completed
// and its writes are visible (at once when no such grid is in flight).
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// TMEM allocation by one whole warp; the base address lands in *holder.
__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t cols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(holder)),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_free(uint32_t base, uint32_t cols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols));
}

// 32 consecutive columns of this warp's 32 lanes (lane quarter = warp % 4): thread = lane.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
__device__ __forceinline__ void st4(uint32_t taddr, const uint32_t (&r)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]));
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of (lane quarter of this warp, column col).
__device__ __forceinline__ uint32_t taddr(uint32_t base, int warp, int col)
{
    return base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)col;
}

// tf32 split: hi = x with its 13 low mantissa bits cleared (truncation, one integer op),
// lo = x - hi (exact in fp32, |lo| < 2^-10 |x|).  The tensor core reads lo as tf32, keeping
// its 10 leading mantissa bits, so the split represents x to within 2^-21 |x|, and the
// three-pass product misses only the lo lo term, below 2^-20 |a b|.
__device__ __forceinline__ uint32_t to_tf32(float x)
{
    return __float_as_uint(x) & 0xFFFFE000u;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo)
{
    hi = to_tf32(x);
    lo = __float_as_uint(__fsub_rn(x, __uint_as_float(hi)));
}
// Two fp32 values as one 32-bit word of bf16 values rounded to nearest: x0 in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float x0, float x1)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x1), "f"(x0));
    return r;
}
// x0, x1 (consecutive K elements, x0 the even one) split into bf16 hi and lo words:
// x = hi + lo + O(2^-16 |x|).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16x2(x0, x1);
    lo = pack_bf16x2(__fsub_rn(x0, __uint_as_float(hi << 16)), __fsub_rn(x1, __uint_as_float(hi & 0xFFFF0000u)));
}

// 8 consecutive K elements of one row (one 16-byte unit of a bf16 tile in the layouts above)
// as bf16 hi at hi_base + 4 unit and lo `half` floats further.
__device__ __forceinline__ void put_bf16x8(float* hi_base, int half, int unit, const float (&x)[8])
{
    uint4 hi, lo;
    split_bf16x2(x[0], x[1], hi.x, lo.x);
    split_bf16x2(x[2], x[3], hi.y, lo.y);
    split_bf16x2(x[4], x[5], hi.z, lo.z);
    split_bf16x2(x[6], x[7], hi.w, lo.w);
    *reinterpret_cast<uint4*>(hi_base + 4 * unit) = hi;
    *reinterpret_cast<uint4*>(hi_base + half + 4 * unit) = lo;
}

// Barrier among the first `threads` threads of the CTA (named barrier 1), leaving the rest
// of the CTA free to run.
__device__ __forceinline__ void bar_sync_first(int threads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// ---- mbarriers and bulk copies ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Polls the phase with parity `parity` until it completes; false once kWaitLimitNs of
// wall-clock time (%globaltimer) have passed without it, far beyond any legitimate wait.
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    uint64_t start = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 255) == 0) {
            const uint64_t now = global_ns();
            if (it == 0)
                start = now;
            else if (now - start > kWaitLimitNs)
                return false;
        }
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Bulk copy global -> shared (TMA engine, no tensor map): both addresses 16-byte aligned,
// bytes a multiple of 16.  Completion is counted on `bar` in bytes.
// One m16n8k8 tf32 product C += A B issued by a whole warp (mma.sync; for the small
// products of the CUDA-core kernels, where a TMEM accumulator and an issuing thread do not
// pay).  A: rows g, g + 8 and columns tq, tq + 4 of the 16 x 8 tile (g = lane / 4,
// tq = lane % 4); B: rows tq, tq + 4 of column g of the 8 x 8 tile; C: rows g, g + 8 and
// columns 2 tq, 2 tq + 1.  Operand registers hold fp32 bit patterns, of which the tensor
// pipe reads the top 19 bits (tf32).
__device__ __forceinline__ void mma_warp_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// An L2 prefetch hint for one line through the load/store path.  A CTA whose first global
// access is a bulk copy ran its memory-bound steps measurably slower on GB300 than one that
// touched global memory through the load/store path first (cause unknown); the kernels issue
// one of these before their first bulk copies.
__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

#endif  // __CUDACC__

}  // namespace tc
}  // namespace gdn
