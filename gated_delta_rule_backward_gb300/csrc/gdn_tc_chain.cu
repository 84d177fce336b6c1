// gdn_tc_chain.cu -- the two serial chains of the chunked scalar gate at head size 128 on
// the 5th-generation tensor cores (tcgen05, kind::f16 with bf16 hi/lo operands, three-pass
// split for fp32-level accuracy): the forward's state chain and the dM chain of the
// backward.
//
// State chain:
//
// one CTA owns one head's whole state M (128 x 128, rows j = value index) and walks its
// chunks in order.  Per chunk (32 tokens; "metal: GATED_DELTA_NET_BACK" row form regrouped
// by chunks, see gdn_chunk.cu for the derivation):
//   D1  = M [W; Q]^T                    128 x 64, K = 128    (A = M from TMEM, B = [W; Q])
//   Delta^T = U^T - D1[:, 0:32]         in registers, split to bf16 hi/lo in TMEM
//   D23 = Delta^T [scale QD; (r K)^T]^T 128 x 160, K = 32    (A = Delta^T, B from smem)
//   y^T = scale gamma (.) D1[:, 32:64] + D23[:, 0:32]
//   M   <- gamma_last M + D23[:, 32:160]
// M itself stays in registers in fp32 (thread = row j, 64 columns); each chunk it is split
// into bf16 hi/lo parts written to TMEM as the A operand of the next D1.  The chunk
// operands ([W; Q], [scale QD; (r K)^T] as bf16 hi/lo, U^T in fp32, gamma) are written by
// the prep kernel in the tensor-core operand layout and arrive by bulk copies (TMA), the
// next chunk's as soon as the current one's buffer is free.  In bf16 (K = 16 per
// instruction) the chunk's two products take 30 MMAs instead of 60 in tf32; M, the
// accumulators and every sum outside the products stay fp32.
//
// Grid: (head, sequence); the chain writes y, the checkpoints and state_T (or, between
// chunk ranges, the carried state).  The backward needs no rerun of it: its gradient step
// rebuilds the chunk-entry states it needs (gdn_tc_grad.cu).
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

// Status word of the tensor-core kernels on this device: 0, or after a bounded wait gave up
// GDN_ERR_TIMEOUT (6) | kernel << 4 | wait sites << 8 (bits kW* of the CTAs that gave up,
// OR-ed).  Read and cleared by tc_take_status.
__device__ int g_tc_status;

namespace {

constexpr int TD = 128;                       // head size
constexpr int TCT = 288;                      // 8 compute warps (row j, column half) + 1 issuer warp
constexpr int kIssuer = 256;                  // issues the MMAs and bulk copies
constexpr uint32_t kColMhi = 0;               // TMEM columns: M hi  (bf16 A operand, K = 128)
constexpr uint32_t kColMlo = 64;              //               M lo
constexpr uint32_t kColDh = 128;              //               Delta^T hi (bf16 A of D23, K = 32)
constexpr uint32_t kColDl = 144;              //               Delta^T lo
constexpr uint32_t kColD1 = 256;              //               D1 (64 columns)
constexpr uint32_t kColD23 = 320;             //               D23 (160 columns)
constexpr uint32_t kTmemCols = 512;
constexpr int kStatusTimeout = 6;
// kernel field of the status word
constexpr int kKerState = 1, kKerDstate = 3, kKerSelftest = 4;  // 2: no longer used
// wait sites (s_err bits): the issuer's waits on copies and operand handoffs, and the
// compute warps' waits on MMA completion
constexpr int kWCopyA = 1 << 0, kWCopyB = 1 << 1, kWHandoff1 = 1 << 2, kWHandoff2 = 1 << 3,
              kWMma1 = 1 << 4, kWMma2 = 1 << 5, kWMma3 = 1 << 6,
              kWTmem = 1 << 7;  // an MMA committed before a give-up did not complete either:
                                // the tensor memory may still be written after its release
__device__ __forceinline__ void raise_timeout(int kernel, int sites)
{
    atomicOr(&g_tc_status, kStatusTimeout | kernel << 4 | sites << 8);
}

// Shared memory, in floats.
constexpr int kSB1 = 0;                            // [W; Q] bf16 hi, then lo: 2 x 64 x 128, row-group-major
constexpr int kSB23 = kSB1 + kTcWElems + kTcQElems;  // [sQD; rK^T] bf16 hi, lo  2 x 160 x 32
constexpr int kSU = kSB23 + kTcB23Elems;           // U^T, operand layout (R = 128), fp32
constexpr int kSDel = kSU + BC * TD;               // staging of checkpoint rows (32 x kStageLd)
constexpr int kSGam = kSDel + 2 * BC * TD;         // gamma (32)
constexpr int kStageLd = TD + 4;                   // staging rows for coalesced global writes
constexpr int kSY = kSGam + BC;                    // y of two chunks, rows t (forward)
constexpr int kSGl = kSY + 2 * BC * kStageLd;      // KDA: gamma_last per column, two buffers by
                                                   // chunk parity (the next chunk's lands while
                                                   // this one's update reads)
constexpr int kSFloats = kSGl + 2 * TD;
constexpr size_t kSmemBytes = sizeof(float) * kSFloats + 128;  // + barriers (6 used)

constexpr uint32_t kB1Bytes = sizeof(float) * (kTcWElems + kTcQElems);
constexpr int kHalfW = kTcWElems / 2;  // 32 x 128 bf16 values
constexpr uint32_t kB23Bytes = sizeof(float) * kTcB23Elems + sizeof(float) * BC * TD + sizeof(float) * BC;

// [W; Q] hi then lo: W of the value head and Q of its key head (KDA: Q (.) gamma of the value
// head; the caller passes that block's index as ck), stacked by row groups.
__device__ __forceinline__ void load_b1(const ChunkArgs& A, long long ch, long long ck, float* sm, uint64_t* bar)
{
    const float* w = A.ws + A.o_W1 + ch * kTcWElems;
    const float* q = A.ws + A.o_Q1 + ck * kTcQElems;
    constexpr uint32_t part = sizeof(float) * kHalfW;
    tc::mbar_expect_tx(bar, kB1Bytes);
    tc::bulk_g2s(sm + kSB1, w, part, bar);
    tc::bulk_g2s(sm + kSB1 + kHalfW, q, part, bar);
    tc::bulk_g2s(sm + kSB1 + 2 * kHalfW, w + kHalfW, part, bar);
    tc::bulk_g2s(sm + kSB1 + 3 * kHalfW, q + kHalfW, part, bar);
}

// [scale QD; (r K)^T], U^T and gamma of chunk c; KDA: also gamma_last (per column) into the
// buffer of c's parity.
template <bool KDA>
__device__ __forceinline__ void load_b23(const ChunkArgs& A, long long ch, int c, float* sm, uint64_t* bar)
{
    tc::mbar_expect_tx(bar, kB23Bytes + (KDA ? (uint32_t)sizeof(float) * TD : 0u));
    tc::bulk_g2s(sm + kSB23, A.ws + A.o_B23 + ch * kTcB23Elems, sizeof(float) * kTcB23Elems, bar);
    tc::bulk_g2s(sm + kSU, A.ws + A.o_U + ch * (BC * TD), sizeof(float) * BC * TD, bar);
    tc::bulk_g2s(sm + kSGam, A.ws + A.o_gam + ch * BC, sizeof(float) * BC, bar);
    if (KDA) tc::bulk_g2s(sm + kSGl + (c & 1) * TD, A.ws + A.o_gL + ch * TD, sizeof(float) * TD, bar);
}

}  // namespace

// The state chain of one head (bx = head, by = sequence); sm is the dynamic shared memory.
// KDA: the per-key-column gate (operands per value head, M decayed column by column).
template <bool KDA>
__device__ __forceinline__ void state_chain(const ChunkArgs& A, float* sm, int bx, int by)
{
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSFloats);  // b1, b23, mma, a[8]
    uint64_t* bar_b1 = bars;
    uint64_t* bar_b23 = bars + 1;
    uint64_t* bar_mma = bars + 2;
    uint64_t* bar_a = bars + 3;  // bar_a[g]: columns [32 g, 32 g + 32) of both halves of M are in TMEM
    uint64_t* bar_d = bars + 5;  // Delta^T (the A operand of D23) is in TMEM, and every compute
                                 // warp has seen D1 complete
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool compute = warp < 8;          // warps 0-7 hold M; warp 8 issues MMAs and copies
    const bool issuer = tid == kIssuer;
    const int j = 32 * (warp & 3) + lane;   // row of M (compute warps)
    const int hc = (warp >> 2) & 1;         // column half: columns [64 hc, 64 hc + 64)

    const int h = bx, n = by, c_begin = A.c_lo, c_end = A.c_hi;
    const long long head = (long long)n * A.H_v + h;
    const long long khead = KDA ? head : (long long)n * A.H_k + h % A.H_k;

    if (tid == 0) {
        tc::mbar_init(bar_b1, 1);
        tc::mbar_init(bar_b23, 1);
        tc::mbar_init(bar_mma, 1);
        for (int g = 0; g < 2; ++g) tc::mbar_init(bar_a + g, 8);  // one arrival per compute warp
        tc::mbar_init(bar_d, 8);                                  // one per compute warp
        tc::mbar_fence_init();
        s_err = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;

    uint32_t ph_b1 = 0, ph_b23 = 0, ph_mma = 0;
    bool mma_out = false;  // issuer: a committed MMA group not yet seen complete, phase ph_out
    uint32_t ph_out = 0;
    bool b1_pending = false, b23_pending = false;
    if (issuer) {
        tc::prefetch_l2(A.ws + A.o_U + (head * A.n_chunks + c_begin) * (BC * TD));  // see prefetch_l2
        load_b1(A, head * A.n_chunks + c_begin, khead * A.n_chunks + c_begin, sm, bar_b1);
        load_b23<KDA>(A, head * A.n_chunks + c_begin, c_begin, sm, bar_b23);
        b1_pending = b23_pending = true;
    }

    // entry state: this thread's 64 columns of row j
    float m[64];
    if (compute) {
        const float* src = c_begin == 0 ? A.state0 + (head * TD + j) * TD : A.carry + (head * TD + j) * TD;
        const float4* s4 = reinterpret_cast<const float4*>(src + 64 * hc);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 x = __ldg(s4 + q);
            m[4 * q] = x.x;
            m[4 * q + 1] = x.y;
            m[4 * q + 2] = x.z;
            m[4 * q + 3] = x.w;
        }
    }
    // y of a chunk is assembled in shared memory (rows t, one of two buffers by chunk parity)
    // by the column-half 1 threads: the Q part in (3), the QD Delta part added in (5).  It
    // goes to global memory during the next chunk's D23, when the compute warps would only
    // wait (the buffer is next written two chunks later, after the CTA barrier of (5)).
    int y_t0 = 0, y_nb = 0;
    const float* y_buf = sm + kSY;  // the buffer of the chunk whose y is pending
    float* stage = sm + kSDel;   // idle while D1 runs: 32 rows of kStageLd floats (checkpoints)
    const int ctid = tid;        // 0..255 for the compute warps
    auto store_y = [&]() {       // the global writes are whole 512-byte rows
        tc::bar_sync_first(256);  // the column-half 1 threads' adds to y_buf are complete
        float* yp = A.y + (((long long)n * A.T + y_t0) * A.H_v + h) * TD;
        const long long ys = (long long)A.H_v * TD;
        for (int idx = ctid; idx < y_nb * (TD / 4); idx += 256) {
            const int t = idx / (TD / 4), q = idx - t * (TD / 4);
            const float4 v = *reinterpret_cast<const float4*>(y_buf + t * kStageLd + 4 * q);
            float* yq = yp + t * ys + 4 * q;
            if (A.vec_y) {  // y is only required to be 4-byte aligned
                *reinterpret_cast<float4*>(yq) = v;
            } else {
                yq[0] = v.x; yq[1] = v.y; yq[2] = v.z; yq[3] = v.w;
            }
        }
    };
    auto store_ckpt = [&](float* dst) {  // row-major M through `stage`, 32 rows at a time
#pragma unroll 1
        for (int r = 0; r < 4; ++r) {
            if ((warp & 3) == r) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<float4*>(stage + lane * kStageLd + 64 * hc + 4 * q) =
                        make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
            }
            tc::bar_sync_first(256);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int idx = ctid + 256 * k, row = idx >> 5, q = idx & 31;
                *reinterpret_cast<float4*>(dst + (long long)(32 * r + row) * TD + 4 * q) =
                    *reinterpret_cast<const float4*>(stage + row * kStageLd + 4 * q);
            }
            tc::bar_sync_first(256);
        }
    };
    // Columns [8 q, 8 q + 8) of this thread's half of M -> bf16 hi/lo in TMEM (4 columns
    // each): half of the K = 16 slice 4 hc + q / 2 of the next D1's A operand.
    auto split_store = [&](int q) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) tc::split_bf16x2(m[8 * q + 2 * e], m[8 * q + 2 * e + 1], hi[e], lo[e]);
        tc::st4(tc::taddr(tmem, warp, kColMhi + 32 * hc + 4 * q), hi);
        tc::st4(tc::taddr(tmem, warp, kColMlo + 32 * hc + 4 * q), lo);
    };
    // Columns [32 g, 32 g + 32) of this thread's half of the next D1's A operand are written:
    // the issuer may use k-slices 2 g, 2 g + 1, 4 + 2 g and 5 + 2 g (one arrival per compute
    // warp, after the warp's stores are complete).
    auto release_group = [&](int g) {
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar_a + g);
    };
    if (compute) {
#pragma unroll
        for (int q = 0; q < 8; ++q) split_store(q);
        release_group(0);
        release_group(1);
    }

    const float* sU = sm + kSU;
    const float* sGam = sm + kSGam;
    const uint32_t id64 = tc::idesc_bf16(64), id160 = tc::idesc_bf16(160);

    int c = c_begin;
    for (; c < c_end; ++c) {
        const int seg = c / A.cps;
        const int loc = c - seg * A.cps;
        const int t0 = seg * A.C + loc * BC;
        const int nb = min(BC, min(A.T, seg * A.C + A.C) - t0);
        const long long ch = head * A.n_chunks + c;
        float* sY = sm + kSY + (c & 1) * (BC * kStageLd);  // this chunk's y
        // (1) M (bf16 hi/lo, the A operand of D1) goes into TMEM slice by slice (release_group)
        // (2) D1 = M [W; Q]^T on the tensor cores, each k-slice issued as soon as its columns of
        //     M are in TMEM; meanwhile the compute warps store the checkpoint at a segment's
        //     first chunk
        const uint32_t ph_a = (uint32_t)(c - c_begin) & 1u;
        if (issuer) {
            if (!tc::mbar_wait(bar_b1, ph_b1)) atomicOr(&s_err, kWCopyA);
            ph_b1 ^= 1;
            b1_pending = false;
            if (!s_err) {
                const uint64_t bhi = tc::tile_desc16_rg(sm + kSB1, TD);
                const uint64_t blo = tc::tile_desc16_rg(sm + kSB1 + 2 * kHalfW, TD);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if ((q & 1) == 0) {
                        if (!tc::mbar_wait(bar_a + (q >> 1), ph_a)) {
                            atomicOr(&s_err, kWHandoff1);
                            break;
                        }
                        tc::fence_after();
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int s = q + 4 * h2;
                        const uint32_t ahi = tmem + kColMhi + 8 * s, alo = tmem + kColMlo + 8 * s;
                        tc::mma_ts16(tmem + kColD1, ahi, tc::desc_kslice_rg(bhi, s), id64, s > 0);
                        tc::mma_ts16(tmem + kColD1, ahi, tc::desc_kslice_rg(blo, s), id64, 1);
                        tc::mma_ts16(tmem + kColD1, alo, tc::desc_kslice_rg(bhi, s), id64, 1);
                    }
                }
                if (!s_err) {
                    tc::commit(bar_mma);
                    mma_out = true;
                    ph_out = ph_mma;
                }
            }
        } else if (compute) {
            if (loc == 0) store_ckpt(A.ckpt_out + (head * A.n_ck + seg) * (long long)(TD * TD));
        }
        // (3) Delta^T (rows j) and the Q part of y^T.  Only the compute warps and the issuer
        // wait on bar_mma: every waiter must have seen a phase complete before the next commit
        // on it can land (else it would wait on the phase after), and only the bar_d arrivals
        // of the compute warps order that for D23.
        bool ok = !(compute || issuer) || tc::mbar_wait(bar_mma, ph_mma);
        if (issuer && ok) mma_out = false;
        ph_mma ^= 1;
        tc::fence_after();
        float gl = 0.f;
        if (issuer) {
            if (ok && c + 1 < c_end) {
                load_b1(A, ch + 1, khead * A.n_chunks + c + 1, sm, bar_b1);
                b1_pending = true;
            }
        } else if (compute) {
            if (hc == 1) {  // D23 overwrites nothing these warps read: release it at once
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar_d);
            }
            ok = tc::mbar_wait(bar_b23, ph_b23) && ok;
            gl = sGam[BC - 1];
            if (hc == 0) {
                // Delta^T[j][t] = U^T[j][t] - D1[j][t], split into bf16 hi/lo in TMEM: the A
                // operand of D23 (K = t, 16 tokens per 8 columns)
#pragma unroll
                for (int q = 0; q < BC / 16; ++q) {
                    float x[16];
                    tc::ld16(tc::taddr(tmem, warp, kColD1 + 16 * q), x);
                    tc::wait_ld();
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int h4 = 0; h4 < 4; ++h4) {
                        const int b = 4 * q + h4;
                        const float4 u = *reinterpret_cast<const float4*>(sU + 4 * (b * TD + j));
                        tc::split_bf16x2(__fsub_rn(u.x, x[4 * h4]), __fsub_rn(u.y, x[4 * h4 + 1]), hi[2 * h4], lo[2 * h4]);
                        tc::split_bf16x2(__fsub_rn(u.z, x[4 * h4 + 2]), __fsub_rn(u.w, x[4 * h4 + 3]), hi[2 * h4 + 1],
                                         lo[2 * h4 + 1]);
                    }
                    tc::st8(tc::taddr(tmem, warp, kColDh + 8 * q), hi);
                    tc::st8(tc::taddr(tmem, warp, kColDl + 8 * q), lo);
                }
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar_d);
            } else {  // the Q part of y
                float x[32];
                tc::ld32(tc::taddr(tmem, warp, kColD1 + BC), x);
                tc::wait_ld();
#pragma unroll
                for (int t = 0; t < BC; ++t) sY[t * kStageLd + j] = __fmul_rn(__fmul_rn(A.scale, sGam[t]), x[t]);
            }
            if (y_nb > 0) store_y();  // the previous chunk's y, while D23 runs
        }
        ph_b23 ^= 1;
        if (!ok) atomicOr(&s_err, kWMma1);
        // (4) D23 = Delta^T [scale QD; (r K)^T]^T, issued as soon as Delta^T is in TMEM
        if (issuer) {
            b23_pending = false;
            if (!tc::mbar_wait(bar_d, (uint32_t)(c - c_begin) & 1u)) atomicOr(&s_err, kWHandoff2);
            tc::fence_after();
            if (!s_err) {
                const uint64_t bhi = tc::tile_desc(sm + kSB23, 160);
                const uint64_t blo = tc::tile_desc(sm + kSB23 + kTcB23Elems / 2, 160);
#pragma unroll
                for (int s = 0; s < BC / 16; ++s) {
                    const uint32_t a_h = tmem + kColDh + 8 * s, a_l = tmem + kColDl + 8 * s;
                    const uint64_t b_h = tc::desc_kslice(bhi, 160, s), b_l = tc::desc_kslice(blo, 160, s);
                    tc::mma_ts16(tmem + kColD23, a_h, b_h, id160, s > 0);
                    tc::mma_ts16(tmem + kColD23, a_h, b_l, id160, 1);
                    tc::mma_ts16(tmem + kColD23, a_l, b_h, id160, 1);
                }
                tc::commit(bar_mma);
                mma_out = true;
                ph_out = ph_mma;
            }
        }
        // (5) y and the state update
        ok = !(compute || issuer) || tc::mbar_wait(bar_mma, ph_mma);
        if (issuer && ok) mma_out = false;
        ph_mma ^= 1;
        tc::fence_after();
        if (!__syncthreads_and(ok)) {
            if (!ok) atomicOr(&s_err, kWMma2);
            __syncthreads();
            break;
        }
        if (issuer) {
            if (c + 1 < c_end) {
                tc::fence_async_smem();
                load_b23<KDA>(A, ch + 1, c + 1, sm, bar_b23);
                b23_pending = true;
            }
        } else if (compute) {
            if (hc == 1) {  // y += D23[:, 0:32]
                float x[32];
                tc::ld32(tc::taddr(tmem, warp, kColD23), x);
                tc::wait_ld();
#pragma unroll
                for (int t = 0; t < BC; ++t) sY[t * kStageLd + j] = __fadd_rn(sY[t * kStageLd + j], x[t]);
            }
            y_t0 = t0;
            y_nb = nb;
            y_buf = sY;
            // M <- gamma_last M + D23[:, 32:160], split at once into the next D1's A operand and
            // released to the issuer in two column groups
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float x[8];
                tc::ld8(tc::taddr(tmem, warp, kColD23 + BC + 64 * hc + 8 * q), x);
                tc::wait_ld();
                if (KDA) {  // column 64 hc + 8 q + e decays by its own gamma_last
                    const float* sgl = sm + kSGl + (c & 1) * TD + 64 * hc + 8 * q;
#pragma unroll
                    for (int e = 0; e < 8; ++e) m[8 * q + e] = __fmaf_rn(sgl[e], m[8 * q + e], x[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) m[8 * q + e] = __fmaf_rn(gl, m[8 * q + e], x[e]);
                }
                split_store(q);
                if ((q & 3) == 3) release_group(q >> 2);
            }
        }
    }

    if (s_err) {
        // give the copies in flight a bounded chance to land before the TMEM is released
        if (issuer) {
            raise_timeout(kKerState, s_err);
            // the products in flight must be done before the tensor memory is released
            if (mma_out && !tc::mbar_wait(bar_mma, ph_out)) raise_timeout(kKerState, kWTmem);
            if (b1_pending) tc::mbar_wait(bar_b1, ph_b1);
            if (b23_pending) tc::mbar_wait(bar_b23, ph_b23);
        }
    } else if (compute) {
        if (y_nb > 0) store_y();
        store_ckpt((c_end == A.n_chunks ? A.state_T : A.carry) + head * (long long)(TD * TD));
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_free(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------
// The dM chain in reverse on the tensor cores.  One CTA per head owns dM (128 x 128, rows j;
// fp32 in registers, bf16 hi/lo in TMEM as an A operand).  Per chunk, last first:
//   park dM (the gradient of the chunk's end state)
//   Da = dM K^T                 128 x 32,  K = 128   (B: K rows t)
//   dDelta^T = r (.) Da + E     E = scale dY^T QD, precomputed by the prep kernel
//   Db = dDelta^T T             128 x 32,  K = 32    (B: T^T rows t)
//   dX^T = Db
//   Dc = [scale gamma dY^T | -gamma dX^T] [Q; K]     128 x 128, K = 64   (B: [Q^T | K^T]);
//        the dY half does not depend on the chain and is issued right after Da
//   dM <- gamma_last dM + Dc
// Parks dM, dDelta^T and dX^T for the gradient kernel in the unit layout (float4 unit
// (c / 4) * 128 + j holds row j, columns c .. c + 3); writes dstate0 at the end.
namespace {
// TMEM columns: dM as bf16 hi/lo pairs (A of Da, K = 128), Da, Db, Dc, and the bf16 A operand
// of Db, then of Dc's second half (K = 32)
constexpr uint32_t kDsColHi = 0, kDsColLo = 64, kDsColA = 256, kDsColB = 288, kDsColC = 320;
constexpr uint32_t kDsColXh = 448, kDsColXl = 480;
// shared memory (floats): K | T^T | [Q^T | K^T] | scale gamma dY^T | E | r | gamma
constexpr int kSmKb = 0;
constexpr int kSmTT = kSmKb + kDkQKT - kDkKb;
constexpr int kSmQKT = kSmTT + kDsG - kDsTT;
constexpr int kSmG = kSmQKT + kTcDkElems - kDkQKT;
constexpr int kSmE = kSmG + kDsE - kDsG;
constexpr int kSmR = kSmE + kDsR - kDsE;
constexpr int kSmGam = kSmR + kDsGam - kDsR;
constexpr int kSmGl = kSmGam + BC;  // KDA: gamma_last per column, two buffers by chunk parity
constexpr int kDsFloats = kSmGl + 2 * TD;
constexpr size_t kDsSmemBytes = sizeof(float) * kDsFloats + 64;
constexpr uint32_t kDsBytesKb = sizeof(float) * (kDkQKT - kDkKb);
constexpr uint32_t kDsBytesTT = sizeof(float) * (kDsG - kDsTT);
constexpr uint32_t kDsBytesQKT = sizeof(float) * (kTcDkElems - kDkQKT);
constexpr uint32_t kDsBytesTail = sizeof(float) * (kTcDsElems - kDsG);

__device__ __forceinline__ void ds_load_kb(const ChunkArgs& A, long long ck, float* sm, uint64_t* bar)
{
    tc::mbar_expect_tx(bar, kDsBytesKb);
    tc::bulk_g2s(sm + kSmKb, A.ws + A.o_DK + ck * kTcDkElems + kDkKb, kDsBytesKb, bar);
}
template <bool KDA>
__device__ __forceinline__ void ds_load_rest(const ChunkArgs& A, long long ch, long long ck, int c, float* sm,
                                             uint64_t* bar)
{
    tc::mbar_expect_tx(bar, kDsBytesTT + kDsBytesQKT + kDsBytesTail + (KDA ? (uint32_t)sizeof(float) * TD : 0u));
    tc::bulk_g2s(sm + kSmTT, A.ws + A.o_DS + ch * kTcDsElems + kDsTT, kDsBytesTT, bar);
    tc::bulk_g2s(sm + kSmQKT, A.ws + A.o_DK + ck * kTcDkElems + kDkQKT, kDsBytesQKT, bar);
    tc::bulk_g2s(sm + kSmG, A.ws + A.o_DS + ch * kTcDsElems + kDsG, kDsBytesTail, bar);
    if (KDA) tc::bulk_g2s(sm + kSmGl + (c & 1) * TD, A.ws + A.o_gL + ch * TD, sizeof(float) * TD, bar);
}
}  // namespace

// KDA: the per-key-column gate (K (.) R and [Q (.) gamma; K (.) gamma] per value head, r = gamma = 1,
// dM decayed column by column).
template <bool KDA>
__device__ __forceinline__ void dstate_chain(const ChunkArgs& A, float* sm, int h, int n)
{
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kDsFloats);  // kb, rest, mma, x, y
    uint64_t* bar_kb = bars;
    uint64_t* bar_rest = bars + 1;
    uint64_t* bar_mma = bars + 2;
    uint64_t* bar_x = bars + 3;   // dDelta^T, the A operand of Db, is in TMEM
    uint64_t* bar_y = bars + 4;   // -gamma dX^T, the A operand of Dc's second half, is in TMEM
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool compute = warp < 8;
    const bool issuer = tid == kIssuer;
    const int j = 32 * (warp & 3) + lane;   // row of dM
    const int hc = (warp >> 2) & 1;         // dM columns [64 hc, 64 hc + 64); chunk columns [16 hc, 16 hc + 16)
    const long long head = (long long)n * A.H_v + h;
    const long long khead = KDA ? head : (long long)n * A.H_k + h % A.H_k;

    if (tid == 0) {
        tc::mbar_init(bar_kb, 1);
        tc::mbar_init(bar_rest, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init(bar_x, 8);  // one arrival per compute warp
        tc::mbar_init(bar_y, 8);
        tc::mbar_fence_init();
        s_err = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;

    const int c_last = A.c_hi - 1;
    uint32_t ph_kb = 0, ph_rest = 0, ph_mma = 0;
    bool mma_out = false;  // issuer: a committed MMA group not yet seen complete, phase ph_out
    uint32_t ph_out = 0;
    bool kb_pending = false, rest_pending = false;
    if (issuer) {
        tc::prefetch_l2(A.ws + A.o_DS + (head * A.n_chunks + c_last) * kTcDsElems);  // see prefetch_l2
        ds_load_kb(A, khead * A.n_chunks + c_last, sm, bar_kb);
        ds_load_rest<KDA>(A, head * A.n_chunks + c_last, khead * A.n_chunks + c_last, c_last, sm, bar_rest);
        kb_pending = rest_pending = true;
    }
    float m[64];
    if (compute) {
        const float* seed = A.c_hi == A.n_chunks ? A.dstate_T : A.carry;
        if (seed) {
            const float4* s4 = reinterpret_cast<const float4*>(seed + (head * TD + j) * TD + 64 * hc);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 x = __ldg(s4 + q);
                m[4 * q] = x.x;
                m[4 * q + 1] = x.y;
                m[4 * q + 2] = x.z;
                m[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) m[e] = 0.f;
        }
    }
    const float* sE = sm + kSmE;
    const float* sR = sm + kSmR;
    const float* sGam = sm + kSmGam;
    const uint32_t id32 = tc::idesc_bf16(32), id128 = tc::idesc_bf16(128);
    // Row j of a 128 x 32 (rows j, K = t) A operand in TMEM: this thread's columns t in
    // [16 hc, 16 hc + 16), bf16 hi at kDsColXh and lo at kDsColXl (two t per column); then
    // one arrival on `bar` per warp once the warp's stores are complete.
    auto put_a = [&](const float (&v)[16], uint64_t* bar) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) tc::split_bf16x2(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
        tc::st8(tc::taddr(tmem, warp, kDsColXh + 8 * hc), hi);
        tc::st8(tc::taddr(tmem, warp, kDsColXl + 8 * hc), lo);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar);
    };
    auto park16 = [&](long long off, const float (&v)[16]) {  // unit layout, 128 x 32
        float4* d = reinterpret_cast<float4*>(A.ws + off);
#pragma unroll
        for (int b = 0; b < 4; ++b)
            d[(4 * hc + b) * TD + j] = make_float4(v[4 * b], v[4 * b + 1], v[4 * b + 2], v[4 * b + 3]);
    };

    int c = c_last;
    for (; c >= A.c_lo; --c) {
        const long long ch = head * A.n_chunks + c;
        // (1) dM -> bf16 hi/lo in TMEM (two columns i per TMEM column)
        if (compute) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) tc::split_bf16x2(m[8 * q + 2 * e], m[8 * q + 2 * e + 1], hi[e], lo[e]);
                tc::st4(tc::taddr(tmem, warp, kDsColHi + 32 * hc + 4 * q), hi);
                tc::st4(tc::taddr(tmem, warp, kDsColLo + 32 * hc + 4 * q), lo);
            }
            tc::wait_st();
        }
        tc::fence_before();
        __syncthreads();
        // (2) Da = dM K^T, then the chain-free half of Dc; meanwhile park dM
        if (issuer) {
            tc::fence_after();
            if (!tc::mbar_wait(bar_kb, ph_kb)) atomicOr(&s_err, kWCopyA);
            ph_kb ^= 1;
            kb_pending = false;
            if (!s_err) {
                const uint64_t bhi = tc::tile_desc(sm + kSmKb, 32);
                const uint64_t blo = tc::tile_desc(sm + kSmKb + 32 * TD / 2, 32);
#pragma unroll
                for (int s = 0; s < TD / 16; ++s) {
                    const uint32_t ahi = tmem + kDsColHi + 8 * s, alo = tmem + kDsColLo + 8 * s;
                    tc::mma_ts16(tmem + kDsColA, ahi, tc::desc_kslice(bhi, 32, s), id32, s > 0);
                    tc::mma_ts16(tmem + kDsColA, ahi, tc::desc_kslice(blo, 32, s), id32, 1);
                    tc::mma_ts16(tmem + kDsColA, alo, tc::desc_kslice(bhi, 32, s), id32, 1);
                }
                tc::commit(bar_mma);
                mma_out = true;
                ph_out = ph_mma;
                if (!tc::mbar_wait(bar_rest, ph_rest)) atomicOr(&s_err, kWCopyB);
                if (!s_err) {
                    const uint64_t ahi = tc::tile_desc(sm + kSmG, TD), alo = tc::tile_desc(sm + kSmG + BC * TD / 2, TD);
                    const uint64_t qhi = tc::tile_desc(sm + kSmQKT, TD);
                    const uint64_t qlo = tc::tile_desc(sm + kSmQKT + BC * TD, TD);
#pragma unroll
                    for (int s = 0; s < BC / 16; ++s) {
                        const uint64_t a_h = tc::desc_kslice(ahi, TD, s), a_l = tc::desc_kslice(alo, TD, s);
                        const uint64_t b_h = tc::desc_kslice(qhi, TD, s), b_l = tc::desc_kslice(qlo, TD, s);
                        tc::mma_ss16(tmem + kDsColC, a_h, b_h, id128, s > 0);
                        tc::mma_ss16(tmem + kDsColC, a_h, b_l, id128, 1);
                        tc::mma_ss16(tmem + kDsColC, a_l, b_h, id128, 1);
                    }
                }
            }
        } else if (compute) {
            float4* dst = reinterpret_cast<float4*>(A.ws + A.o_dM + ch * (long long)(TD * TD));
#pragma unroll
            for (int q = 0; q < 16; ++q)
                dst[(16 * hc + q) * TD + j] = make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
        }
        // (3) dDelta^T = r (.) Da + E.  Only the compute warps and the issuer wait on bar_mma,
        // and each compute warp arrives on bar_x / bar_y after its wait: so every waiter has
        // seen a phase complete before the issuer commits the next one (a waiter that missed
        // a phase would wait on the one after it).
        bool ok = !(compute || issuer) || tc::mbar_wait(bar_mma, ph_mma);
        if (issuer && ok) mma_out = false;
        ph_mma ^= 1;
        tc::fence_after();
        if (issuer) {
            if (ok && c > A.c_lo) {
                ds_load_kb(A, khead * A.n_chunks + c - 1, sm, bar_kb);
                kb_pending = true;
            }
        } else if (compute) {
            ok = tc::mbar_wait(bar_rest, ph_rest) && ok;
            float x[16];
            tc::ld16(tc::taddr(tmem, warp, kDsColA + 16 * hc), x);
            tc::wait_ld();
            float v[16];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float4 e = *reinterpret_cast<const float4*>(sE + 4 * ((4 * hc + b) * TD + j));
                const int t = 16 * hc + 4 * b;
                v[4 * b] = __fmaf_rn(sR[t], x[4 * b], e.x);
                v[4 * b + 1] = __fmaf_rn(sR[t + 1], x[4 * b + 1], e.y);
                v[4 * b + 2] = __fmaf_rn(sR[t + 2], x[4 * b + 2], e.z);
                v[4 * b + 3] = __fmaf_rn(sR[t + 3], x[4 * b + 3], e.w);
            }
            park16(A.o_dDel + ch * (BC * TD), v);
            put_a(v, bar_x);
        }
        ph_rest ^= 1;
        if (!ok) atomicOr(&s_err, kWMma1);
        const uint32_t ph_xy = (uint32_t)(c_last - c) & 1u;
        // (4) Db = dDelta^T T, issued as soon as dDelta^T is in TMEM
        if (issuer) {
            rest_pending = false;
            if (!tc::mbar_wait(bar_x, ph_xy)) atomicOr(&s_err, kWHandoff1);
            tc::fence_after();
            if (!s_err) {
                const uint64_t bhi = tc::tile_desc(sm + kSmTT, 32), blo = tc::tile_desc(sm + kSmTT + 32 * 32 / 2, 32);
#pragma unroll
                for (int s = 0; s < BC / 16; ++s) {
                    const uint32_t a_h = tmem + kDsColXh + 8 * s, a_l = tmem + kDsColXl + 8 * s;
                    const uint64_t b_h = tc::desc_kslice(bhi, 32, s), b_l = tc::desc_kslice(blo, 32, s);
                    tc::mma_ts16(tmem + kDsColB, a_h, b_h, id32, s > 0);
                    tc::mma_ts16(tmem + kDsColB, a_h, b_l, id32, 1);
                    tc::mma_ts16(tmem + kDsColB, a_l, b_h, id32, 1);
                }
                tc::commit(bar_mma);
                mma_out = true;
                ph_out = ph_mma;
            }
        }
        // (5) dX^T = Db;  A operand <- -gamma dX^T
        ok = !(compute || issuer) || tc::mbar_wait(bar_mma, ph_mma);
        if (issuer && ok) mma_out = false;
        ph_mma ^= 1;
        tc::fence_after();
        float gl = 0.f;
        if (compute) {
            gl = sGam[BC - 1];
            float x[16];
            tc::ld16(tc::taddr(tmem, warp, kDsColB + 16 * hc), x);
            tc::wait_ld();
            park16(A.o_dX + ch * (BC * TD), x);
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = -__fmul_rn(sGam[16 * hc + e], x[e]);
            put_a(v, bar_y);  // Db is done: its A operand's columns are free
        }
        if (!ok) atomicOr(&s_err, kWMma3);
        // (6) Dc += (-gamma dX^T) K, issued as soon as -gamma dX^T is in TMEM
        if (issuer) {
            if (!tc::mbar_wait(bar_y, ph_xy)) atomicOr(&s_err, kWHandoff2);
            tc::fence_after();
            if (!s_err) {
                const uint64_t qhi = tc::tile_desc(sm + kSmQKT, TD);
                const uint64_t qlo = tc::tile_desc(sm + kSmQKT + BC * TD, TD);
#pragma unroll
                for (int s = 0; s < BC / 16; ++s) {
                    const uint32_t a_h = tmem + kDsColXh + 8 * s, a_l = tmem + kDsColXl + 8 * s;
                    const uint64_t b_h = tc::desc_kslice(qhi, TD, s + BC / 16), b_l = tc::desc_kslice(qlo, TD, s + BC / 16);
                    tc::mma_ts16(tmem + kDsColC, a_h, b_h, id128, 1);
                    tc::mma_ts16(tmem + kDsColC, a_h, b_l, id128, 1);
                    tc::mma_ts16(tmem + kDsColC, a_l, b_h, id128, 1);
                }
                tc::commit(bar_mma);
                mma_out = true;
                ph_out = ph_mma;
            }
        }
        // (7) dM <- gamma_last dM + Dc
        ok = !(compute || issuer) || tc::mbar_wait(bar_mma, ph_mma);
        if (issuer && ok) mma_out = false;
        ph_mma ^= 1;
        tc::fence_after();
        if (!__syncthreads_and(ok)) {
            if (!ok) atomicOr(&s_err, kWMma2);
            __syncthreads();
            break;
        }
        if (issuer) {
            if (c > A.c_lo) {
                tc::fence_async_smem();
                ds_load_rest<KDA>(A, ch - 1, khead * A.n_chunks + c - 1, c - 1, sm, bar_rest);
                rest_pending = true;
            }
        } else if (compute) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float x[32];
                tc::ld32(tc::taddr(tmem, warp, kDsColC + 64 * hc + 32 * q), x);
                tc::wait_ld();
                if (KDA) {  // column 64 hc + 32 q + e decays by its own gamma_last
                    const float* sgl = sm + kSmGl + (c & 1) * TD + 64 * hc + 32 * q;
#pragma unroll
                    for (int e = 0; e < 32; ++e) m[32 * q + e] = __fmaf_rn(sgl[e], m[32 * q + e], x[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) m[32 * q + e] = __fmaf_rn(gl, m[32 * q + e], x[e]);
                }
            }
        }
    }

    if (s_err) {
        if (issuer) {
            raise_timeout(kKerDstate, s_err);
            if (mma_out && !tc::mbar_wait(bar_mma, ph_out)) raise_timeout(kKerDstate, kWTmem);
            if (kb_pending) tc::mbar_wait(bar_kb, ph_kb);
            if (rest_pending) tc::mbar_wait(bar_rest, ph_rest);
        }
    } else if (compute) {
        // dstate0 lies in the caller's packed buffer after the dbeta region, so it is 16-byte
        // aligned only when the regions before it hold a multiple of 4 floats
        float* out = (A.c_lo == 0 ? A.dstate0 : A.carry) + (head * TD + j) * TD + 64 * hc;
        if (A.c_lo != 0 || A.vec_ds0) {
            float4* d4 = reinterpret_cast<float4*>(out);
#pragma unroll
            for (int q = 0; q < 16; ++q) d4[q] = make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) out[e] = m[e];
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_free(tmem, kTmemCols);
}

// The forward's state chain: one CTA per (head, sequence).
template <bool KDA>
__global__ void __launch_bounds__(TCT, 1) gdn_tc_state_kernel(const ChunkArgs A)
{
    extern __shared__ __align__(1024) float sm[];
    state_chain<KDA>(A, sm, blockIdx.x, blockIdx.y);
}

// The backward's dM chain: one CTA per (value head, sequence), over the chunks [c_lo, c_hi).
template <bool KDA>
__global__ void __launch_bounds__(TCT, 1) gdn_tc_dstate_kernel(const ChunkArgs A)
{
    extern __shared__ __align__(1024) float sm[];
    dstate_chain<KDA>(A, sm, blockIdx.x, blockIdx.y);
}

template <bool KDA>
static int launch_tc_state_t(const ChunkArgs& a, cudaStream_t s)
{
    int e = (int)cudaFuncSetAttribute(gdn_tc_state_kernel<KDA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kSmemBytes);
    if (e) return e;
    gdn_tc_state_kernel<KDA><<<dim3(a.H_v, a.N), TCT, kSmemBytes, s>>>(a);
    return (int)cudaGetLastError();
}

template <bool KDA>
static int launch_tc_dstate_t(const ChunkArgs& a, cudaStream_t s)
{
    int e = (int)cudaFuncSetAttribute(gdn_tc_dstate_kernel<KDA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kDsSmemBytes);
    if (e) return e;
    gdn_tc_dstate_kernel<KDA><<<dim3(a.H_v, a.N), TCT, kDsSmemBytes, s>>>(a);
    return (int)cudaGetLastError();
}

int launch_tc_state(const ChunkArgs& a, void* stream)
{
    return a.kda ? launch_tc_state_t<true>(a, (cudaStream_t)stream) : launch_tc_state_t<false>(a, (cudaStream_t)stream);
}

int launch_tc_dstate(const ChunkArgs& a, void* stream)
{
    return a.kda ? launch_tc_dstate_t<true>(a, (cudaStream_t)stream) : launch_tc_dstate_t<false>(a, (cudaStream_t)stream);
}

// A bounded wait on a barrier that nothing completes: gives up and records the timeout.
__global__ void gdn_selftest_wait_kernel()
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0)) raise_timeout(kKerSelftest, kWHandoff1);
}

int launch_selftest_wait(void* stream)
{
    gdn_selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>();
    return (int)cudaGetLastError();
}

int tc_take_status(void* stream, int* status)
{
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    int e = (int)cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (!e) e = (int)cudaStreamSynchronize(s);
    if (e) return e;
    if (v) {
        const int zero = 0;
        e = (int)cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (!e) e = (int)cudaStreamSynchronize(s);
    }
    *status = v;
    return e;
}

}  // namespace gdn
