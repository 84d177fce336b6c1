// gdn_internal.h -- host/device shared declarations of libgdn (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#if defined(__CUDACC__)
#define GDN_HD __host__ __device__
#else
#define GDN_HD
#endif

namespace gdn {

// Thread layout shared by every recurrence kernel: a warp holds 4 row groups of 8
// column lanes; lane = 8 * group + column_lane.  Column lane c owns the float4 blocks
// starting at columns 32 v + 4 c (v < S/32) of each row the thread holds.
constexpr int kColLanes = 8;
constexpr int kGroups = 4;

// GB300 facts the launch planner sizes for.
constexpr int kNumSMs = 152;
constexpr int kSmemPerSM = 228 * 1024;     // shared memory per SM
constexpr int kSmemPerCtaMax = 227 * 1024; // opt-in maximum per CTA
constexpr int kSmemReservePerCta = 1024;   // driver-reserved per resident CTA

struct FwdArgs {
    const float* q;
    const float* k;
    const float* v;
    const float* g;
    const float* beta;
    const float* state0;
    float* y;
    float* state_T;
    float* ckpt;
    long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2;
    int N, T, H_k, H_v, C, n_ck;
    int SK, DV;  // key head size (the state's columns) and value head size (its rows)
    int rep;     // value sequences per q/k sequence: q, k of sequence n are those of n / rep
    float scale;
    int tc;  // tokens per shared-memory tile
    int vec_q, vec_k, vec_v, vec_g;
};

struct BwdArgs {
    const float* q;
    const float* k;
    const float* v;
    const float* g;
    const float* beta;
    const float* ckpt;
    const float* gy;
    const float* dstate_T;  // may be null
    float* dv;              // packed dv region
    float* dstate0;         // packed dstate region
    float* sub;             // workspace: level-1 sub-checkpoints
    float* ws_col;          // workspace: per-CTA column partials [N*T*H_v][P][NQ*D]
    float* ws_sc;           // workspace: per-CTA scalar partials [N*T*H_v][P][2]
    long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2, gys0, gys1, gys2;
    int N, T, H_k, H_v, C, n_ck, c2, nsub_max;
    int SK, DV;  // key head size (the state's columns) and value head size (its rows)
    int rep;     // value sequences per q/k sequence: q, k of sequence n are those of n / rep
    float scale;
    int vec_q, vec_k, vec_v, vec_gy, vec_g, vec_ds0;
};

struct ReduceArgs {
    const float* ws_col;
    const float* ws_sc;
    float* dq;
    float* dk;
    float* dg;
    float* dbeta;
    int N, T, H_k, H_v, D, P, NQ, kda;
    int SK;  // output column width (S_k); the partials are D wide
    int rep; // value sequences per q/k sequence: dq, dk sum over each group of rep
};

// Chunked (WY) form, scalar gate: chunk length and the arguments of its kernels.
constexpr int BC = 32;

struct ChunkArgs {
    const float* q;
    const float* k;
    const float* v;
    const float* g;
    const float* beta;
    const float* state0;    // forward input
    const float* ckpt;      // backward input (checkpoints of the forward)
    const float* gy;        // backward input
    const float* dstate_T;  // backward input, may be null
    float* y;               // forward outputs
    float* state_T;
    float* ckpt_out;
    float* dq;              // backward outputs (packed regions)
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dstate0;
    float* ws;              // workspace base
    long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2, gys0, gys1, gys2;
    int N, T, H_k, H_v, C, n_ck, cps, n_chunks;
    int rep;                // value sequences per q/k sequence (q, k of n are those of n / rep)
    float scale;
    // workspace sub-arrays (float offsets from ws), per (sequence, value head, chunk)
    long long o_T, o_QKD, o_QDT, o_gam, o_r, o_W, o_U, o_Mc, o_dM, o_dDel, o_dX;
    long long o_Tr, o_Z, o_KK, o_QK, o_Dm;  // backward: chunk factors for the gradient kernel
    long long o_W1, o_Q1, o_B23;            // tensor-core operands of the state chain
    long long o_DK, o_DS;                   // tensor-core operands of the dM chain
    long long o_dqM, o_dkM;                 // tensor-core gradient step: per value head dq, dk
    // per-key-column (KDA) gate, head size 128, per (sequence, value head, chunk): gamma_last
    // (128 floats), the bf16 hi/lo tiles K (.) gamma (rows t) and (K (.) R)^T (rows i), and
    // gamma, R in fp32 (rows t)
    long long o_gL, o_KG, o_KRT, o_kGam, o_kR;
    // sequence broadcast at head sizes 32, 64: each value sequence's dq, dk [N][T][H_k][D]
    // before the sum over the sequences that share q, k
    long long o_dqS, o_dkS;
    int kda;
    int want_wu;
    int want_factors;
    int want_tc;                            // head size 128: state chain on the tensor cores
    int c_lo, c_hi;                         // chunk range of this launch (prep and chains)
    int grad_loc;                           // gradient launch: -1 for every chunk of [c_lo, c_hi),
                                            // else only the chunks at this place in their segment
    float* carry;                           // [N][H_v][D][D] state (or dM) between ranges
    int vec_q, vec_k, vec_v, vec_gy, vec_g;
    int vec_ds0;                            // the packed dstate region is 16-byte aligned
    int vec_y;                              // y is 16-byte aligned
};

// Records caller-provided timing events around the stages of one call: mark() before
// the first stage and after each one, while events remain.
struct EventTap {
    void* const* ev;
    int n;
    int i;
    void mark(void* stream);
};

// Library streams of one device for the pipelined tensor-core path: the serial chains on
// a high-priority stream, the chunk-range preps (then, backward, the value-head sums) on a
// middle one and the gradient steps on a low one.  Created on first use; the lock
// serialises the enqueueing of calls that use them.
constexpr int kMaxRanges = 4;
// The backward's value-head sums run on their own stream.  Below the gradient steps'
// priority (kSumBelowGrads) their CTAs take what the gradient CTAs leave free on an SM (a sum
// CTA fits beside a gradient CTA) instead of holding the next gradient launch back until
// they are placed: 1.744 against 1.755 ms per step (4096 tokens, 48 heads of 128, three runs
// each).  With kSumByPlace, and at most kMaxPlaces places of a chunk in its segment, each
// gradient launch's chunks are summed as soon as it is done (measured 1.825 against 1.808 ms
// with the sums above the gradient steps); otherwise each chunk range's once all its
// gradient launches are.
constexpr int kMaxPlaces = 4;
constexpr bool kSumBelowGrads = true;
constexpr bool kSumByPlace = false;
struct Pipeline {
    void* hi;   // chains
    void* lo;   // preps
    void* bg;   // gradient steps
    void* sum;  // value-head sums, the least urgent
    void* fork;
    void* join_hi;
    void* join_lo;
    void* join_bg;
    void* join_sum;
    void* prep_done[kMaxRanges];
    void* chain_go[kMaxRanges];
    void* ds_done[kMaxRanges];
    void* grad_done[kMaxRanges];
    void* place_done[kMaxRanges][kMaxPlaces];
};
// Returns the current device's pipeline (creating it on first use) with its lock held;
// release_pipeline() unlocks.  Returns a cudaError_t as int.
int acquire_pipeline(Pipeline** out);
void release_pipeline();
// Chunk ranges of the pipelined path: segment-aligned, at most kMaxRanges.  (A backward
// call with timing events runs its stages one after another instead, as one range.)
int pipeline_ranges(int n_ck, bool backward);
// Checkpoint segments [s_lo, s_hi) of range r of R.  The forward's 4 ranges grow (10, 20,
// 30, 40 % of the segments, from 40 segments up): the state chain cannot start before the
// first range's prep, and each later prep is shorter than the chain range it runs beside.
// The backward's 2 ranges take 35 and 65 % of the segments in walk order (the last
// segments first), from 40 segments up.  Otherwise equal.
void range_segments(int n_ck, int R, bool backward, int r, int* s_lo, int* s_hi);

// Tensor-core operands of the state chain (head size 128), in the bf16 operand layouts of
// gdn_tc.cuh, sizes in floats: W = T diag(gamma) K per (chunk, value head) and Q per (chunk,
// key head), each 32 x 128 as bf16 hi then lo in the row-group-major layout (the two stack
// into the 64-row B operand [W; Q]); [scale QD; (r K)^T] per (chunk, value head) as bf16 hi
// then lo (2 x 160 x 32, k-chunk-major).
constexpr int kTcWElems = 32 * 128;
constexpr int kTcQElems = 32 * 128;
constexpr int kTcB23Elems = 160 * 32;
// Tensor-core operands of the dM chain and the gradient step, sizes in floats.  Per (chunk,
// key head): K (32 x 128, B of dM K^T and of M K^T) and [Q^T | K^T] (128 x 64, B of the dM
// update, A of the gradient's last product) as bf16 hi then lo.  Per (chunk, value head):
// T^T (32 x 32, B of dDelta^T T) and scale gamma dY^T (128 x 32, A of the update) as bf16
// hi then lo, E = scale dY^T QD (128 x 32, fp32, rows j), r and gamma (32 each).
constexpr int kDkKb = 0;
constexpr int kDkQKT = kDkKb + 32 * 128;
constexpr int kTcDkElems = kDkQKT + 128 * 64;
constexpr int kDsTT = 0;
constexpr int kDsG = kDsTT + 32 * 32;
constexpr int kDsE = kDsG + 128 * 32;
constexpr int kDsR = kDsE + 128 * 32;
constexpr int kDsGam = kDsR + 32;
constexpr int kTcDsElems = kDsGam + 32;
// KDA gate: floats of one 32 x 128 bf16 hi/lo tile (K (.) gamma, or (K (.) R)^T).
constexpr int kTcKdaTile = 32 * 128;

int launch_chunk_forward(const ChunkArgs& a, int D, void* stream, EventTap& tap);
// The chains on the tensor cores (gdn_tc_chain.cu): the forward's state chain and the
// backward's dM chain over [c_lo, c_hi).
int launch_tc_state(const ChunkArgs& a, void* stream);
int launch_tc_dstate(const ChunkArgs& a, void* stream);
// The gradient step on the tensor cores (gdn_tc_grad.cu): per (chunk, value head) every
// gradient of the chunk (dv, dg, dbeta written; this value head's dq, dk parked row-major
// [t][i] at o_dqM, o_dkM), then the sum of the value heads of each key head.
// With grad_loc = k >= 0 a launch covers the chunks at place k of the segments of
// [c_lo, c_hi) and parks the entry state of each one's successor in its segment (the
// launch for k + 1 reads it), so the launches for k = 0, 1, .. run in order.
int launch_tc_grad(const ChunkArgs& a, void* stream);
int tc_grad_units(const ChunkArgs& a);  // the launch's chunks per (value head, sequence)
int launch_tc_dqdk_sum(const ChunkArgs& a, void* stream);
int tc_grad_take_status(void* stream, int* status);
// Reads and clears the tensor-core kernels' device status word (0 or GDN_ERR_TIMEOUT),
// synchronising `stream`.  Returns a cudaError_t as int.
int tc_take_status(void* stream, int* status);
// One kernel whose bounded wait gives up, recording a timeout (test of that path).
int launch_selftest_wait(void* stream);
int launch_chunk_backward(const ChunkArgs& a, int D, void* stream, EventTap& tap);

// Shared-memory layout of the backward kernel, in floats (every offset a multiple of 4).
struct BwdSmem {
    int ring, sk, sq, sa, sb, sv, sgy, sdel, svmu, sdd, scol, sdg, total;
};

GDN_HD inline int round4(int x) { return (x + 3) & ~3; }

GDN_HD inline BwdSmem bwd_smem_layout(int D, int RT, int W, int c2, bool kda)
{
    const int NT = 32 * W, R = 4 * RT * W, NV = D / 32, NQ = kda ? 3 : 2;
    BwdSmem s;
    int o = 0;
    s.ring = o; o += c2 * RT * NV * NT * 4;
    s.sk = o;   o += c2 * D;
    s.sq = o;   o += c2 * D;
    s.sa = o;   o += kda ? c2 * D : round4(c2);
    s.sb = o;   o += round4(c2);
    s.sv = o;   o += round4(c2 * R);
    s.sgy = o;  o += round4(c2 * R);
    s.sdel = o; o += round4(c2 * R);
    s.svmu = o; o += round4(c2 * R);
    s.sdd = o;  o += round4(c2 * R);
    s.scol = o; o += W * c2 * NQ * D;
    s.sdg = o;  o += kda ? 0 : W * c2 * 32;
    s.total = o;
    return s;
}

struct FwdSmem {
    int sk, sq, sa, sb, sv, sy, total;
};

GDN_HD inline FwdSmem fwd_smem_layout(int D, int RT, int W, int tc, bool kda)
{
    const int R = 4 * RT * W;
    FwdSmem s;
    int o = 0;
    s.sk = o; o += tc * D;
    s.sq = o; o += tc * D;
    s.sa = o; o += kda ? tc * D : round4(tc);
    s.sb = o; o += round4(tc);
    s.sv = o; o += round4(tc * R);
    s.sy = o; o += round4(tc * R);
    s.total = o;
    return s;
}

// Launchers (defined in gdn_fwd.cu / gdn_bwd.cu).  Return a cudaError_t as int.
int launch_forward(const FwdArgs& a, int D, int RT, int W, bool kda, void* stream);
int launch_backward(const BwdArgs& a, int D, int RT, int W, bool kda, void* stream);
int launch_reduce(const ReduceArgs& a, void* stream);

// Widens a bf16 (in_dtype 1) or fp16 (2) tensor [N][T][H][D] with element strides s (last
// dim contiguous) into dense fp32 at dst (gdn_widen.cu).  Returns a cudaError_t as int.
int launch_widen(const void* src, int in_dtype, const long long s[3], int N, int T, int H, int D, float* dst,
                 void* stream);

// Sets the text gdn_last_error() returns on the calling thread.
void set_last_error(const char* msg);

}  // namespace gdn
