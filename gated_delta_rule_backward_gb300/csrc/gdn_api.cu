// gdn_api.cu -- host side of libgdn: argument validation, launch planning, the C ABI.
//
// The operation and its citations are stated in include/gdn.h.  Nothing here computes
// any part of the recurrence: every step runs in the kernels of gdn_fwd.cu / gdn_bwd.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

thread_local std::string g_last_error;
thread_local void* const* g_events = nullptr;
thread_local int g_n_events = 0;

gdn_status_t fail(gdn_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gdn_status_t fail(gdn_status_t s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

int64_t ceil_sqrt(int64_t T)
{
    if (T <= 1) return 1;
    int64_t r = 1;
    while (r * r < T) ++r;
    return r;
}

// Launch plan: everything the kernels and the workspace sizes depend on.  The scalar gate,
// and the per-key-column (KDA) gate at head size 128, run the chunked (WY) kernels; the KDA
// gate at head sizes 32 and 64 and the degenerate T = 0 case run the token recurrence.
struct Plan {
    int D = 0, RT = 1, W = 4, R = 16, P = 1, tc = 32, c2 = 1, nsub_max = 1;
    int SK = 0, DV = 0;  // the state's columns (key head size) and rows (value head size)
    int rep = 1;         // value sequences per q/k sequence
    bool kda = false;
    bool chunked = false;
    int64_t C = 1, n_ck = 0;
    size_t off_sub = 0, off_col = 0, off_sc = 0, ws_bytes = 0;  // recurrence backward
    // chunked form
    int cps = 1;          // chunks per checkpoint segment
    int64_t n_chunks = 0; // chunks per (sequence, value head)
    long long o_T = 0, o_QKD = 0, o_QDT = 0, o_gam = 0, o_r = 0, o_W = 0, o_U = 0, o_Mc = 0, o_dM = 0,
              o_dDel = 0, o_dX = 0, o_Tr = 0, o_Z = 0, o_KK = 0, o_QK = 0, o_Dm = 0, o_W1 = 0, o_Q1 = 0, o_B23 = 0, o_DK = 0, o_DS = 0,
              o_dqM = 0, o_dkM = 0, o_carry = 0, o_carry_b = 0, o_gL = 0, o_KG = 0, o_KRT = 0, o_kGam = 0,
              o_kR = 0, o_dqS = 0, o_dkS = 0;
    bool tensor = false;  // head size 128: the state chain runs on the tensor cores
    size_t fwd_ws_bytes = 0, bwd_ws_bytes = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

gdn_status_t check_sizes(const gdn_params_t* p)
{
    if (!p) return fail(GDN_ERR_INVALID_ARG, "params is NULL");
    if (p->seq_rep < 0) return fail(GDN_ERR_INVALID_ARG, "negative seq_rep");
    if (p->n_seq % (p->seq_rep > 1 ? p->seq_rep : 1) != 0)
        return fail(GDN_ERR_INVALID_ARG, "n_seq (%lld) is not a multiple of seq_rep (%d)", (long long)p->n_seq,
                    (int)p->seq_rep);
    if (p->in_dtype != GDN_F32 && p->in_dtype != GDN_BF16 && p->in_dtype != GDN_F16)
        return fail(GDN_ERR_INVALID_ARG, "unknown input dtype %d", (int)p->in_dtype);
    if (p->n_seq < 0 || p->T < 0) return fail(GDN_ERR_INVALID_ARG, "negative n_seq or T");
    if (p->H_k < 1 || p->H_v < 1) return fail(GDN_ERR_INVALID_ARG, "H_k and H_v must be >= 1");
    if (p->H_v % p->H_k != 0)
        return fail(GDN_ERR_INVALID_ARG, "H_v (%lld) is not a multiple of H_k (%lld)",
                    (long long)p->H_v, (long long)p->H_k);
    if (p->gate != GDN_GATE_SCALAR && p->gate != GDN_GATE_KDA)
        return fail(GDN_ERR_INVALID_ARG, "unknown gate kind %d", (int)p->gate);
    if (p->S_k < 1 || p->S_v < 1) return fail(GDN_ERR_INVALID_ARG, "head sizes must be >= 1");
    if (p->S_k != 16 && p->S_k != 32 && p->S_k != 64 && p->S_k != 128 && p->S_k != 256)
        return fail(GDN_ERR_UNSUPPORTED, "key head size S_k = %lld is not supported (16, 32, 64, 128, 256)",
                    (long long)p->S_k);
    if (p->S_v % 16 != 0 || p->S_v > 256)
        return fail(GDN_ERR_UNSUPPORTED, "value head size S_v = %lld is not supported (a multiple of 16 up to 256)",
                    (long long)p->S_v);
    if (p->T > INT_MAX / 2 || p->H_v > 65535 || p->n_seq > 65535)
        return fail(GDN_ERR_UNSUPPORTED, "sizes beyond the kernels' index range");
    for (int i = 0; i < 3; ++i)
        if (p->q_s[i] < 0 || p->k_s[i] < 0 || p->v_s[i] < 0 || p->gy_s[i] < 0)
            return fail(GDN_ERR_INVALID_ARG, "negative stride");
    return GDN_OK;
}

Plan make_plan(const gdn_params_t* p)
{
    Plan pl;
    // the token recurrence computes at column width D: S_k, or 32 for S_k = 16 (zero padding)
    pl.SK = (int)p->S_k;
    pl.DV = (int)p->S_v;
    pl.D = pl.SK < 32 ? 32 : pl.SK;
    pl.rep = p->seq_rep > 1 ? p->seq_rep : 1;
    pl.kda = p->gate == GDN_GATE_KDA;
    pl.C = p->C > 0 ? p->C : ceil_sqrt(p->T);
    if (pl.C > INT_MAX / 2) pl.C = INT_MAX / 2;
    pl.n_ck = p->T > 0 ? (p->T + pl.C - 1) / pl.C : 0;
    pl.RT = 1;
    pl.W = 4;
    pl.R = 4 * pl.RT * pl.W;
    pl.P = pl.DV / pl.R;
    pl.tc = 32;
    // Sub-segment length c2: as many ring slots as fit the shared memory of the number
    // of CTAs each SM must hold for the whole grid to be resident (at most 4 per SM).
    const long long ctas = (long long)p->n_seq * p->H_v * pl.P;
    long long per_sm = (ctas + gdn::kNumSMs - 1) / gdn::kNumSMs;
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 4) per_sm = 4;
    long long budget = gdn::kSmemPerSM / per_sm - gdn::kSmemReservePerCta;
    if (budget > gdn::kSmemPerCtaMax) budget = gdn::kSmemPerCtaMax;
    const int cmax = (int)(pl.C < 64 ? pl.C : 64);
    int c2 = 1;
    for (int c = cmax; c >= 1; --c) {
        const gdn::BwdSmem L = gdn::bwd_smem_layout(pl.D, pl.RT, pl.W, c, pl.kda);
        if ((long long)L.total * 4 <= budget) { c2 = c; break; }
    }
    pl.c2 = c2;
    pl.nsub_max = (int)((pl.C + c2 - 1) / c2);
    if (p->T > 0 && pl.nsub_max > (p->T + c2 - 1) / c2) pl.nsub_max = (int)((p->T + c2 - 1) / c2);
    // workspace: sub-checkpoints | column partials | scalar partials
    const size_t NQ = pl.kda ? 3 : 2;
    const size_t cta_state = (size_t)pl.R * pl.D;  // floats per CTA per stored state
    const size_t sub_f = (size_t)ctas * (pl.nsub_max > 1 ? pl.nsub_max - 1 : 0) * cta_state;
    const size_t toks = (size_t)p->n_seq * p->T * p->H_v;
    const size_t col_f = toks * pl.P * NQ * pl.D;
    const size_t sc_f = toks * pl.P * 2;
    pl.off_sub = 0;
    pl.off_col = align256(sub_f * 4);
    pl.off_sc = pl.off_col + align256(col_f * 4);
    pl.ws_bytes = pl.off_sc + align256(sc_f * 4);

    // chunked (WY) kernels: square heads of size 32, 64 or 128 (the per-key-column gate at
    // 128 only); every other shape runs the token recurrence
    pl.chunked = p->T > 0 && pl.SK == pl.DV && (pl.SK == 32 || pl.SK == 64 || pl.SK == 128) &&
                 (!pl.kda || pl.SK == 128);
    if (pl.chunked) {
        const int64_t BC = gdn::BC;
        pl.cps = (int)((pl.C + BC - 1) / BC);
        const int64_t last_len = p->T - (pl.n_ck - 1) * pl.C;
        pl.n_chunks = (pl.n_ck - 1) * pl.cps + (last_len + BC - 1) / BC;
        const int64_t CH = p->n_seq * p->H_v * pl.n_chunks;
        const int64_t CK = p->n_seq * p->H_k * pl.n_chunks;
        const int64_t D = pl.D;
        pl.tensor = (D == 128);
        // the blocks the scalar gate keeps once per key head (Q, K, [Q^T | K^T]) carry the
        // per-value-head decay with the KDA gate: one per value head
        const int64_t CKq = pl.kda ? CH : CK;
        // float offsets, each sub-array 256-byte aligned
        auto al = [](int64_t f) { return (long long)((f + 63) & ~int64_t(63)); };
        long long o = 0;
        if (!pl.tensor) {  // the FP32 chains' operands T^T, QD, QD^T
            pl.o_T = o;   o += al(CH * BC * BC);
            pl.o_QKD = o; o += al(CH * BC * BC);
            pl.o_QDT = o; o += al(CH * BC * BC);
        }
        pl.o_gam = o; o += al(CH * BC);
        pl.o_r = o;   o += al(CH * BC);
        if (pl.kda) {  // gamma_last per column, written by both preps
            pl.o_gL = o; o += al(CH * D);
        }
        const long long common = o;
        if (pl.tensor) {  // U^T in fp32 and the tf32 hi/lo operands, tensor-core layout
            pl.o_U = o;   o += al(CH * BC * D);
            pl.o_W1 = o;  o += al(CH * gdn::kTcWElems);
            pl.o_Q1 = o;  o += al(CKq * gdn::kTcQElems);
            pl.o_B23 = o; o += al(CH * gdn::kTcB23Elems);
            pl.o_carry = o; o += al(p->n_seq * p->H_v * D * D);  // forward: state between ranges
        } else {
            pl.o_W = o;   o += al(CH * BC * D);
            pl.o_U = o;   o += al(CH * BC * D);
        }
        pl.fwd_ws_bytes = (size_t)o * 4;
        // backward: W, U and the chunk-entry states only when segments hold several chunks
        if (pl.cps > 1) {
            pl.o_Mc = o; o += al(CH * D * D);
        } else {
            o = common;
        }
        pl.o_Tr = o;   o += al(CH * BC * BC);
        pl.o_Z = o;    o += al(CH * BC * BC);
        pl.o_KK = o;   o += al(CH * BC * BC);
        pl.o_QK = o;   o += al(CH * BC * BC);
        if (!pl.kda) {
            pl.o_Dm = o; o += al(CH * BC * BC);
        }
        pl.o_dM = o;   o += al(CH * D * D);
        pl.o_dDel = o; o += al(CH * BC * D);
        pl.o_dX = o;   o += al(CH * BC * D);
        if (pl.tensor) {
            pl.o_DK = o;  o += al(CKq * gdn::kTcDkElems);
            pl.o_DS = o;  o += al(CH * gdn::kTcDsElems);
            pl.o_dqM = o; o += al(CH * BC * D);
            pl.o_dkM = o; o += al(CH * BC * D);
            pl.o_carry_b = o; o += al(p->n_seq * p->H_v * D * D);  // dM between ranges
            if (pl.kda) {  // the gradient step's K (.) gamma, (K (.) R)^T tiles, gamma and R
                pl.o_KG = o;   o += al(CH * gdn::kTcKdaTile);
                pl.o_KRT = o;  o += al(CH * gdn::kTcKdaTile);
                pl.o_kGam = o; o += al(CH * BC * D);
                pl.o_kR = o;   o += al(CH * BC * D);
            }
        } else if (pl.rep > 1) {  // each value sequence's dq, dk before the sequence sums
            pl.o_dqS = o; o += al(p->n_seq * p->T * p->H_k * D);
            pl.o_dkS = o; o += al(p->n_seq * p->T * p->H_k * D);
        }
        pl.bwd_ws_bytes = (size_t)o * 4;
        pl.ws_bytes = pl.bwd_ws_bytes;
    }
    return pl;
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

// Byte extent of a [N][T][H][D] tensor with element strides {s0, s1, s2, 1} and elements of
// `es` bytes.
Range extent4(const void* ptr, int64_t N, int64_t T, int64_t H, int64_t D, const int64_t s[3], size_t es = 4)
{
    const uintptr_t lo = (uintptr_t)ptr;
    if (!ptr || N == 0 || T == 0 || H == 0 || D == 0) return {lo, lo};
    const uint64_t last = (uint64_t)(s[0] * (N - 1) + s[1] * (T - 1) + s[2] * (H - 1) + D);
    return {lo, lo + last * es};
}

Range extent_dense(const void* ptr, size_t elems, size_t es = 4)
{
    const uintptr_t lo = (uintptr_t)ptr;
    return {lo, ptr ? lo + elems * es : lo};
}

// 16-bit input storage: the dense fp32 copies of q, k, v, g, beta (and, backward, gy) the
// call widens its inputs into, at the start of its workspace (byte offsets).
struct Wide {
    size_t q = 0, k = 0, v = 0, g = 0, b = 0, gy = 0, total = 0;
};

Wide wide_layout(const gdn_params_t* p, bool backward)
{
    Wide w;
    if (p->in_dtype == GDN_F32) return w;
    const size_t N = (size_t)p->n_seq, T = (size_t)p->T, Hk = (size_t)p->H_k, Hv = (size_t)p->H_v;
    const size_t Sk = (size_t)p->S_k, Sv = (size_t)p->S_v, gw = p->gate == GDN_GATE_KDA ? Sk : 1;
    const size_t Nq = (size_t)p->n_seq / (size_t)(p->seq_rep > 1 ? p->seq_rep : 1);
    size_t o = 0;
    w.q = o; o += align256(Nq * T * Hk * Sk * 4);
    w.k = o; o += align256(Nq * T * Hk * Sk * 4);
    w.v = o; o += align256(N * T * Hv * Sv * 4);
    w.g = o; o += align256(N * T * Hv * gw * 4);
    w.b = o; o += align256(N * T * Hv * 4);
    if (backward) {
        w.gy = o; o += align256(N * T * Hv * Sv * 4);
    }
    w.total = o;
    return w;
}

// The fp32 parameters of the widened copies: dense strides, in_dtype fp32.
gdn_params_t dense_f32(const gdn_params_t* p)
{
    gdn_params_t q = *p;
    q.in_dtype = GDN_F32;
    const int64_t T = p->T, Hk = p->H_k, Hv = p->H_v, Sk = p->S_k, Sv = p->S_v;
    const int64_t qs[3] = {T * Hk * Sk, Hk * Sk, Sk}, vs[3] = {T * Hv * Sv, Hv * Sv, Sv};
    for (int i = 0; i < 3; ++i) {
        q.q_s[i] = q.k_s[i] = qs[i];
        q.v_s[i] = q.gy_s[i] = vs[i];
    }
    return q;
}

bool overlap(Range a, Range b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

bool vec_ok(const void* ptr, const int64_t s[3])
{
    return aligned(ptr, 16) && s[0] % 4 == 0 && s[1] % 4 == 0 && s[2] % 4 == 0;
}

// The q/k sequences: n_seq / seq_rep (the sequence broadcast), else n_seq.
int64_t qk_seqs(const gdn_params_t* p) { return p->n_seq / (p->seq_rep > 1 ? p->seq_rep : 1); }

void packed_offsets(const gdn_params_t* p, size_t off[7])
{
    const size_t N = (size_t)p->n_seq, T = (size_t)p->T, Hk = (size_t)p->H_k, Hv = (size_t)p->H_v;
    const size_t Sk = (size_t)p->S_k, Sv = (size_t)p->S_v, Nq = (size_t)qk_seqs(p);
    off[0] = 0;
    off[1] = off[0] + Nq * T * Hk * Sk;
    off[2] = off[1] + Nq * T * Hk * Sk;
    off[3] = off[2] + N * T * Hv * Sv;
    off[4] = off[3] + N * T * Hv * (p->gate == GDN_GATE_KDA ? Sk : 1);
    off[5] = off[4] + N * T * Hv;
    off[6] = off[5] + N * Hv * Sv * Sk;
}

gdn_status_t cuda_status(int err, const char* what)
{
    if (err == 0) return GDN_OK;
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString((cudaError_t)err));
}

void fill_chunk_common(gdn::ChunkArgs& c, const gdn_params_t* p, const Plan& pl)
{
    c.qs0 = p->q_s[0]; c.qs1 = p->q_s[1]; c.qs2 = p->q_s[2];
    c.ks0 = p->k_s[0]; c.ks1 = p->k_s[1]; c.ks2 = p->k_s[2];
    c.vs0 = p->v_s[0]; c.vs1 = p->v_s[1]; c.vs2 = p->v_s[2];
    c.gys0 = p->gy_s[0]; c.gys1 = p->gy_s[1]; c.gys2 = p->gy_s[2];
    c.N = (int)p->n_seq; c.T = (int)p->T; c.H_k = (int)p->H_k; c.H_v = (int)p->H_v;
    c.C = (int)pl.C; c.n_ck = (int)pl.n_ck; c.cps = pl.cps; c.n_chunks = (int)pl.n_chunks;
    c.scale = p->scale;
    c.o_T = pl.o_T; c.o_QKD = pl.o_QKD; c.o_QDT = pl.o_QDT; c.o_gam = pl.o_gam; c.o_r = pl.o_r; c.o_W = pl.o_W;
    c.o_U = pl.o_U; c.o_Mc = pl.o_Mc; c.o_dM = pl.o_dM; c.o_dDel = pl.o_dDel; c.o_dX = pl.o_dX;
    c.o_Tr = pl.o_Tr; c.o_Z = pl.o_Z; c.o_KK = pl.o_KK; c.o_QK = pl.o_QK; c.o_Dm = pl.o_Dm;
    c.o_W1 = pl.o_W1; c.o_Q1 = pl.o_Q1; c.o_B23 = pl.o_B23; c.o_DK = pl.o_DK; c.o_DS = pl.o_DS;
    c.o_dqM = pl.o_dqM; c.o_dkM = pl.o_dkM;
    c.o_gL = pl.o_gL; c.o_KG = pl.o_KG; c.o_KRT = pl.o_KRT; c.o_kGam = pl.o_kGam; c.o_kR = pl.o_kR;
    c.o_dqS = pl.o_dqS; c.o_dkS = pl.o_dkS;
    c.kda = pl.kda;
    c.rep = pl.rep;
    c.want_tc = pl.tensor;
    c.c_lo = 0;
    c.c_hi = (int)pl.n_chunks;
    c.grad_loc = -1;
}

// Chunk ranges the pipelined tensor-core path launches (non-empty ones).
int tc_ranges(const Plan& pl, bool backward)
{
    const int R = gdn::pipeline_ranges((int)pl.n_ck, backward);
    int n = 0;
    for (int r = 0; r < R; ++r) {
        int s_lo = 0, s_hi = 0;
        gdn::range_segments((int)pl.n_ck, R, backward, r, &s_lo, &s_hi);
        if (std::min<int64_t>(pl.n_chunks, (int64_t)s_hi * pl.cps) > std::min<int64_t>(pl.n_chunks, (int64_t)s_lo * pl.cps))
            ++n;
    }
    return n;
}

// Kernels of a tensor-core backward call: per non-empty range the prep, the dM chain, one
// gradient launch per place in a segment that has chunks there, and the sums over value heads
// (one per gradient launch, or one per range).
int tc_backward_launches(const Plan& pl)
{
    const int R = gdn::pipeline_ranges((int)pl.n_ck, true);
    int n = 0;
    for (int r = 0; r < R; ++r) {
        int s_lo = 0, s_hi = 0;
        gdn::range_segments((int)pl.n_ck, R, true, r, &s_lo, &s_hi);
        gdn::ChunkArgs a{};
        a.cps = pl.cps;
        a.c_lo = (int)std::min<int64_t>(pl.n_chunks, (int64_t)s_lo * pl.cps);
        a.c_hi = (int)std::min<int64_t>(pl.n_chunks, (int64_t)s_hi * pl.cps);
        if (a.c_hi <= a.c_lo) continue;
        n += 2;  // prep, dM chain
        int places = 0;  // gradient launches, one per place with chunks
        for (a.grad_loc = 0; a.grad_loc < pl.cps; ++a.grad_loc) places += gdn::tc_grad_units(a) > 0 ? 1 : 0;
        const bool by_place = gdn::kSumByPlace && pl.cps <= gdn::kMaxPlaces;
        n += places + (by_place ? places : 1);  // and the sums over value heads
    }
    return n;
}

}  // namespace

void gdn::set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

namespace {
constexpr int kMaxDevices = 64;
gdn::Pipeline g_pipes[kMaxDevices];
bool g_pipe_ready[kMaxDevices];
std::mutex g_pipe_mu[kMaxDevices];
thread_local int g_pipe_held = -1;
}  // namespace

int gdn::acquire_pipeline(gdn::Pipeline** out)
{
    int dev = 0;
    int e = (int)cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    g_pipe_mu[dev].lock();
    g_pipe_held = dev;
    if (!g_pipe_ready[dev]) {
        gdn::Pipeline& P = g_pipes[dev];
        int least = 0, greatest = 0;
        e = (int)cudaDeviceGetStreamPriorityRange(&least, &greatest);
        // numerically lower is more urgent: chains first, then preps; the gradient steps and
        // the sums in the order kSumBelowGrads sets (levels the device lacks fall back to the
        // least urgent one)
        auto level = [&](int k) { return greatest + k < least ? greatest + k : least; };
        const int grads = gdn::kSumBelowGrads ? level(2) : least;
        const int sums = gdn::kSumBelowGrads ? least : level(1);
        cudaStream_t hi = nullptr, lo = nullptr, bg = nullptr, sm = nullptr;
        if (!e) e = (int)cudaStreamCreateWithPriority(&hi, cudaStreamNonBlocking, greatest);
        if (!e) e = (int)cudaStreamCreateWithPriority(&lo, cudaStreamNonBlocking, level(1));
        if (!e) e = (int)cudaStreamCreateWithPriority(&bg, cudaStreamNonBlocking, grads);
        if (!e) e = (int)cudaStreamCreateWithPriority(&sm, cudaStreamNonBlocking, sums);
        constexpr int kEv = 5 + 4 * gdn::kMaxRanges + gdn::kMaxRanges * gdn::kMaxPlaces;
        cudaEvent_t ev[kEv] = {};
        for (int i = 0; i < kEv && !e; ++i)
            e = (int)cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
        if (e) {
            release_pipeline();
            return e;
        }
        P.hi = hi;
        P.lo = lo;
        P.bg = bg;
        P.sum = sm;
        P.fork = ev[0];
        P.join_hi = ev[1];
        P.join_lo = ev[2];
        P.join_bg = ev[3];
        P.join_sum = ev[4];
        for (int i = 0; i < gdn::kMaxRanges; ++i) {
            P.prep_done[i] = ev[5 + i];
            P.chain_go[i] = ev[5 + gdn::kMaxRanges + i];
            P.ds_done[i] = ev[5 + 2 * gdn::kMaxRanges + i];
            P.grad_done[i] = ev[5 + 3 * gdn::kMaxRanges + i];
            for (int k = 0; k < gdn::kMaxPlaces; ++k)
                P.place_done[i][k] = ev[5 + 4 * gdn::kMaxRanges + i * gdn::kMaxPlaces + k];
        }
        g_pipe_ready[dev] = true;
    }
    *out = &g_pipes[dev];
    return 0;
}

void gdn::release_pipeline()
{
    if (g_pipe_held >= 0) {
        const int dev = g_pipe_held;
        g_pipe_held = -1;
        g_pipe_mu[dev].unlock();
    }
}

namespace {
// The backward's ranges and their shares of the segments, in the order the backward walks
// them (the last segments first).  The first range is the smaller: its prep and dM chain
// run with nothing beside them, while the second range's run beside the first range's
// gradient step.  At the 4096-token, 64-segment workload, on one GB300: 40/60 1.833 ms per
// step, 45/55 1.840, 35/65 1.870, 30/70 1.880, 50/50 1.881 (three runs each; three ranges
// were 1.90-1.94 when last tried).  After the gradient step's code shrank (it shares its SMs
// with the second range's prep and dM chain) 35/65 took the lead: 1.713-1.715 ms against
// 1.714-1.740 for 40/60 (four alternating runs each), 45/55 1.726-1.747.
constexpr int kBwdRanges = 2;
constexpr int kBwdWalkPct[gdn::kMaxRanges] = {35, 65, 0, 0};
}  // namespace

int gdn::pipeline_ranges(int n_ck, bool backward)
{
    const int m = backward ? kBwdRanges : gdn::kMaxRanges;
    return n_ck < m ? (n_ck < 1 ? 1 : n_ck) : m;
}

void gdn::range_segments(int n_ck, int R, bool backward, int r, int* s_lo, int* s_hi)
{
    if (!backward && R == 4 && n_ck >= 40) {  // every range keeps at least 4 segments
        static const int kCum[5] = {0, 10, 30, 60, 100};  // percent of the segments
        *s_lo = (int)((long long)n_ck * kCum[r] / 100);
        *s_hi = (int)((long long)n_ck * kCum[r + 1] / 100);
        return;
    }
    if (backward && R == kBwdRanges && R > 1 && n_ck >= 40) {
        const int w = R - 1 - r;  // walk position of range r
        int cum_lo = 0;
        for (int i = 0; i < w; ++i) cum_lo += kBwdWalkPct[i];
        const int cum_hi = w == R - 1 ? 100 : cum_lo + kBwdWalkPct[w];
        *s_hi = n_ck - (int)((long long)n_ck * cum_lo / 100);
        *s_lo = n_ck - (int)((long long)n_ck * cum_hi / 100);
        return;
    }
    const int per = (n_ck + R - 1) / R;
    *s_lo = std::min(n_ck, r * per);
    *s_hi = std::min(n_ck, (r + 1) * per);
}

void gdn::EventTap::mark(void* stream)
{
    if (ev && i < n) cudaEventRecord((cudaEvent_t)ev[i], (cudaStream_t)stream);
    ++i;
}

extern "C" {

gdn_status_t gdn_forward(const gdn_params_t* p, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* state0, float* y,
                         float* state_T, float* ckpt, void* workspace, size_t workspace_bytes,
                         void* stream);

int64_t gdn_checkpoint_interval(const gdn_params_t* p)
{
    if (!p) return 0;
    return p->C > 0 ? p->C : ceil_sqrt(p->T);
}

int64_t gdn_num_checkpoints(const gdn_params_t* p)
{
    if (!p || p->T <= 0) return 0;
    const int64_t C = gdn_checkpoint_interval(p);
    return (p->T + C - 1) / C;
}

size_t gdn_ckpt_elems(const gdn_params_t* p)
{
    if (!p) return 0;
    return (size_t)p->n_seq * p->H_v * gdn_num_checkpoints(p) * p->S_v * p->S_k;
}

size_t gdn_packed_grad_elems(const gdn_params_t* p)
{
    if (!p) return 0;
    size_t off[7];
    packed_offsets(p, off);
    return off[6];
}

void gdn_packed_grad_offsets(const gdn_params_t* p, size_t off[6])
{
    if (!p || !off) return;
    size_t o[7];
    packed_offsets(p, o);
    for (int i = 0; i < 6; ++i) off[i] = o[i];
}

size_t gdn_backward_workspace_bytes(const gdn_params_t* p)
{
    if (check_sizes(p) != GDN_OK) return 0;
    return wide_layout(p, true).total + make_plan(p).ws_bytes;
}

size_t gdn_forward_workspace_bytes(const gdn_params_t* p)
{
    if (check_sizes(p) != GDN_OK) return 0;
    const Plan pl = make_plan(p);
    return wide_layout(p, false).total + (pl.chunked ? pl.fwd_ws_bytes : 0);
}

int gdn_forward_launches(const gdn_params_t* p)
{
    if (check_sizes(p) != GDN_OK) return 0;
    if (p->n_seq == 0) return 0;
    if (p->in_dtype != GDN_F32) {  // the widening kernels, then the fp32 path
        const gdn_params_t q = dense_f32(p);
        return (p->T > 0 ? 5 : 0) + gdn_forward_launches(&q);
    }
    const Plan pl = make_plan(p);
    if (pl.chunked && pl.tensor) return 2 * tc_ranges(pl, false);  // prep + state chain per range
    return pl.chunked ? 2 : 1;
}

int gdn_timing_stages(const gdn_params_t* p, int backward)
{
    if (check_sizes(p) != GDN_OK) return 0;
    if (p->n_seq == 0) return 0;
    const Plan pl = make_plan(p);
    if (pl.chunked && pl.tensor) return backward ? 3 : 1;
    return backward ? gdn_backward_launches(p) : gdn_forward_launches(p);
}

int gdn_backward_launches(const gdn_params_t* p)
{
    if (check_sizes(p) != GDN_OK) return 0;
    if (p->n_seq == 0) return 0;
    if (p->in_dtype != GDN_F32) {
        const gdn_params_t q = dense_f32(p);
        return (p->T > 0 ? 6 : 0) + gdn_backward_launches(&q);
    }
    const Plan pl = make_plan(p);
    // chunked: prep, [recompute], dM chain, gradients.  On the tensor-core path, per chunk
    // range: prep, dM chain, a gradient launch per place in a segment, and the sums over value
    // heads.  (A call with timing events runs its stages as one range, with one sum.)
    if (pl.chunked) return pl.tensor ? tc_backward_launches(pl) : (pl.cps > 1 ? 4 : 3) + (pl.rep > 1 ? 1 : 0);
    return p->T > 0 ? 2 : 1;
}

gdn_status_t gdn_device_status(void* stream)
{
    int a = 0, b = 0;
    int e = gdn::tc_take_status(stream, &a);
    if (!e) e = gdn::tc_grad_take_status(stream, &b);
    if (e) return cuda_status(e, "device status");
    if (!a && !b) return GDN_OK;
    // chain status word: 6 | kernel << 4 | wait-site bits << 8 (gdn_tc_chain.cu)
    static const char* const kernels[] = {"?", "state chain", "?", "dM chain", "selftest"};
    const int ker = (a >> 4) & 15;
    // wait-site bit 0x80 (chains) and gradient-kernel bit 8: a product was still running when
    // its kernel gave up and released the tensor memory
    const char* grad = !b ? "ok" : ((b >> 8) & 1) ? "timed out, a product still in flight at exit" : "timed out";
    return fail(GDN_ERR_TIMEOUT,
                "a kernel's bounded wait gave up; that call's outputs are invalid (chains: %s, "
                "wait sites 0x%x; gradient kernel: %s)",
                a ? kernels[ker < 5 ? ker : 0] : "ok", (unsigned)a >> 8, grad);
}

gdn_status_t gdn_selftest_wait_timeout(void* stream)
{
    return cuda_status(gdn::launch_selftest_wait(stream), "selftest launch");
}

const char* gdn_status_str(gdn_status_t s)
{
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    }
    return "unknown gdn status";
}

const char* gdn_last_error(void) { return g_last_error.c_str(); }

void gdn_set_timing_events(void* const* events, int n_events)
{
    g_events = events;
    g_n_events = events ? n_events : 0;
}

}  // extern "C"

namespace {

// Widens one 16-bit input [N][T][H][D] (element strides s, last dim contiguous) into its
// dense fp32 copy.
gdn_status_t widen_one(const gdn_params_t* p, const void* src, const int64_t s[3], int64_t N, int64_t H, int64_t D,
                       float* dst, void* stream)
{
    const long long ss[3] = {(long long)s[0], (long long)s[1], (long long)s[2]};
    return cuda_status(gdn::launch_widen(src, p->in_dtype, ss, (int)N, (int)p->T, (int)H, (int)D, dst, stream),
                       "widening launch");
}

// The caller's 16-bit inputs against the buffers the call writes: no overlap.
gdn_status_t check_16bit_inputs(const gdn_params_t* p, const void* const* in, int n_in, const Range* out, int n_out)
{
    const int64_t N = p->n_seq, T = p->T, Hk = p->H_k, Hv = p->H_v, Sk = p->S_k, Sv = p->S_v;
    const int64_t gw = p->gate == GDN_GATE_KDA ? Sk : 1;
    for (int i = 0; i < n_in; ++i)
        if (!aligned(in[i], 2)) return fail(GDN_ERR_INVALID_ARG, "16-bit input not 2-byte aligned");
    const Range r[6] = {extent4(in[0], qk_seqs(p), T, Hk, Sk, p->q_s, 2), extent4(in[1], qk_seqs(p), T, Hk, Sk, p->k_s, 2),
                        extent4(in[2], N, T, Hv, Sv, p->v_s, 2), extent_dense(in[3], (size_t)(N * T * Hv * gw), 2),
                        extent_dense(in[4], (size_t)(N * T * Hv), 2),
                        n_in > 5 ? extent4(in[5], N, T, Hv, Sv, p->gy_s, 2) : Range{0, 0}};
    for (int i = 0; i < n_in; ++i)
        for (int j = 0; j < n_out; ++j)
            if (overlap(r[i], out[j])) return fail(GDN_ERR_ALIAS, "an output or the workspace overlaps an input");
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status_t gdn_forward(const gdn_params_t* p, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* state0, float* y,
                         float* state_T, float* ckpt, void* workspace, size_t workspace_bytes,
                         void* stream)
{
    gdn_status_t st = check_sizes(p);
    if (st != GDN_OK) return st;
    g_last_error.clear();
    if (p->in_dtype != GDN_F32 && p->n_seq > 0) {
        // 16-bit inputs: widen them into the workspace, then run the fp32 path on the copies
        const int64_t N = p->n_seq, T = p->T, Hv = p->H_v, Sk = p->S_k, Sv = p->S_v;
        if (T > 0 && (!q || !k || !v || !g || !beta))
            return fail(GDN_ERR_INVALID_ARG, "q, k, v, g and beta must be non-NULL");
        const Wide w = wide_layout(p, false);
        const gdn_params_t p32 = dense_f32(p);
        const size_t need = w.total + gdn_forward_workspace_bytes(&p32);
        if (workspace_bytes < need)
            return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
        if (!workspace || !aligned(workspace, 256))
            return fail(GDN_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
        const void* in[5] = {q, k, v, g, beta};
        const Range out[4] = {extent_dense(y, (size_t)(N * T * Hv * Sv)), extent_dense(state_T, (size_t)(N * Hv * Sv * Sk)),
                              extent_dense(ckpt, gdn_ckpt_elems(p)), {(uintptr_t)workspace, (uintptr_t)workspace + need}};
        st = check_16bit_inputs(p, in, 5, out, 4);
        if (st != GDN_OK) return st;
        char* ws = (char*)workspace;
        float *wq = (float*)(ws + w.q), *wk = (float*)(ws + w.k), *wv = (float*)(ws + w.v);
        float *wg = (float*)(ws + w.g), *wb = (float*)(ws + w.b);
        if (T > 0) {
            const int64_t gs[3] = {T * Hv * (p->gate == GDN_GATE_KDA ? Sk : 1), Hv * (p->gate == GDN_GATE_KDA ? Sk : 1),
                                   p->gate == GDN_GATE_KDA ? Sk : 1};
            const int64_t bs[3] = {T * Hv, Hv, 1};
            if ((st = widen_one(p, q, p->q_s, qk_seqs(p), p->H_k, Sk, wq, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, k, p->k_s, qk_seqs(p), p->H_k, Sk, wk, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, v, p->v_s, p->n_seq, Hv, Sv, wv, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, g, gs, p->n_seq, Hv, gs[2], wg, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, beta, bs, p->n_seq, Hv, 1, wb, stream)) != GDN_OK) return st;
        }
        return gdn_forward(&p32, wq, wk, wv, wg, wb, state0, y, state_T, ckpt, ws + w.total, workspace_bytes - w.total,
                           stream);
    }
    const Plan pl = make_plan(p);
    const int64_t N = p->n_seq, T = p->T, Hk = p->H_k, Hv = p->H_v, D = p->S_k, DV = p->S_v;
    if (N == 0) return GDN_OK;
    const bool tok = T > 0;
    if (tok && (!q || !k || !v || !g || !beta))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, g and beta must be non-NULL");
    if (!state0 || !state_T) return fail(GDN_ERR_INVALID_ARG, "state0 and state_T must be non-NULL");
    if (tok && (!y || !ckpt)) return fail(GDN_ERR_INVALID_ARG, "y and ckpt must be non-NULL");
    for (const void* ptr : {(const void*)q, (const void*)k, (const void*)v, (const void*)g,
                            (const void*)beta, (const void*)y})
        if (!aligned(ptr, 4)) return fail(GDN_ERR_INVALID_ARG, "pointer not 4-byte aligned");
    if (!aligned(state0, 16) || !aligned(state_T, 16) || !aligned(ckpt, 16))
        return fail(GDN_ERR_INVALID_ARG, "state0, state_T and ckpt must be 16-byte aligned");

    const int64_t gw = pl.kda ? D : 1;
    const Range rq = extent4(q, qk_seqs(p), T, Hk, D, p->q_s), rk = extent4(k, qk_seqs(p), T, Hk, D, p->k_s);
    const Range rv = extent4(v, N, T, Hv, DV, p->v_s);
    const Range rg = extent_dense(g, (size_t)(N * T * Hv * gw));
    const Range rb = extent_dense(beta, (size_t)(N * T * Hv));
    const Range rs0 = extent_dense(state0, (size_t)(N * Hv * DV * D));
    const Range ry = extent_dense(y, (size_t)(N * T * Hv * DV));
    const Range rsT = extent_dense(state_T, (size_t)(N * Hv * DV * D));
    const Range rck = extent_dense(ckpt, (size_t)(N * Hv * pl.n_ck * DV * D));
    for (Range out : {ry, rsT, rck})
        for (Range in : {rq, rk, rv, rg, rb, rs0})
            if (overlap(out, in)) return fail(GDN_ERR_ALIAS, "a forward output overlaps an input");
    if (overlap(ry, rsT) || overlap(ry, rck) || overlap(rsT, rck))
        return fail(GDN_ERR_ALIAS, "forward outputs overlap one another");
    const size_t need = pl.chunked ? pl.fwd_ws_bytes : 0;
    if (workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (!workspace || !aligned(workspace, 256)))
        return fail(GDN_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
    const Range rws = {(uintptr_t)workspace, (uintptr_t)workspace + (workspace ? need : 0)};
    for (Range other : {rq, rk, rv, rg, rb, rs0, ry, rsT, rck})
        if (overlap(rws, other)) return fail(GDN_ERR_ALIAS, "workspace overlaps a tensor");

    gdn::EventTap tap{g_events, g_n_events, 0};
    if (pl.chunked) {
        gdn::ChunkArgs c{};
        c.q = (const float*)q; c.k = (const float*)k; c.v = (const float*)v; c.g = (const float*)g;
        c.beta = (const float*)beta; c.state0 = state0;
        c.y = y; c.state_T = state_T; c.ckpt_out = ckpt; c.ws = (float*)workspace;
        fill_chunk_common(c, p, pl);
        c.carry = pl.tensor ? c.ws + pl.o_carry : nullptr;
        c.want_wu = 1;
        c.vec_q = vec_ok(q, p->q_s); c.vec_k = vec_ok(k, p->k_s); c.vec_v = vec_ok(v, p->v_s);
        c.vec_g = aligned(g, 16);
        c.vec_y = aligned(y, 16);
        return cuda_status(gdn::launch_chunk_forward(c, pl.D, stream, tap), "forward launch");
    }

    gdn::FwdArgs a{};
    a.q = (const float*)q; a.k = (const float*)k; a.v = (const float*)v; a.g = (const float*)g;
    a.beta = (const float*)beta; a.state0 = state0;
    a.y = y; a.state_T = state_T; a.ckpt = ckpt;
    a.qs0 = p->q_s[0]; a.qs1 = p->q_s[1]; a.qs2 = p->q_s[2];
    a.ks0 = p->k_s[0]; a.ks1 = p->k_s[1]; a.ks2 = p->k_s[2];
    a.vs0 = p->v_s[0]; a.vs1 = p->v_s[1]; a.vs2 = p->v_s[2];
    a.N = (int)N; a.T = (int)T; a.H_k = (int)Hk; a.H_v = (int)Hv;
    a.C = (int)pl.C; a.n_ck = (int)pl.n_ck; a.scale = p->scale; a.tc = pl.tc;
    a.SK = pl.SK; a.DV = pl.DV; a.rep = pl.rep;
    a.vec_q = vec_ok(q, p->q_s); a.vec_k = vec_ok(k, p->k_s); a.vec_v = vec_ok(v, p->v_s);
    a.vec_g = aligned(g, 16);
    tap.mark(stream);
    st = cuda_status(gdn::launch_forward(a, pl.D, pl.RT, pl.W, pl.kda, stream), "forward launch");
    tap.mark(stream);
    return st;
}

gdn_status_t gdn_backward(const gdn_params_t* p, const void* q, const void* k, const void* v,
                          const void* g, const void* beta, const float* ckpt, const void* gy,
                          const float* dstate_T, float* packed, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    gdn_status_t st = check_sizes(p);
    if (st != GDN_OK) return st;
    g_last_error.clear();
    if (p->in_dtype != GDN_F32 && p->n_seq > 0) {
        // 16-bit inputs: widen them into the workspace, then run the fp32 path on the copies
        const int64_t T = p->T, Hv = p->H_v, Sk = p->S_k, Sv = p->S_v;
        if (T > 0 && (!q || !k || !v || !g || !beta || !gy))
            return fail(GDN_ERR_INVALID_ARG, "q, k, v, g, beta and gy must be non-NULL");
        const Wide w = wide_layout(p, true);
        const gdn_params_t p32 = dense_f32(p);
        const size_t need = w.total + gdn_backward_workspace_bytes(&p32);
        if (workspace_bytes < need)
            return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
        if (!workspace || !aligned(workspace, 256))
            return fail(GDN_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
        const void* in[6] = {q, k, v, g, beta, gy};
        const Range out[2] = {extent_dense(packed, gdn_packed_grad_elems(p)),
                              {(uintptr_t)workspace, (uintptr_t)workspace + need}};
        st = check_16bit_inputs(p, in, 6, out, 2);
        if (st != GDN_OK) return st;
        char* ws = (char*)workspace;
        float *wq = (float*)(ws + w.q), *wk = (float*)(ws + w.k), *wv = (float*)(ws + w.v);
        float *wg = (float*)(ws + w.g), *wb = (float*)(ws + w.b), *wgy = (float*)(ws + w.gy);
        if (T > 0) {
            const int64_t gw = p->gate == GDN_GATE_KDA ? Sk : 1;
            const int64_t gs[3] = {T * Hv * gw, Hv * gw, gw};
            const int64_t bs[3] = {T * Hv, Hv, 1};
            if ((st = widen_one(p, q, p->q_s, qk_seqs(p), p->H_k, Sk, wq, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, k, p->k_s, qk_seqs(p), p->H_k, Sk, wk, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, v, p->v_s, p->n_seq, Hv, Sv, wv, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, g, gs, p->n_seq, Hv, gw, wg, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, beta, bs, p->n_seq, Hv, 1, wb, stream)) != GDN_OK) return st;
            if ((st = widen_one(p, gy, p->gy_s, p->n_seq, Hv, Sv, wgy, stream)) != GDN_OK) return st;
        }
        return gdn_backward(&p32, wq, wk, wv, wg, wb, ckpt, wgy, dstate_T, packed, ws + w.total,
                            workspace_bytes - w.total, stream);
    }
    const Plan pl = make_plan(p);
    const int64_t N = p->n_seq, T = p->T, Hk = p->H_k, Hv = p->H_v, D = p->S_k, DV = p->S_v;
    if (N == 0) return GDN_OK;
    const bool tok = T > 0;
    if (tok && (!q || !k || !v || !g || !beta || !ckpt || !gy))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, g, beta, ckpt and gy must be non-NULL");
    if (!packed) return fail(GDN_ERR_INVALID_ARG, "packed_grads must be non-NULL");
    for (const void* ptr : {(const void*)q, (const void*)k, (const void*)v, (const void*)g,
                            (const void*)beta, (const void*)gy})
        if (!aligned(ptr, 4)) return fail(GDN_ERR_INVALID_ARG, "pointer not 4-byte aligned");
    if (!aligned(ckpt, 16) || !aligned(dstate_T, 16) || !aligned(packed, 16))
        return fail(GDN_ERR_INVALID_ARG, "ckpt, dstate_T and packed_grads must be 16-byte aligned");
    if (workspace_bytes < pl.ws_bytes)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    pl.ws_bytes);
    if (pl.ws_bytes > 0 && (!workspace || !aligned(workspace, 256)))
        return fail(GDN_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");

    size_t off[7];
    packed_offsets(p, off);
    const int64_t gw = pl.kda ? D : 1;
    const Range rq = extent4(q, qk_seqs(p), T, Hk, D, p->q_s), rk = extent4(k, qk_seqs(p), T, Hk, D, p->k_s);
    const Range rv = extent4(v, N, T, Hv, DV, p->v_s), rgy = extent4(gy, N, T, Hv, DV, p->gy_s);
    const Range rg = extent_dense(g, (size_t)(N * T * Hv * gw));
    const Range rb = extent_dense(beta, (size_t)(N * T * Hv));
    const Range rck = extent_dense(ckpt, (size_t)(N * Hv * pl.n_ck * DV * D));
    const Range rdsT = extent_dense(dstate_T, (size_t)(N * Hv * DV * D));
    const Range rpk = extent_dense(packed, off[6]);
    const Range rws = {(uintptr_t)workspace, (uintptr_t)workspace + (workspace ? pl.ws_bytes : 0)};
    for (Range out : {rpk, rws})
        for (Range in : {rq, rk, rv, rgy, rg, rb, rck, rdsT})
            if (overlap(out, in)) return fail(GDN_ERR_ALIAS, "a backward output overlaps an input");
    if (overlap(rpk, rws)) return fail(GDN_ERR_ALIAS, "workspace overlaps packed_grads");

    gdn::EventTap tap{g_events, g_n_events, 0};
    if (pl.chunked) {
        gdn::ChunkArgs c{};
        c.q = (const float*)q; c.k = (const float*)k; c.v = (const float*)v; c.g = (const float*)g;
        c.beta = (const float*)beta; c.ckpt = ckpt; c.gy = (const float*)gy;
        c.dstate_T = dstate_T; c.ws = (float*)workspace;
        c.dq = packed + off[0]; c.dk = packed + off[1]; c.dv = packed + off[2];
        c.dg = packed + off[3]; c.dbeta = packed + off[4]; c.dstate0 = packed + off[5];
        fill_chunk_common(c, p, pl);
        c.carry = pl.tensor ? c.ws + pl.o_carry_b : nullptr;
        c.want_wu = pl.cps > 1 && !pl.tensor;  // the tensor-core gradient parks the states itself
        c.want_factors = 1;
        c.vec_q = vec_ok(q, p->q_s); c.vec_k = vec_ok(k, p->k_s); c.vec_v = vec_ok(v, p->v_s);
        c.vec_gy = vec_ok(gy, p->gy_s);
        c.vec_g = aligned(g, 16);
        c.vec_ds0 = aligned(c.dstate0, 16);
        return cuda_status(gdn::launch_chunk_backward(c, pl.D, stream, tap), "backward launch");
    }

    char* ws = (char*)workspace;
    gdn::BwdArgs a{};
    a.q = (const float*)q; a.k = (const float*)k; a.v = (const float*)v; a.g = (const float*)g;
    a.beta = (const float*)beta; a.ckpt = ckpt; a.gy = (const float*)gy;
    a.dstate_T = dstate_T;
    a.dv = packed + off[2];
    a.dstate0 = packed + off[5];
    a.sub = (float*)(ws + pl.off_sub);
    a.ws_col = (float*)(ws + pl.off_col);
    a.ws_sc = (float*)(ws + pl.off_sc);
    a.qs0 = p->q_s[0]; a.qs1 = p->q_s[1]; a.qs2 = p->q_s[2];
    a.ks0 = p->k_s[0]; a.ks1 = p->k_s[1]; a.ks2 = p->k_s[2];
    a.vs0 = p->v_s[0]; a.vs1 = p->v_s[1]; a.vs2 = p->v_s[2];
    a.gys0 = p->gy_s[0]; a.gys1 = p->gy_s[1]; a.gys2 = p->gy_s[2];
    a.N = (int)N; a.T = (int)T; a.H_k = (int)Hk; a.H_v = (int)Hv;
    a.C = (int)pl.C; a.n_ck = (int)pl.n_ck; a.c2 = pl.c2; a.nsub_max = pl.nsub_max;
    a.SK = pl.SK; a.DV = pl.DV; a.rep = pl.rep;
    a.scale = p->scale;
    a.vec_q = vec_ok(q, p->q_s); a.vec_k = vec_ok(k, p->k_s); a.vec_v = vec_ok(v, p->v_s);
    a.vec_gy = vec_ok(gy, p->gy_s); a.vec_g = aligned(g, 16);
    a.vec_ds0 = aligned(packed + off[5], 16);
    tap.mark(stream);
    st = cuda_status(gdn::launch_backward(a, pl.D, pl.RT, pl.W, pl.kda, stream), "backward launch");
    tap.mark(stream);
    if (st != GDN_OK || !tok) return st;

    gdn::ReduceArgs r{};
    r.ws_col = a.ws_col; r.ws_sc = a.ws_sc;
    r.dq = packed + off[0]; r.dk = packed + off[1]; r.dg = packed + off[3]; r.dbeta = packed + off[4];
    r.N = (int)N; r.T = (int)T; r.H_k = (int)Hk; r.H_v = (int)Hv; r.D = pl.D; r.P = pl.P;
    r.SK = pl.SK;
    r.rep = pl.rep;
    r.NQ = pl.kda ? 3 : 2; r.kda = pl.kda;
    st = cuda_status(gdn::launch_reduce(r, stream), "reduce launch");
    tap.mark(stream);
    return st;
}

}  // extern "C"
