/* ssm_oracle.c -- float64 CPU oracle of the selective scan and its reverse walk.
 *
 * TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU legs load it;
 * the product library never does.
 *
 * Source: "dillon-blake llama.cpp PR #26", the SSM_SCAN_BACK section: the selective scan's
 * gradient is a reverse recurrence that walks the tokens from the last to the first while
 * carrying the state gradient; it returns five gradients (d_s, d_x, d_dt, d_B, d_C) packed
 * the way the forward packs y with the final states; Mamba-2 has one scalar decay per head and
 * Mamba-1 one per state; the decay is exponential in dt * A; the cotangent of the final states
 * is part of the incoming gradient and seeds the walk; the walk needs s_{t-1} for d(dt)
 * through the decay, so the states are recomputed (all of them, or from checkpoints, which
 * must give the same bits); heads fold into their group's dB, dC slab with g = h / (nh / ng).
 *
 * Readings where the section leaves a step open (the plainest one the rest supports):
 *   - per token t, head h, channel p (0 <= p < P) and state index j (0 <= j < S), with
 *     g = h / (H / G):
 *         a_t[j]     = exp(dt[t][h] * A[h][j])          (Mamba-2: A[h] for every j)
 *         s_t[p][j]  = a_t[j] s_{t-1}[p][j] + B[t][g][j] x[t][h][p] dt[t][h]
 *         y[t][h][p] = sum_j s_t[p][j] C[t][g][j]
 *     dt enters as given (no softplus inside the scan), there is no skip term D x, and A is not
 *     among the gradients (the section lists five);
 *   - the walk, t = T-1 .. 0, with ds seeded by the final-state cotangent:
 *         ds          += dy_t C_t^T                     (ds = dL/ds_t)
 *         dC[t][g][j] += sum_{h in g, p} dy[t][h][p] s_t[p][j]
 *         dx[t][h][p]  = sum_j ds[p][j] B[t][g][j] dt[t][h]
 *         dB[t][g][j] += sum_{h in g, p} ds[p][j] x[t][h][p] dt[t][h]
 *         ddt[t][h]    = sum_{p, j} ds[p][j] (B[t][g][j] x[t][h][p] + A[h][j] a_t[j] s_{t-1}[p][j])
 *         ds           = a_t (.) ds                     (now dL/ds_{t-1})
 *     and d_s = ds after token 0.
 *
 * Layouts (row-major, float64): s0, sT, ds0 [N][H][P][S]; x, y, dy, dx [N][T][H][P];
 * dt, ddt [N][T][H]; A [H] (a_per_state = 0) or [H][S]; B, C, dB, dC [N][T][G][S];
 * checkpoints [N][H][n_ck][P][S], checkpoint k holding the state entering token k * K.
 *
 * Planted defects for the kill-list tests (SSM_ORACLE_MUTATION, compiled in on request):
 *   1 the walk starts from a zero state gradient (the final-state cotangent ignored)
 *   2 d(dt) without the decay path
 *   3 the decay path reads s_t where it needs s_{t-1} (a state one token late)
 *   4 dC from s_{t-1} instead of s_t
 *   5 heads routed to groups by h % G
 *   6 dx without its dt factor
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef SSM_ORACLE_MUTATION
#define SSM_ORACLE_MUTATION 0
#endif

typedef struct {
    int64_t N, T, H, P, S, G;
    int64_t a_per_state; /* 1: A is [H][S] (Mamba-1); 0: A is [H] (Mamba-2) */
    int64_t K;           /* checkpoint interval in tokens (>= 1) */
} ssm_dims;

int ssm_oracle_mutation(void) { return SSM_ORACLE_MUTATION; }

int64_t ssm_oracle_num_checkpoints(int64_t T, int64_t K) { return T <= 0 ? 1 : (T + K - 1) / K; }

static int64_t group_of(const ssm_dims* d, int64_t h)
{
#if SSM_ORACLE_MUTATION == 5
    return h % d->G;
#else
    return h / (d->H / d->G);
#endif
}

static double a_coef(const ssm_dims* d, const double* A, int64_t h, int64_t j) { return d->a_per_state ? A[h * d->S + j] : A[h]; }

static int check(const ssm_dims* d)
{
    if (d->N < 0 || d->T < 0 || d->H < 1 || d->P < 1 || d->S < 1 || d->G < 1 || d->K < 1) return 1;
    if (d->H % d->G) return 1;
    return 0;
}

/* One token of the scan for one (sequence, head): st[P][S] <- a st + B x dt. */
static void step(const ssm_dims* d, const double* A, int64_t h, double dtv, const double* xrow, const double* Brow,
                 double* st)
{
    const int64_t P = d->P, S = d->S;
    for (int64_t p = 0; p < P; ++p)
        for (int64_t j = 0; j < S; ++j) {
            const double a = exp(dtv * a_coef(d, A, h, j));
            st[p * S + j] = a * st[p * S + j] + Brow[j] * xrow[p] * dtv;
        }
}

static void forward_unit(const ssm_dims* d, int64_t n, int64_t h, double* st, const double* s0, const double* x,
                         const double* dt, const double* A, const double* B, const double* C, double* y, double* sT,
                         double* ckpt)
{
    const int64_t T = d->T, H = d->H, P = d->P, S = d->S, G = d->G, K = d->K;
    const int64_t nck = ssm_oracle_num_checkpoints(T, K);
    const int64_t g = group_of(d, h);
    memcpy(st, s0 + (n * H + h) * P * S, sizeof(double) * P * S);
    for (int64_t t = 0; t < T; ++t) {
        if (ckpt && t % K == 0) memcpy(ckpt + ((n * H + h) * nck + t / K) * P * S, st, sizeof(double) * P * S);
        const double dtv = dt[(n * T + t) * H + h];
        step(d, A, h, dtv, x + ((n * T + t) * H + h) * P, B + ((n * T + t) * G + g) * S, st);
        const double* Crow = C + ((n * T + t) * G + g) * S;
        for (int64_t p = 0; p < P; ++p) {
            double acc = 0.0;
            for (int64_t j = 0; j < S; ++j) acc += st[p * S + j] * Crow[j];
            y[((n * T + t) * H + h) * P + p] = acc;
        }
    }
    if (ckpt && T == 0) memcpy(ckpt + (n * H + h) * nck * P * S, st, sizeof(double) * P * S);
    memcpy(sT + (n * H + h) * P * S, st, sizeof(double) * P * S);
}

int ssm_oracle_forward(const ssm_dims* d, const double* s0, const double* x, const double* dt, const double* A,
                       const double* B, const double* C, double* y, double* sT, double* ckpt)
{
    if (check(d)) return 1;
    const int64_t N = d->N, H = d->H, PS = d->P * d->S;
    int err = 0;
#pragma omp parallel
    {
        double* st = malloc(sizeof(double) * PS);
        if (!st) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for collapse(2) schedule(static)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t h = 0; h < H; ++h)
                if (st) forward_unit(d, n, h, st, s0, x, dt, A, B, C, y, sT, ckpt);
        free(st);
    }
    return err;
}

/* The walk of one (sequence, head); states holds span + 1 states, ds P x S. */
static void backward_unit(const ssm_dims* d, int store_all, int64_t n, int64_t h, double* states, double* ds,
                          const double* s0, const double* x, const double* dt, const double* A, const double* B,
                          const double* C, const double* ckpt, const double* dy, const double* dsT, double* ds0,
                          double* dx, double* ddt, double* dB, double* dC)
{
    const int64_t T = d->T, H = d->H, P = d->P, S = d->S, G = d->G, K = d->K;
    const int64_t nck = ssm_oracle_num_checkpoints(T, K);
    const int64_t PS = P * S;
    const int64_t g = group_of(d, h);
#if SSM_ORACLE_MUTATION == 1
    (void)dsT;
    memset(ds, 0, sizeof(double) * PS);
#else
    memcpy(ds, dsT + (n * H + h) * PS, sizeof(double) * PS);
#endif
    /* segments [t0, t1), last first; store-all: one segment of every token */
    const int64_t nseg = store_all ? 1 : nck;
    for (int64_t sgi = nseg - 1; sgi >= 0; --sgi) {
        const int64_t t0 = store_all ? 0 : sgi * K;
        const int64_t t1 = store_all ? T : (t0 + K < T ? t0 + K : T);
        if (store_all)
            memcpy(states, s0 + (n * H + h) * PS, sizeof(double) * PS);
        else
            memcpy(states, ckpt + ((n * H + h) * nck + sgi) * PS, sizeof(double) * PS);
        for (int64_t t = t0; t < t1; ++t) {  /* states[t - t0 + 1]: the state after token t */
            memcpy(states + (t - t0 + 1) * PS, states + (t - t0) * PS, sizeof(double) * PS);
            step(d, A, h, dt[(n * T + t) * H + h], x + ((n * T + t) * H + h) * P, B + ((n * T + t) * G + g) * S,
                 states + (t - t0 + 1) * PS);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const double* s_prev = states + (t - t0) * PS;     /* state entering token t */
            const double* s_cur = states + (t - t0 + 1) * PS;  /* state after token t */
            (void)s_prev;  /* (each is unused in one planted defect) */
            (void)s_cur;
            const double dtv = dt[(n * T + t) * H + h];
            const double* xr = x + ((n * T + t) * H + h) * P;
            const double* Br = B + ((n * T + t) * G + g) * S;
            const double* Cr = C + ((n * T + t) * G + g) * S;
            const double* dyr = dy + ((n * T + t) * H + h) * P;
            double* dBr = dB + ((n * T + t) * G + g) * S;
            double* dCr = dC + ((n * T + t) * G + g) * S;
            /* the output term y = s_t C */
            for (int64_t p = 0; p < P; ++p)
                for (int64_t j = 0; j < S; ++j) {
                    ds[p * S + j] += dyr[p] * Cr[j];
#if SSM_ORACLE_MUTATION == 4
                    dCr[j] += dyr[p] * s_prev[p * S + j];
#else
                    dCr[j] += dyr[p] * s_cur[p * S + j];
#endif
                }
            /* the write term B x dt */
            double gdt = 0.0;
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t j = 0; j < S; ++j) {
                    acc += ds[p * S + j] * Br[j];
                    dBr[j] += ds[p * S + j] * xr[p] * dtv;
                    gdt += ds[p * S + j] * Br[j] * xr[p];
                }
#if SSM_ORACLE_MUTATION == 6
                dx[((n * T + t) * H + h) * P + p] = acc;
#else
                dx[((n * T + t) * H + h) * P + p] = acc * dtv;
#endif
            }
            /* the decay a = exp(dt A): d a / d dt = A a, against s_{t-1} */
            for (int64_t p = 0; p < P; ++p)
                for (int64_t j = 0; j < S; ++j) {
                    const double Av = a_coef(d, A, h, j);
                    const double a = exp(dtv * Av);
#if SSM_ORACLE_MUTATION == 2
                    (void)a;
#elif SSM_ORACLE_MUTATION == 3
                    gdt += ds[p * S + j] * Av * a * s_cur[p * S + j];
#else
                    gdt += ds[p * S + j] * Av * a * s_prev[p * S + j];
#endif
                }
            ddt[(n * T + t) * H + h] = gdt;
            /* carry to s_{t-1} */
            for (int64_t p = 0; p < P; ++p)
                for (int64_t j = 0; j < S; ++j) ds[p * S + j] *= exp(dtv * a_coef(d, A, h, j));
        }
    }
    memcpy(ds0 + (n * H + h) * PS, ds, sizeof(double) * PS);
}

/* Reverse walk.  store_all = 1: every state s_0 .. s_T recomputed from s0 and kept;
 * store_all = 0: the states of each checkpoint segment recomputed from its checkpoint
 * (ckpt, as the forward wrote it).  dB and dC are zeroed, then accumulated head by head in
 * ascending h within each group (one thread per (sequence, group), so the sums' order is
 * fixed); the store-all and checkpointed walks therefore give the same bits. */
int ssm_oracle_backward(const ssm_dims* d, int store_all, const double* s0, const double* x, const double* dt,
                        const double* A, const double* B, const double* C, const double* ckpt, const double* dy,
                        const double* dsT, double* ds0, double* dx, double* ddt, double* dB, double* dC)
{
    if (check(d)) return 1;
    if (!store_all && !ckpt) return 1;
    if (store_all && !s0) return 1;
    const int64_t N = d->N, T = d->T, H = d->H, G = d->G, K = d->K;
    const int64_t PS = d->P * d->S;
    const int64_t span = store_all ? T : K;
    memset(dB, 0, sizeof(double) * N * T * G * d->S);
    memset(dC, 0, sizeof(double) * N * T * G * d->S);
    int err = 0;
#pragma omp parallel
    {
        double* states = malloc(sizeof(double) * (span + 1) * PS);
        double* ds = malloc(sizeof(double) * PS);
        if (!states || !ds) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for collapse(2) schedule(static)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t g = 0; g < G; ++g)
                for (int64_t h = 0; h < H; ++h)
                    if (states && ds && group_of(d, h) == g)
                        backward_unit(d, store_all, n, h, states, ds, s0, x, dt, A, B, C, ckpt, dy, dsT, ds0, dx,
                                      ddt, dB, dC);
        free(states);
        free(ds);
    }
    return err;
}

int ssm_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ssm_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
