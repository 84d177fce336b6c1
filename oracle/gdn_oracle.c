/*
 * gdn_oracle.c -- plain float64 CPU oracle of the gated delta rule (Gated DeltaNet
 * with a scalar gate, Kimi Delta Attention with a per-key-column gate): forward and
 * backward.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU-baseline
 * leg call it; the product path (the CUDA library) never does.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it follows:
 *   - Forward, row form: "metal: GATED_DELTA_NET_BACK" (llama.cpp fork PR #16), review
 *     comment "APPROVED at 739b9bf": thread j owns row j of M = S^T;
 *     u_j = sum_i M[j][i] a_i k_i, M[j][i] <- a_i M[j][i] + k_i delta_j.
 *   - Forward, matrix form: meTile "Training kernels and gradients", section
 *     "Recurrent delta attention": decayed = exp(log_decay) * previous,
 *     error = value - decayed^T key, state = decayed + beta * outer(key, error),
 *     output = scale * state^T query.
 *   - Backward: PR #16 review comments ("Math, read term by term against the CPU
 *     reference" and "APPROVED at 739b9bf"): the output term, dd/dv/du/dbeta, the key
 *     term with dM read before the du update, dM += k du^T, dg = sum dS'.*S' (per
 *     column for KDA, summed for the scalar gate), dS_prev = a .* dS'.
 *   - Checkpointed recompute with C ~ sqrt(T): PR #16 body; store-all as the honest
 *     starting point that checkpointing must match bit-for-bit: llama.cpp PR #26
 *     (SSM_SCAN_BACK section).
 *
 * Readings taken where the pages leave a step open:
 *   - S' is the decayed previous state a (.) M_{t-1} (the matrix u is computed from);
 *     it is the S' of the dk and dg terms.
 *   - The q/k head of value head h_v is h_v mod H_k (PR #16: "iv1 % neq1"), and the q/k
 *     sequence of value sequence n is n / rep when q, k hold N / rep sequences (PR #16:
 *     "iv3/rq3"); dq/dk then sum over the rep value sequences that share one.
 *   - g and beta are per value head; the KDA gate indexes the key column i.
 *   - ckpt[c] is the state entering token c*C, c = 0..ceil(T/C)-1; the last segment
 *     may be partial.
 *   - y = scale * M_t q (scale on the output), so dq carries scale and the output
 *     term adds scale * gy_j q_i to dM.
 *   - The only cotangents are gy (per token output) and dstate_T (final state).
 *
 * Layouts (contiguous float64; M = S^T has S_v rows j and S_k columns i; N_q = N / rep):
 *   q, k    [N_q][T][H_k][S_k]      v, y     [N][T][H_v][S_v]
 *   g       [N][T][H_v]  (scalar)  or [N][T][H_v][S_k] (KDA)
 *   beta    [N][T][H_v]             state    [N][H_v][S_v][S_k]
 *   ckpt    [N][H_v][n_ck][S_v][S_k]
 *   dq, dk  as q, k;  dv as v;  dg as g;  dbeta as beta;  dstate0 as state
 *
 * Mutations: building with -DGDN_ORACLE_MUTATION=m (m = 1..7) plants one known defect.
 * Only the tests build such copies, to prove that the pins catch each defect.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef GDN_ORACLE_MUTATION
#define GDN_ORACLE_MUTATION 0
#endif

typedef struct {
    int64_t N, T, H_k, H_v, S_k, S_v;
    int64_t kda; /* 0: scalar gate g[N][T][H_v]; 1: per-key-column gate g[N][T][H_v][S_k] */
    int64_t C;   /* checkpoint interval, >= 1 */
    double scale;
    int64_t rep; /* value sequences per q/k sequence (>= 1); q, k hold N / rep sequences */
} gdn_oracle_dims;

int64_t gdn_oracle_num_checkpoints(int64_t T, int64_t C)
{
    if (T <= 0 || C <= 0) return 0;
    return (T + C - 1) / C;
}

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Host-side thread count of the OpenMP loops over (sequence, value head); n < 1 leaves it
 * unchanged.  Lets a timing run use all host cores or one.  No arithmetic depends on it:
 * every unit is computed by one thread in the same order whatever the count. */
void gdn_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int gdn_oracle_mutation(void) { return GDN_ORACLE_MUTATION; }

/* The key head that serves value head hv. */
static int64_t key_head(const gdn_oracle_dims* d, int64_t hv)
{
#if GDN_ORACLE_MUTATION == 5
    return hv / (d->H_v / d->H_k); /* planted defect: contiguous grouping */
#else
    return hv % d->H_k;
#endif
}

/* The q/k sequence that serves value sequence n. */
static int64_t key_seq(const gdn_oracle_dims* d, int64_t n)
{
#if GDN_ORACLE_MUTATION == 7
    return n % (d->N / d->rep); /* planted defect: interleaved grouping */
#else
    return n / d->rep;
#endif
}

/* Per-token inputs of one (sequence, value head) unit, gathered as plain vectors. */
typedef struct {
    const double* q;  /* [S_k] */
    const double* k;  /* [S_k] */
    const double* v;  /* [S_v] */
    double beta;
    double* a;        /* [S_k], a_i = exp(g_i) (all equal for the scalar gate) */
} token_in;

static void gather_token(const gdn_oracle_dims* d, const double* q, const double* k,
                         const double* v, const double* g, const double* beta, int64_t n,
                         int64_t t, int64_t hv, token_in* tk)
{
    const int64_t hk = key_head(d, hv), nq = key_seq(d, n);
    const int64_t S_k = d->S_k, S_v = d->S_v;
    tk->q = q + ((nq * d->T + t) * d->H_k + hk) * S_k;
    tk->k = k + ((nq * d->T + t) * d->H_k + hk) * S_k;
    tk->v = v + ((n * d->T + t) * d->H_v + hv) * S_v;
    tk->beta = beta[(n * d->T + t) * d->H_v + hv];
    if (d->kda) {
        const double* gt = g + ((n * d->T + t) * d->H_v + hv) * S_k;
        for (int64_t i = 0; i < S_k; ++i) tk->a[i] = exp(gt[i]);
    } else {
        const double a = exp(g[(n * d->T + t) * d->H_v + hv]);
        for (int64_t i = 0; i < S_k; ++i) tk->a[i] = a;
    }
}

/* One forward step (meTile "Recurrent delta attention", decay before correction):
 *   Sp = a (.) M           (Sp[j][i] = a_i M[j][i], the decayed state S')
 *   u_j = sum_i Sp[j][i] k_i,  delta_j = beta (v_j - u_j)
 *   M[j][i] = Sp[j][i] + k_i delta_j
 * M is updated in place.  u and delta (length S_v) are returned when non-NULL. */
static void forward_step(const gdn_oracle_dims* d, const token_in* tk, double* M,
                         double* u, double* delta)
{
    const int64_t S_k = d->S_k, S_v = d->S_v;
    for (int64_t j = 0; j < S_v; ++j) {
        double* row = M + j * S_k;
        for (int64_t i = 0; i < S_k; ++i) row[i] = tk->a[i] * row[i];
        double uj = 0.0;
        for (int64_t i = 0; i < S_k; ++i) uj += row[i] * tk->k[i];
        const double dj = tk->beta * (tk->v[j] - uj);
        for (int64_t i = 0; i < S_k; ++i) row[i] = row[i] + tk->k[i] * dj;
        if (u) u[j] = uj;
        if (delta) delta[j] = dj;
    }
}

/* y_j = scale * sum_i M[j][i] q_i, with M the state after the token. */
static void readout(const gdn_oracle_dims* d, const token_in* tk, const double* M, double* y)
{
    const int64_t S_k = d->S_k, S_v = d->S_v;
    for (int64_t j = 0; j < S_v; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < S_k; ++i) acc += M[j * S_k + i] * tk->q[i];
        y[j] = d->scale * acc;
    }
}

/* ------------------------------------------------------------------------------ */
/* Forward                                                                          */
/* ------------------------------------------------------------------------------ */

static void forward_unit(const gdn_oracle_dims* d, int64_t n, int64_t hv, const double* q,
                         const double* k, const double* v, const double* g,
                         const double* beta, const double* state0, double* y,
                         double* state_T, double* ckpt)
{
    const int64_t S_k = d->S_k, S_v = d->S_v, SS = S_k * S_v;
    const int64_t n_ck = gdn_oracle_num_checkpoints(d->T, d->C);
    double* M = (double*)malloc(sizeof(double) * (size_t)SS);
    double* a = (double*)malloc(sizeof(double) * (size_t)S_k);
    token_in tk;
    tk.a = a;
    memcpy(M, state0 + (n * d->H_v + hv) * SS, sizeof(double) * (size_t)SS);
    for (int64_t t = 0; t < d->T; ++t) {
        if (ckpt && t % d->C == 0)
            memcpy(ckpt + ((n * d->H_v + hv) * n_ck + t / d->C) * SS, M,
                   sizeof(double) * (size_t)SS);
        gather_token(d, q, k, v, g, beta, n, t, hv, &tk);
        forward_step(d, &tk, M, NULL, NULL);
        if (y) readout(d, &tk, M, y + ((n * d->T + t) * d->H_v + hv) * S_v);
    }
    if (state_T) memcpy(state_T + (n * d->H_v + hv) * SS, M, sizeof(double) * (size_t)SS);
    free(a);
    free(M);
}

/* y, state_T and ckpt may each be NULL.  Returns 0 on success. */
int gdn_oracle_forward(const gdn_oracle_dims* d, const double* q, const double* k,
                       const double* v, const double* g, const double* beta,
                       const double* state0, double* y, double* state_T, double* ckpt)
{
    if (!d || d->H_k <= 0 || d->H_v % d->H_k != 0 || d->C <= 0 || d->T < 0 || d->N < 0 ||
        d->rep < 1 || d->N % d->rep != 0)
        return 1;
    const int64_t units = d->N * d->H_v;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t uidx = 0; uidx < units; ++uidx)
        forward_unit(d, uidx / d->H_v, uidx % d->H_v, q, k, v, g, beta, state0, y, state_T,
                     ckpt);
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* Backward                                                                         */
/* ------------------------------------------------------------------------------ */

/* Reverse step for token t.  Mprev = M_{t-1}, Mcur = M_t, dM = dL/dM_t on entry and
 * dL/dM_{t-1} on exit.  Writes dq_h/dk_h (this value head's contribution, length
 * S_k), dv (S_v), dg (S_k for KDA, 1 for the scalar gate) and dbeta. */
static void backward_step(const gdn_oracle_dims* d, const token_in* tk, const double* Mprev,
                          const double* Mcur, const double* gy, double* dM, double* Sp,
                          double* u, double* delta, double* dd, double* du, double* dq_h,
                          double* dk_h, double* dv, double* dg, double* dbeta)
{
    const int64_t S_k = d->S_k, S_v = d->S_v;
    const double* a = tk->a;
    const double* kk = tk->k;
    const double beta = tk->beta;

    /* The decayed previous state S' and the token's u, delta (recomputed). */
    for (int64_t j = 0; j < S_v; ++j) {
        double uj = 0.0;
        for (int64_t i = 0; i < S_k; ++i) {
            Sp[j * S_k + i] = a[i] * Mprev[j * S_k + i];
            uj += Sp[j * S_k + i] * kk[i];
        }
        u[j] = uj;
        delta[j] = beta * (tk->v[j] - uj);
    }

    /* Output term: dq_i = scale sum_j M_t[j][i] gy_j; dM[j][i] += scale gy_j q_i. */
    for (int64_t i = 0; i < S_k; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < S_v; ++j) {
#if GDN_ORACLE_MUTATION == 6
            acc += Mcur[j * S_k + i]; /* planted defect: gy ignored */
#else
            acc += Mcur[j * S_k + i] * gy[j];
#endif
        }
#if GDN_ORACLE_MUTATION == 4
        dq_h[i] = acc; /* planted defect: scale dropped from dq */
#else
        dq_h[i] = d->scale * acc;
#endif
    }
    for (int64_t j = 0; j < S_v; ++j) {
#if GDN_ORACLE_MUTATION == 6
        const double sg = d->scale;
#else
        const double sg = d->scale * gy[j];
#endif
        for (int64_t i = 0; i < S_k; ++i) dM[j * S_k + i] += sg * tk->q[i];
    }

    /* Delta terms: dd = dM k; dv = beta dd; du = -beta dd; dbeta = sum_j dd_j (v_j - u_j). */
    double db = 0.0;
    for (int64_t j = 0; j < S_v; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < S_k; ++i) acc += dM[j * S_k + i] * kk[i];
        dd[j] = acc;
        dv[j] = beta * acc;
        du[j] = -beta * acc;
        db += acc * (tk->v[j] - u[j]);
    }
    *dbeta = db;

    /* Key term, with dM read before the du update:
     * dk_i = sum_j dM[j][i] delta_j + sum_j S'[j][i] du_j. */
#if GDN_ORACLE_MUTATION == 3
    for (int64_t j = 0; j < S_v; ++j) /* planted defect: du update applied first */
        for (int64_t i = 0; i < S_k; ++i) dM[j * S_k + i] += kk[i] * du[j];
#endif
    for (int64_t i = 0; i < S_k; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < S_v; ++j) {
#if GDN_ORACLE_MUTATION == 2
            acc += dM[j * S_k + i] * delta[j] + Mprev[j * S_k + i] * du[j]; /* defect */
#else
            acc += dM[j * S_k + i] * delta[j] + Sp[j * S_k + i] * du[j];
#endif
        }
        dk_h[i] = acc;
    }

    /* Outer update: dS' = dM + k du^T. */
#if GDN_ORACLE_MUTATION != 3
    for (int64_t j = 0; j < S_v; ++j)
        for (int64_t i = 0; i < S_k; ++i) dM[j * S_k + i] += kk[i] * du[j];
#endif

    /* Gate: dg = sum dS' (.) S', per key column for KDA, summed for the scalar gate. */
    if (d->kda) {
        for (int64_t i = 0; i < S_k; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < S_v; ++j) acc += dM[j * S_k + i] * Sp[j * S_k + i];
            dg[i] = acc;
        }
    } else {
        double acc = 0.0;
        for (int64_t j = 0; j < S_v; ++j)
            for (int64_t i = 0; i < S_k; ++i) acc += dM[j * S_k + i] * Sp[j * S_k + i];
        dg[0] = acc;
    }

    /* Decay: dS_prev = a (.) dS'. */
    for (int64_t j = 0; j < S_v; ++j)
        for (int64_t i = 0; i < S_k; ++i) dM[j * S_k + i] *= a[i];
}

/* mode 0: store-all (recompute every state from state0 and keep all T+1 of them).
 * mode 1: checkpointed (recompute each segment from ckpt[s], keeping C+1 states). */
static void backward_unit(const gdn_oracle_dims* d, int mode, int64_t n, int64_t hv,
                          const double* q, const double* k, const double* v, const double* g,
                          const double* beta, const double* state0, const double* ckpt,
                          const double* gy, const double* dstate_T, double* dqh, double* dkh,
                          double* dv, double* dg, double* dbeta, double* dstate0)
{
    const int64_t T = d->T, S_k = d->S_k, S_v = d->S_v, SS = S_k * S_v;
    const int64_t C = d->C, n_ck = gdn_oracle_num_checkpoints(T, C);
    const int64_t span = (mode == 0) ? T : C; /* tokens covered by one stored block */
    double* states = (double*)malloc(sizeof(double) * (size_t)(SS * (span + 1)));
    double* dM = (double*)malloc(sizeof(double) * (size_t)SS);
    double* Sp = (double*)malloc(sizeof(double) * (size_t)SS);
    double* a = (double*)malloc(sizeof(double) * (size_t)S_k);
    double* u = (double*)malloc(sizeof(double) * (size_t)S_v);
    double* delta = (double*)malloc(sizeof(double) * (size_t)S_v);
    double* dd = (double*)malloc(sizeof(double) * (size_t)S_v);
    double* du = (double*)malloc(sizeof(double) * (size_t)S_v);
    token_in tk;
    tk.a = a;

    /* Seed: dM(T) = dstate_T (the final-state cotangent), zero when absent. */
#if GDN_ORACLE_MUTATION == 1
    memset(dM, 0, sizeof(double) * (size_t)SS); /* planted defect: seed dropped */
    (void)dstate_T;
#else
    if (dstate_T)
        memcpy(dM, dstate_T + (n * d->H_v + hv) * SS, sizeof(double) * (size_t)SS);
    else
        memset(dM, 0, sizeof(double) * (size_t)SS);
#endif

    const int64_t n_blocks = (mode == 0) ? (T > 0 ? 1 : 0) : n_ck;
    for (int64_t b = n_blocks - 1; b >= 0; --b) {
        const int64_t t0 = (mode == 0) ? 0 : b * C;
        const int64_t t1 = (mode == 0) ? T : (t0 + C < T ? t0 + C : T);
        /* states[s] = M_{t0 + s - 1}, i.e. states[0] = state entering token t0. */
        if (mode == 0)
            memcpy(states, state0 + (n * d->H_v + hv) * SS, sizeof(double) * (size_t)SS);
        else
            memcpy(states, ckpt + ((n * d->H_v + hv) * n_ck + b) * SS,
                   sizeof(double) * (size_t)SS);
        for (int64_t t = t0; t < t1; ++t) {
            gather_token(d, q, k, v, g, beta, n, t, hv, &tk);
            double* next = states + (t - t0 + 1) * SS;
            memcpy(next, states + (t - t0) * SS, sizeof(double) * (size_t)SS);
            forward_step(d, &tk, next, NULL, NULL);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            gather_token(d, q, k, v, g, beta, n, t, hv, &tk);
            const int64_t row = (n * T + t) * d->H_v + hv;
            backward_step(d, &tk, states + (t - t0) * SS, states + (t - t0 + 1) * SS,
                          gy + row * S_v, dM, Sp, u, delta, dd, du, dqh + row * S_k,
                          dkh + row * S_k, dv + row * S_v, dg + (d->kda ? row * S_k : row),
                          dbeta + row);
        }
    }
    memcpy(dstate0 + (n * d->H_v + hv) * SS, dM, sizeof(double) * (size_t)SS);
    free(du);
    free(dd);
    free(delta);
    free(u);
    free(a);
    free(Sp);
    free(dM);
    free(states);
}

/* Backward.  mode 0 needs state0, mode 1 needs ckpt (written by gdn_oracle_forward
 * with the same C).  dstate_T may be NULL (zero cotangent).  dq/dk are the sums over
 * the units that share a key head and a q/k sequence: the rep value sequences in
 * ascending order, and within each the H_v/H_k value heads in ascending h_v order.
 * Returns 0 on success. */
int gdn_oracle_backward(const gdn_oracle_dims* d, int mode, const double* q, const double* k,
                        const double* v, const double* g, const double* beta,
                        const double* state0, const double* ckpt, const double* gy,
                        const double* dstate_T, double* dq, double* dk, double* dv,
                        double* dg, double* dbeta, double* dstate0)
{
    if (!d || d->H_k <= 0 || d->H_v % d->H_k != 0 || d->C <= 0 || d->T < 0 || d->N < 0 ||
        d->rep < 1 || d->N % d->rep != 0)
        return 1;
    if ((mode == 0 && !state0) || (mode == 1 && !ckpt) || (mode != 0 && mode != 1)) return 2;
    const int64_t N = d->N, T = d->T, H_k = d->H_k, H_v = d->H_v, S_k = d->S_k;
    const size_t per_head = (size_t)(N * T * H_v * S_k);
    double* dqh = (double*)calloc(per_head ? per_head : 1, sizeof(double));
    double* dkh = (double*)calloc(per_head ? per_head : 1, sizeof(double));
    const int64_t units = N * H_v;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t uidx = 0; uidx < units; ++uidx)
        backward_unit(d, mode, uidx / H_v, uidx % H_v, q, k, v, g, beta, state0, ckpt, gy,
                      dstate_T, dqh, dkh, dv, dg, dbeta, dstate0);
    /* Fold the units onto their q/k sequence and key head: ascending value sequence, then
     * ascending h_v. */
    for (int64_t nq = 0; nq < N / d->rep; ++nq)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t hk = 0; hk < H_k; ++hk)
                for (int64_t i = 0; i < S_k; ++i) {
                    double sq = 0.0, sk = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        if (key_seq(d, n) != nq) continue;
                        for (int64_t hv = 0; hv < H_v; ++hv) {
                            if (key_head(d, hv) != hk) continue;
                            sq += dqh[((n * T + t) * H_v + hv) * S_k + i];
                            sk += dkh[((n * T + t) * H_v + hv) * S_k + i];
                        }
                    }
                    dq[((nq * T + t) * H_k + hk) * S_k + i] = sq;
                    dk[((nq * T + t) * H_k + hk) * S_k + i] = sk;
                }
    free(dkh);
    free(dqh);
    return 0;
}
