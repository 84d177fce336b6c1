/* ssm.h -- C ABI of the selective scan (Mamba-1 / Mamba-2) forward and its reverse walk
 * (SSM_SCAN_BACK), part of libgdn.
 *
 * Source: "dillon-blake llama.cpp PR #26", the SSM_SCAN_BACK section.  The scan's gradient is
 * a reverse recurrence carrying the state gradient from the last token to the first; it
 * returns five gradients (d_s, d_x, d_dt, d_B, d_C) packed the way the forward packs y with
 * the final states; Mamba-2 has one scalar decay per head, Mamba-1 one per state; the decay
 * is exponential in dt * A; the incoming gradient's state region is not zero and seeds the
 * walk; the walk needs s_{t-1} for d(dt), so states are recomputed from checkpoints; heads
 * fold into their group's B, C slab with g = h / (H / G).
 *
 * What is computed, per sequence n, token t, head h, channel p < P, state j < S, with
 * g = h / (H / G) (dt as given: the caller applies any softplus; no skip term D x):
 *     a_t[j]     = exp(dt[t][h] * A[h][j])            (Mamba-2: A[h] for every j)
 *     s_t[p][j]  = a_t[j] s_{t-1}[p][j] + B[t][g][j] (x[t][h][p] dt[t][h])
 *     y[t][h][p] = sum_j s_t[p][j] C[t][g][j]
 * and, walking t = T-1 .. 0 with ds seeded by the final-state cotangent ds_T:
 *     ds += dy_t C_t^T;  dC[t][g] += sum_{h in g, p} dy[t][h][p] s_t[p];
 *     dx[t][h][p] = dt[t][h] sum_j ds[p][j] B[t][g][j];  dB[t][g] += sum_{h in g, p} ds[p] x[t][h][p] dt[t][h];
 *     ddt[t][h] = sum_{p, j} ds[p][j] (B[t][g][j] x[t][h][p] + A[h][j] a_t[j] s_{t-1}[p][j]);
 *     ds = a_t (.) ds;    and d_s = ds after token 0.
 * Arithmetic: fp32 throughout (FP32 pipe, expf); every sum over channels, heads and states
 * runs in a fixed order (no atomics), so a call's results do not change from run to run.
 *
 * Three forms compute this (ssm_form() says which runs; each regroups the same sums, so
 * results agree within rounding):
 *   - the token-serial walk follows the recurrences above token by token (its results do not
 *     depend on K);
 *   - the chunked form (one decay per head, P = 64, S = 128, K a multiple of 64) groups 64
 *     tokens into a chunk and writes each chunk's part of the recurrence as dense products,
 *     with l_t = dt_t A, the running sum c_t of l over the chunk, Q = C B^T and the mask
 *     exp(c_t - c_tau) for tau <= t; only the state passes from chunk to chunk;
 *   - the segmented form (a decay per state, P = 1, S = 16, H / G a multiple of 16, and
 *     ceil(T / K) * 16 <= T) runs every (channel, state) recurrence by checkpoint segments:
 *     a segment maps its entry state s to G s + dS (G the product of its decays, dS its scan
 *     from zero), and 32-token blocks of the reverse walk map the gradient arriving from the
 *     right, c, to U + G c the same way.
 * The last two forms' results depend on K through the segments.
 *
 * Layouts: dense, row-major, fp32, device memory, no strides:
 *     s0 [N][H][P][S]   x [N][T][H][P]   dt [N][T][H]   A [H] or [H][S]   B, C [N][T][G][S]
 *     checkpoints [N][H][n_ck][P][S]: checkpoint k is the state entering token k * K
 *     forward output, packed:  [ y [N][T][H][P] | s_T [N][H][P][S] ]
 *     backward input, packed:  [ dy [N][T][H][P] | ds_T [N][H][P][S] ]   (the forward's layout)
 *     backward output, packed: [ d_s [N][H][P][S] | d_x [N][T][H][P] | d_dt [N][T][H] |
 *                                d_B [N][T][G][S] | d_C [N][T][G][S] ]
 * Every pointer must be 16-byte aligned.
 *
 * Ownership and streams: the caller owns every buffer and the stream (a cudaStream_t; NULL is
 * the legacy default stream).  Calls only enqueue work; the library keeps no pointer after a
 * call returns and allocates nothing.
 *
 * Errors (gdn.h's codes; text in gdn_last_error()), returned before any work is enqueued:
 *   GDN_ERR_INVALID_ARG  NULL pointer, a size below 1 (T may be 0; N may be 0), H % G != 0,
 *                        K < 0, a misaligned pointer
 *   GDN_ERR_UNSUPPORTED  S not one of 16, 32, 64, 128, 256; the channels of a group not a
 *                        multiple of the rows a block of the walk covers, or P neither a
 *                        multiple nor a divisor of them (ssm_supported() says which)
 *   GDN_ERR_ALIAS        an output overlaps an input
 *   GDN_ERR_WORKSPACE    workspace smaller than ssm_backward_workspace_bytes()
 *   GDN_ERR_CUDA         a launch failed
 */
#ifndef SSM_H
#define SSM_H

#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int64_t N;            /* sequences */
    int64_t T;            /* tokens per sequence (>= 0) */
    int64_t H;            /* heads */
    int64_t P;            /* channels per head (Mamba-2 head dim; 1 for Mamba-1) */
    int64_t S;            /* states per channel (d_state) */
    int64_t G;            /* groups of B and C (H % G == 0) */
    int32_t a_per_state;  /* 1: A is [H][S] (Mamba-1); 0: A is [H] (Mamba-2) */
    int32_t K;            /* checkpoint interval in tokens; 0 = ceil(sqrt(T)), rounded up
                             to a multiple of 64 for the chunked form's sizes */
    int32_t reserved0;    /* 0 */
    int32_t reserved1;    /* 0 */
} ssm_params_t;

/* The checkpoint interval in use (K; for K = 0, ceil(sqrt(T)), rounded up to a multiple of
 * 64 where the chunked form runs; at least 1). */
int64_t ssm_checkpoint_interval(const ssm_params_t* p);
/* Checkpoints per (sequence, head): ceil(T / K), and 1 when T = 0. */
int64_t ssm_num_checkpoints(const ssm_params_t* p);
/* Floats of the packed forward output, and of the packed backward output. */
size_t ssm_packed_out_elems(const ssm_params_t* p);
size_t ssm_packed_grad_elems(const ssm_params_t* p);
/* Bytes of device workspace ssm_backward needs. */
size_t ssm_backward_workspace_bytes(const ssm_params_t* p);
/* GDN_OK when the sizes are supported, else the code ssm_forward / ssm_backward would return. */
int ssm_supported(const ssm_params_t* p);
/* 1 when these sizes run the chunked form (one decay per head, P = 64, S = 128, T >= 1, K a
 * multiple of 64), 0 when they run another form or are unsupported. */
int ssm_chunked(const ssm_params_t* p);
/* The form these sizes run: 0 token-serial walk, 1 chunked, 2 segmented (a decay per state);
 * -1 when unsupported. */
int ssm_form(const ssm_params_t* p);
/* Kernels a forward / backward call with these params launches (0 when the call would
 * launch none: unsupported sizes, N = 0, or the backward at T = 0). */
int ssm_forward_launches(const ssm_params_t* p);
int ssm_backward_launches(const ssm_params_t* p);

/* Forward: y and s_T into out_packed, the checkpoints into ckpt (n_ck states per head). */
int ssm_forward(const ssm_params_t* p, const float* s0, const float* x, const float* dt, const float* A,
                const float* B, const float* C, float* out_packed, float* ckpt, void* stream);

/* Reverse walk: from the forward's checkpoints and the packed cotangent [dy | ds_T], the
 * packed gradients [d_s | d_x | d_dt | d_B | d_C]. */
int ssm_backward(const ssm_params_t* p, const float* x, const float* dt, const float* A, const float* B,
                 const float* C, const float* ckpt, const float* grad_in, float* grad_out, void* workspace,
                 size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_H */
