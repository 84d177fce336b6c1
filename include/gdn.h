/*
 * gdn.h -- C ABI of libgdn: the gated delta rule (Gated DeltaNet with a scalar gate,
 * Kimi Delta Attention with a per-key-column gate), forward and backward, as CUDA
 * kernels for sm_103a (GB300).
 *
 * The operation
 * -------------
 * Per sequence n and value head h (its key head is h mod H_k), with the state kept as
 * M = S^T (S_v rows j = value index, S_k columns i = key index) and a = exp(g):
 *     S'      = a (.) M_{t-1}                 (S'[j][i] = a_i M_{t-1}[j][i])
 *     u_j     = sum_i S'[j][i] k_i,   delta_j = beta (v_j - u_j)
 *     M_t     = S' + k delta^T        (M_t[j][i] = S'[j][i] + k_i delta_j)
 *     y_j     = scale sum_i M_t[j][i] q_i
 * Sources: "metal: GATED_DELTA_NET_BACK" (llama.cpp fork PR #16), review comment
 * "APPROVED at 739b9bf" (row form); meTile "Training kernels and gradients", section
 * "Recurrent delta attention" (matrix form, decay before correction).
 *
 * The backward walks the tokens in reverse from dM = dstate_T (PR #16 review "Math,
 * read term by term"): dM += scale gy q^T; dq = scale M_t^T gy; dd = dM k;
 * dv = beta dd; du = -beta dd; dbeta = sum_j dd_j (v_j - u_j);
 * dk = dM^T delta + S'^T du (dM read before the du update); dM += k du^T (= dS');
 * dg = sum_j dS' (.) S' per key column (KDA) or summed (scalar gate); dM = a (.) dS'.
 * dq/dk are summed over the H_v/H_k value heads that share a key head, in ascending
 * value-head order (and, with the sequence broadcast, over the value sequences that share
 * a q/k sequence, ascending), without atomics.
 *
 * Checkpointed recompute (PR #16 body: "checkpointed recompute (C ~ sqrt(T))"): the
 * forward stores ckpt[c] = the state entering token c*C for c = 0..n_ck-1,
 * n_ck = ceil(T/C); the backward recomputes every segment from its checkpoint.  The
 * backward returns one packed buffer [dq|dk|dv|dg|dbeta|dstate] (PR #16 body).
 *
 * Layouts (M = S^T; fp32 unless gdn_params_t.in_dtype makes q, k, v, g, beta, gy 16-bit)
 * ----------------------------------------------------------------------------------
 *   q, k      [N_q][T][H_k][S_k] element strides q_s/k_s = {seq, token, head}; the
 *                               S_k elements of one (seq, token, head) are contiguous
 *                               (so q, k may be row views of a packed qkv buffer);
 *                               N_q = N / seq_rep (N without the sequence broadcast)
 *   v         [N][T][H_v][S_v]  strides v_s, last dim contiguous
 *   gy        [N][T][H_v][S_v]  strides gy_s, last dim contiguous
 *   g         [N][T][H_v] (scalar gate) or [N][T][H_v][S_k] (KDA), contiguous
 *   beta      [N][T][H_v] contiguous
 *   state0, state_T, dstate_T    [N][H_v][S_v][S_k] contiguous
 *   y         [N][T][H_v][S_v] contiguous
 *   ckpt      [N][H_v][n_ck][S_v][S_k] contiguous
 *   packed    dq [N_q][T][H_k][S_k] | dk [N_q][T][H_k][S_k] | dv [N][T][H_v][S_v] |
 *             dg (like g) | dbeta [N][T][H_v] | dstate [N][H_v][S_v][S_k], back to back
 *             (element offsets from gdn_packed_grad_offsets)
 *
 * Arithmetic
 * ----------
 * Inputs, outputs, the state and every accumulator are fp32.  The products are computed
 * as follows: at head size 128 (scalar gate) the state-sized products run on the tcgen05
 * tensor cores as three-pass split products -- each operand split x = hi + lo into bf16
 * (kind::f16) or, for one product of the gradient step, tf32 parts, and a b taken as
 * hi hi + hi lo + lo hi with an fp32 accumulator, about 2^-16 (bf16) or 2^-20 (tf32) of
 * |a b| -- and the chunk-sized products as three-pass tf32 warp-level MMAs; elsewhere
 * every product is fp32 on the FP32 pipe (and three-pass tf32 warp-level MMAs for the
 * chunk-sized ones).  Gates use the accurate expf; nothing is built with fast-math.
 *
 * Ownership and ordering
 * ----------------------
 * The caller owns every buffer and the stream; the library allocates no device memory
 * and keeps no pointer after a call returns.  Work is enqueued on `stream` (a
 * cudaStream_t; NULL is the legacy default stream): GDN_OK means "validated and
 * launched".  At head size 128 the chunked path also uses four library streams per
 * device (created on first use): the call's stream forks into them and joins back with
 * events, so everything the call enqueues is ordered after earlier work on `stream` and
 * before later work on it.  Those streams are shared by every caller on the device, so
 * such calls are serialised on the GPU even when their own streams are independent (and
 * their host-side enqueueing takes a per-device lock).  The inputs and
 * ckpt must stay unchanged between gdn_forward and gdn_backward; the backward never
 * writes its inputs.  Inputs must be finite.
 *
 * Errors (no call ever writes an output when it returns an error)
 * ------
 *   GDN_ERR_INVALID_ARG  NULL pointer, negative size, H_v % H_k != 0, n_seq % seq_rep != 0,
 *                        a stride that is
 *                        negative, an input that is not aligned to its element (4 bytes,
 *                        2 for 16-bit inputs), a state or output buffer that is not
 *                        16-byte aligned, bad gate kind or input dtype
 *   GDN_ERR_UNSUPPORTED  S_k != S_v, or a head size other than 32, 64, 128
 *   GDN_ERR_ALIAS        an output overlaps an input (state_T over state0 included)
 *   GDN_ERR_WORKSPACE    workspace smaller than gdn_backward_workspace_bytes()
 *   GDN_ERR_CUDA         a CUDA launch failed (text in gdn_last_error())
 * gdn_last_error() returns a description of the last failure on the calling thread.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,
    GDN_ERR_UNSUPPORTED = 2,
    GDN_ERR_ALIAS = 3,
    GDN_ERR_WORKSPACE = 4,
    GDN_ERR_CUDA = 5,
    GDN_ERR_TIMEOUT = 6
} gdn_status_t;

typedef enum { GDN_GATE_SCALAR = 0, GDN_GATE_KDA = 1 } gdn_gate_t;

/* Storage type of the inputs q, k, v, g, beta and gy (meTile "Training kernels and
 * gradients": 16-bit inputs beside fp32 state and fp32 gradients).  States (state0,
 * dstate_T, state_T, ckpt) and every output are fp32 whatever the input type.  A call with
 * 16-bit inputs widens them (exactly: every bf16 and fp16 value is an fp32 value) into
 * dense fp32 copies at the start of its workspace, then runs the fp32 path on them; the
 * workspace queries include those copies. */
typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 } gdn_dtype_t;

typedef struct {
    int64_t n_seq, T, H_k, H_v, S_k, S_v; /* sizes; H_v = r H_k, key head = h_v mod H_k */
    int32_t gate;                         /* gdn_gate_t */
    int32_t in_dtype;                     /* gdn_dtype_t of q, k, v, g, beta, gy (0: fp32) */
    int64_t C;                            /* checkpoint interval; <= 0: ceil(sqrt(T)) */
    float scale;                          /* output scale, usually 1/sqrt(S_k) */
    int32_t seq_rep;                      /* 0 or 1: q, k have n_seq sequences.  r > 1: the
                                             sequence broadcast (PR #16 "iv3/rq3"): q, k
                                             (and dq, dk) hold n_seq / r sequences and value
                                             sequence n reads q/k sequence n / r */
    int64_t q_s[3], k_s[3], v_s[3], gy_s[3]; /* element strides of {seq, token, head} */
} gdn_params_t;

/* Effective checkpoint interval (C, or ceil(sqrt(T)) when C <= 0) and count ceil(T/C). */
int64_t gdn_checkpoint_interval(const gdn_params_t* p);
int64_t gdn_num_checkpoints(const gdn_params_t* p);
/* Elements of the ckpt buffer: N * H_v * n_ck * S_v * S_k. */
size_t gdn_ckpt_elems(const gdn_params_t* p);

/* Device workspace the forward needs (bytes; 0 when it needs none).  Scratch owned by
 * the caller for the duration of the enqueued work; 256-byte aligned start required. */
size_t gdn_forward_workspace_bytes(const gdn_params_t* p);

/* Forward (meTile "Recurrent delta attention"; PR #16 row form).  Reads q, k, v, g,
 * beta, state0; writes y, state_T and ckpt (each must be non-NULL unless its size is
 * zero).  state_T may not overlap state0 (llama.cpp PR #26: an in-place state update
 * destroyed the initial state the backward needed).  The scalar gate runs the chunked
 * (WY) regrouping of the recurrence (exact, chunks of 32 tokens aligned to the
 * checkpoint segments); the per-key-column gate runs the token recurrence. */
gdn_status_t gdn_forward(const gdn_params_t* p, const void* q, const void* k,
                         const void* v, const void* g, const void* beta,
                         const float* state0, float* y, float* state_T, float* ckpt,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Packed gradient buffer: total elements, and the element offsets of its six regions
 * in the order dq, dk, dv, dg, dbeta, dstate (PR #16 body: "[dq|dk|dv|dg|dbeta|dstate]"). */
size_t gdn_packed_grad_elems(const gdn_params_t* p);
void gdn_packed_grad_offsets(const gdn_params_t* p, size_t off[6]);

/* Device workspace the backward needs (bytes, 256-byte aligned start required). */
size_t gdn_backward_workspace_bytes(const gdn_params_t* p);

/* Backward (PR #16, GATED_DELTA_NET_BACK).  Reads q, k, v, g, beta, ckpt (from
 * gdn_forward with the same params), gy and dstate_T (NULL = zero cotangent for the
 * final state); writes every element of packed_grads.  The workspace is scratch owned
 * by the caller for the duration of the enqueued work. */
gdn_status_t gdn_backward(const gdn_params_t* p, const void* q, const void* k,
                          const void* v, const void* g, const void* beta,
                          const float* ckpt, const void* gy, const float* dstate_T,
                          float* packed_grads, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Backward without a caller workspace.  The paper has no counterpart: this entry point
 * exists for callers that cannot allocate device memory when they run the backward (a
 * host framework that has already handed out its whole memory budget, a plugin host
 * that gives extensions no device allocator, a call site that must not trigger an
 * allocator).  Its scratch is one fixed 64 MiB array in device memory that every GPU
 * which loads libgdn holds until the process exits; it allocates nothing itself.
 * Arguments and results are those of gdn_backward, less the workspace.  Problems whose
 * gdn_backward_workspace_bytes() exceeds 64 MiB return GDN_ERR_WORKSPACE (text in
 * gdn_last_error()) before any work is enqueued.  The first call on a device, with that
 * device current, looks up the array's address; make it before any stream capture.  All
 * calls on a device share the array (no call needs it zeroed: every scratch element a
 * call reads, it wrote first), so calls whose work overlaps on the GPU race on it:
 * order them on one stream or with events.  The address is looked up once per device and
 * kept: a process that calls cudaDeviceReset on a device must not use this entry point on
 * it afterwards.  A device index of 64 or more returns GDN_ERR_UNSUPPORTED. */
gdn_status_t gdn_backward_noalloc(const gdn_params_t* p, const void* q, const void* k,
                                  const void* v, const void* g, const void* beta,
                                  const float* ckpt, const void* gy, const float* dstate_T,
                                  float* packed_grads, void* stream);

/* Static text of a status code, and the detail of the calling thread's last error. */
const char* gdn_status_str(gdn_status_t s);
const char* gdn_last_error(void);

/* Optional per-stage timing for the calling thread: while `events` is non-NULL, every
 * gdn_forward / gdn_backward call records events[0] on its stream before its first
 * stage and events[i] after its i-th stage, for i < n_events (stages: see
 * gdn_timing_stages).  The events are cudaEvent_t handles the caller created and owns;
 * NULL turns the recording off.  Not part of the operation: it lets a caller time the
 * kernels of a call. */
void gdn_set_timing_events(void* const* events, int n_events);

/* Kernels a forward / backward call with these params launches (0 when the call would
 * fail validation).  Lets callers account for the work they enqueue.  On the head-size-128
 * path this is the count without timing events.  A backward call with timing events set
 * runs its stages one after another as one chunk range: the prep, the dM chain, one
 * gradient launch per place of a chunk in its segment, and the sum. */
int gdn_forward_launches(const gdn_params_t* p);
int gdn_backward_launches(const gdn_params_t* p);

/* Timed stages of a forward (backward = 0) or backward (backward = 1) call with these
 * params: gdn_set_timing_events records one event before the first stage and one after
 * each stage.  A stage is one kernel, except on the head-size-128 path.  There the
 * forward's chunk preps and state chain run pipelined over chunk ranges on library
 * streams and form 1 stage.  The backward normally overlaps all of its kernels across
 * chunk ranges; with timing events set it runs them one after another instead, in 3
 * stages (prep and both chains, the gradient step, the sum over value heads), so that
 * each kernel can be timed.  0 when the call would fail validation. */
int gdn_timing_stages(const gdn_params_t* p, int backward);

/* Device-side status of the work enqueued so far on the current device.  The
 * tensor-core kernels (head size 128) wait on hardware barriers for their operand copies
 * and products; every such wait is bounded (0.2 s of wall clock, far beyond any
 * legitimate wait), and a wait that gives up makes its kernel return early and record
 * GDN_ERR_TIMEOUT in a device status word, leaving that call's outputs invalid.  This
 * call synchronises `stream` (a cudaStream_t, NULL = legacy default stream), then reads
 * and clears the status words: GDN_OK, GDN_ERR_TIMEOUT, or GDN_ERR_CUDA if the stream or
 * the read failed (text in gdn_last_error()).  No counterpart on the pages; it exists
 * because a GPU kernel cannot return an error code by itself. */
gdn_status_t gdn_device_status(void* stream);

/* Test hook for the timeout path: enqueues one single-CTA kernel whose bounded wait on a
 * barrier that nothing completes gives up, as above, so that the next gdn_device_status
 * returns GDN_ERR_TIMEOUT.  Touches no caller memory; takes about 0.2 s of GPU time.
 * Returns GDN_ERR_CUDA if the launch failed. */
gdn_status_t gdn_selftest_wait_timeout(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
