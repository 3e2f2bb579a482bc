/*
 * gdn.h — C ABI of the GB300 (sm_103a) chunked forward pass of the gated
 * delta rule (Gated DeltaNet).
 *
 * The operation (page "WarpDrive", kernels 3-5 and section "Pipeline", chunk
 * size C = 64): for every batch b and head h, with a per-head state h of shape
 * [K, V] carried across the sequence in chunks of 64 tokens,
 *
 *   A      = (I + L)^-1, L_ij = beta_i (k_i . k_j) exp(g_i - g_j) for i > j
 *            (the chunk's "[64,64] WY matrix", kernel 5),
 *   u      = A (v * beta),  w = A (k * beta * exp(g))          (recompute_w_u, kernel 5)
 *   per chunk, in order (chunk_fwd_h, kernel 3):
 *            store h; v_new = u - w @ h; v_gated = v_new * exp(g_last - g_t);
 *            h *= exp(g_last); h += k^T @ v_gated
 *   o      = scale * (q @ h * exp(g)) + causal(q @ k^T * exp(g_i - g_j)) @ v_new
 *            with the causal mask i >= j                     (chunk_fwd_o, kernel 4)
 *
 * which equals, token by token, S <- exp(gamma_t) S; S += k_t (beta_t (v_t - S^T k_t))^T;
 * o_t = scale S^T q_t with h0 the state before the first token and h_final
 * the state after the last.
 *
 * Conventions shared by every entry point:
 *  - Every tensor argument is a DEVICE pointer on the current CUDA device,
 *    contiguous, row-major, 16-byte aligned. The caller owns all memory; the
 *    library allocates nothing. Apart from two documented exceptions (the
 *    fixed scratch array of gdn_chunk_fwd_noalloc and the one-shot test hook
 *    gdn_debug_arm_stall) it keeps no mutable global state between calls, so
 *    calls on different streams are independent as long as each has its own
 *    workspace.
 *  - Layouts: q, k [B,T,H,K]; v, o [B,T,H,V]; g, beta [B,T,H] fp32;
 *    h0, h_final [B,H,K,V] fp32.
 *  - g is the per-token log-decay summed cumulatively *within each 64-token
 *    chunk* (restarting at t = 0, 64, 128, ...), unless the problem's flags
 *    hold GDN_FLAG_RAW_G (below). Values should be <= 0 and non-increasing
 *    inside a chunk; exp(g_i - g_j) is only evaluated for i >= j.
 *  - T need not be a multiple of 64: the last chunk is partial and g_last is
 *    the g of its last valid token. T = 0 is valid: h_final = h0 (or zeros).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously. Argument errors are reported
 *    synchronously before anything is enqueued; a launch error is reported as
 *    GDN_ERR_CUDA. No C++ exception crosses this boundary.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,    /* NULL required pointer, negative size, bad enum */
    GDN_ERR_UNSUPPORTED = 2,    /* shape or dtype/algorithm combination not built */
    GDN_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
    GDN_ERR_WORKSPACE = 4,      /* workspace NULL or smaller than required */
    GDN_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
    GDN_ERR_DEVICE_TIMEOUT = 6  /* a bounded device-side wait gave up */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum {
    GDN_ALGO_AUTO = 0,   /* fastest built path for the problem */
    GDN_ALGO_SIMT = 1,   /* CUDA-core fp32 pipeline, four kernels, any dtype */
    GDN_ALGO_TC = 2,     /* tensor-core (tcgen05/TMEM, TMA) path, bf16 only: a
                          * kernel building every chunk's WY matrix (in parallel,
                          * to the workspace), then the forward kernel */
    GDN_ALGO_TC_SINGLE = 3, /* the same in one kernel: each CTA builds its chunks'
                          * WY matrices itself, one chunk ahead of their use, so
                          * A never reaches HBM (slower today: the build is a
                          * serial chain inside the CTA). Without the output stage
                          * and without the A export (else GDN_ERR_UNSUPPORTED) */
    GDN_ALGO_TC_WIDE = 4 /* GDN_ALGO_TC with the wide forward kernel: one CTA per
                          * 128 V columns of a head (W, q k^T and the operand
                          * loads shared by both 64-column halves). GDN_ALGO_TC
                          * and GDN_ALGO_AUTO pick it by themselves when the
                          * 64-column grid would take more than one wave of SMs.
                          * V a multiple of 128; without the output stage (else
                          * GDN_ERR_UNSUPPORTED) */
} gdn_algo;

/* Input front-end options (gdn_problem.flags), a bit set; 0 = inputs as
 * described above. Both steps sit before the WY build: they are the
 * normalisation and gate steps that a Gated DeltaNet layer applies to its
 * projections ("KdaSplit" decode kernel page, its q/k normalisation), done
 * inside the kernels so that no separate pass over q, k or g is needed.
 *  - GDN_FLAG_RAW_G: g holds the per-token log decays gamma_t themselves;
 *    the chunk-local cumulative sum is taken in the kernels (restarting at
 *    t = 0, 64, 128, ...). Without it g is that cumulative sum already.
 *  - GDN_FLAG_QK_L2NORM: every q and k row (one token of one head, K values)
 *    is replaced by x / sqrt(sum_i x_i^2 + 1e-6) before use; scale still
 *    multiplies o, i.e. it scales the normalised q. The normalised rows are
 *    never rounded back to the input dtype.
 *  - GDN_FLAG_PER_CHANNEL_DECAY: the decay is a K-vector per token (the KDA
 *    variant of the "KdaSplit" decode kernel page, where each state row decays
 *    by its own factor): g is [B,T,H,K] fp32 and the decay step becomes
 *    S[i, :] <- exp(gamma_t[i]) S[i, :]; in the chunked form every
 *    exp(g_i - g_j) becomes a per-channel factor inside the k and q products.
 *    It combines with the other flags (the cumulative sum is then per
 *    channel). The chunked forward runs it on the CUDA-core pipeline or, for
 *    bf16, on a tensor-core form of its own under GDN_ALGO_TC (a prep kernel
 *    per chunk building the decay-weighted WY and attention products, then
 *    the forward kernel over the chunks); GDN_ALGO_TC_SINGLE and
 *    GDN_ALGO_TC_WIDE give GDN_ERR_UNSUPPORTED. That form runs the output
 *    stage too, but of the stage exports it has only A_beta: with GDN_ALGO_TC
 *    a call asking for the others gives GDN_ERR_UNSUPPORTED, with
 *    GDN_ALGO_AUTO it runs on the CUDA-core pipeline, and the workspace size
 *    for GDN_ALGO_AUTO covers both.
 * gdn_decode_step always takes raw gamma and accepts either g flag; it
 * honours GDN_FLAG_QK_L2NORM and GDN_FLAG_PER_CHANNEL_DECAY (gamma [B,T,H,K]). */
enum {
    GDN_FLAG_RAW_G = 1,
    GDN_FLAG_QK_L2NORM = 2,
    GDN_FLAG_PER_CHANNEL_DECAY = 4
};

/* Problem description. K in {64, 128}; V a multiple of 64 in [64, 256];
 * dtype is the element type of q, k, v and o; flags a set of GDN_FLAG_*
 * (unknown bits give GDN_ERR_INVALID_ARG). */
typedef struct {
    int32_t B, T, H, K, V;
    int32_t dtype;   /* gdn_dtype */
    int32_t algo;    /* gdn_algo */
    int32_t flags;   /* GDN_FLAG_* bits */
} gdn_problem;

/* Bytes of device workspace gdn_chunk_fwd needs for this problem (0 if the
 * problem is invalid). The workspace is scratch: its contents on entry do not
 * matter and are undefined on exit, except where gdn_chunk_fwd_stages says. */
GDN_API size_t gdn_chunk_fwd_workspace_bytes(const gdn_problem *p);

/* Chunked forward. q, k, v, g, beta, o are required; h0 == NULL means a zero
 * initial state; h_final == NULL means the final state is not written.
 * scale multiplies both the inter-chunk (q @ h) and intra-chunk terms of o.
 * o is written in `dtype` (round to nearest even from fp32); h_final in fp32. */
GDN_API gdn_status gdn_chunk_fwd(const gdn_problem *p,
                                 const void *q, const void *k, const void *v,
                                 const float *g, const float *beta, float scale,
                                 const float *h0, void *o, float *h_final,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* Stage export for testing: same computation as gdn_chunk_fwd, then copies the
 * intermediates of the pipeline into the given device buffers (each may be
 * NULL = not exported), all fp32 and indexed with T_pad = ceil(T/64)*64 rows
 * per (b, h) (rows >= T are padding):
 *   A      [B,T_pad,H,64]  the chunk's WY matrix, row t, column = token index in its chunk
 *   w      [B,T_pad,H,K]   u [B,T_pad,H,V]   v_new [B,T_pad,H,V] (ungated)
 *   h      [B,NT,H,K,V]    the state entering each chunk, NT = ceil(T/64)
 *   A_beta [B,T_pad,H,64]  A diag(beta), the WY stage the tensor-core path keeps (bf16 there)
 * The SIMT path materialises A, w, u, v_new and h; the tensor-core path only
 * A_beta. Requesting a stage the chosen path never materialises returns
 * GDN_ERR_UNSUPPORTED before anything is enqueued. */
typedef struct {
    float *A, *w, *u, *v_new, *h, *A_beta;
} gdn_stage_exports;

GDN_API gdn_status gdn_chunk_fwd_stages(const gdn_problem *p,
                                        const void *q, const void *k, const void *v,
                                        const float *g, const float *beta, float scale,
                                        const float *h0, void *o, float *h_final,
                                        void *workspace, size_t workspace_bytes,
                                        const gdn_stage_exports *ex, void *stream);

/* Number of kernels one gdn_chunk_fwd call on this problem launches, in launch
 * order (0 if the problem is invalid); names[i] receives a static name of
 * kernel i when names != NULL and i < max_names. */
GDN_API int32_t gdn_chunk_fwd_launches(const gdn_problem *p, const char **names,
                                       int32_t max_names);

/* gdn_chunk_fwd with timing markers for measurement: `events` holds
 * n_events >= gdn_chunk_fwd_launches(p) + 1 cudaEvent_t handles created by the
 * caller; events[0] is recorded on `stream` before the first kernel and
 * events[i + 1] right after kernel i. Same results as gdn_chunk_fwd. */
GDN_API gdn_status gdn_chunk_fwd_profiled(const gdn_problem *p,
                                          const void *q, const void *k, const void *v,
                                          const float *g, const float *beta, float scale,
                                          const float *h0, void *o, float *h_final,
                                          void *workspace, size_t workspace_bytes,
                                          void *const *events, int32_t n_events, void *stream);

/* The forward from and to HOST memory, for callers whose tensors live there:
 * q, k, v, g, beta, h0 (or NULL) are host buffers in the layouts above; o and
 * h_final (or NULL) are host buffers the results are written to. Page-locked
 * (pinned) host buffers let the copies run asynchronously and overlap.
 *
 * The sequence is cut into up to `pieces` spans of T (1..16 spans, each a
 * multiple of 64 tokens, all batch rows and heads at once; pieces == 0 lets
 * the library pick about one span per 32 MiB of inputs, 3 to 16) so that the
 * host-to-device copies of one span (on `stream_a`) overlap the kernels and the
 * device-to-host copies of the previous one (on `stream_b`); each span starts
 * from the previous span's final state. The call creates and destroys one
 * event per span to order the two streams. `device_buffer` (device memory of at
 * least gdn_chunk_fwd_host_bytes(p, pieces) bytes, 256-byte aligned) holds the
 * device copies of the inputs and outputs, two state buffers and one span's
 * workspace. Both streams must be distinct, caller-created streams of the
 * current device. The call returns when o and h_final are in host memory (it
 * synchronises both streams); errors are reported as for gdn_chunk_fwd, and a
 * bounded device wait that gave up in any span's kernels is returned as
 * GDN_ERR_DEVICE_TIMEOUT (the outputs are then garbage). Same results as
 * gdn_chunk_fwd up to rounding (the state crosses a span boundary in fp32;
 * with one span they are identical). */
GDN_API size_t gdn_chunk_fwd_host_bytes(const gdn_problem *p, int32_t pieces);
GDN_API gdn_status gdn_chunk_fwd_host(const gdn_problem *p,
                                      const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float scale,
                                      const float *h0, void *o, float *h_final,
                                      void *device_buffer, size_t device_bytes,
                                      int32_t pieces, void *stream_a, void *stream_b);

/* Waits for `stream`, then reads and clears the device status word kept in the
 * first bytes of `workspace`: GDN_ERR_DEVICE_TIMEOUT if a bounded device wait
 * of an earlier call on this workspace gave up, GDN_OK otherwise (or
 * GDN_ERR_CUDA if the stream itself reports an error). Every gdn_chunk_fwd
 * call clears the word when it starts, so it reports on the last call. */
GDN_API gdn_status gdn_check_device_status(void *workspace, void *stream);

/* Test hook for the device-timeout path; the method's pages have no
 * counterpart. Arms a one-shot fault for the next launch of the tensor-core
 * forward in this process: that launch withholds the input loads of its first
 * chunk, so every role's first wait on them runs out after `wait_ns`
 * nanoseconds (0 means 1 ns), the roles leave their loops, whatever was
 * issued drains, and the launch records the timeout in the workspace's status
 * word (read it with gdn_check_device_status). The outputs of that call are
 * garbage; later calls are unaffected. Nothing traps and no wait is unbounded.
 * Process-global: for tests only, never with concurrent callers. */
GDN_API void gdn_debug_arm_stall(uint64_t wait_ns);

/* gdn_chunk_fwd without a workspace argument, for callers that cannot allocate
 * device memory at all: code running where cudaMalloc is unavailable or
 * forbidden (a plugin handed only its input and output buffers by a host
 * framework that owns every allocation, or code that must not allocate after
 * start-up). The method's pages have no counterpart to this call; it is a
 * deployment convenience.
 *
 * The scratch lives in a fixed 64 MiB array inside the library's device image,
 * present on every GPU that loads the library until the process exits. It runs
 * the CUDA-core (SIMT) pipeline; p->algo must be GDN_ALGO_AUTO or
 * GDN_ALGO_SIMT (else GDN_ERR_UNSUPPORTED). Problems whose SIMT workspace
 * (gdn_chunk_fwd_workspace_bytes with algo SIMT) exceeds 64 MiB are rejected
 * with GDN_ERR_WORKSPACE before anything is enqueued. Nothing here calls
 * cudaMalloc, cudaFree or an allocating library routine.
 *
 * Every call looks up the array's device address on the current device (a
 * host-side lookup, so the address stays right after a cudaDeviceReset); the
 * first call on a device may also load the library's device code, so make
 * that first call before any stream capture. `stream` must belong to the
 * current device (else GDN_ERR_INVALID_ARG): the array used is the current
 * device's. Every call on a device shares the one array: calls whose work
 * overlaps on the GPU (on different streams, or from different threads) race
 * and give wrong results; serialise them. The array keeps the last call's
 * contents; no call depends on them. Pointer conventions, layouts and other
 * errors are those of gdn_chunk_fwd. */
GDN_API gdn_status gdn_chunk_fwd_noalloc(const gdn_problem *p,
                                         const void *q, const void *k, const void *v,
                                         const float *g, const float *beta, float scale,
                                         const float *h0, void *o, float *h_final,
                                         void *stream);

/* One or a few tokens of the recurrent (decode) form of the same rule, for
 * generation after a prefill: for every batch b and head h, token by token,
 *
 *   S <- exp(gamma_t) S;   delta_t = beta_t (v_t - S^T k_t);   S += k_t delta_t^T;
 *   o_t = scale S^T q_t
 *
 * i.e. the state is decayed first, then read at k_t, written, and read at q_t
 * (the order of the delta-rule row update of the "KdaSplit" decode kernel page,
 * its `update` step, with the scalar per-head decay of Gated DeltaNet). Tokens
 * after the first of a call see the state left by the one before.
 *
 *  - p->T >= 0 tokens per sequence (1 for plain decode; a few for multi-token
 *    verification); every sequence of the batch advances by the same T.
 *    T = 0 copies state_in to state_out (nothing when they are the same).
 *  - q, k [B,T,H,K] and v, o [B,T,H,V] in p->dtype; gamma, beta [B,T,H] fp32.
 *    gamma is the per-token log decay log(alpha_t) <= 0 itself, NOT the
 *    chunk-local cumulative sum gdn_chunk_fwd takes (for T = 1 the two agree).
 *  - state_in, state_out [B,H,K,V] fp32, in the layout of h0 / h_final, so a
 *    prefill's h_final is a decode's state_in. They may be the same pointer
 *    (update in place) or non-overlapping buffers; partial overlap is
 *    undefined. state_in is required (a zero state is a zeroed buffer).
 *  - Limits: K a multiple of 64 up to 256; V a multiple of 16 up to 4096;
 *    p->algo GDN_ALGO_AUTO or GDN_ALGO_SIMT (the step is a matrix-vector
 *    product with no tensor-core form; GDN_ALGO_TC gives GDN_ERR_UNSUPPORTED).
 *  - No workspace; nothing is allocated. For long T the chunked forward is
 *    the faster route to the same result.
 * Pointer, alignment, stream and error conventions are those above. */
GDN_API gdn_status gdn_decode_step(const gdn_problem *p,
                                   const void *q, const void *k, const void *v,
                                   const float *gamma, const float *beta, float scale,
                                   const float *state_in, float *state_out, void *o,
                                   void *stream);

/* Number of kernels one gdn_decode_step call on this problem launches: 1 for
 * T >= 1, 0 for T = 0 (the state copy is a cudaMemcpyAsync) or an invalid
 * problem. names[0] receives the kernel's static name when names != NULL,
 * max_names > 0 and the count is 1. */
GDN_API int32_t gdn_decode_step_launches(const gdn_problem *p, const char **names,
                                         int32_t max_names);

/* Output stage (optional): the gated RMSNorm that a Gated DeltaNet layer applies
 * to the rule's output (the output stage of the "KdaSplit" decode kernel page:
 * root of the mean square over the head's channels plus eps, norm weight, and
 * the token's gate through a sigmoid). Each row o_t of one token and head
 * (V values) becomes
 *     o_t[v] * rsqrt(mean_u o_t[u]^2 + eps) * weight[v] * sigmoid(gate_t[v]),
 * formed from the fp32 o before its one rounding to the output dtype. On the
 * tensor-core path, the heads that the 128-column forward kernel takes
 * (GDN_ALGO_TC_WIDE, or GDN_ALGO_TC / AUTO on grids that take it) get the mean
 * square from the fp32 o too, but weight and gate are applied to o rounded to
 * the output dtype: one more rounding, at most one unit in the last place. */
typedef struct {
    const void *gate;      /* [B,T,H,V] in p->dtype, required, 16-byte aligned */
    const float *weight;   /* [V] fp32, required, 16-byte aligned */
    float eps;             /* >= 0 */
} gdn_output_norm;

/* gdn_chunk_fwd with the optional output stage (norm == NULL: the plain o of
 * gdn_chunk_fwd) and optional timing markers as in gdn_chunk_fwd_profiled
 * (events == NULL: none). On the tensor-core path the forward kernels apply
 * the stage themselves, the CTAs of one head's V tiles forming a thread-block
 * cluster to share the row sums, so a call launches the kernels that
 * gdn_chunk_fwd_launches names. Every other contract is gdn_chunk_fwd's. */
GDN_API gdn_status gdn_chunk_fwd_ex(const gdn_problem *p,
                                    const void *q, const void *k, const void *v,
                                    const float *g, const float *beta, float scale,
                                    const float *h0, const gdn_output_norm *norm,
                                    void *o, float *h_final,
                                    void *workspace, size_t workspace_bytes,
                                    void *const *events, int32_t n_events, void *stream);

/* gdn_decode_step with the optional output stage (norm == NULL: plain o).
 * With it, one CTA holds a head's whole [K, V] state, so K * V <= 32768
 * (else GDN_ERR_UNSUPPORTED). */
GDN_API gdn_status gdn_decode_step_ex(const gdn_problem *p,
                                      const void *q, const void *k, const void *v,
                                      const float *gamma, const float *beta, float scale,
                                      const float *state_in, float *state_out,
                                      const gdn_output_norm *norm, void *o, void *stream);

/* Static description of a status code. Never NULL. */
GDN_API const char *gdn_status_string(gdn_status s);

/* Library version, (major << 16) | (minor << 8) | patch. */
GDN_API uint32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
