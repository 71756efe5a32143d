/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) Kimi Delta Attention core.
 *
 * The library computes the gated delta rule with a per-key-channel decay, the
 * mixer core of the Kimi-Linear / Kimi-K3 KDA layers, for every independent
 * (sequence, head) unit:
 *
 *     q^ = q / sqrt(|q|^2 + 1e-6),  k^ = k / sqrt(|k|^2 + 1e-6)     (if use_qk_l2norm)
 *     S_t = (I - beta_t k^_t k^_t^T) Diag(exp g_t) S_{t-1} + beta_t k^_t v_t^T
 *     o_t = scale * S_t^T q^_t
 *
 * optionally followed by the head-wise sigmoid-gated RMSNorm
 *
 *     y = o / sqrt(mean_v(o^2) + eps) * w * sigmoid(gate)
 *
 * Sources (page title, section):
 *   nnterp encyclopedia "Kimi-Linear": section 02 "support()" (the kernel's
 *   arguments attention_queries/keys/values, decays, betas, state_input and its
 *   outputs attention_head_outputs, state_output, with their layouts); section 03
 *   "Kimi Delta Attention decays each key channel" (g per key channel, fp32,
 *   non-positive; beta = sigmoid(b_proj); L2 norm and 1/sqrt(key_dim) applied in
 *   the kernel; state [batch, heads, key_dim, value_dim]); section 03 "Loading"
 *   (a prompt runs a chunked kernel that carries the state from one 64-token
 *   chunk to the next, a decode step the token-by-token kernel); section 04
 *   "From the family module" (the state decays channel by channel before each
 *   delta-rule update; call contract (query, key, value, g=, beta=,
 *   initial_state=) -> (core_attn_out, last_recurrent_state)).
 *   Kimi-K3 atlas "gate-project (decode, P = 1000)": sections "Parameters" (the
 *   gated RMSNorm holds 128 weights shared by the 96 heads) and "Code" (o_norm(o,
 *   gate) with activation 'sigmoid', heads then flattened to heads * head_dim).
 *
 * Conventions for every entry point:
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc, or any memory the
 *     GPU can address) unless its name ends in _host.  Tensors are dense,
 *     row-major, contiguous, 16-byte aligned.  The caller owns every buffer; the
 *     library allocates no device memory and keeps no pointer after the call.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and returns without synchronising.  Outputs are valid once the
 *     stream reaches that point.
 *   - Arguments are validated on the host before anything is launched.  A bad
 *     argument returns KDA_ERR_INVALID_ARG, an unsupported but well-formed
 *     request KDA_ERR_UNSUPPORTED, a CUDA launch/runtime error KDA_ERR_CUDA;
 *     nothing is launched in the first two cases.  kda_last_error() then holds a
 *     message for the calling thread.  No C++ exception crosses the ABI.
 *   - Precondition (not checked on the device): g lies in [-5, 0] (the layer's
 *     gate_lower_bound is -5), beta in [0, 1].  Out-of-range values give
 *     numerically meaningless but memory-safe results.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED = 2,  /* well-formed but not built (dims, dtype, chunk, mode) */
    KDA_ERR_CUDA = 3,         /* a CUDA runtime / launch error */
    KDA_ERR_TIMEOUT = 4       /* a bounded device wait gave up (returned by kda_device_status) */
} kda_status;

typedef enum kda_dtype {
    KDA_BF16 = 0,
    KDA_F32 = 1
} kda_dtype;

typedef enum kda_mode {
    KDA_MODE_AUTO = 0,    /* tensor-core path where supported, else the fp32 path */
    KDA_MODE_TENSOR = 1,  /* tcgen05 path only (K = V = 128, chunk = 64); else UNSUPPORTED */
    KDA_MODE_FP32 = 2,    /* CUDA-core fp32 chunked path (any supported K, V, chunk) */
    KDA_MODE_SPLIT = 3    /* tcgen05 path, the two-kernel split form (needs a workspace) */
} kda_mode;

/* Library version (major * 10000 + minor * 100 + patch). */
int kda_version(void);

/* Message describing the last failed call on this thread ("" if none). */
const char *kda_last_error(void);

/* Static name of a status code. */
const char *kda_status_string(int status);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t kda_launch_count(void);

/*
 * kda_device_status -- failures detected on the device since the last call.
 *
 * Every wait inside the kernels (on a bulk or TMA copy, or on the tensor core) is
 * bounded.  A CTA whose wait gives up lets the copies it started land, writes NaN
 * into every output it was responsible for (the state, o and y of its (sequence,
 * head) units, or the y and state rows of its convolution tiles; a decode CTA also
 * poisons every later unit it owned), and counts the event in a device-side counter.
 * The compute calls are asynchronous and cannot see this, so this call synchronises
 * `stream` (a cudaStream_t; NULL = the legacy default stream), reads the counters of
 * the current device and clears them.  Returns KDA_ERR_TIMEOUT if any wait gave up
 * (kda_last_error() names the kernels and counts), KDA_ERR_CUDA if the stream or a
 * counter read failed, KDA_OK otherwise.  The counters are shared by all streams of
 * the device: call it when the work to be checked has been enqueued on `stream` or
 * has finished.  No counterpart on the pages: it is the library's failure detection.
 */
kda_status kda_device_status(void *stream);

/*
 * kda_set_wait_limit -- bound on the first-line waits on copies from global memory.
 *
 * The decode step's copy waits (kda_recurrent_step, kda_recurrent_step_logits with
 * K = V = 128), the short convolution's tile waits (kda_short_conv_fwd over a prompt)
 * and the fused tensor-core prefill's tile and blob waits (kda_chunk_fwd,
 * kda_chunk_fwd_logits without a workspace or with one in the concurrent form) poll
 * their mbarrier at most this many times before they give up, for the calls made after
 * this one (process-wide).  polls < 0 restores the default (2^26); 0 makes every such
 * wait give up at once, which tests of the failure handling use (kda_device_status then
 * reports KDA_ERR_TIMEOUT and the outputs hold NaN).  The waits that let copies in
 * flight land before a CTA exits, the tensor-core waits, and the split form's kernels
 * always keep their full bound.  Returns KDA_OK, or
 * KDA_ERR_INVALID_ARG above 2^32 - 1.  No counterpart on the pages.
 */
kda_status kda_set_wait_limit(int64_t polls);

/*
 * kda_chunk_prepass_hits -- how many chunks of the concurrent form (kda_chunk_fwd with a
 * workspace) took their state-independent operands from the pre-pass rather than
 * forming them in the fused kernel, since the last call (a diagnostic of how much
 * of the work the idle SMs took over).  Synchronises `stream`, reads the current
 * device's counter into *chunks and clears it.  KDA_ERR_INVALID_ARG for a NULL
 * chunks, KDA_ERR_CUDA if the stream or the read failed.  No counterpart on the pages.
 */
kda_status kda_chunk_prepass_hits(void *stream, uint64_t *chunks);

/*
 * kda_chunk_fwd -- chunked prefill over whole prompts.
 *
 * Pages: nnterp "Kimi-Linear" section 03 "Loading" (the chunked kernel carries
 * the state from one 64-token chunk to the next and never holds it per token),
 * section 02 (argument and output layouts), section 04 (call contract).
 *
 * Dense mode (cu_seqlens == NULL): N = B sequences of T tokens.
 *   q, k   [B, T, H, K]  qkv_dtype          v [B, T, H, V] qkv_dtype
 *   g      [B, T, H, K]  float, log decay    beta [B, T, H] float
 *   initial_state [N, H, K, V] float or NULL (zero state)
 *   final_state   [N, H, K, V] float or NULL; may be the same buffer as
 *                 initial_state (updated in place)
 *   o      [B, T, H, V]  o_dtype, the per-head outputs (head outputs before the
 *                        gated norm); may be NULL when y is given
 * Varlen mode (cu_seqlens != NULL): B must be 1, T is the packed token count and
 *   sequence n covers tokens [cu_seqlens[n], cu_seqlens[n+1]), n < n_seqs;
 *   initial_state / final_state are [n_seqs, H, K, V].  cu_seqlens is a device
 *   int32 array of n_seqs + 1 entries.  cu_seqlens_host, if not NULL, is a host
 *   copy of it: it is checked (starts at 0, non-decreasing, ends at T) and used to
 *   start the longest sequences first.  Without it the device array is trusted;
 *   kernels still clamp every sequence to [0, T] so a bad array cannot make them
 *   read or write out of bounds.
 * Gated norm (gate != NULL): gate [B, T, H, V] gate_dtype, norm_w [V] float,
 *   eps > 0, y [B, T, H * V] o_dtype, y = RMSNorm_v(o) * norm_w * sigmoid(gate).
 * chunk: tokens per chunk, 16, 32 or 64 (the tensor path needs 64).
 * scale: applied to q^ (1/sqrt(K) for the layer).  use_qk_l2norm: 0 or 1.
 * Supported K, V: 32, 64, 128 (fp32 path); 128 (tensor path).
 * workspace: caller-owned device scratch of workspace_bytes, or NULL.  With NULL
 *   the tensor path runs one fused kernel per (sequence, head).  A workspace of at
 *   least kda_chunk_workspace_size(B, T, H, n_seqs) bytes lets it use the SMs that
 *   kernel leaves idle (N * H below the SM count): a pre-pass kernel on a stream the
 *   call creates forms chunks' state-independent operands (grams, UT transform) ahead
 *   of the fused kernel, which takes each one that is ready when it gets there and
 *   forms the rest itself, never waiting (the concurrent form; the caller's stream
 *   covers both kernels).  With mode KDA_MODE_SPLIT the pre-pass instead forms every
 *   chunk's operands first, then one CTA per (sequence, head) runs the state through
 *   the chunks (the split form).  All forms give the same bits.  A workspace that is
 *   too small, misaligned or overlaps a tensor of the call is KDA_ERR_INVALID_ARG; the
 *   fp32 path ignores it.  Its contents are scratch: overwritten by the call,
 *   meaningless after it.  Calls that may overlap on the GPU need workspaces of
 *   their own.
 * mode: a kda_mode.  Returns a kda_status.
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                         const float *g, const float *beta, const float *initial_state,
                         float *final_state, void *o, kda_dtype o_dtype,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int n_seqs,
                         int B, int T, int H, int K, int V, int chunk, float scale,
                         int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                         const float *norm_w, float eps, void *y, void *workspace,
                         size_t workspace_bytes, int mode, void *stream);

/*
 * kda_chunk_workspace_size -- bytes of the workspace kda_chunk_fwd and
 * kda_chunk_fwd_logits take for the concurrent and split tensor-core forms: 32 KiB per
 * (chunk slot, head) for (ceil(B * T / 64) + N) slots, N = n_seqs in varlen mode
 * (n_seqs > 0), else B, then a 4-byte flag per (slot, head) and a 4-byte progress
 * word per (sequence, head), each array 256-byte aligned.  0 for arguments no call
 * accepts.  Host only; launches nothing.
 */
size_t kda_chunk_workspace_size(int B, int T, int H, int n_seqs);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd for callers that cannot allocate device memory.
 *
 * The concurrent and split tensor-core prefill forms keep chunks' state-independent
 * operands in scratch memory between their two kernels, and kda_chunk_fwd takes that
 * scratch from the caller as a workspace.  Some callers have no way to provide one: code behind a
 * fixed operator or plugin interface that passes only input and output tensors, and
 * code that runs where device allocation is not allowed or not possible (a memory
 * pool owned by another component, a latency-critical path that must not allocate).
 * This entry point takes the same arguments as kda_chunk_fwd without the workspace
 * and uses a fixed 64 MiB array in the library's own device memory instead.  It makes
 * no allocation of any kind: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 *   - Limit: a call may need at most 64 MiB of scratch, i.e. 2048 (chunk slot, head)
 *     blobs of 32 KiB (kda_chunk_workspace_size gives a call's need); for example one
 *     prompt of up to 1280 tokens at 96 heads.  A larger call returns
 *     KDA_ERR_UNSUPPORTED with a message giving both sizes, and launches nothing.
 *   - The array exists on every GPU that loads the library and stays there until the
 *     process exits.  The first call on a device, with that device current, looks up
 *     the array's device address (cudaGetSymbolAddress, once per device); make that
 *     first call before any stream capture.
 *   - Every call shares the one array and leaves its contents behind.  Nothing in it
 *     needs to start at zero: a call clears the flags it uses itself and writes every
 *     other byte before reading it.  Calls whose work can overlap on the GPU
 *     (different streams, different host threads) race on the array and must be
 *     ordered by the caller.
 *   - Results are identical to kda_chunk_fwd with a workspace (the same kernels).
 * No counterpart on the pages: it is an interface for a class of callers.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                 const float *g, const float *beta, const float *initial_state,
                                 float *final_state, void *o, kda_dtype o_dtype,
                                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int n_seqs,
                                 int B, int T, int H, int K, int V, int chunk, float scale,
                                 int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                 const float *norm_w, float eps, void *y, int mode, void *stream);

/*
 * kda_chunk_fwd_logits -- kda_chunk_fwd with the decay and the write strength
 * computed inside the kernels from the logits the layer's projections produce,
 * instead of read as fp32 g and beta (halves the g traffic with bf16 logits).
 *
 * Pages: Kimi-K3 atlas "gate-project (decode, P = 1000)", section "Code" (the
 * layer holds A_log = log U(1, 16) per head, f_a_proj / f_b_proj producing one
 * decay logit per key channel of each head, dt_bias with one bias per such logit,
 * b_proj with one write-strength logit per head, gate_lower_bound); nnterp
 * encyclopedia "Kimi-Linear", section 03 (g per key channel, fp32, non-positive;
 * beta = sigmoid(b_proj)).  The line combining them is not on the pages; this
 * library reads it as
 *     g[t][h][c] = max(g_lower_bound, -exp(A_log[h]) * softplus(g_logits[t][h][c] + dt_bias[h][c]))
 *     beta[t][h] = sigmoid(beta_logits[t][h])
 *
 *   g_logits    [B, T, H, K] g_logits_dtype     A_log [H] float
 *   dt_bias     [H, K] float or NULL (zero)     g_lower_bound <= 0; -INFINITY for none
 *   beta_logits [B, T, H] beta_logits_dtype
 * Everything else as kda_chunk_fwd.
 */
kda_status kda_chunk_fwd_logits(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                kda_dtype beta_logits_dtype, const float *initial_state, float *final_state,
                                void *o, kda_dtype o_dtype, const int32_t *cu_seqlens,
                                const int32_t *cu_seqlens_host, int n_seqs, int B, int T, int H, int K, int V,
                                int chunk, float scale, int use_qk_l2norm, const void *gate,
                                kda_dtype gate_dtype, const float *norm_w, float eps, void *y, void *workspace,
                                size_t workspace_bytes, int mode, void *stream);

/*
 * kda_chunk_fwd_host / kda_chunk_fwd_logits_host -- kda_chunk_fwd (_logits) for a
 * caller whose tensors are in HOST memory: a dense prompt (B sequences of T tokens)
 * streamed through the device in segments of `segment` tokens.
 *
 * Page: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (the chunked kernel
 * carries the state from one 64-token chunk to the next; a segment boundary is a
 * chunk boundary, so the outputs equal those of one kda_chunk_fwd call on device
 * copies of the same tensors, bit for bit).
 *
 * Every tensor argument -- q, k, v, g, beta (or g_logits, beta_logits, A_log,
 * dt_bias), initial_state, final_state, o, gate, norm_w, y -- is a HOST pointer with
 * the layout of kda_chunk_fwd (dense only: no cu_seqlens).  Page-locked memory
 * (cudaHostAlloc / cudaHostRegister) lets the copies overlap the kernels; pageable
 * memory works, with copies that do not overlap.  Outputs must not overlap inputs.
 *
 *   segment    tokens per segment, a multiple of 64; 0 = 1024.
 *   workspace  DEVICE memory of at least kda_chunk_fwd_host_workspace_size(B, H, K,
 *              V, segment) bytes, 256-byte aligned: the state, two buffers of each
 *              tensor's segment, the small parameters.  Owned by the caller; in use
 *              until `stream` reaches the end of the call.
 *   stream     the caller's stream: the kernels run on it, the copies on two streams
 *              the call creates and destroys, and `stream` waits for the last copy, so
 *              the outputs are in host memory once `stream` has completed
 *              (cudaStreamSynchronize).  The host buffers must stay valid until then.
 * Other arguments and errors as kda_chunk_fwd.
 */
size_t kda_chunk_fwd_host_workspace_size(int B, int H, int K, int V, int segment);

kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v, kda_dtype qkv_dtype, const float *g,
                              const float *beta, const float *initial_state, float *final_state, void *o,
                              kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk, float scale,
                              int use_qk_l2norm, const void *gate, kda_dtype gate_dtype, const float *norm_w,
                              float eps, void *y, int segment, void *workspace, size_t workspace_bytes, int mode,
                              void *stream);

kda_status kda_chunk_fwd_logits_host(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                     const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                     const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                     kda_dtype beta_logits_dtype, const float *initial_state, float *final_state,
                                     void *o, kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk,
                                     float scale, int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                     const float *norm_w, float eps, void *y, int segment, void *workspace,
                                     size_t workspace_bytes, int mode, void *stream);

/*
 * kda_recurrent_fwd -- the token-by-token form over T tokens (fp32 arithmetic).
 *
 * Pages: nnterp "Kimi-Linear" section 03 "Loading" (the token-by-token kernel;
 * the per-token `states` readout needs it) and section 02 (`state` / `states`
 * [batch seq heads key_dim value_dim]).
 *
 * Same arguments and layouts as kda_chunk_fwd, without chunk and mode, plus
 *   states [B, T, H, K, V] float or NULL: the state after every token (varlen:
 *          [1, T, H, K, V] indexed by packed token).
 */
kda_status kda_recurrent_fwd(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                             const float *g, const float *beta, const float *initial_state,
                             float *final_state, void *o, kda_dtype o_dtype, float *states,
                             const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                             int n_seqs, int B, int T, int H, int K, int V, float scale,
                             int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                             const float *norm_w, float eps, void *y, void *stream);

/*
 * kda_recurrent_step -- one decode token per sequence, gated norm fused.
 *
 * Pages: nnterp "Kimi-Linear" section 03 "Loading" (a decode step runs the
 * token-by-token kernel); Kimi-K3 atlas "gate-project (decode, P = 1000)"
 * (decode shapes [B, 96, 1, 128] in, [B, 1, 12288] after the flatten).
 *
 *   q, k  [B, H, K] qkv_dtype     v [B, H, V] qkv_dtype
 *   g     [B, H, K] float         beta [B, H] float
 *   state_in  [B, H, K, V] float or NULL (zero state)
 *   state_out [B, H, K, V] float; may be the same buffer as state_in (in place)
 *   o     [B, H, V] o_dtype or NULL when y is given
 *   gate  [B, H, V] gate_dtype or NULL; norm_w [V]; eps; y [B, H * V] o_dtype
 * Supported K, V: 32, 64, 128.
 */
kda_status kda_recurrent_step(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                              const float *g, const float *beta, const float *state_in,
                              float *state_out, void *o, kda_dtype o_dtype, int B, int H, int K,
                              int V, float scale, int use_qk_l2norm, const void *gate,
                              kda_dtype gate_dtype, const float *norm_w, float eps, void *y,
                              void *stream);

/*
 * kda_recurrent_step_logits -- kda_recurrent_step with g and beta computed from
 * their logits, as kda_chunk_fwd_logits defines them:
 *   g_logits [B, H, K] g_logits_dtype, A_log [H], dt_bias [H, K] or NULL,
 *   g_lower_bound, beta_logits [B, H] beta_logits_dtype.
 */
kda_status kda_recurrent_step_logits(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                     const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                     const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                     kda_dtype beta_logits_dtype, const float *state_in, float *state_out,
                                     void *o, kda_dtype o_dtype, int B, int H, int K, int V, float scale,
                                     int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                     const float *norm_w, float eps, void *y, void *stream);

/*
 * kda_recurrent_step_conv -- the decode step with the q, k and v short
 * convolutions (+ SiLU) fused ahead of it, in one kernel.
 *
 * Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Kimi Delta Attention
 * decays each key channel" (a width-4 convolution before the delta rule, whose
 * last inputs are carried outside the recurrent state) and section "Printout"
 * (depthwise Conv1d, kernel 4, padding 3, no bias); Kimi-K3 atlas "gate-project
 * (decode, P = 1000)", section "Code" (q_conv1d, k_conv1d, v_conv1d =
 * ShortConvolution(..., activation='silu') applied to the projections).
 *
 * As kda_recurrent_step (or kda_recurrent_step_logits: give exactly one of the
 * pairs g, beta / g_logits, beta_logits with A_log; the other pointers NULL), but
 *   q, k  [B, H, K] qkv_dtype, v [B, H, V] qkv_dtype are the RAW projections of
 *         this token; the step uses silu(conv(.)) of each, then (optionally) the
 *         L2 norm of q and k, as the layer does.
 *   conv_weight[f]    [H*128, W] float: f = 0 for q, 1 for k, 2 for v (the Conv1d
 *                     weight [D, 1, W] without its middle axis); no bias.
 *   conv_state_in[f]  [B, W-1, H*128] float: the W-1 raw inputs before this token,
 *                     oldest first, as kda_short_conv_fwd keeps them; the array
 *                     pointer NULL (or all three entries NULL) = zero history.
 *   conv_state_out[f] [B, W-1, H*128] float, required: the new history (the old
 *                     one shifted by this token).  Each may be conv_state_in[f]
 *                     itself (in place); no other overlap is allowed.
 * conv_weight, conv_state_in and conv_state_out are HOST arrays of three device
 * pointers, read during the call only.  The convolution output stays in fp32 in
 * the kernel (no rounding to qkv_dtype between the two steps).  Supported: K = V =
 * 128, W in {2, 3, 4}; other shapes return KDA_ERR_UNSUPPORTED.  Returns a kda_status.
 */
kda_status kda_recurrent_step_conv(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                   const float *const conv_weight[3], int W,
                                   const float *const conv_state_in[3], float *const conv_state_out[3],
                                   const float *g, const float *beta,
                                   const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                   const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                   kda_dtype beta_logits_dtype, const float *state_in, float *state_out,
                                   void *o, kda_dtype o_dtype, int B, int H, int K, int V, float scale,
                                   int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                   const float *norm_w, float eps, void *y, void *stream);

/*
 * kda_gated_rmsnorm -- the head-wise sigmoid-gated RMSNorm on its own.
 *
 * Page: Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters"
 * and "Code".
 *   o    [rows, H, V] o_dtype       gate [rows, H, V] gate_dtype
 *   w    [V] float                  y    [rows, H * V] y_dtype
 *   y = o / sqrt(mean_v(o^2) + eps) * w * sigmoid(gate); rows may be 0.
 * Supported V: 32, 64, 128.
 */
kda_status kda_gated_rmsnorm(const void *o, kda_dtype o_dtype, const void *gate,
                             kda_dtype gate_dtype, const float *w, float eps, void *y,
                             kda_dtype y_dtype, int64_t rows, int H, int V, void *stream);

/*
 * kda_short_conv_fwd -- causal depthwise short convolution along the sequence,
 * with an optional SiLU: the preprocessing of q, k and v before the delta rule.
 *
 * Pages: nnterp encyclopedia "Kimi-Linear", section "Printout" (the layer's conv1d
 * is Conv1d(12288, 12288, kernel_size=(4,), padding=(3,), groups=12288,
 * bias=False): one filter per channel, padded by 3 before the first token, the
 * first T outputs kept); Kimi-K3 atlas "gate-project (decode, P = 1000)", section
 * "Code" (q_conv1d, k_conv1d, v_conv1d = ShortConvolution(hidden_size,
 * kernel_size=short_conv_kernel_size = 4, activation='silu')).
 *
 *   y[t][c] = act( bias[c] + sum_{w<W} weight[c][w] * x[t - (W-1) + w][c] )
 *
 * Positions before a sequence read its conv state (the W-1 inputs before it,
 * oldest first) or zero; act is SiLU (z / (1 + e^-z)) when activation = 1, the
 * identity when 0.
 *
 * Dense mode (cu_seqlens == NULL): N = B sequences of T tokens.
 *   x       [B, T, D] x_dtype      y [B, T, D] y_dtype (must not overlap x)
 *   weight  [D, W] float (the Conv1d weight [D, 1, W] without its middle axis)
 *   bias    [D] float or NULL
 *   conv_state_in  [N, W-1, D] float or NULL (zero history)
 *   conv_state_out [N, W-1, D] float or NULL: the last W-1 inputs of each
 *                  sequence, oldest first (a sequence shorter than W-1 keeps part
 *                  of its old state).  It may be the same buffer as
 *                  conv_state_in only for a decode step (dense, T = 1); otherwise
 *                  the two must not overlap.
 * Varlen mode: as kda_chunk_fwd (B = 1, T packed, cu_seqlens device int32
 *   [n_seqs + 1], optional host copy cu_seqlens_host, which is then checked).
 * A decode step is T = 1 with both states given.  Supported: W in {2, 3, 4},
 * D a multiple of 8, B * T <= INT32_MAX.  Returns a kda_status.
 */
kda_status kda_short_conv_fwd(const void *x, kda_dtype x_dtype, const float *weight, const float *bias,
                              const float *conv_state_in, float *conv_state_out, void *y,
                              kda_dtype y_dtype, const int32_t *cu_seqlens,
                              const int32_t *cu_seqlens_host, int n_seqs, int B, int T, int D, int W,
                              int activation, void *stream);

/*
 * kda_o_proj -- the layer's output projection applied to the gated-norm output y.
 *
 * Page: Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters"
 * (output projection: 88,080,384 weights = 12288 inputs x 7168 outputs) and "Code"
 * (o = o_proj(o) after o_norm and the heads flattened to heads * head_dim).
 *
 *   out[r][n] = sum_c y[r][c] * w_o[n][c]            (nn.Linear, no bias)
 *
 *   y     [rows, in_features] bf16 (the y of kda_chunk_fwd / kda_recurrent_step with a
 *         bf16 output dtype)
 *   w_o   [out_features, in_features] bf16 (the nn.Linear weight layout)
 *   out   [rows, out_features] out_dtype; must not overlap y or w_o
 * A dense GEMM on the tensor cores (this library's own tcgen05 kernel, bf16 operands,
 * fp32 accumulation, one rounding to out_dtype).  in_features must be a multiple of
 * 64 and out_features of 128 (KDA_ERR_UNSUPPORTED otherwise); rows may be 0.  Keeps
 * no state between calls.
 */
kda_status kda_o_proj(const void *y, const void *w_o, void *out, kda_dtype out_dtype, int64_t rows,
                      int in_features, int out_features, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
