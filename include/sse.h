/*
 * sse.h -- C ABI of libsse, a GB300 (sm_103a) CUDA library for the Sparse
 * State Expansion (SSE) linear-attention layer.
 *
 * Method: "Scaling Linear Attention with Sparse State Expansion" (arXiv
 * 2507.16577; close-reading notes, sections 2.3-2.6).  Per token t and head
 * h, with N routed partition states S_i (each c x d, key rows by value
 * columns) and one always-on shared state S_N:
 *
 *   e_t  = softmax(router_logits_t)              over the N partitions (eq. 9)
 *   T_t  = the top_k partitions by logit, equal logits ordered by
 *          ascending partition index                                  (eq. 10)
 *   a_t  = exp(log_gate_t), one decay per key row (diagonal gate, eq. 6)
 *   S_i <- diag(a_t) S_i + e_t[i] k_t^T v_t      for i in T_t         (eq. 13)
 *   S_i    unchanged (no write, no decay)        for i not in T_t
 *   S_N <- diag(a_t) S_N + ks_t^T v_t            (shared, section 2.5)
 *   o_t  = sum_{i in T_t} e_t[i] (scale q_t) S_i + (scale qs_t) S_N   (eq. 14)
 *
 * e_t is the full-N softmax (not renormalised over T_t).  k_t is taken as
 * given (the caller applies the key softmax of eq. 12); q is linear.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - All array pointers are DEVICE pointers owned by the caller.  The library
 *   allocates no device or host memory, keeps no state between calls and
 *   never synchronizes the stream (except sse_read_device_status and
 *   sse_get_last_device_error).  Calls are
 *   asynchronous on `stream` (NULL = legacy default stream) and thread-safe.
 * - Token tensors are packed over all sequences, head-interleaved, row-major:
 *   q, k, log_gate, q_shared, k_shared : [total_tokens, H, c]
 *   v, out                             : [total_tokens, H, d]
 *   router_logits                      : [total_tokens, H, N]
 *   in the dtype of cfg->dtype (float32 or bfloat16); out has that dtype too.
 * - States are float32 [num_seqs, H, P, c, d] with P = N + use_shared; slot N
 *   is the shared partition.
 * - cu_seqlens is a device int32 array [num_seqs + 1]: cu_seqlens[0] = 0,
 *   non-decreasing, cu_seqlens[num_seqs] = total_tokens (zero-length
 *   sequences allowed).  The host passes num_seqs and total_tokens for sizing;
 *   the device values are trusted, not checked.
 * - Arguments are validated on the host before any launch; a rejected call
 *   launches nothing and returns SSE_ERR_INVALID_ARG / SSE_ERR_UNSUPPORTED /
 *   SSE_ERR_WORKSPACE.  SSE_ERR_CUDA reports a launch error (the CUDA error is
 *   left to cudaGetLastError of the caller's runtime).
 * - Every token-tensor pointer must be 16-byte aligned; c and d must make a
 *   row a multiple of 16 bytes.
 */
#ifndef SSE_H
#define SSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, without including the CUDA headers. */
typedef struct CUstream_st *sse_stream_t;

typedef enum {
    SSE_OK = 0,
    SSE_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, top_k out of range */
    SSE_ERR_UNSUPPORTED = 2, /* well-formed but not supported (c, d, N, dtype, algo) */
    SSE_ERR_WORKSPACE = 3,   /* workspace null, misaligned (256 B) or too small */
    SSE_ERR_CUDA = 4,        /* a kernel launch failed */
    SSE_ERR_DEVICE = 5,      /* a device-side check failed (sse_read_device_status) */
    SSE_ERR_DEVICE_TIMEOUT = 6 /* a bounded wait inside a kernel expired: the affected work
                                  stopped early and its results are invalid */
} sse_status_t;

typedef enum { SSE_F32 = 0, SSE_BF16 = 1 } sse_dtype_t;

/* Forward algorithm selection (cfg->algo). */
typedef enum {
    SSE_ALGO_AUTO = 0,      /* tensor-core chunked path where supported, else recurrent */
    SSE_ALGO_CHUNKED = 1,   /* tcgen05 chunked path: bf16, c in {64,128}, d in {64,128} */
    SSE_ALGO_RECURRENT = 2, /* CUDA-core per-token recurrence: any supported dtype/shape */
    SSE_ALGO_MASKED = 3     /* tcgen05 chunked path on the masking schedule ("Scaling Linear
                               Attention with Sparse State Expansion", section 2.6, short
                               sequences): every routed partition runs over the whole
                               sequence; tokens it did not select add nothing and leave its
                               state undecayed.  Same results as the grouped (varlen)
                               schedule, no token->partition sort; same shapes as CHUNKED. */
} sse_algo_t;

typedef struct {
    int32_t num_heads;      /* H >= 1 */
    int32_t key_dim;        /* c: query/key width = rows of every state */
    int32_t value_dim;      /* d: value width = columns of every state */
    int32_t num_partitions; /* N routed partitions, 1..64 */
    int32_t top_k;          /* k selected per token and head, 1..min(N, 8) */
    int32_t use_shared;     /* 0 or 1: the always-on shared partition (slot N) */
    float scale;            /* multiplies q and q_shared at the read (1.0 = none) */
    int32_t dtype;          /* sse_dtype_t of all token tensors and of out */
    int32_t algo;           /* sse_algo_t, forward only */
} sse_config_t;

/* Version of this ABI (incremented on any incompatible change). */
int32_t sse_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *sse_status_string(sse_status_t status);

/* ---------------------------------------------------------------------------
 * sse_route -- router and token->partition grouping (eqs. 9-10; the varlen
 * grouping of section 2.6 that gathers, per sequence and partition, the
 * tokens routed to it in their original time order).
 *
 * Outputs (device, caller-owned, fully overwritten):
 *   topk_idx [total_tokens, H, k] int32  selected partitions, descending logit,
 *                                        equal logits by ascending index
 *   topk_w   [total_tokens, H, k] float  e_t at those partitions (fp32 softmax)
 *   seg_off  [num_seqs*H*N + 1]   int32  start of segment s = (b*H + h)*N + i
 *                                        in perm; seg_off[last] = H*k*total_tokens
 *   perm     [H*k*total_tokens]   int32  token indices of each segment, ascending
 * topk_w, seg_off and perm may be NULL (not written).  The grouping is exact
 * (integer) and deterministic.  Workspace: sse_route_workspace_size bytes,
 * 256-byte aligned, contents undefined on entry and exit.
 * ------------------------------------------------------------------------- */
size_t sse_route_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs);

sse_status_t sse_route(const sse_config_t *cfg, const void *router_logits,
                       const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t *topk_idx, float *topk_w, int32_t *seg_off, int32_t *perm,
                       void *workspace, size_t workspace_bytes, sse_stream_t stream);

/* sse_route_noalloc -- sse_route for callers that cannot allocate device
 * memory (a plugin inside a host application that owns every device
 * allocation, a latency-critical loop that cannot afford the device-wide
 * synchronisation of cudaMalloc, a language without a CUDA allocator
 * binding).  The source paper has no counterpart; this is an interface
 * convenience.  Same arguments, outputs and results as sse_route, without the
 * workspace: the routing scratch lives in a 4 MiB array inside the library's
 * device image, reserved on every GPU that loads the library until the
 * process exits.  Limit: (num_seqs + 1) + 4 B + H * N * (B + 1) int32
 * entries, B = ceil(total_tokens / 256) + num_seqs (plus 256-byte alignment
 * padding), must fit in 4 MiB -- about one million tokens at H = 16, N = 16;
 * larger calls return
 * SSE_ERR_WORKSPACE before any launch.  The configuration and size checks are
 * those of sse_route (same status for the same bad argument).  Every call
 * looks up the array's device address in the current device's context (a
 * host-side query, never cached, so a device reset or another context on the
 * same device is safe); the first call on a device also loads the array, so
 * make that first call before any stream capture.  Nothing is allocated or
 * freed.  All calls on a device share the array and it keeps the previous
 * call's contents (no entry needs to start at zero); calls that overlap on
 * the GPU race on it and must be serialised. */
sse_status_t sse_route_noalloc(const sse_config_t *cfg, const void *router_logits,
                               const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                               int32_t *topk_idx, float *topk_w, int32_t *seg_off, int32_t *perm,
                               sse_stream_t stream);

/* ---------------------------------------------------------------------------
 * sse_forward -- the SSE layer over packed varlen sequences (eqs. 9-14 and
 * the shared partition of section 2.5), computed per (sequence, head,
 * partition) segment in chunks (section 2.6, varlen schedule), with the
 * gated sum of the partial read-outs scattered back to token order.
 *
 *   q_shared, k_shared  may be NULL: the shared partition then reads q, k.
 *   initial_state       may be NULL: all states start at zero.
 *   final_state         may be NULL: not written.  May alias initial_state.
 *   out                 [total_tokens, H, d] in cfg->dtype.
 *   topk_idx, topk_w    may be NULL; when given they receive the routing of
 *                       every token (same contents as sse_route).
 * Workspace: sse_forward_workspace_size bytes (256-byte aligned).
 * Numerics: float32 states and accumulation.  The chunked path rounds its
 * tensor-core operands to bfloat16 and splits the decay factors of each
 * 128-row chunk of a segment around its midpoint, which takes the summed
 * log-gate of each half chunk to stay above -64 per key row.  A segment with a
 * chunk past that (strong decays: e.g. log-gates of -2 on every row) is
 * recomputed in the same call, token by token in float32 on the CUDA cores,
 * so every decay in (0, 1] gives a valid result; sse_read_device_status then
 * reports the informational SSE_DEVICE_RECOMPUTED bit.  The range check takes
 * the log-gates to be <= 0 (decays in (0, 1], as in the method); positive
 * log-gates are outside the method and not checked.
 * ------------------------------------------------------------------------- */
size_t sse_forward_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs);

sse_status_t sse_forward(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                         const void *log_gate, const void *router_logits,
                         const void *q_shared, const void *k_shared,
                         const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                         const float *initial_state, float *final_state, void *out,
                         int32_t *topk_idx, float *topk_w,
                         void *workspace, size_t workspace_bytes, sse_stream_t stream);

/* sse_forward with timing hooks and a launch count (for benchmarks).
 * stage_events (NULL = none): four caller-created cudaEvent_t handles, each
 * recorded on `stream`: [0] before the first launch, [1] after the routing and
 * grouping kernels, [2] after the main segment kernel, [3] after the last
 * kernel.  num_launches (NULL = none) receives the number of kernels the call
 * launched.  Everything else is exactly sse_forward. */
sse_status_t sse_forward_timed(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                               const void *log_gate, const void *router_logits,
                               const void *q_shared, const void *k_shared,
                               const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                               const float *initial_state, float *final_state, void *out,
                               int32_t *topk_idx, float *topk_w,
                               void *workspace, size_t workspace_bytes, sse_stream_t stream,
                               void *const *stage_events, int32_t *num_launches);

/* ---------------------------------------------------------------------------
 * sse_decode_step -- one token per sequence on states resident in device
 * memory (section 2.6: decoding recurs only on the selected states).  Reads
 * and rewrites, in place, only the top_k selected states and the shared
 * state of each (sequence, head); every other state is left untouched.
 *
 *   q, k, log_gate, q_shared, k_shared : [batch, H, c]
 *   v, out                              : [batch, H, d]
 *   router_logits                       : [batch, H, N]
 *   state   [batch, H, P, c, d] float32, updated in place
 *   topk_idx, topk_w  [batch, H, k], may be NULL
 * No workspace.  cfg->algo is ignored.
 * ------------------------------------------------------------------------- */
sse_status_t sse_decode_step(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                             const void *log_gate, const void *router_logits,
                             const void *q_shared, const void *k_shared, int32_t batch,
                             float *state, void *out, int32_t *topk_idx, float *topk_w,
                             sse_stream_t stream);

/* ---------------------------------------------------------------------------
 * sse_backward -- gradients of the SSE layer (eqs. 9-14 and the shared
 * partition of section 2.5) for L = <d_out, out> + <d_final_state,
 * final_state>, the forward of sse_forward with the same arguments.  The
 * router weight e_t[i] receives gradient from both the write and the read
 * (section 2.3: the same e_t[i] appears in eq. 13 and eq. 14) and flows to the
 * logits through the softmax over all N partitions; the top-k selection is
 * piecewise constant and carries none.
 *
 *   d_out          [total_tokens, H, d] in cfg->dtype
 *   d_final_state  float32 [num_seqs, H, P, c, d], may be NULL (zero)
 *   dq, dk, d_log_gate [total_tokens, H, c]; dv [total_tokens, H, d];
 *   d_router_logits [total_tokens, H, N]: all in cfg->dtype, fully written
 *   dq_shared, dk_shared  [total_tokens, H, c]: given exactly when q_shared /
 *                  k_shared are; with NULL q_shared the shared partition's
 *                  query gradient is added into dq (likewise dk)
 *   d_initial_state float32 [num_seqs, H, P, c, d], may be NULL (not written)
 * The routing is recomputed from router_logits.  Every (token, head) gets
 * one contribution per selected partition and one from the shared
 * partition (dq, dk, dv in cfg->dtype, d_log_gate in float32), summed in
 * float32 in a fixed order (deterministic).
 *
 * Two computations, chosen by cfg->algo:
 *  - chunked (SSE_ALGO_AUTO, SSE_ALGO_CHUNKED, SSE_ALGO_MASKED; bf16, c = 128,
 *    d in {64, 128}): chunks of 128 grouped rows on the tensor cores -- each
 *    chunk's state contributions, a scan over the chunks in float32, then the
 *    chunk's gradient products (bf16 operands, float32 accumulation) with the
 *    decay referenced to the chunk's midpoint row.  A work item with a chunk
 *    whose summed log-gate leaves that form's range (|G_m| or |G_l - G_m| above
 *    64) is recomputed token by token, as below.  SSE_ALGO_CHUNKED on another
 *    shape returns SSE_ERR_UNSUPPORTED.
 *  - recurrent (SSE_ALGO_RECURRENT, and AUTO / MASKED on other shapes): token
 *    by token in float32 on the CUDA cores, any shape the recurrent forward
 *    takes.
 * Workspace: sse_backward_workspace_size bytes (256-byte aligned); the chunked
 * form adds about 192 KB per chunk of 128 grouped rows (states, their
 * gradients and the bf16 operand tiles) plus 16 MB of per-CTA scratch.
 * ------------------------------------------------------------------------- */
size_t sse_backward_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs);

sse_status_t sse_backward(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                          const void *log_gate, const void *router_logits,
                          const void *q_shared, const void *k_shared,
                          const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                          const float *initial_state, const void *d_out, const float *d_final_state,
                          void *dq, void *dk, void *dv, void *d_log_gate, void *d_router_logits,
                          void *dq_shared, void *dk_shared, float *d_initial_state,
                          void *workspace, size_t workspace_bytes, sse_stream_t stream);

/* ---------------------------------------------------------------------------
 * sse_delta_forward / sse_delta_decode_step -- SSE on a gated delta-rule
 * transition: the close-reading notes of "Scaling Linear Attention with
 * Sparse State Expansion" name Gated DeltaNet's structured transition
 * (section 2.1, eq. 6) as the alternative to GLA's diagonal decay and the
 * combination as future work (section 6); DeltaNet's update is on the
 * "动态线性注意力" page (section 2.1, eq. 4).  Same router, grouping, shared
 * partition and read-out as sse_forward; the state update of a selected
 * partition i becomes
 *   S_i <- alpha_t (I - e_t[i] beta_t k_t^T k_t) S_i + e_t[i] beta_t k_t^T v_t
 * (the router weight scales the delta write), the shared one the same with
 * weight 1, unselected partitions untouched.  alpha_t = exp(log_alpha_t) and
 * beta_t are one scalar each per (token, head); the caller normalises the
 * keys (DeltaNet takes unit keys).
 *
 *   log_alpha, beta   [total_tokens, H] (decode: [batch, H]) in cfg->dtype
 *   everything else   as sse_forward / sse_decode_step
 * Forward, two computations chosen by cfg->algo:
 *  - chunked (every algo but SSE_ALGO_RECURRENT; bf16, c = d = 128): chunks
 *    of 128 rows on the tensor cores -- the chunk's write strengths solved as
 *    a unit lower-triangular system (its inverse in float32 up to 64-row
 *    blocks, the rest by bf16 tensor-core products), bf16 operands, float32
 *    accumulation and a float32 state held on chip for each segment;
 *  - token by token in float32 on the CUDA cores (SSE_ALGO_RECURRENT and every
 *    other shape).
 * The decode step is token by token in float32.  Read-outs are summed per
 * (token, head) in a fixed order.  Shapes: d in {16, 32, 64, 128, 256},
 * c <= 256 (and c <= 4 * 256 * 16 / d).  Workspace (forward only):
 * sse_delta_forward_workspace_size bytes, 256-byte aligned; its first word is
 * the status word sse_read_device_status reads (SSE_DEVICE_TIMEOUT when a
 * bounded wait of the chunked form ran out).
 * ------------------------------------------------------------------------- */
size_t sse_delta_forward_workspace_size(const sse_config_t *cfg, int64_t total_tokens, int32_t num_seqs);

sse_status_t sse_delta_forward(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                               const void *log_alpha, const void *beta, const void *router_logits,
                               const void *q_shared, const void *k_shared,
                               const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                               const float *initial_state, float *final_state, void *out,
                               int32_t *topk_idx, float *topk_w,
                               void *workspace, size_t workspace_bytes, sse_stream_t stream);

sse_status_t sse_delta_decode_step(const sse_config_t *cfg, const void *q, const void *k, const void *v,
                                   const void *log_alpha, const void *beta, const void *router_logits,
                                   const void *q_shared, const void *k_shared, int32_t batch,
                                   float *state, void *out, int32_t *topk_idx, float *topk_w,
                                   sse_stream_t stream);

/* ---------------------------------------------------------------------------
 * sse_front_end -- the layer's projections from the hidden states
 * ("Scaling Linear Attention with Sparse State Expansion", eqs. 9-10; the
 * shared partition's rank-64 Q/K LoRA of section 2.5; GLA's diagonal gate).
 * Per token t and head h, with y = x W^T for each weight W:
 *   q = y_q;  k = softmax(y_k) over the c keys;  v = y_v;
 *   log_gate = logsigmoid(y_g) * gate_inv_tau   (GLA: alpha = sigmoid^(1/tau));
 *   router_logits = y_e  (the router softmax and top-k stay in sse_route /
 *   sse_forward);
 *   with the LoRA factors: q_shared = y_q + (x A_q^T) B_q^T and
 *   k_shared = softmax(y_k + (x A_k^T) B_k^T).
 * The outputs are exactly the token tensors sse_forward and sse_decode_step
 * take.  bf16 only (cfg->dtype == SSE_BF16); fp32 accumulation on the tensor
 * cores; one rounding of x A to bf16 before the LoRA's second factor.
 *
 *   x                  [T, D] bf16 (D = hidden, a multiple of 64, >= 64)
 *   w_q, w_k, w_g      [H*c, D]      w_v [H*d, D]      w_e [H*N, D]
 *   a_q, a_k           [64, D]       b_q, b_k [H*c, 64]   (all four NULL: no LoRA)
 *   q, k, log_gate, q_shared, k_shared [T, H, c]   v [T, H, d]
 *   router_logits      [T, H, N]
 * Weights use the [out_features, in_features] layout (row n holds the D
 * weights of output n).  All pointers are device pointers, 16-byte aligned;
 * q_shared / k_shared are required with the LoRA factors and ignored without.
 * Supported: c, d in {64, 128}; H*N a multiple of 16 and at most 256; T >= 128.
 * Workspace: sse_front_end_workspace_size bytes (256-byte aligned); its first
 * word holds the device-check flags (sse_read_device_status reads them).
 * ------------------------------------------------------------------------- */
size_t sse_front_end_workspace_size(const sse_config_t *cfg, int32_t hidden, int64_t total_tokens);

sse_status_t sse_front_end(const sse_config_t *cfg, int32_t hidden, int64_t total_tokens, const void *x,
                           const void *w_q, const void *w_k, const void *w_v, const void *w_g,
                           const void *w_e, const void *a_q, const void *b_q, const void *a_k,
                           const void *b_k, float gate_inv_tau, void *q, void *k, void *v,
                           void *log_gate, void *router_logits, void *q_shared, void *k_shared,
                           void *workspace, size_t workspace_bytes, sse_stream_t stream);

/* Device-side status bits (bit mask), written by the kernels into the first
 * word of the workspace of sse_forward, sse_backward, sse_delta_forward and
 * sse_front_end (each call clears them first).
 *   SSE_DEVICE_TIMEOUT      error: a bounded wait on the tensor-core pipeline
 *                           expired; the affected segments stopped early and
 *                           the call's results are invalid
 *   SSE_DEVICE_RECOMPUTED   information only: at least one segment had a chunk
 *                           whose summed log-gate left the chunked path's
 *                           factorised range and was recomputed token by token
 *                           (results valid) */
enum { SSE_DEVICE_TIMEOUT = 2, SSE_DEVICE_RECOMPUTED = 4 };

/* Reads the device-status bits of the last sse_forward, sse_backward,
 * sse_delta_forward or sse_front_end that used `workspace`.  Synchronizes `stream`.  *flags receives the bit mask.
 * Returns SSE_ERR_DEVICE_TIMEOUT if the timeout bit is set, SSE_ERR_DEVICE for
 * any other error bit, SSE_OK otherwise (informational bits included), and
 * SSE_ERR_CUDA if the copy fails. */
sse_status_t sse_read_device_status(void *workspace, int32_t *flags, sse_stream_t stream);

/* The status alone: sse_read_device_status without the bit mask
 * ("Scaling Linear Attention with Sparse State Expansion" has no counterpart;
 * this is the failure-detection hook of the library). */
sse_status_t sse_get_last_device_error(void *workspace, sse_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSE_H */
