/*
 * spec_verify.h -- C ABI of libspecverify: batched speculative-decoding
 * verification over vocabulary-sized logits on one GB300 (sm_103a).
 *
 * Operations (source pages, by title and section):
 *   spec_verify_greedy  mini-sglang PR #134 "[Feature] Vanilla speculative
 *                       decoding", Modifications (verify.py): accept the
 *                       longest prefix of the K drafts that matches the
 *                       target argmax over the K+1 verify-pass logits, then
 *                       append the bonus token (argmax of the next row).
 *   spec_verify_sample  spec-decode README, "How it works": accept draft t with
 *                       probability min(1, p(t)/q(t)), stop at the first
 *                       rejection and draw from normalize(relu(p - q)); if all
 *                       K are accepted draw a bonus token from p. nanospec
 *                       README, acceptance rules: exact / relaxed (p >= tau or
 *                       top-k) / power (min(1, p/rest)^alpha), and a target
 *                       log-prob and behaviour probability mu per token.
 *   spec_verify_tree    nanospec README, EAGLE-3 tree configuration (depth 5,
 *                       topk 4): walk a draft tree given by parent indices,
 *                       accepting one root-to-node path.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, except
 *     where a comment says otherwise. The library allocates nothing, keeps no
 *     state between calls and never synchronises the stream.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream). Argument errors the host can see are returned
 *     synchronously and nothing is launched. SV_ERR_CUDA means a launch failed.
 *   - Logit rows: row r of a [rows, V] matrix starts at
 *     base + r * row_stride ELEMENTS (row_stride >= V). bf16 rows need only
 *     2-byte alignment and fp32 rows 4-byte alignment; the kernels handle
 *     rows that do not start on a 16-byte boundary.
 *   - Argmax ties go to the lowest vocabulary index; argmax is taken on raw
 *     logits. Logits may contain -inf (masked tokens). A row whose maximum is
 *     not finite, or that contains NaN, is flagged (SV_STATUS_NONFINITE_ROW)
 *     when the decision reads it, and that request's outputs are unspecified.
 *   - Temperature T scales both p = softmax(x/T) and q = softmax(y/T).
 *     Log-probs are natural-log p_T(token) of the distribution used
 *     (temperature 1 for the greedy rules).
 *   - Output slots after the emitted tokens hold token -1, log-prob 0, mu 0.
 *   - out_logprob, out_mu and out_status may be NULL.
 *   - The workspace (device memory, 16-byte aligned, at least the size the
 *     matching *_workspace_size function returns) needs no initialisation
 *     and may be reused by later calls on the same stream. Two calls that
 *     run concurrently must not share a workspace.
 *   - A device-side problem found in one request sets bits in out_status[b]
 *     (SV_STATUS_*); other requests are unaffected. Kernels never trap; every
 *     wait inside them is bounded (SV_STATUS_TIMEOUT if one gives up).
 *   - Calls are asynchronous, so a wait that gives up inside a kernel cannot
 *     be a return code of the call that launched it: it is the per-request bit
 *     SV_STATUS_TIMEOUT. A caller that reads the status array back can turn it
 *     into the return code SV_ERR_TIMEOUT with spec_verify_check_status.
 *     A wait gives up after 20 ms of polling; time the context spends switched
 *     out (time-slicing, preemption) is not counted beyond 1 ms per gap, so a
 *     preempted call does not time out spuriously. A request with the bit set
 *     has unspecified outputs: re-run the call once; a second timeout means
 *     the device is not making progress and should be treated as failed.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_VERIFY_ABI_VERSION 3

/* Return codes. */
typedef int32_t sv_status;
#define SV_OK                      0
#define SV_ERR_INVALID_ARG         1  /* a pointer, size, stride or parameter is invalid */
#define SV_ERR_UNSUPPORTED_DTYPE   2  /* dtype is neither SV_F32 nor SV_BF16 */
#define SV_ERR_WORKSPACE_TOO_SMALL 3  /* workspace_bytes below the required size */
#define SV_ERR_CUDA                4  /* a CUDA launch or attribute call failed */
#define SV_ERR_NOT_SUPPORTED       5  /* valid request this build does not implement
                                         (no call of this version returns it) */
#define SV_ERR_TIMEOUT             6  /* a bounded wait inside a kernel gave up (returned
                                         only by spec_verify_check_status) */

/* Logit element types. */
#define SV_F32  0
#define SV_BF16 1

/* Acceptance rules (nanospec README, acceptance rules). */
#define SV_RULE_EXACT   0  /* lossless: accept with min(1, p/q) */
#define SV_RULE_RELAXED 1  /* accept iff p >= tau or rank < top_k; mu = 1 on accepted drafts */
#define SV_RULE_POWER   2  /* accept with probability min(1, p/rest)^alpha */

/* Per-request status bits written to out_status[b]. */
#define SV_STATUS_BAD_TOKEN      1   /* a consulted draft / node token is outside [0, V) */
#define SV_STATUS_BAD_PARENT     2   /* parents[0] != -1 or some parents[n] not in [0, n) */
#define SV_STATUS_NONFINITE_ROW  4   /* a consulted row has a non-finite max or a NaN */
#define SV_STATUS_ZERO_MASS      8   /* a draft token with p(t) = q(t) = 0 (rejected) */
#define SV_STATUS_DEPTH_EXCEEDED 16  /* the walk reached max_depth at a node with children */
#define SV_STATUS_TIMEOUT        32  /* a bounded wait in a kernel gave up */
#define SV_STATUS_STOPPED        64  /* finish step: a stop token ended the request */
#define SV_STATUS_CAPPED         128 /* finish step: max_new removed emitted tokens */

/* Rule parameters. tau: relaxed threshold on p. top_k: relaxed rank bound
 * (0 disables it; rank = number of logits strictly greater, so top_k = 1
 * accepts the argmax). alpha > 0: power exponent (alpha = 1 is the exact
 * rule). */
typedef struct sv_rule_params {
  int32_t rule;
  float tau;
  int32_t top_k;
  float alpha;
} sv_rule_params;

/* Optional finish step of the *_ex entry points (mini-sglang PR #134: Known
 * limitations, multi-token stop sets, and engine.py's accept_length /
 * accept_rate counters; spec-decode README CLI: tokens per target pass and
 * acceptance rate). A call emits tokens[0..n]; the request stops at the first
 * emitted token in stop_ids (that token is kept); max_new[b] (clamped at 0)
 * caps the tokens kept; positions kept..n are cleared (token -1, log-prob 0,
 * mu 0, tree node -1) and out_len[b] = kept. num_accepted still reports the
 * rule's n. counters[b] (int64, 4 per request, running totals owned by the
 * caller) gain (1 round, drafts offered = K or max_depth, n, kept): tokens
 * per pass = counters[3] / counters[0], acceptance rate = counters[2] /
 * counters[1]. All pointers are device memory; stop_ids may be NULL when
 * n_stop = 0, max_new and counters may be NULL; out_len is required. The
 * step runs inside the call's last kernel; two calls on the same counters
 * must not overlap on the GPU. */
#define SV_MAX_STOP_IDS 16
typedef struct sv_finish_params {
  const int32_t* stop_ids;   /* [n_stop] token ids */
  int32_t n_stop;            /* 0 .. SV_MAX_STOP_IDS */
  const int32_t* max_new;    /* [B] tokens each request may still emit, or NULL */
  int32_t* out_len;          /* [B] tokens kept */
  int64_t* counters;         /* [B, 4] running totals, or NULL */
} sv_finish_params;

/* Largest top_k the relaxed rule supports. */
#define SV_MAX_TOP_K 16
/* Largest node count a tree may have. */
#define SV_MAX_TREE_NODES 1024

/* ABI version of the loaded library (SPEC_VERIFY_ABI_VERSION). */
int32_t spec_verify_abi_version(void);

/* Static, NUL-terminated description of a return code. */
const char* spec_verify_status_string(sv_status s);

/* Workspace bytes for a call with these sizes; 0 if the sizes are invalid.
 * Pure host functions: they touch no device. */

/* One size for every verification entry point (mini-sglang PR #134,
 * verify_drafts: one buffer serves any call): bytes that suffice for
 * spec_verify_greedy / _greedy_ex / _greedy_early with K = rows_per_req - 1,
 * spec_verify_sample / _sample_ex with K = rows_per_req - 1 (with or without
 * draft logits, any rule), and spec_verify_tree / _tree_ex with
 * N = rows_per_req when rows_per_req <= SV_MAX_TREE_NODES. 0 if B < 0,
 * rows_per_req < 1, V < 1 or dtype is invalid. */
size_t spec_verify_workspace_size(int32_t B, int32_t rows_per_req, int32_t V, int32_t dtype);

size_t spec_verify_greedy_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype);
size_t spec_verify_sample_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype,
                                         int32_t has_draft_logits);
size_t spec_verify_tree_workspace_size(int32_t B, int32_t N, int32_t V, int32_t dtype);

/* Greedy chain verification (mini-sglang PR #134, verify_drafts).
 *   target_logits  [B, K+1, V] rows of `dtype`, row (b, i) at row b*(K+1)+i.
 *   draft_tokens   [B, K] int32, row-major.
 *   B >= 0, K >= 0, V >= 1.
 * Outputs (row-major, B rows):
 *   out_tokens        [B, K+1] int32: d_0..d_{n-1}, argmax(row n), then -1.
 *   out_num_accepted  [B] int32: n, the accepted draft count (n+1 tokens).
 *   out_logprob       [B, K+1] float: log_softmax(row j)[token j] at T = 1.
 *   out_mu            [B, K+1] float: 1 for emitted tokens (deterministic rule).
 *   out_status        [B] int32: SV_STATUS_* bits.
 * A draft outside [0, V) counts as a mismatch and sets SV_STATUS_BAD_TOKEN. */
sv_status spec_verify_greedy(const void* target_logits, int32_t dtype, int64_t row_stride,
                             const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                             int32_t* out_tokens, int32_t* out_num_accepted,
                             float* out_logprob, float* out_mu, int32_t* out_status,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Stochastic chain verification (spec-decode README "How it works";
 * nanospec README rules).
 *   target_logits  [B, K+1, V]; draft_logits [B, K, V] of the same dtype with
 *                  its own row stride, or NULL for deterministic drafts
 *                  (q = one-hot of the draft token).
 *   draft_tokens   [B, K] int32.  temperature: finite, >= 1e-4.
 *   uniforms       [B, K+1] float in [0, 1): column i < K tests draft i
 *                  (accepted iff u < acceptance), column K drives the single
 *                  final draw (residual or bonus), which is the smallest
 *                  index j whose inclusive prefix sum of the weights exceeds
 *                  u * (total weight), in ascending vocabulary order.
 * With draft logits: exact acceptance min(1, p/q); p(t) = q(t) = 0 rejects
 * (SV_STATUS_ZERO_MASS); residual normalize(relu(p - q)), or p when that mass
 * is zero; mu = p(token). The power rule accepts with min(1, p/q)^alpha and
 * the relaxed rule with [p >= tau or rank < top_k]; the residual is the same,
 * and mu_j(a) = q_j(a) acc_j(a) + (1 - sum_s q_j(s) acc_j(s)) res_j(a) for
 * every emitted draft row j (the bonus token after K acceptances keeps
 * mu = p). These two rules add one more pass over rows 0..n of both logit
 * arrays for those sums.
 * Relaxed with top_k > 0 adds a per-row selection of the top_k-th largest
 * logit (rank(t) < top_k iff x_t is at least that value), reading each tested
 * row two (bf16) or four (fp32) more times.
 * Without draft logits (deterministic drafts): exact a = p(d), power
 * a = p(d)^alpha, relaxed a = [p(d) >= tau or rank(d) < top_k]; mu = a for
 * an accepted draft; on rejection the draw is from p with d removed and mu is
 * (1 - a) p(j) / (1 - p(d)).
 * Outputs as for spec_verify_greedy. */
sv_status spec_verify_sample(const void* target_logits, int32_t dtype, int64_t row_stride,
                             const void* draft_logits, int64_t draft_row_stride,
                             const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                             float temperature, const float* uniforms, sv_rule_params rule,
                             int32_t* out_tokens, int32_t* out_num_accepted,
                             float* out_logprob, float* out_mu, int32_t* out_status,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Tree verification (nanospec README, EAGLE-3 tree configuration).
 *   target_logits  [B, N, V]: row n is the target's next-token logits after
 *                  the path root..n (node 0 is the root).
 *   node_tokens    [B, N] int32: token of node n (node 0's is unused).
 *   parents        [B, N] int32: parents[b, 0] = -1, 0 <= parents[b, n] < n.
 *                  A node with an invalid link is ignored (SV_STATUS_BAD_PARENT).
 *   1 <= N <= SV_MAX_TREE_NODES, max_depth >= 0: at most max_depth nodes are
 *   accepted; outputs have max_depth + 1 columns.
 *   temperature == 0 selects the greedy walk (uniforms may be NULL): from the
 *   current node move to the lowest-index child whose token is the argmax of
 *   the current row; stop when none; append the argmax of the last row.
 *   temperature > 0 (>= 1e-4) selects the stochastic walk with `rule`:
 *   children are tested in increasing node index with uniforms[b, c]; with
 *   rest_1 = 1 and rest_{j+1} = rest_j - p(c_j) over rejected distinct tokens,
 *   exact a_j = min(1, p/rest_j), power a_j = min(1, p/rest_j)^alpha, relaxed
 *   a_j = [p >= tau or rank < top_k]; a duplicate of a rejected sibling's
 *   token has a_j = 0. On acceptance the walk descends; when every child is
 *   rejected, or at a leaf, one token is drawn with uniforms[b, 0] from p with
 *   the rejected tokens removed. mu is the probability of the branch taken.
 * Outputs ([B, max_depth+1] unless noted):
 *   out_tokens, out_logprob, out_mu as above; out_nodes: the path node whose
 *   row scored each emitted token (out_nodes[b, 0] = 0; accepted nodes are
 *   out_nodes[b, 1..n]); out_num_accepted [B]; out_status [B]. */
sv_status spec_verify_tree(const void* target_logits, int32_t dtype, int64_t row_stride,
                           const int32_t* node_tokens, const int32_t* parents,
                           int32_t B, int32_t N, int32_t V, int32_t max_depth,
                           float temperature, const float* uniforms, sv_rule_params rule,
                           int32_t* out_tokens, int32_t* out_nodes, int32_t* out_num_accepted,
                           float* out_logprob, float* out_mu, int32_t* out_status,
                           void* workspace, size_t workspace_bytes, void* stream);

/* The three entry points above with the finish step (sv_finish_params);
 * finish = NULL behaves exactly like the plain call. Invalid finish
 * parameters (out_len NULL, n_stop outside 0..SV_MAX_STOP_IDS, stop_ids NULL
 * with n_stop > 0, misaligned pointers) return SV_ERR_INVALID_ARG. */
sv_status spec_verify_greedy_ex(const void* target_logits, int32_t dtype, int64_t row_stride,
                                const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                int32_t* out_tokens, int32_t* out_num_accepted,
                                float* out_logprob, float* out_mu, int32_t* out_status,
                                const sv_finish_params* finish,
                                void* workspace, size_t workspace_bytes, void* stream);
sv_status spec_verify_sample_ex(const void* target_logits, int32_t dtype, int64_t row_stride,
                                const void* draft_logits, int64_t draft_row_stride,
                                const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                float temperature, const float* uniforms, sv_rule_params rule,
                                int32_t* out_tokens, int32_t* out_num_accepted,
                                float* out_logprob, float* out_mu, int32_t* out_status,
                                const sv_finish_params* finish,
                                void* workspace, size_t workspace_bytes, void* stream);
sv_status spec_verify_tree_ex(const void* target_logits, int32_t dtype, int64_t row_stride,
                              const int32_t* node_tokens, const int32_t* parents,
                              int32_t B, int32_t N, int32_t V, int32_t max_depth,
                              float temperature, const float* uniforms, sv_rule_params rule,
                              int32_t* out_tokens, int32_t* out_nodes, int32_t* out_num_accepted,
                              float* out_logprob, float* out_mu, int32_t* out_status,
                              const sv_finish_params* finish,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Early-exit greedy chain verification (mini-sglang PR #134, verify.py: rows
 * after a request's first mismatch never reach the outputs). Same arguments,
 * outputs and workspace size (spec_verify_greedy_workspace_size) as
 * spec_verify_greedy, with identical tokens, num_accepted and status (log-
 * probs agree to rounding: each row is summed by one CTA); the row-statistics kernel
 * reads rows position by position across the batch and stops reading a
 * request's rows once a mismatch at an earlier position is known, so a long
 * chain that is rejected early costs a fraction of its logit bytes.
 *   state           [2B] int32 device array owned by the caller (per request
 *                   the smallest known mismatch, then the rows finished):
 *                   zero-filled before its first use; every call leaves it
 *                   zero again. Calls that overlap on the GPU need separate
 *                   state arrays.
 *   out_bytes_read  [1] uint64 device: logit bytes this call actually read
 *                   (at least the bytes of rows 0..n of every request, at
 *                   most all rows); may be NULL. */
sv_status spec_verify_greedy_early(const void* target_logits, int32_t dtype, int64_t row_stride,
                                   const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                   int32_t* out_tokens, int32_t* out_num_accepted,
                                   float* out_logprob, float* out_mu, int32_t* out_status,
                                   int32_t* state, uint64_t* out_bytes_read,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* EAGLE-style draft-tree construction, the step before spec_verify_tree
 * (nanospec README: EAGLE-3 tree speculation, depth 5, topk 4).
 *   draft_logits  [B, R, V], R = 1 + (depth - 1) * topk draft rows per
 *                 request in rank order: row 0 is the root's; row
 *                 1 + (d - 2) * topk + r belongs to the r-th best node of
 *                 level d - 1 (d = 2..depth).
 *   1 <= topk <= 8 and topk <= V; depth >= 1; the candidate count
 *   topk + (depth - 1) * topk^2 is at most 1024 and R at most 128; 1 <= n_nodes <=
 *   min(1 + candidates, SV_MAX_TREE_NODES); temperature finite, >= 1e-4.
 * A node's score is its path's cumulative draft log-prob
 * (log_softmax(y / T)). Level 1 holds the root row's topk tokens (largest
 * logits, lower id first on ties); each later level expands the topk best
 * nodes of the level above (score descending, earlier candidate first) into
 * the topk tokens of their rows. The n_nodes - 1 best candidates are kept with
 * the root and written in BFS order (level, then score descending, then
 * creation order):
 *   out_tokens [B, n_nodes] (root -1), out_parents [B, n_nodes] (root -1,
 *   parents[n] < n), out_scores [B, n_nodes] (root 0; may be NULL),
 *   out_status [B] (SV_STATUS_NONFINITE_ROW if a used row has no finite
 *   maximum; may be NULL).
 * out_tokens / out_parents feed spec_verify_tree directly. */
size_t spec_tree_build_workspace_size(int32_t B, int32_t depth, int32_t topk, int32_t V);
sv_status spec_tree_build(const void* draft_logits, int32_t dtype, int64_t row_stride,
                          int32_t B, int32_t V, int32_t depth, int32_t topk, int32_t n_nodes,
                          float temperature, int32_t* out_tokens, int32_t* out_parents,
                          float* out_scores, int32_t* out_status,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Accepted-path KV compaction, the step after spec_verify_tree (nanospec
 * README: paged KV cache; mini-sglang PR #134, draft.py: the cache keeps the
 * accepted prefix and the rest is truncated). The verify pass wrote tree node
 * n's key/value row at logical position seq_base[b] + n; logical position p
 * of request b is slot p % page_size of page page_table[b, p / page_size] in
 * a cache of pages of page_size rows, token_stride_bytes apart, each row
 * row_bytes long (both multiples of 16; kv 16-byte aligned). The path
 * path_nodes[b, 0..n] (out_nodes of spec_verify_tree, n = num_accepted[b],
 * path_cols its row length; node ids strictly increasing along the path, as
 * a tree walk writes them, otherwise the moved rows are unspecified) is moved
 * so its j-th node lands at position seq_base[b] + j, in place; rows off the
 * path are untouched; out_len[b] =
 * seq_base[b] + n + 1 (the root and the accepted nodes). A path node outside
 * [0, max_nodes), n outside [0, path_cols), or a page id < 0 or past
 * max_pages leaves the request untouched, out_len[b] = seq_base[b] and
 * out_status[b] = SV_STATUS_BAD_PAGE (out_status may be NULL). Requests must
 * not share pages. All pointers are device memory. */
#define SV_STATUS_BAD_PAGE 256
sv_status spec_kv_compact(void* kv, int64_t token_stride_bytes, int32_t row_bytes,
                          const int32_t* page_table, int32_t max_pages, int32_t page_size,
                          const int32_t* seq_base, const int32_t* path_nodes, int32_t path_cols,
                          const int32_t* num_accepted, int32_t B, int32_t max_nodes,
                          int32_t* out_len, int32_t* out_status, void* stream);

/* Host-side reduction of a status array the caller has copied back to host
 * memory (status_host[0..B-1], the out_status of a finished call):
 * SV_ERR_TIMEOUT if any request has SV_STATUS_TIMEOUT, SV_ERR_INVALID_ARG if
 * status_host is NULL with B > 0 or B < 0, else SV_OK (the other bits are
 * per-request outcomes, not errors). Touches no device. */
sv_status spec_verify_check_status(const int32_t* status_host, int32_t B);

/* Self-test of the kernels' failure path, for health checks: enqueues one
 * one-thread-block kernel that waits on an mbarrier phase nothing completes,
 * with the same bounded wait the verification kernels use. The wait gives up
 * after its limit (about 20 ms), the kernel writes SV_STATUS_TIMEOUT to
 * out_status[0] (device memory, int32) and returns normally, so the context
 * stays usable. No bulk copy or other asynchronous work is outstanding when
 * the kernel exits. Returns SV_ERR_INVALID_ARG for a NULL or misaligned
 * out_status, SV_ERR_CUDA if the launch fails. */
sv_status spec_verify_selftest_wait(int32_t* out_status, void* stream);

/* Bytes of the library's static scratch array used by
 * spec_verify_greedy_static (one array per GPU that loads the library). */
#define SV_STATIC_SCRATCH_BYTES (4u << 20)

/* Greedy chain verification that allocates nothing and takes no workspace.
 * The pages have no counterpart to this entry point: it exists for callers
 * that hold only their input and output buffers and cannot allocate device
 * memory themselves -- plugin hosts that hand a custom op fixed buffers,
 * serving loops that forbid allocation after start-up (an allocation can
 * synchronise the device or fail under memory pressure), or code running
 * while another component owns the allocator.
 * Arguments, outputs and results are exactly those of spec_verify_greedy; the
 * scratch is a file-scope static device array of SV_STATIC_SCRATCH_BYTES,
 * which holds B*(K+1) <= 33353 rows. Larger requests return
 * SV_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address once; make that first call before any stream
 * capture. The address is kept for the life of the process: after
 * cudaDeviceReset (or anything else that destroys the device's primary
 * context) it is stale, and this entry point must not be called again on that
 * device in the same process. Every call shares the one array per device, and it keeps the last
 * call's contents: nothing in it has to start at zero (each call writes all it
 * reads), but two calls whose work overlaps on the GPU (different streams, or
 * concurrent host threads) race on it and must be serialised by the caller. */
sv_status spec_verify_greedy_static(const void* target_logits, int32_t dtype, int64_t row_stride,
                                    const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                    int32_t* out_tokens, int32_t* out_num_accepted,
                                    float* out_logprob, float* out_mu, int32_t* out_status,
                                    void* stream);

/* Greedy chain verification of logits that sit in HOST memory (the same
 * verification as spec_verify_greedy, mini-sglang PR #134, verify_drafts;
 * the transfer schedule is this library's). The requests go to the GPU in
 * groups of `group` (0: the library picks groups of about
 * SV_HOST_GROUP_BYTES of logits): group i is copied into one of two device
 * staging slots on a copy stream of the library's while group i - 1 is
 * verified on `stream`, and each group's outputs are copied back to the host
 * outputs on `stream` after its verification. The copy engine then carries
 * the logits back to back and the kernels run in its shadow.
 *   target_logits, draft_tokens: host memory, laid out as for
 *     spec_verify_greedy (request b's K+1 rows contiguous at row b*(K+1)).
 *     Page-locked (cudaHostAlloc / cudaHostRegister) memory copies at full
 *     speed; pageable memory works but each copy then blocks the host.
 *   out_*: host memory, as for spec_verify_greedy (out_logprob, out_mu,
 *     out_status may be NULL).
 *   workspace: device memory of spec_verify_greedy_host_workspace_size(B, K,
 *     V, dtype, group) bytes, 256-byte aligned; nothing in it needs to start
 *     at zero. Results are the same as spec_verify_greedy's on the same
 *     groups of requests: tokens, counts and status are identical to a
 *     single device call; log-probabilities agree to float rounding.
 * The call returns once the work is enqueued; the host outputs are valid
 * after `stream` completes (cudaStreamSynchronize). Calls on one device
 * share the library's copy stream, and each call orders its copies after
 * the work already enqueued on `stream`. The copy stream is created by the
 * first call on each device (with that device current) and kept for the life
 * of the process; after cudaDeviceReset (or anything else that destroys the
 * device's primary context) it is stale, and this entry point must not be
 * called again on that device in the same process. Errors as for
 * spec_verify_greedy; SV_ERR_CUDA also when the copy stream or an event
 * cannot be created. */
#define SV_HOST_GROUP_BYTES (256ull << 20)
size_t spec_verify_greedy_host_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype,
                                              int32_t group);
sv_status spec_verify_greedy_host(const void* target_logits, int32_t dtype, int64_t row_stride,
                                  const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                  int32_t group, int32_t* out_tokens, int32_t* out_num_accepted,
                                  float* out_logprob, float* out_mu, int32_t* out_status,
                                  void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
