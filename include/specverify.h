/*
 * specverify.h -- C ABI of libspecverify: batched speculative-decoding
 * verification on one GB300 (sm_103a).
 *
 * Source of the method: "Accelerating Sonar through speculation"
 * (Perplexity blog), sections "Speculative decoding", "Target-Draft",
 * "EAGLE", "MTP" and "MTP schedule for a single token", and the rule of the
 * work it cites first, "Fast Inference from Transformers via Speculative
 * Decoding": accept a drafted token x with probability min(1, p(x)/q(x));
 * at the first rejection draw from norm(max(0, p - q)); after a full accept
 * draw a bonus token from the target's last row.
 *
 * Conventions shared by every call:
 *  - Every array argument is a DEVICE pointer owned by the caller, except
 *    `params`, which is a host pointer read before the call returns.  The
 *    library allocates nothing and keeps no state between calls.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and
 *    the call returns without synchronising.  Outputs are valid once the
 *    stream reaches that point.
 *  - Host-detectable errors (NULL required pointer, bad size, unsupported
 *    combination, workspace too small) are returned synchronously and
 *    nothing is enqueued.  SPEC_ERR_CUDA reports a failed launch.
 *  - Data-dependent errors found on the device (token id outside [0, V),
 *    NaN or +inf logits, a row with no finite entry, a malformed parent
 *    array, an out-of-range accepted length) OR a SPEC_DEVERR_* bit into
 *    *dev_error (zeroed by the call first) and give that request a defined
 *    fallback result (see each call).  The library never traps.
 *  - Logit rows are contiguous: element (b, i, v) sits at
 *    ((b * rows + i) * V + v).  V need not be a multiple of 8.
 *  - Random draws use counter-based Philox4x32-10 (Salmon, Moraes, Dror,
 *    Shaw, SC'11): key = (seed lo32, seed hi32), counter = (request lo32,
 *    position lo32, purpose | round << 8, request hi32), u = (word0 >> 8) *
 *    2^-24.  Results depend only on (inputs, seed, request id, position),
 *    not on the batch size or on a request's slot in the batch: bit for bit
 *    when every row starts on a 16-byte boundary (V * element size a
 *    multiple of 16 and 16-byte aligned base pointers); otherwise rows in
 *    different slots are summed in a different order, and only decisions
 *    that sit within rounding of a threshold can differ.
 *  - Calls that overlap on the GPU must not share output or workspace
 *    buffers.
 *  - Each call makes the device that holds its logits (or hidden states)
 *    current for its own launches and puts the caller's current device
 *    back before it returns.
 *  - The linear calls and the draft-side sampler use dependent launches:
 *    a launch may be scheduled while the kernel before it on the stream is
 *    ending, and waits for that kernel to complete before it reads or
 *    writes anything.  Stream order is kept; after any other stream
 *    operation (a copy, an event) they are ordinary launches.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* spec_stream_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,  /* NULL required pointer, negative size, bad params */
    SPEC_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. size limits) */
    SPEC_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than spec_workspace_size() */
    SPEC_ERR_CUDA = 4          /* a CUDA call or kernel launch failed */
} spec_status;

typedef enum { SPEC_BF16 = 0, SPEC_F32 = 1 } spec_dtype;

/* How the children of a draft-tree node were drawn from the draft model
 * (section "EAGLE": Top-K candidates per node).  The residual update after
 * a rejected child depends on it. */
typedef enum {
    SPEC_CHILD_WOR = 0,           /* sampled without replacement */
    SPEC_CHILD_IID = 1,           /* sampled with replacement */
    SPEC_CHILD_DETERMINISTIC = 2  /* the K most likely draft tokens; draft logits unused */
} spec_child_mode;

typedef enum { SPEC_OP_LINEAR = 0, SPEC_OP_TREE = 1 } spec_op;

/* Philox purposes (counter word 2, low byte). */
#define SPEC_PURPOSE_ACCEPT 1
#define SPEC_PURPOSE_RESIDUAL 2
#define SPEC_PURPOSE_BONUS 3
#define SPEC_PURPOSE_DRAFT 4

/* Bits OR-ed into *dev_error. */
#define SPEC_DEVERR_TOKEN 1      /* a draft/node token outside [0, V) */
#define SPEC_DEVERR_NONFINITE 2  /* NaN or +inf logit, or no finite logit in a row */
#define SPEC_DEVERR_PARENT 4     /* parent[] not a tree rooted at 0 with parent[i] < i, deeper than max_depth,
                                    or a node with more than 64 children */
#define SPEC_DEVERR_LENGTH 8     /* compaction: accepted length or source row out of range */
#define SPEC_DEVERR_TIMEOUT 16   /* a wait for a bulk copy ran out (2 s); the rows it left were
                                    recomputed by the two-pass route, so the results stand */

typedef struct {
    float temperature;  /* 0 => greedy (argmax, ties to the lowest index); > 0 => sampled */
    float top_p;        /* in (0, 1): nucleus filter on p and q; >= 1 => off */
    uint64_t seed;      /* Philox key */
    int32_t child_mode; /* spec_child_mode; tree only */
} spec_sampling_params;

/*
 * Bytes of device workspace a call needs (16-byte alignment suffices).
 * op = SPEC_OP_LINEAR: k_or_N = k.  op = SPEC_OP_TREE: k_or_N = N.
 * Returns 0 for invalid sizes.
 */
size_t spec_workspace_size(spec_op op, int B, int k_or_N, int V, spec_dtype dtype);

/*
 * Linear verification (sections "Speculative decoding" and "Target-Draft":
 * the target scores every prefix of the k drafted tokens; the longest
 * accepted prefix is kept and the target's logits after it give one more
 * token, so k drafts yield at most k+1 tokens).
 *
 *  target_logits [B, k+1, V]  row i scores the token after the prefix plus
 *                             d_1..d_i (row k: after all k drafts).
 *  draft_logits  [B, k, V]    row i is the distribution d_{i+1} was drawn
 *                             from.  Unused (may be NULL) when
 *                             temperature == 0.
 *  draft_tokens  [B, k] int32 d_1..d_k.
 *  request_ids   [B] int64 or NULL (=> b); positions [B] int64 or NULL
 *                (=> 0): drafted token i (1-based) is at position
 *                positions[b] + i; the emitted token t* at
 *                positions[b] + a + 1.
 *  params        temperature T, top_p, seed (child_mode ignored).
 *  p = filter(softmax(target / T)), q = filter(softmax(draft / T)), filter
 *  = the top-p nucleus in (logit desc, index asc) order (a token is kept
 *  when the mass before it is < top_p), renormalised.
 *  Sampled (T > 0): d_i is accepted iff u_i < p_{i-1}(d_i) / q_{i-1}(d_i)
 *  (q == 0, a token outside q's nucleus, rejects; the ratio is taken from
 *  the logits' exponents when p or q only underflows fp32, so drafts far in
 *  the tail are decided by their true ratio), u_i from purpose ACCEPT; a =
 *  number of leading
 *  accepts.  If a < k, t* is the smallest v with C(v) > u * C(V-1), C the
 *  running sum of max(0, p_a - q_a) in index order and u from purpose
 *  RESIDUAL (if that residual is all zero, of p_a instead); if a == k, the
 *  same over p_k with purpose BONUS.
 *  Greedy (T == 0): d_i is accepted iff it is the lowest-index argmax of
 *  target row i-1; t* = argmax of target row a.
 *
 *  Outputs: accepted_len [B] (a), out_tokens [B, k+1] (d_1..d_a, t*, then
 *  -1), accept_prob [B, k] = min(1, p/q) for every drafted token (greedy:
 *  1 or 0) or NULL, token_probs [B, k, 2] = (p_{i}(d_{i+1}),
 *  q_{i}(d_{i+1})) or NULL, len_hist [k+1] histogram of a over the batch
 *  (zeroed by the call) or NULL, dev_error [1] or NULL.
 *  Invalid request (bad token, non-finite row): a = 0, t* = lowest-index
 *  argmax of target row 0 over entries that are neither NaN nor +inf,
 *  accept_prob and token_probs 0.
 *  workspace: spec_workspace_size(SPEC_OP_LINEAR, B, k, V, dtype) bytes.
 *  Limits: 1 <= B, 1 <= k <= 64, 1 <= V < 2^31 / (2k+1) / B rows*V.
 */
spec_status spec_verify_linear(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, int B, int k, int V,
                               const int64_t* request_ids, const int64_t* positions,
                               const spec_sampling_params* params,
                               int32_t* accepted_len, int32_t* out_tokens, float* accept_prob,
                               float* token_probs, int32_t* len_hist, int32_t* dev_error,
                               void* workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * Linear verification followed by the compaction of the accepted positions
 * for the next draft step, in the same launches (section "MTP": token
 * t_{i+1} is drawn from logits computed from hidden state H_i; section "MTP
 * schedule for a single token": a kernel inserts the next target tokens,
 * with no host synchronisation).  Results as spec_verify_linear followed by
 * spec_compact_accepted(hidden, B, k+1, H, accepted_len, NULL, out_tokens,
 * k+1, out_hidden, offsets, next_tokens, ...), without the compaction's own
 * launch: the launch after the row statistics takes every request's
 * decisions and the packed offsets, and each request's draw CTA copies its
 * a_b + 1 hidden rows and writes their next tokens.
 *
 *  hidden       [B, k+1, H] bf16 (2-byte elements, copied bit for bit):
 *               row i is the hidden state after the prefix plus d_1..d_i.
 *  out_hidden   [B*(k+1), H] out: row offsets[b] + r = hidden[b, r, :],
 *               r = 0..a_b (rows past offsets[B] untouched).
 *  offsets      [B+1] out: offsets[0] = 0, offsets[b+1] = offsets[b] + a_b + 1.
 *  next_tokens  [B*(k+1)] out: next_tokens[offsets[b] + r] = out_tokens[b, r].
 *  An invalid request (see spec_verify_linear) contributes its row 0 and
 *  its fallback token.  Other arguments, outputs, limits and workspace as
 *  spec_verify_linear; the vector path wants H * 2 a multiple of 16 and
 *  16-byte aligned hidden pointers (else 2-byte copies).  B * (k+1) < 2^31.
 */
spec_status spec_verify_linear_compact(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                       const int32_t* draft_tokens, int B, int k, int V,
                                       const int64_t* request_ids, const int64_t* positions,
                                       const spec_sampling_params* params, const void* hidden, int H,
                                       int32_t* accepted_len, int32_t* out_tokens, float* accept_prob,
                                       float* token_probs, int32_t* len_hist, void* out_hidden, int32_t* offsets,
                                       int32_t* next_tokens, int32_t* dev_error, void* workspace,
                                       size_t workspace_bytes, spec_stream_t stream);

/*
 * The two launch groups of spec_verify_linear (and of
 * spec_verify_linear_compact), for callers that want to time them apart or
 * start the streaming pass as soon as the logits exist.
 * spec_linear_stats_decide reads every target row (and every draft row when
 * T > 0) once, writes per-row statistics into `workspace`, and in a
 * finishing launch runs every request's accept tests: it writes
 * accepted_len, accept_prob, token_probs, len_hist and dev_error (zeroing
 * len_hist and dev_error first) and keeps each request's decision and the
 * packed offsets in the workspace.  spec_linear_draw then draws every
 * request's t* and writes out_tokens and, when hidden is not NULL, the
 * compaction outputs of spec_verify_linear_compact (hidden NULL: H,
 * out_hidden, offsets and next_tokens are ignored).  Called in that order
 * on one stream with identical inputs, params and workspace, they give
 * exactly the results of the one-call forms (which are these two calls).
 * The workspace must not be reused between them.  Arguments as above.
 */
spec_status spec_linear_stats_decide(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                     const int32_t* draft_tokens, int B, int k, int V,
                                     const int64_t* request_ids, const int64_t* positions,
                                     const spec_sampling_params* params, int32_t* accepted_len, float* accept_prob,
                                     float* token_probs, int32_t* len_hist, int32_t* dev_error, void* workspace,
                                     size_t workspace_bytes, spec_stream_t stream);
spec_status spec_linear_draw(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                             const int32_t* draft_tokens, int B, int k, int V, const int64_t* request_ids,
                             const int64_t* positions, const spec_sampling_params* params, const void* hidden, int H,
                             int32_t* out_tokens, void* out_hidden, int32_t* offsets, int32_t* next_tokens,
                             const void* workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_linear for callers that cannot allocate device memory at the
 * point where they verify (code inside a custom allocator or memory pool,
 * code whose device memory is fixed at start-up, code that only receives
 * buffers from a host framework).  The page describes no such variant; it
 * exists for those callers only.
 *
 * Same arguments and results as spec_verify_linear, without the workspace:
 * the workspace (per-row statistics, decisions, offsets, a counter) lives in
 * a fixed array of about 2.3 MiB inside the library's device image, which
 * every GPU that loads the library keeps until the process exits.  Limits: B * (2k + 1) <= 65536 rows, else
 * SPEC_ERR_UNSUPPORTED (nothing is enqueued).  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).  The first call
 * on each device looks up the array's device address once; make that first
 * call before any stream capture.  Every call shares the one array, so
 * calls that overlap on the GPU (different streams or host threads) race on
 * it; each call clears the counter and writes every record it later reads,
 * so no state carries over.
 */
spec_status spec_verify_linear_noalloc(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                       const int32_t* draft_tokens, int B, int k, int V,
                                       const int64_t* request_ids, const int64_t* positions,
                                       const spec_sampling_params* params, int32_t* accepted_len,
                                       int32_t* out_tokens, float* accept_prob, float* token_probs,
                                       int32_t* len_hist, int32_t* dev_error, spec_stream_t stream);

/*
 * Tree verification (section "EAGLE": a static draft tree explored with the
 * Top-K candidates of every node; the longest accepted root-to-leaf path is
 * kept plus one target token).
 *
 *  target_logits [B, N, V]   row n scores the token after node n's path
 *                            (node 0 = the root, the last committed token).
 *  draft_logits  [B, N, V]   row n is the draft distribution the children of
 *                            n were drawn from; may be NULL when T == 0 or
 *                            child_mode == SPEC_CHILD_DETERMINISTIC.
 *  node_tokens   [B, N] int32 token of each node (node 0's is ignored).
 *  parent        [N] int32   parent[0] = -1, 0 <= parent[i] < i.  The
 *                            children of n are tested in increasing index
 *                            order.
 *  max_depth     depth of the deepest node (host value; checked on the
 *                device); outputs have W = max_depth + 1 columns.
 *  At node n of depth t, with P = p_n and Q = q_n: child j (0-based) with
 *  token x is accepted iff u < P(x) / Q(x) (DETERMINISTIC: u < P(x)), u from
 *  purpose ACCEPT, round j, position positions[b] + t + 1.  After a reject:
 *  P <- norm(max(0, P - Q)) (DETERMINISTIC: P with x removed, renormalised;
 *  a zero residual leaves P unchanged), and Q <- Q with x removed,
 *  renormalised (WOR) or unchanged (IID).  An accept moves to that child.
 *  A leaf draws the bonus token from p_leaf (purpose BONUS); a node whose
 *  children are all rejected draws t* from the final P (purpose RESIDUAL),
 *  both by the inverse CDF above.  Greedy: descend into the first child
 *  whose token is the lowest-index argmax of p_n, else emit that argmax.
 *
 *  Outputs: accepted_len [B] (accepted depth a), path_nodes [B, W] (0, the
 *  accepted nodes, then -1), out_tokens [B, W] (their tokens, t*, then -1),
 *  dev_error [1] or NULL.  Invalid request: a = 0, path = [0], t* = argmax
 *  of target row 0 as for the linear call.
 *  workspace: spec_workspace_size(SPEC_OP_TREE, B, N, V, dtype) bytes.
 *  Limits: 1 <= N <= 1024, max_depth < N, at most 64 children per node.
 */
spec_status spec_verify_tree(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                             const int32_t* node_tokens, const int32_t* parent, int B, int N, int V,
                             int max_depth, const int64_t* request_ids, const int64_t* positions,
                             const spec_sampling_params* params, int32_t* accepted_len, int32_t* path_nodes,
                             int32_t* out_tokens, int32_t* dev_error, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/*
 * Tree verification with a tree of its own for every request (section
 * "EAGLE": the tree explored is fixed (EAGLE) or dynamically shaped
 * (EAGLE-2, in the page's citation); each request's tree is then its own).
 * The walk at every node is spec_verify_tree's; only the shape differs:
 *
 *  parent  [B, N] int32   row b is request b's parent array over its nodes
 *                         (parent[b, 0] = -1, 0 <= parent[b, i] < i).
 *  n_nodes [B] int32      request b has nodes 0 .. n_nodes[b]-1; its rows,
 *                         tokens and parent entries past them are not read.
 *  target_logits, draft_logits [B, N, V] and node_tokens [B, N] as for
 *  spec_verify_tree, N the largest tree; max_depth bounds every request's
 *  depth (outputs have W = max_depth + 1 columns).
 *  A request with n_nodes outside 1 .. N, or an invalid parent row, is
 *  invalid (SPEC_DEVERR_PARENT) with the defined fallback.  n_nodes NULL
 *  returns SPEC_ERR_INVALID_ARG; other host checks and limits as above.
 */
spec_status spec_verify_tree_dynamic(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                     const int32_t* node_tokens, const int32_t* parent, const int32_t* n_nodes,
                                     int B, int N, int V, int max_depth, const int64_t* request_ids,
                                     const int64_t* positions, const spec_sampling_params* params,
                                     int32_t* accepted_len, int32_t* path_nodes, int32_t* out_tokens,
                                     int32_t* dev_error, void* workspace, size_t workspace_bytes,
                                     spec_stream_t stream);

/*
 * Compaction for the next draft step (section "MTP": token t_{i+1} is drawn
 * from logits computed from hidden state H_i, so token buffers sit one step
 * left of the hidden states; section "MTP schedule for a single token": a
 * kernel inserts the next target tokens into their slots with no host
 * synchronisation).
 *
 *  hidden       [B, T, H] 2-byte elements (bf16), copied bit for bit.
 *  accepted_len [B]; out_tokens [B, W]; path_nodes [B, W] or NULL (NULL =>
 *               rows 0..a_b, the linear layout).
 *  offsets      [B+1] out: offsets[0] = 0, offsets[b+1] = offsets[b] +
 *               a_b + 1.
 *  out_hidden   [B*W, H] out: row offsets[b] + r = hidden[b, src_r, :],
 *               src_r = path_nodes[b, r] (or r), r = 0..a_b.
 *  next_tokens  [B*W] out: next_tokens[offsets[b] + r] = out_tokens[b, r]
 *               (the token that follows the hidden row it is paired with).
 *  A request with a_b outside [0, W-1], or a source row outside [0, T),
 *  contributes no rows and sets SPEC_DEVERR_LENGTH.  Rows past
 *  offsets[B] are left untouched.
 *  Limits: H * 2 bytes must be a multiple of 16 when the hidden and output
 *  pointers are 16-byte aligned for the vector path; other cases use a
 *  2-byte path.  B * W < 2^31.
 */
spec_status spec_compact_accepted(const void* hidden, int B, int T, int H, const int32_t* accepted_len,
                                  const int32_t* path_nodes, const int32_t* out_tokens, int W, void* out_hidden,
                                  int32_t* offsets, int32_t* next_tokens, int32_t* dev_error,
                                  spec_stream_t stream);

/*
 * Draft-side sampling: one token per logit row drawn from
 * filter(softmax(row / T)), the draft model's own sampling of its tokens
 * (section "Target-Draft"), done on the GPU so that a token drawn from
 * logits carried over from the previous step reaches the next draft run
 * without a host round trip (section "MTP schedule for a single token").
 *
 *  logits       [R, V] bf16 or fp32, row-major.
 *  request_ids  [R] int64 or NULL (NULL => r); positions [R] int64 or NULL
 *               (NULL => 0).  Row r draws u = Philox(seed, request_ids[r],
 *               positions[r], purpose 4 = DRAFT, round 0) and returns the
 *               smallest v with C(v) > u * C(V-1), C the running sum of the
 *               filtered probabilities in index order (the filter as in
 *               spec_verify_linear: temperature, then the exact top-p
 *               nucleus with ties at the boundary kept in index order).
 *  out_tokens   [R] int32 out.
 *  params       temperature == 0: the lowest-index maximum over entries
 *               that are neither NaN nor +inf (0 when there is none), with
 *               no error.  temperature > 0: a row holding a NaN or +inf, or
 *               no finite entry, sets SPEC_DEVERR_NONFINITE and yields that
 *               argmax.  child_mode is ignored.
 *  dev_error    [1] or NULL.
 *  Errors: SPEC_ERR_INVALID_ARG (NULL logits / out_tokens / params, R < 1,
 *  V < 1, temperature < 0 or not finite, top_p <= 0 or NaN, dtype not
 *  bf16 or fp32); SPEC_ERR_UNSUPPORTED (V above 524,280).
 */
spec_status spec_sample_rows(const void* logits, spec_dtype dtype, int R, int V, const int64_t* request_ids,
                             const int64_t* positions, const spec_sampling_params* params, int32_t* out_tokens,
                             int32_t* dev_error, spec_stream_t stream);

/* Static, human-readable name of a status code. */
const char* spec_status_string(spec_status status);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
