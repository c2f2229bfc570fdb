/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library, libspecverify.so.
 *
 * The library implements the target-side verification step of speculative
 * decoding as described on these pages (cited by title and section):
 *   [LZ] "3.5 Speculative Decoding" (llm-learning-path)
 *   [MN] "246 Speculative Decoding" (ai_in_action)
 *   [LB] "Speculative Decoding: Mathematical Foundations, Rejection Sampling
 *        Dynamics, Draft Architectures, and Serving Latency" (llms.blog)
 *   [SS] "Speculative Decoding from First Principles" (theservingstack.com)
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers into memory the caller owns
 *     (e.g. PyTorch tensors).  The library never allocates, frees or
 *     synchronises, except spec_verify_last_error, which synchronises the
 *     given stream.  Work is enqueued on `stream` (NULL = the legacy default
 *     stream) and completes asynchronously.
 *   - Logit arrays are row-major with the vocabulary innermost and
 *     contiguous; their base pointers must be aligned to their element size
 *     (4 bytes for SPEC_F32, 2 for SPEC_BF16 -- bf16 is stored as its 16-bit
 *     pattern).  Token arrays are int32, uniforms fp32.
 *   - Argument errors are returned synchronously as a negative status and
 *     nothing is enqueued.  A call with B = 0 is valid, enqueues nothing and
 *     may pass NULL for every array.  Data errors found on the device (a NaN or +inf
 *     logit, a row that is entirely -inf, a token outside [0, V), a uniform
 *     outside [0, 1), a malformed tree) never trap: the affected sequence's
 *     outputs are set to -1 and a bit is OR-ed into the workspace's error
 *     word, read back by spec_verify_last_error.
 *   - A workspace is caller-owned device memory of at least the size the
 *     matching *_workspace_size function reports.  It must be zero-filled
 *     before its first use (spec_verify_workspace_init, or any zero fill);
 *     the library returns its internal counters to zero at the end of every
 *     call.  After a call that returned SPEC_ERR_CUDA, zero-fill it again.
 *     Calls that share one workspace must be ordered (one stream, or
 *     events): two calls running at the same time on one workspace race.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t). */
typedef struct CUstream_st *spec_stream_t;

/* Logit storage types. */
enum { SPEC_F32 = 0, SPEC_BF16 = 1 };

/* Verification rules for spec_verify_sample. */
enum {
    SPEC_STOCHASTIC = 0, /* rejection sampling with residual / bonus draw */
    SPEC_GREEDY = 1      /* draft kept iff it equals the target argmax     */
};

/* Synchronous status codes (negative: nothing was enqueued). */
enum {
    SPEC_OK = 0,
    SPEC_ERR_NULL = -1,      /* a required pointer is NULL                 */
    SPEC_ERR_SHAPE = -2,     /* B, k, V, N or D outside the supported range */
    SPEC_ERR_PARAM = -3,     /* temperature <= 0 or not finite, top_p not
                                in (0, 1]                                  */
    SPEC_ERR_DTYPE = -4,     /* dtype not SPEC_F32 / SPEC_BF16             */
    SPEC_ERR_MODE = -5,      /* mode not SPEC_STOCHASTIC / SPEC_GREEDY     */
    SPEC_ERR_ALIGN = -6,     /* a pointer misaligned for its element type  */
    SPEC_ERR_WORKSPACE = -7, /* workspace NULL or smaller than required    */
    SPEC_ERR_CUDA = -8       /* a CUDA runtime call failed                 */
};

/* Data-error bits of the workspace error word (device-detected). */
enum {
    SPEC_DATA_ROW_NONFINITE = 1 << 1,   /* a NaN or +inf logit in a row    */
    SPEC_DATA_ROW_ALL_NEG_INF = 1 << 2, /* every logit of a row is -inf    */
    SPEC_DATA_TOKEN_RANGE = 1 << 3,     /* a draft or node token not in
                                           [0, V)                          */
    SPEC_DATA_UNIFORM_RANGE = 1 << 4,   /* a uniform not in [0, 1)         */
    SPEC_DATA_TREE_SHAPE = 1 << 5,      /* parents not a rooted tree in
                                           topological order, or a node
                                           deeper than D                   */
    SPEC_DATA_PROB_RANGE = 1 << 6       /* a gathered draft probability
                                           q_i(x~_i) not in [0, 1]         */
};

/* Supported ranges. */
#define SPEC_MAX_K 31          /* draft length k in [1, 31]: the k+1
                                  positions fit one warp                  */
#define SPEC_MAX_V (1 << 22)   /* vocabulary size V in [1, 2^22]           */
#define SPEC_MAX_TREE_NODES 1024

/*
 * Workspace bytes needed by spec_verify_sample for batch B, draft length k
 * and vocabulary V (either mode, either dtype), and by every other chain
 * call on the same shape (top-k included).  The top-k calls' row summaries
 * are laid out last, so calls without top-k also accept a workspace that
 * stops before them (the size of the other parts, ~16 KB per target row
 * plus small records).  Returns SPEC_OK or SPEC_ERR_NULL / SPEC_ERR_SHAPE.
 */
int spec_verify_workspace_size(int B, int k, int V, size_t *bytes);

/* Workspace bytes needed by spec_verify_tree for B trees of N nodes. */
int spec_verify_tree_workspace_size(int B, int N, int V, size_t *bytes);

/* Zero-fill `bytes` of a workspace on `stream` (cudaMemsetAsync). */
int spec_verify_workspace_init(void *workspace, size_t bytes, spec_stream_t stream);

/*
 * One verification step for B independent sequences.
 *
 * SPEC_STOCHASTIC -- [LZ] "The algorithm (one step)", steps 3 and 4; [MN]
 * 2.2 "The acceptance test for one token" and 3.3 "The full block loop";
 * [LB] "The Modified Rejection Sampling Algorithm":
 *   p_i = the target distribution at position i (row i of target_logits),
 *   q_i = the draft distribution (row i of draft_logits), both after the
 *   same processing ([LZ] "Notation"; [MN] 6 "Pitfalls"): divide the logits
 *   by `temperature`, softmax, then -- if top_p < 1 -- keep the smallest set
 *   of most likely tokens whose mass reaches top_p (all tokens tied with the
 *   last one kept) and renormalise.
 *   For i = 1..k, left to right: accept draft x~_i iff
 *     u_i * q_i(x~_i) < p_i(x~_i)        (u_i = uniforms[b][i-1])
 *   and stop at the first rejection.  j = number accepted.
 *   If j < k: draw from the residual max(0, p_{j+1} - q_{j+1}) normalised
 *   (if it is zero everywhere, from p_{j+1}); if j = k: draw the bonus
 *   token from p_{k+1}.  The draw uses u = uniforms[b][k] by inverse CDF in
 *   token order: the smallest x whose cumulative weight exceeds u * (total
 *   weight).
 * SPEC_GREEDY -- [LZ] end of "Proof that the output distribution is exactly
 * p"; [SS] "Draft, verify, keep what matches": g_i = first argmax of the raw
 * target row i; j = number of leading i with x~_i == g_i; the emitted token
 * after them is g_{j+1}.  draft_logits, uniforms, temperature and top_p are
 * ignored (may be NULL / any value).
 *
 * Arguments
 *   target_logits    [B, k+1, V] dtype, device
 *   draft_logits     [B, k, V]   dtype, device (STOCHASTIC)
 *   draft_tokens     [B, k]      int32, device
 *   uniforms         [B, k+1]    fp32 in [0, 1), device (STOCHASTIC)
 *   B >= 0, 1 <= k <= SPEC_MAX_K, 1 <= V <= SPEC_MAX_V
 *   temperature > 0, 0 < top_p <= 1 (STOCHASTIC)
 *   mode             SPEC_STOCHASTIC or SPEC_GREEDY
 *   dtype            SPEC_F32 or SPEC_BF16 (both logit arrays)
 *   out_tokens       [B, k+1] int32, device: x~_1..x~_j, then the drawn
 *                    (or argmax) token, then -1; all -1 on a data error
 *   out_num_accepted [B] int32, device: j in [0, k], -1 on a data error
 *   workspace        >= spec_verify_workspace_size(B, k, V) bytes, zeroed
 *                    before first use
 * Returns SPEC_OK or a negative status.
 */
int spec_verify_sample(const void *target_logits, const void *draft_logits,
                       const int32_t *draft_tokens, const float *uniforms,
                       int B, int k, int V, float temperature, float top_p,
                       int mode, int dtype, int32_t *out_tokens,
                       int32_t *out_num_accepted, void *workspace,
                       size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_sample with top-k as well ([MN] 6 "Pitfalls": target and
 * draft must share temperature, top-p, top-k and every other logit
 * processor; the pages never define top-k).  Reading: after temperature,
 * keep the tokens whose logit is at least the top_k-th largest of the row
 * (every tie of it kept) and renormalise; top-p then applies to that
 * renormalised distribution.  top_k <= 0 or top_k >= V: no top-k (the call
 * is then spec_verify_sample).  Same processing on target and draft rows;
 * ignored in SPEC_GREEDY mode.  Other arguments and results as for
 * spec_verify_sample.
 */
int spec_verify_sample_topk(const void *target_logits, const void *draft_logits,
                            const int32_t *draft_tokens, const float *uniforms,
                            int B, int k, int V, float temperature, float top_p, int top_k,
                            int mode, int dtype, int32_t *out_tokens,
                            int32_t *out_num_accepted, void *workspace,
                            size_t workspace_bytes, spec_stream_t stream);

/*
 * The two phases of spec_verify_sample, with the same arguments.
 * spec_verify_sample gives the results of spec_verify_sample_rows followed,
 * on the same stream and workspace, by spec_verify_sample_finish, bit for
 * bit.  (On a small call with short rows it launches no separate draw: the
 * row kernel's deciding warp draws.)
 *   _rows    streams every logit row once, leaves per-row statistics
 *            (max, normaliser, nucleus threshold, argmax) in the workspace
 *            and takes every sequence's accept decision; with top-p it also
 *            draws from the nucleus list and writes those outputs;
 *   _finish  runs the remaining final draws (residual or bonus row) and
 *            writes out_tokens / out_num_accepted for them.
 * The split lets a caller time or overlap the phases; _finish must follow a
 * _rows call with identical arguments, with no other call on the workspace
 * in between.  In SPEC_GREEDY mode _rows does all the work and _finish
 * enqueues nothing.
 */
int spec_verify_sample_rows(const void *target_logits, const void *draft_logits,
                            const int32_t *draft_tokens, const float *uniforms,
                            int B, int k, int V, float temperature, float top_p,
                            int mode, int dtype, int32_t *out_tokens,
                            int32_t *out_num_accepted, void *workspace,
                            size_t workspace_bytes, spec_stream_t stream);
int spec_verify_sample_finish(const void *target_logits, const void *draft_logits,
                              const int32_t *draft_tokens, const float *uniforms,
                              int B, int k, int V, float temperature, float top_p,
                              int mode, int dtype, int32_t *out_tokens,
                              int32_t *out_num_accepted, void *workspace,
                              size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_sample (SPEC_STOCHASTIC) with the draft given as
 * probabilities instead of logits: the step takes "draft logits (or
 * probabilities)".  draft_probs [B, k, V] fp32 is q_1..q_k itself -- the
 * distributions the drafter sampled x~_i from -- and is used as given: no
 * temperature, no top-p, no top-k, no renormalisation.  temperature, top_k
 * and top_p process the target rows only (p_i as in
 * spec_verify_sample_topk).  Draft rows
 * are read only where the step needs them: q_i(x~_i) at each draft token,
 * and the rejecting position's row for the residual max(0, p - q).
 *
 * Arguments as for spec_verify_sample, except
 *   draft_probs      [B, k, V] fp32, device, 4-byte aligned (any dtype of
 *                    target_logits)
 *   dtype            storage type of target_logits
 * Data errors as for spec_verify_sample, plus SPEC_DATA_PROB_RANGE: a
 * gathered q_i(x~_i) that is NaN or outside [0, 1] fails the sequence.  The
 * rest of each row is not checked: it must hold finite, non-negative values
 * (a NaN there weighs zero in the residual).
 * spec_verify_intermediates after this call: P, Q and S as documented; Z
 * holds the k+1 target rows of each sequence only, packed at stride k+1.
 * spec_verify_acceptance does not apply to this form.
 */
int spec_verify_sample_probs(const void *target_logits, const float *draft_probs,
                             const int32_t *draft_tokens, const float *uniforms,
                             int B, int k, int V, float temperature, float top_p,
                             int top_k, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                             void *workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/*
 * Greedy tree verification for B sequences sharing one candidate tree --
 * [LZ] "Tree verification": the flattened tree is scored in one target
 * pass; keep the longest root-to-leaf path that passes verification; [LB]
 * "Tree-Based Verification and Custom Attention Masks".
 *   g_n = first argmax of target row n.  Node c (parent n) is accepted iff
 *   n is accepted and node_tokens[b][c] == g_n; the root is accepted.  The
 *   deepest accepted node wins (ties to the lowest flattened index); its
 *   path's tokens are emitted, then g of that node (the bonus token).
 *
 * Arguments
 *   target_logits    [B, N, V] dtype, device: one row per flattened node
 *   parents          [N] int32, device: parents[0] = -1 (the root, the last
 *                    committed token), 0 <= parents[n] < n otherwise
 *   node_tokens      [B, N] int32, device: candidate token of each node (the
 *                    root's entry is ignored)
 *   1 <= N <= SPEC_MAX_TREE_NODES, 0 <= D < N: every node's depth <= D
 *   out_tokens       [B, D+1] int32, device: path tokens, bonus, -1 pad
 *   out_num_accepted [B] int32, device: accepted depth d, -1 on a data error
 *   out_path         [B, D+1] int32, device, or NULL: node ids root, n_1,
 *                    ..., n_d, then -1
 *   workspace        >= spec_verify_tree_workspace_size(B, N, V) bytes
 * Returns SPEC_OK or a negative status.
 */
int spec_verify_tree(const void *target_logits, const int32_t *parents,
                     const int32_t *node_tokens, int B, int N, int V, int D,
                     int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                     int32_t *out_path, void *workspace, size_t workspace_bytes,
                     spec_stream_t stream);

/*
 * Stochastic tree verification for B sequences sharing one tree shape --
 * [LZ] "Tree verification" names SpecInfer's lossless multi-candidate
 * acceptance rule for sampling, without stating it.  Reading: the children
 * of node n are candidates drawn independently from q_n (draft row n,
 * processed like the target).  From the root, the current node's children
 * are tried in flattened order: child c is accepted iff
 *   u_c * q_n(x_c) < p'(x_c)
 * where p' starts as p_n (target row n) and becomes, after each rejected
 * child, the residual max(0, p' - q_n) normalised (kept as it is if that
 * residual is zero everywhere).  An accepted child becomes the current
 * node; when every child is rejected, or there is none, the final token is
 * drawn from p' by inverse CDF in token order.  Every emitted position
 * then follows the target's distribution.
 *
 * Arguments
 *   target_logits    [B, N, V] dtype, device: target row of each node
 *   draft_logits     [B, N, V] dtype, device: row n is the law the children
 *                    of node n were drawn from (a leaf's row is not used)
 *   parents          [N] int32, device (as spec_verify_tree); at most 64
 *                    children per node
 *   node_tokens      [B, N] int32, device (the root's entry is ignored)
 *   uniforms         [B, N] fp32 in [0, 1), device: entry c >= 1 is node
 *                    c's test, entry 0 the final draw
 *   1 <= N <= SPEC_MAX_TREE_NODES, 0 <= D < N; temperature, top_p, top_k
 *                    process target and draft rows alike (as
 *                    spec_verify_sample_topk)
 *   out_tokens, out_num_accepted, out_path: as spec_verify_tree
 *   workspace        >= spec_verify_tree_sample_workspace_size(B, N, V)
 * Data errors: as spec_verify_tree, plus a uniform outside [0, 1) and a node
 * with more than 64 children (SPEC_DATA_TREE_SHAPE).
 * Returns SPEC_OK or a negative status.
 */
int spec_verify_tree_sample_workspace_size(int B, int N, int V, size_t *bytes);
int spec_verify_tree_sample(const void *target_logits, const void *draft_logits,
                            const int32_t *parents, const int32_t *node_tokens,
                            const float *uniforms, int B, int N, int V, int D,
                            float temperature, float top_p, int top_k, int dtype,
                            int32_t *out_tokens, int32_t *out_num_accepted,
                            int32_t *out_path, void *workspace, size_t workspace_bytes,
                            spec_stream_t stream);

/*
 * Tree attention inputs for B candidate trees -- the step just before the
 * target pass whose logits spec_verify_tree verifies.  [LZ] "Tree
 * verification": the flattened tree is scored in one target pass where
 * every node attends to the context and to its own ancestors only, and
 * nodes at the same depth share one position index (for RoPE); [LB]
 * "Tree-Based Verification and Custom Attention Masks": M_ij = 0 where
 * node j is an ancestor of node i, -inf elsewhere.  A node counts as its
 * own ancestor here (the diagonal is visible), as in [LZ]'s mask.
 *
 * Arguments
 *   parents    [B, N] int32, device: one tree per sequence, flattened as
 *              for spec_verify_tree (parents[b][0] = -1, 0 <= parents[b][n]
 *              < n otherwise)
 *   pos0       [B] int32, device, or NULL (all 0): position index of each
 *              tree's root (the last committed token)
 *   1 <= N <= SPEC_MAX_TREE_NODES, B >= 0
 *   out_mask   [B, N, N] uint8, device, or NULL: 1 where node i (row) may
 *              attend to node j (column), 0 elsewhere
 *   out_bias   [B, N, N] fp32, device, or NULL: the same as 0 / -inf
 *   out_pos    [B, N] int32, device, or NULL: pos0[b] + depth(n)
 * The context (the tokens before the root) is visible to every node and is
 * not part of these outputs.  A sequence whose parents are not a rooted
 * tree in topological order gets an all-zero mask, an all -inf bias and
 * positions -1 (no error word: this call takes no workspace).
 * Returns SPEC_OK or a negative status; nothing is enqueued on error.
 */
int spec_verify_tree_mask(const int32_t *parents, const int32_t *pos0, int B, int N,
                          uint8_t *out_mask, float *out_bias, int32_t *out_pos,
                          spec_stream_t stream);

/*
 * spec_verify_sample for callers that cannot allocate device memory (no
 * counterpart on the pages: it is a deployment variant).  A serving engine
 * that plans all device memory ahead and forbids allocation on its decode
 * path, or a plugin whose host framework gives it no allocator, cannot pass
 * a workspace; this entry point instead uses a fixed 4 MiB scratch array in
 * the library's own device image, held by every GPU that loads the library
 * until the process exits.  It calls no allocator.
 *   - Same arguments and results as spec_verify_sample, without the
 *     workspace.  Batches whose workspace without the top-k part (see
 *     spec_verify_workspace_size) exceeds 4 MiB are rejected with
 *     SPEC_ERR_WORKSPACE.
 *   - Each call zero-fills the part of the scratch it uses on `stream`
 *     first.  All calls on a device share the one array: calls whose work
 *     overlaps on the GPU race and give wrong results; order them.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make it before any stream capture begins.  The
 *     address is kept for the process and belongs to the device's primary
 *     context (the one the CUDA runtime uses): do not call this entry point
 *     from another context on that device, nor after resetting the device
 *     (cudaDeviceReset) once it has been called there.
 *   - Data errors show as -1 outputs; the error word is not kept.
 */
int spec_verify_sample_noalloc(const void *target_logits, const void *draft_logits,
                               const int32_t *draft_tokens, const float *uniforms,
                               int B, int k, int V, float temperature, float top_p,
                               int mode, int dtype, int32_t *out_tokens,
                               int32_t *out_num_accepted, spec_stream_t stream);

/*
 * Synchronise `stream`, then return the workspace's data-error word (an OR
 * of SPEC_DATA_* bits accumulated since the previous call of this function;
 * 0 if none) and clear it.  Negative on an argument or CUDA error.
 */
int spec_verify_last_error(void *workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * Debug read-out of the intermediates of the last spec_verify_sample call
 * (STOCHASTIC) made with this workspace and the same B, k, V:
 *   P [B, k]    p_i(x~_i), processed target probability of each draft
 *   Q [B, k]    q_i(x~_i)
 *   Z [B, 2k+1] per-row normaliser sum_x exp((l(x) - max l) / T) over the
 *               kept tokens (target rows 0..k, then draft rows 0..k-1)
 *   S [B]       total weight of the final draw (residual or bonus row)
 * All four are device fp32 arrays (any may be NULL).  Enqueued on `stream`.
 */
int spec_verify_intermediates(const void *workspace, size_t workspace_bytes,
                              int B, int k, int V, float *P, float *Q, float *Z,
                              float *S, spec_stream_t stream);

/*
 * Per-position acceptance rate of the last verification step -- [LZ]
 * "Proof that the output distribution is exactly p": once position i is
 * tested it accepts with probability
 *   beta_i = sum_x min(p_i(x), q_i(x)) = 1 - TV(p_i, q_i),
 * and [LB] "Acceptance Rate and Total Variation Distance": TV(p, q) =
 * (1/2) sum_x |p(x) - q(x)|.  Engines log beta to track how well the draft
 * matches the target.
 *
 * Reads the per-row statistics that the last spec_verify_sample,
 * spec_verify_sample_topk (or spec_verify_sample_rows) call left in
 * `workspace`; that call must have been SPEC_STOCHASTIC, with the same
 * target_logits, draft_logits, B, k, V, temperature, top_p, top_k (0 for
 * spec_verify_sample) and dtype, on this stream (or ordered before it).
 * Otherwise the results are meaningless (never out of bounds).  It changes
 * nothing that spec_verify_sample_finish reads, so it may run between
 * _rows and _finish.
 *
 * Arguments
 *   target_logits, draft_logits, B, k, V, temperature, top_p, top_k, dtype:
 *                    as for spec_verify_sample_topk (target rows k+1 are
 *                    not read)
 *   out_beta         [B, k] fp32, device: beta_i for i = 1..k; NaN where
 *                    row i of the target or draft has a data error
 *   out_tv           [B, k] fp32, device, or NULL: 1 - beta_i
 *   workspace        the verify call's workspace
 * Returns SPEC_OK or a negative status; nothing is enqueued on error.
 */
int spec_verify_acceptance(const void *target_logits, const void *draft_logits, int B,
                           int k, int V, float temperature, float top_p, int top_k, int dtype,
                           float *out_beta, float *out_tv, void *workspace,
                           size_t workspace_bytes, spec_stream_t stream);

/* Static, human-readable description of a status or data-error bit. */
const char *spec_verify_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
