/*
 * specdec.h -- C ABI of the GB300 (sm_103a) speculative-decoding draft/verify
 * library (libspecdec.so).
 *
 * The path: per-step draft softmax and top-k, expansion of the top-k into a
 * candidate tree, tree build (mask, positions, retrieve links), one batched
 * verification pass over the target logits of every tree node (greedy
 * first-rejection commit with bonus token, or stochastic acceptance with the
 * positive residual), accepted-path KV-slot compaction, and the TLI
 * heterogeneous-vocabulary constraint and id remapping.
 *
 * Sources (web pages, cited by title and section):
 *   [HB]  ai-infra-handbooks, "EAGLE speculative decoding in four parts: why
 *         it became a worker" -- "Drafting, verification and slots".
 *   [ML]  secrett2633 blog, "[SGLang] Multi-Layer EAGLE" -- section 2
 *         (select_top_k_tokens, tree_info) and section 3 (softmax, fast_topk).
 *   [ZS]  zero-to-sglang ch.10 "Speculative decoding (code walk-through)" --
 *         3.2 drafting and EOS, 3.3 row alignment, 4.1 greedy commitment,
 *         5.1 stochastic acceptance and residual, 5.2 verify input and KV.
 *   [TLI] SGLang PR #22883 "TLI (Token-Level Intersection)" -- Modifications.
 *
 * Conventions shared by every call:
 *   - Every pointer is a DEVICE pointer owned by the caller, unless a comment
 *     says otherwise.  The library allocates nothing.  Calls that need
 *     scratch take (ws, ws_bytes), sized by the matching *_ws_size call.
 *   - Work is enqueued asynchronously on the caller's stream (0 = legacy
 *     default stream).  No call synchronises the device.
 *   - Requests b in [0,B); tree nodes n in [0,N); node 0 is the root (the
 *     last committed token).  Logit rows are row-major and contiguous:
 *     target logits [B, N, V], row (b, n) = the target's next-token logits
 *     after the path root..n, which verifies n's children and, at a leaf,
 *     gives the bonus ([ZS] 3.3: row L-1+i verifies draft i).
 *   - dtype: SPEC_F32 or SPEC_BF16 for logit buffers.  Ids are int32;
 *     probabilities are fp32.  NaN logits are treated as -inf; ties in
 *     argmax / top-k go to the lowest index.
 *   - Random numbers are inputs (uniforms in [0,1)), so results are
 *     deterministic: no float atomics, fixed reduction orders.
 *   - Return value: SPEC_OK, or a negative SPEC_ERR_* code.  Arguments are
 *     checked on the host before anything is enqueued; a failed check
 *     enqueues nothing.  Data-dependent anomalies are not errors: they are
 *     counted in the optional stats array (int32[SPEC_NUM_STATS], device,
 *     incremented with integer atomics; the caller zeroes it).
 */
#ifndef SPECDEC_H
#define SPECDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* spec_stream_t; /* same object as cudaStream_t */

#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG (-1)  /* null pointer, bad size or shape, bad option */
#define SPEC_ERR_UNSUPPORTED (-2)  /* dtype, alignment or size beyond a stated limit */
#define SPEC_ERR_CUDA (-3)         /* a launch failed (cudaGetLastError) */
#define SPEC_ERR_WORKSPACE (-4)    /* ws_bytes below the *_ws_size value */

#define SPEC_F32 0
#define SPEC_BF16 1

/* stats[] slots */
#define SPEC_STAT_NONFINITE_ROW 0     /* a row whose maximum is not finite */
#define SPEC_STAT_Q_ZERO 1            /* accept test met q[y] == 0 */
#define SPEC_STAT_RESIDUAL_FALLBACK 2 /* residual had no positive mass; p_cur kept */
#define SPEC_STAT_CDF_FALLBACK 3      /* inverse CDF found no crossing; last positive taken */
#define SPEC_STAT_EMPTY_INTERSECTION 4/* TLI row with no finite intersection logit */
#define SPEC_STAT_BAD_REQUEST 5       /* compaction input out of range; request skipped */
#define SPEC_STAT_WAIT_TIMEOUT 6      /* a CTA gave up waiting on another's row (results void) */
#define SPEC_STAT_BOUNDS 7            /* debug build only: an index outside its buffer (access skipped) */
#define SPEC_NUM_STATS 8

/* Limits (checked on the host; SPEC_ERR_UNSUPPORTED beyond them). */
#define SPEC_MAX_TOPK 32          /* k of spec_softmax_topk / spec_tree_expand */
#define SPEC_MAX_POOL 16384       /* candidate-pool size P of spec_build_tree */
#define SPEC_MAX_NODES 2048       /* tree nodes N per request */
#define SPEC_MAX_VOCAB (1 << 22)  /* V of every logit row */

/* walk_info[b*3 + 2] values */
#define SPEC_FINAL_ACCEPTED 0    /* the last committed token is an accepted draft */
#define SPEC_FINAL_CORRECTION 1  /* drawn after a rejection at the final node */
#define SPEC_FINAL_BONUS 2       /* drawn at a leaf after full acceptance */

/* ------------------------------------------------------------------ draft */

/* Draft-step softmax and top-k.  [ML] section 3: probs = softmax(logits),
 * then top-k; the top-k probabilities are the tree scores, from a plain
 * softmax (T_score = 1 in the draft loop).  [ZS] 5.1: with a temperature,
 * the stored draft distribution q is the processed one (temperature T).
 *   logits     [R, V] (dtype), row-major.
 *   T          temperature > 0 of q (probs_or_null, row_stats_or_null):
 *              p_v = exp((l_v - max l)/T) / sum_u exp((l_u - max l)/T).
 *   T_score    temperature > 0 of topk_p (the same formula at T_score).
 *              When q is written and T_score != T, the one pass over the
 *              row keeps a normaliser at each temperature.
 *   k          1 <= k <= min(V, SPEC_MAX_TOPK).
 *   topk_p     [R, k] fp32 out: probabilities of the top-k tokens at T_score.
 *   topk_idx   [R, k] int32 out: indices by (logit desc, index asc), the
 *              same at every temperature.
 *   probs_or_null [R, V] fp32 out (optional): the full distribution at T
 *              (the draft distribution q that stochastic verify reads).
 *   row_stats_or_null [R, 2] fp32 out (optional): the row's maximum m and
 *              normaliser Z = sum 2^((l - m) log2(e)/T), from which
 *              spec_verify_sample_qlogits recomputes exactly the values
 *              probs_or_null would hold.
 * A row whose maximum is not finite gets zero probabilities and counts in
 * SPEC_STAT_NONFINITE_ROW. */
int spec_softmax_topk(const void* logits, int dtype, int64_t R, int64_t V, float T, float T_score,
                      int k, float* topk_p, int32_t* topk_idx, float* probs_or_null,
                      float* row_stats_or_null, int32_t* stats_or_null, spec_stream_t stream);

/* Draft sampling with caller uniforms (chain drafts drawn from q; [ZS] 5.1
 * "a candidate y drawn from the draft distribution q").  One token per row
 * by inverse CDF over vocabulary order: the smallest v whose inclusive prefix
 * sum of the row's weights exceeds u[r] times their total.
 *   probs_or_null  [R, V] fp32 weights; if NULL, weights are
 *                  exp((l - max l)/T) of logits_or_null [R, V] (dtype).
 *   u              [R] fp32 uniforms in [0,1).
 *   out_token      [R] int32 out.
 *   out_prob_or_null [R] fp32 out: the drawn token's normalised weight.
 *   row_stats_or_null [R, 2] fp32 in (logits only, optional): each row's
 *                  maximum as spec_softmax_topk recorded it; the row is
 *                  then read once instead of twice.  The result is the same.
 * If rounding leaves no crossing, the last index with positive weight is
 * taken (SPEC_STAT_CDF_FALLBACK). */
int spec_sample(const void* logits_or_null, int dtype, const float* probs_or_null, int64_t R,
                int64_t V, float T, const float* u, int32_t* out_token, float* out_prob_or_null,
                const float* row_stats_or_null, int32_t* stats_or_null, spec_stream_t stream);

/* Draft softmax and sampling in one pass, for sampled chains (drafts drawn
 * from q, [ZS] 5.1).  Per row: m, Z as spec_softmax_topk defines them and
 * one token by inverse CDF over vocabulary order with the uniform u[r] (the
 * smallest v whose inclusive prefix sum of 2^((l - m) log2(e)/T) exceeds
 * u[r] times the total), reading the row once.
 *   logits     [R, V] (dtype), V <= 524288 for bf16, 262144 for fp32
 *              (SPEC_ERR_UNSUPPORTED above).
 *   u          [R] fp32 uniforms in [0,1).
 *   out_token  [R] int32 out; out_prob_or_null [R] fp32 out: its weight
 *              divided by the total.
 *   row_stats_or_null [R, 2] fp32 out: (m, Z) for spec_verify_sample_qlogits.
 *   probs_or_null [R, V] fp32 out: the distribution, with the same m and Z.
 * A row with no finite max gets token 0, probability 0, zero probabilities
 * and counts in SPEC_STAT_NONFINITE_ROW; no crossing after rounding takes
 * the last index of positive weight (SPEC_STAT_CDF_FALLBACK). */
int spec_softmax_sample(const void* logits, int dtype, int64_t R, int64_t V, float T, const float* u,
                        int32_t* out_token, float* out_prob_or_null, float* row_stats_or_null,
                        float* probs_or_null, int32_t* stats_or_null, spec_stream_t stream);

/* Candidate-pool size P = 1 + k + (num_steps - 1) * k * k. */
int64_t spec_tree_pool_size(int k, int num_steps);

/* One draft step of the tree expansion ([ML] section 2, select_top_k_tokens
 * with tree_info = (scores, tokens, parents)).
 *   step 0: topk_p / topk_idx are [B, 1, k] (the root rows).  Initialises
 *     the pool: id 0 = root (score 1), ids 1..k = the root's children,
 *     score = topk_p.
 *   step s >= 1: topk_p / topk_idx are [B, k, k]: row (b, f) belongs to
 *     frontier slot f.  Child j of frontier node f gets score
 *     frontier_score[f] * topk_p[f][j] (one fp32 multiply, round to nearest)
 *     and pool id 1 + k + (s-1)k^2 + f*k + j.
 *   Every expansion enters the pool; the new frontier is the best k of this
 *   step's candidates by (score desc, pool id asc), written to
 *   frontier_score / frontier_id [B, k] (in/out).
 *   pool_qrow marks each new frontier node with the row of the step-major
 *   draft-row table that will hold its draft distribution: step 0's rows are
 *   [0, B) (the roots, row b), step t >= 1's rows are B + (t-1)*B*k +
 *   b*k + slot.  Not set on the last step.  Candidates never expanded keep -1.
 *   pool_* are [B, P] (P = spec_tree_pool_size(k, num_steps)).
 * 1 <= k <= SPEC_MAX_TOPK, 0 <= step < num_steps. */
int spec_tree_expand(int step, int num_steps, int B, int k, const float* topk_p,
                     const int32_t* topk_idx, float* pool_score, int32_t* pool_token,
                     int32_t* pool_parent, int32_t* pool_qrow, float* frontier_score,
                     int32_t* frontier_id, spec_stream_t stream);

/* One step of the expansion above, fused into a draft launch: the CTA
 * that completes a request's rows of the step (its one row at step 0 or
 * with k = 1, its k rows after) expands the request, so a draft step is
 * one launch instead of two.  The pool, frontier and step fields are those
 * of spec_tree_expand; counters is [B] int32, zero before the first fused
 * step (the expanding CTA returns it to zero), needed when k > 1. */
typedef struct spec_expand {
  int step, num_steps, B, k;
  float* pool_score;
  int32_t* pool_token;
  int32_t* pool_parent;
  int32_t* pool_qrow;
  float* frontier_score;
  int32_t* frontier_id;
  int32_t* counters;
} spec_expand_t;

/* spec_softmax_topk with the step's pool expansion fused (expand->k == k;
 * R = expand->B at step 0, expand->B * k after; topk_p / topk_idx laid out
 * as spec_tree_expand reads them). */
int spec_softmax_topk_expand(const void* logits, int dtype, int64_t R, int64_t V, float T,
                             float T_score, int k, float* topk_p, int32_t* topk_idx, float* probs_or_null,
                             float* row_stats_or_null, int32_t* stats_or_null, const spec_expand_t* expand,
                             spec_stream_t stream);

/* spec_softmax_sample with the step's pool expansion fused, for chains:
 * expand->k == 1, R = expand->B, out_prob required (the drawn token and its
 * probability are the step's top-1). */
int spec_softmax_sample_expand(const void* logits, int dtype, int64_t R, int64_t V, float T, const float* u,
                               int32_t* out_token, float* out_prob, float* row_stats_or_null,
                               float* probs_or_null, int32_t* stats_or_null, const spec_expand_t* expand,
                               spec_stream_t stream);

/* Tree build ([HB] "Drafting, verification and slots": build_eagle_tree
 * produces the attention mask and positions; [ZS] 5.2 lists the verify input
 * draft_token, positions, custom_mask and retrieve_*).  The N-1 best pool
 * candidates by (score desc, pool id asc) become nodes 1..N-1 in ascending
 * pool-id order (parents precede children; siblings in draft-rank order).
 * Inputs: pool [B, P] from spec_tree_expand, root_token [B], seq_lens [B]
 * (tokens already in the KV cache; the root sits at position seq_len).
 * Outputs, all [B, N] int32 unless noted:
 *   draft_token           token of node n (root_token at n = 0)
 *   parent                parent node (-1 at the root)
 *   positions             seq_len + depth(n)
 *   tree_mask [B, N, N] u8  1 iff column m is n or an ancestor of n
 *   retrieve_index        b*N + n
 *   retrieve_next_token   first child of n, -1 if none
 *   retrieve_next_sibling next node with the same parent, -1 if none
 *   q_row                 draft-row table row of n's draft distribution, -1
 * 1 <= N <= min(P, SPEC_MAX_NODES), P <= SPEC_MAX_POOL.
 * A selected candidate whose pool parent is out of range, not a selected
 * candidate, or not an earlier node (a pool that is not a tree) is detached:
 * parent -1, its mask row and depth from its own chain, and no link from the
 * root reaches it or its subtree, so the verify never visits them. */
int spec_build_tree(int B, int k, int num_steps, int N, const float* pool_score,
                    const int32_t* pool_token, const int32_t* pool_parent,
                    const int32_t* pool_qrow, const int32_t* root_token, const int32_t* seq_lens,
                    int32_t* draft_token, int32_t* parent, int32_t* positions, uint8_t* tree_mask,
                    int32_t* retrieve_index, int32_t* retrieve_next_token,
                    int32_t* retrieve_next_sibling, int32_t* q_row, spec_stream_t stream);

/* ----------------------------------------------------------------- verify */

/* The bounded wait the stochastic verify's CTAs use on each other's row
 * flags, exposed for testing its failure path: one thread waits until
 * *flag != 0 (acquire load at GPU scope) or limit_cycles SM clock cycles
 * pass.  *seen = 1 if the flag was seen; on timeout *seen = 0 and
 * SPEC_STAT_WAIT_TIMEOUT is counted in stats_or_null.  The kernel always
 * returns, so a flag that nothing sets costs limit_cycles and leaves the
 * context usable. */
int spec_wait_probe(const int32_t* flag, int64_t limit_cycles, int32_t* stats_or_null, int32_t* seen,
                    spec_stream_t stream);

/* Bounds-check count of the debug build, libspecdec_debug.so (the same
 * sources compiled with -DSPEC_DEBUG).  No page of the method has a
 * counterpart: it stands in for a memory checker.  In that build every kernel
 * tests the indices it reads and writes through that depend on its inputs
 * (token ids, node links, row numbers, pool and slot ids, chunk and slot
 * counters, shared-memory positions) against the extent of the buffer they
 * index, skips an access that falls outside and counts it: in
 * SPEC_STAT_BOUNDS of the call's stats_or_null, and in a device counter
 * kept per source file.  spec_debug_bounds synchronises the device, writes
 * the sum of those counters since the last reset to *count and zeroes them
 * when reset != 0.  The release library returns SPEC_ERR_UNSUPPORTED and
 * writes nothing. */
int spec_debug_bounds(int64_t* count, int reset);

/* Scratch bytes for spec_verify_greedy / spec_verify_sample (per-row
 * max, normaliser, argmax or ready flag and claim of the target logits, and
 * the chain verify's per-request state). */
size_t spec_verify_ws_size(int B, int N);

/* Greedy verify ([ZS] 4.1 greedy_commit, generalised to trees).  One pass
 * over every target row computes its argmax (lowest index on ties); then per
 * request, from the root: t = argmax(row n) is committed; a child carrying t
 * is accepted (its KV is valid); the walk stops when t == eos_id, when the
 * budget is used, or when no child carries t (t is then the correction, or
 * the bonus at a leaf); otherwise it descends into the child.
 *   target_logits [B, N, V] (dtype)
 *   draft_token, retrieve_next_token, retrieve_next_sibling [B, N] int32
 *     (as written by spec_build_tree; any tree whose children have larger
 *     node indices than their parent works)
 *   budget_or_null [B] remaining output tokens (<= 0: commit nothing);
 *     NULL = no limit.  eos_id < 0: none.
 * Outputs: committed [B, N] (-1 padded), num_committed [B], accept_length [B]
 * (accepted drafts), accept_path [B, N] (node ids from 0, -1 padded),
 * next_root [B] (last committed token, -1 if none), walk_info_or_null [B, 3]
 * = (final node, children rejected over the walk, SPEC_FINAL_*).
 * ws: spec_verify_ws_size(B, N) bytes, 256-byte aligned. */
int spec_verify_greedy(int B, int N, int64_t V, int dtype, const void* target_logits,
                       const int32_t* draft_token, const int32_t* retrieve_next_token,
                       const int32_t* retrieve_next_sibling, const int32_t* budget_or_null,
                       int32_t eos_id, int32_t* committed, int32_t* num_committed,
                       int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                       int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                       size_t ws_bytes, spec_stream_t stream);

/* Stochastic verify ([ZS] 5.1).  p_n = softmax(target row n / T).  At node
 * n the children are tried in sibling order: child c with draft token y is
 * accepted iff coins[b, c] < p_cur[y] / q_n[y] (acceptance probability
 * min(1, p/q)); each rejection replaces p_cur by the normalised positive
 * residual (p_cur - q_n)+ and the next sibling is tried; if no child is
 * accepted (or n is a leaf) one token is drawn from p_cur by inverse CDF with
 * u_final[b] (the correction after a rejection, or the bonus from p after
 * full acceptance).  EOS and budget end the walk after any committed token.
 * q[y] == 0 accepts iff p_cur[y] > 0.  A residual without positive mass
 * leaves p_cur unchanged (SPEC_STAT_RESIDUAL_FALLBACK).
 *   q             draft distributions, fp32 rows of length V.  With
 *                 q_row_or_null, node n's row is q + q_row[b*N+n]*V (the
 *                 step-major draft-row table, q_row from spec_build_tree);
 *                 with NULL, q is [B, N, V] in node order.  Only rows of
 *                 nodes with children are read.
 *   coins [B, N]  uniform per child node (index 0 unused); u_final [B].
 * Other arguments and outputs as spec_verify_greedy. */
int spec_verify_sample(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                       const float* q, const int32_t* q_row_or_null, const int32_t* draft_token,
                       const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                       const float* coins, const float* u_final, const int32_t* budget_or_null,
                       int32_t eos_id, int32_t* committed, int32_t* num_committed,
                       int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                       int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                       size_t ws_bytes, spec_stream_t stream);

/* Stochastic verify with the draft distribution given in logit form: node
 * n's q row is q[v] = 2^((l_v - m) log2(e)/T_q) / Z of draft-logit row
 * r = q_row[b*N+n] (NULL: r = b*N+n), with (m, Z) = q_stats[r] as written by
 * spec_softmax_topk's row_stats.  These are bit-for-bit the probabilities
 * spec_softmax_topk would have written (rows whose maximum is not finite
 * give q = 0), so the result equals spec_verify_sample on the materialised
 * q, while the draft side writes no q and verify reads a rejected node's
 * draft row in the logits' dtype instead of fp32.  The rule is [ZS] 5.1's,
 * as in spec_verify_sample ([ZS] 5.2: the verify input carries the draft
 * distributions; their storage form is free).
 *   q_logits [rows, V] (q_dtype), q_stats [rows, 2] fp32, T_q > 0.
 * Other arguments and outputs as spec_verify_sample. */
int spec_verify_sample_qlogits(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                               const void* q_logits, int q_dtype, const float* q_stats, float T_q,
                               const int32_t* q_row_or_null, const int32_t* draft_token,
                               const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                               const float* coins, const float* u_final, const int32_t* budget_or_null,
                               int32_t eos_id, int32_t* committed, int32_t* num_committed,
                               int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                               int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                               size_t ws_bytes, spec_stream_t stream);

/* Sibling update for children drawn without replacement (the variant the
 * pages name beside the sibling-sequential residual rule: the rejected token's
 * q is zeroed and q renormalised).  At a node, q_cur starts as the node's q;
 * after child y is rejected, p_cur becomes the normalised positive residual
 * of p_cur and q_cur, then q_cur[y] = 0 and q_cur is renormalised; the next
 * sibling y' is accepted iff coin < p_cur[y'] / q_cur[y'].  With children
 * drawn from q without replacement this keeps the target's law exactly.  The
 * q row is taken as a distribution (it sums to 1): the renormalisation
 * divides by 1 minus the rejected tokens' q. */
#define SPEC_VERIFY_WITHOUT_REPLACEMENT 1

/* The caller's trees are chains: every node has at most one child (topk = 1
 * drafting, [ZS] 3.3's k drafts in a row).  The acceptance test at node n
 * then reads only row n, q row n and the child's coin, so the launch tests
 * every node right after its row's statistics and resolves each request as
 * soon as the rows on its path are done; the one draw a request needs (the
 * residual at its first rejection, or p at its leaf) is cut into chunks that
 * any CTA takes.  The rule and every decision's arithmetic are those of the
 * tree walk; only the order of the draw's partial sums differs, so a drawn
 * token can differ only at a CDF boundary.  A node with more than one child
 * has only its first child tested and counts SPEC_STAT_BAD_REQUEST.  With one
 * child per node, SPEC_VERIFY_WITHOUT_REPLACEMENT changes nothing. */
#define SPEC_VERIFY_CHAIN 2

/* spec_verify_sample / spec_verify_sample_qlogits with flags: 0 (the same
 * call), SPEC_VERIFY_WITHOUT_REPLACEMENT and / or SPEC_VERIFY_CHAIN; other
 * bits give SPEC_ERR_INVALID_ARG. */
int spec_verify_sample_flags(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                             const float* q, const int32_t* q_row_or_null, const int32_t* draft_token,
                             const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                             const float* coins, const float* u_final, const int32_t* budget_or_null,
                             int32_t eos_id, int32_t* committed, int32_t* num_committed,
                             int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                             int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                             size_t ws_bytes, int flags, spec_stream_t stream);
int spec_verify_sample_qlogits_flags(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                     const void* q_logits, int q_dtype, const float* q_stats, float T_q,
                                     const int32_t* q_row_or_null, const int32_t* draft_token,
                                     const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                     const float* coins, const float* u_final, const int32_t* budget_or_null,
                                     int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                     int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                     int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                     size_t ws_bytes, int flags, spec_stream_t stream);

/* The committed ids mapped back to the draft vocabulary in the same launch
 * ([TLI] Modifications: map_target_to_draft_ids, applied to the accepted and
 * drawn target ids before the next draft step; hook
 * forward_draft_extend_after_decode).  out[b*N + i] = table[committed[b*N +
 * i]] when that id is in [0, table_len) and the entry is >= 0, else
 * fallback_id; -1 where committed is -1. */
typedef struct spec_id_map {
  const int32_t* table;  /* [table_len] device, e.g. t2d */
  int64_t table_len;
  int32_t fallback_id;
  int32_t* out;          /* [B, N] device */
} spec_id_map_t;

/* spec_verify_sample_qlogits_flags with the id map above fused into its
 * epilogue.  flags must include SPEC_VERIFY_CHAIN (TLI drafts are chains:
 * tli_check_config); SPEC_ERR_INVALID_ARG otherwise, or for a NULL map,
 * table or out, or table_len < 1. */
int spec_verify_sample_qlogits_mapped(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                      const void* q_logits, int q_dtype, const float* q_stats, float T_q,
                                      const int32_t* q_row_or_null, const int32_t* draft_token,
                                      const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                      const float* coins, const float* u_final, const int32_t* budget_or_null,
                                      int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                      int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                      int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                      size_t ws_bytes, int flags, const spec_id_map_t* map, spec_stream_t stream);

/* Greedy verify without caller scratch.  No passage of the pages has a
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory at all -- a plugin that receives only its input and output
 * buffers from a host framework that owns every byte of device memory, or a
 * real-time path that must not call cudaMalloc (which can block and
 * synchronise the device).  It behaves exactly like spec_verify_greedy
 * (same arguments, minus ws / ws_bytes), but keeps the per-row argmax in a
 * fixed array of device memory inside the library.  That array holds
 * SPEC_NOALLOC_MAX_ROWS rows (1 MiB), every GPU that loads the library keeps
 * it until the process exits, and calls with B*N above it return
 * SPEC_ERR_UNSUPPORTED.  The array is shared: calls whose work overlaps on
 * the GPU (different streams, no ordering between them) race on it and give
 * undefined results; calls ordered on one stream are safe.  The first call
 * on each device looks up the array's device address (cudaGetSymbolAddress),
 * so make that first call before any stream capture.  Nothing is allocated,
 * by this call or by the library. */
#define SPEC_NOALLOC_MAX_ROWS (1 << 18)
int spec_verify_greedy_noalloc(int B, int N, int64_t V, int dtype, const void* target_logits,
                               const int32_t* draft_token, const int32_t* retrieve_next_token,
                               const int32_t* retrieve_next_sibling, const int32_t* budget_or_null,
                               int32_t eos_id, int32_t* committed, int32_t* num_committed,
                               int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                               int32_t* walk_info_or_null, int32_t* stats_or_null,
                               spec_stream_t stream);

/* Target-side top-k / top-p filtering ([ZS] 5.1: with temperature, top-k or
 * top-p in force, verification uses the processed target probabilities), in
 * place on logit rows.  Per row, with p = softmax(row / T) and tokens ordered
 * by (p desc, index asc) -- the order of the logits: top_k > 0 (and < V)
 * keeps the first top_k; top_p < 1 then keeps every token whose exclusive
 * prefix mass is below top_p times the top-k mass (the first token always
 * stays; top_p <= 0 keeps it alone).  Every other logit is set to -inf, so
 * softmax of the filtered row is the renormalised filtered p, and
 * spec_verify_sample / spec_verify_sample_qlogits run on the filtered rows
 * verify against it.  NaN counts as -inf; rows without a finite maximum are
 * left as they are (SPEC_STAT_NONFINITE_ROW).  Masses are compared in 2^-40
 * fixed point (exact sums, a deterministic cut).
 *   logits [R, V] (dtype), modified in place.  top_k <= 0 and top_p >= 1:
 *   nothing to do. */
int spec_filter_logits(void* logits, int dtype, int64_t R, int64_t V, float T, int64_t top_k, float top_p,
                       int32_t* stats_or_null, spec_stream_t stream);

/* ------------------------------------------------------------- compaction */

/* Capacity (entries) the freed list of spec_compact_slots needs. */
int64_t spec_compact_freed_capacity(int B, int N, int page_size);

/* Accepted-path KV-slot compaction ([HB] "Drafting, verification and
 * slots": slots for every candidate are allocated before drafting, only the
 * accepted path's are kept, and with a page size above 1 data must be
 * copied; [ZS] 5.2: the cache returns to the committed path and the
 * correction/bonus token has no KV yet).
 * Layout: tree node n occupies logical position seq_len + n, physical slot
 * req_to_token[b*max_ctx + seq_len + n]; with page_size P, slot = page*P +
 * position % P.  Root + accepted nodes stay: new_kv_len = seq_len + 1 +
 * accept_length.
 *   page_size == 1: req_to_token[seq_len + i] = old slot of node path[i]
 *     (i = 1..accept_length); the slots of nodes off the path are freed in
 *     node order; no moves.
 *   page_size > 1: for i = 1..accept_length with path[i] != i a move
 *     (src = slot(seq_len + path[i]), dst = slot(seq_len + i)) is emitted in
 *     move_src/move_dst [B, N] (num_moves [B]); with kv_pool_or_null
 *     ([num_slots, bytes_per_slot] bytes) the payload is copied in place
 *     with the semantics of copying in increasing i (sources are read before
 *     any overlapping destination is written).  Pages this step first
 *     touched (first position in [seq_len, seq_len + N)) whose first position
 *     is >= new_kv_len are freed (page id = slot / page_size).
 *   freed [capacity] is compacted across requests in (b, node/page) order;
 *   num_freed [1] receives the count.
 * A request with seq_len < 0, seq_len + N > max_ctx, accept_length outside
 * [0, N), or a slot outside [0, num_slots) when copying, is skipped
 * (new_kv_len = -1, SPEC_STAT_BAD_REQUEST). */
int spec_compact_slots(int B, int N, int page_size, const int32_t* seq_lens,
                       const int32_t* accept_path, const int32_t* accept_length,
                       int32_t* req_to_token, int64_t max_ctx, int32_t* move_src,
                       int32_t* move_dst, int32_t* num_moves, int32_t* freed,
                       int64_t freed_capacity, int32_t* num_freed, int32_t* new_kv_len,
                       void* kv_pool_or_null, int64_t num_slots, int64_t bytes_per_slot,
                       int32_t* stats_or_null, spec_stream_t stream);

/* -------------------------------------------------------------------- TLI */

/* TLI constrain + top-1 + map ([TLI] Modifications: constrain_draft_logits
 * sets non-intersection draft logits to -inf before the top-k;
 * map_draft_to_target_ids maps the chosen id; TLI requires topk == 1).
 *   draft_logits [R, V_d] (dtype).
 *   d2t [V_d] target id of each draft id, -1 outside the intersection.
 *   t2d_or_null [V_t] its inverse on the intersection (-1 elsewhere);
 *     required when q_target_or_null is given.
 *   top1_draft / top1_target [R]: argmax over the intersection by
 *     (logit desc, index asc) and its target id; top1_p [R]: its probability
 *     under the constrained softmax at temperature T.
 *   q_target_or_null [R, V_t] fp32: the constrained draft distribution in
 *     target-vocabulary order (0 off the intersection) -- the q that
 *     stochastic verify reads.
 * A row with no finite intersection logit gets -1 / -1 / 0, a zero q row and
 * counts in SPEC_STAT_EMPTY_INTERSECTION. */
int tli_constrain_map(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                      const int32_t* d2t, const int32_t* t2d_or_null, float T,
                      int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                      float* q_target_or_null, int32_t* stats_or_null, spec_stream_t stream);

/* Map plan of a vocabulary pair ([TLI] Modifications: vocab_mapping.py
 * builds the id maps once per model pair).  The plan is derived from d2t and
 * t2d alone and lets tli_constrain_map_planned keep the intersection in
 * shared memory:
 *   int32 K (the number of ids with d2t >= 0) and 3 pad words;
 *   uint2 mw[Wp], Wp = ceil(V_d / 32) rounded up to even: .x bit j set when
 *     d2t[32 w + j] >= 0, .y the number of set bits in words before w;
 *   int32 t2r[V_t rounded up to 4]: for target id t with d = t2d[t],
 *     0 <= d < V_d and d in the intersection: the rank of d among the
 *     intersection ids in increasing id order; -1 when t2d[t] < 0 or
 *     d >= V_d (and for the pad entries); -2 - d when d is outside the
 *     intersection.
 * tli_plan_bytes: its size in bytes (-1 for sizes out of range).
 * tli_plan_build: fills `plan` (device, 16-byte aligned, caller-owned,
 * tli_plan_bytes(V_d, V_t) bytes) from d2t [V_d] and t2d [V_t], in stream
 * order (three launches). */
int64_t tli_plan_bytes(int64_t V_d, int64_t V_t);
int tli_plan_build(int64_t V_d, int64_t V_t, const int32_t* d2t, const int32_t* t2d, void* plan,
                   spec_stream_t stream);

/* tli_constrain_map with a plan built by tli_plan_build from the same d2t
 * and t2d (the outputs are the same).  Persistent CTAs keep the plan's
 * bitmap and, when they fit, the row's intersection logits in shared
 * memory; a draft vocabulary whose bitmap does not fit falls back to
 * tli_constrain_map. */
int tli_constrain_map_planned(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                              const int32_t* d2t, const int32_t* t2d_or_null, const void* plan, float T,
                              int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                              float* q_target_or_null, int32_t* stats_or_null, spec_stream_t stream);

/* tli_constrain_map_planned with the step's pool expansion fused (a chain:
 * expand->k == 1, R = expand->B; the mapped top-1 and its probability are
 * the step's top-1). */
int tli_constrain_map_planned_expand(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                                     const int32_t* d2t, const int32_t* t2d_or_null, const void* plan, float T,
                                     int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                                     float* q_target_or_null, int32_t* stats_or_null, const spec_expand_t* expand,
                                     spec_stream_t stream);

/* tli_constrain_map with the constrained draft distribution written in logit
 * form instead of fp32 probabilities (half the bytes for bf16 logits), for
 * spec_verify_sample_qlogits:
 *   q_logits_target [R, V_t] (dtype) out: element t is the draft logit (its
 *     raw bits) of t's partner d = t2d[t] when 0 <= d < V_d, -inf otherwise;
 *   q_stats [R, 2] fp32 out: (m, Z), m the row's largest intersection key
 *     (NaN counted as -inf; -inf for a row with no finite intersection
 *     logit) and Z = sum over the intersection of 2^((key - m) log2(e) / T).
 * spec_verify_sample_qlogits(..., q_logits = q_logits_target, q_dtype =
 * dtype, q_stats, T_q = T) then reads q[t] = min(2^((key_t - m) log2(e) / T)
 * / Z, 1), bit for bit the probabilities tli_constrain_map writes.
 * t2d is required.  plan_or_null: a plan from tli_plan_build (the persistent
 * kernel of tli_constrain_map_planned) or NULL (the per-row kernel).
 * expand_or_null: the step's pool expansion, as in
 * tli_constrain_map_planned_expand.  The top-1 outputs and error behaviour
 * are those of tli_constrain_map; q_logits_target must be element aligned
 * (16-byte aligned rows take vector stores). */
int tli_constrain_map_qlogits(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                              const int32_t* d2t, const int32_t* t2d, const void* plan_or_null, float T,
                              int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                              void* q_logits_target, float* q_stats, int32_t* stats_or_null,
                              const spec_expand_t* expand_or_null, spec_stream_t stream);

/* Id remapping in either direction ([TLI] Modifications:
 * map_target_to_draft_ids / map_draft_to_target_ids): out[i] = table[in[i]]
 * when 0 <= in[i] < table_len and that entry is >= 0, else fallback_id (the
 * unk id, or eos for models without one). */
int tli_map_ids(const int32_t* in, int32_t* out, int64_t n, const int32_t* table,
                int64_t table_len, int32_t fallback_id, spec_stream_t stream);

/* Pruned draft LM head ([TLI] Modifications: _try_prune_draft_lm_head /
 * _PrunedReindexLMHead keep only the LM-head weight rows of the
 * intersection's draft ids, so the draft logits cost O(M K H) instead of
 * O(M V_d H); the constrained top-1 and its mapping follow as in
 * tli_constrain_map, over those K logits).  A tensor-core GEMM (tcgen05,
 * bf16 operands, fp32 accumulation in tensor memory) with the reduction
 * fused into its epilogue:
 *   logits[m][k] = sum over h of hidden[m][h] * weight[k][h].
 *   hidden [M, H] bf16, weight [K, H] bf16 (row k: the LM-head row of draft
 *     id ids[k]), both row-major, 16-byte aligned, H a multiple of 8
 *     (SPEC_ERR_UNSUPPORTED otherwise).
 *   ids [K] int32: the draft id of each weight row, ascending (so ties, which
 *     go to the lower row, go to the lower draft id); d2t [V_d].
 *   top1_draft / top1_target [M] int32: ids[k*] and d2t[ids[k*]] of the
 *     largest logit; top1_p [M]: its probability at temperature T over the K
 *     logits; top1_rank_or_null [M]: k*.
 *   row_stats_or_null [M, 2] fp32: each row's max logit and
 *     sum 2^((l - max) log2(e)/T).
 *   logits_or_null [M, K] fp32: the logits themselves.
 *   ws: tli_pruned_head_ws_size(M, K) bytes, 256-byte aligned (per-tile
 *     partials of the reduction).
 * A row with no finite logit gets -1 ids, probability 0 and counts in
 * SPEC_STAT_EMPTY_INTERSECTION.  Its waits are bounded: one that runs out is
 * counted in SPEC_STAT_WAIT_TIMEOUT (results void). */
size_t tli_pruned_head_ws_size(int64_t M, int64_t K);
int tli_pruned_head(int64_t M, int64_t H, int64_t K, const void* hidden, const void* weight,
                    const int32_t* ids, const int32_t* d2t, int64_t V_d, float T, int32_t* top1_draft,
                    int32_t* top1_target, float* top1_p, int32_t* top1_rank_or_null,
                    float* row_stats_or_null, float* logits_or_null, int32_t* stats_or_null, void* ws,
                    size_t ws_bytes, spec_stream_t stream);

/* TLI configuration check ([TLI] Modifications, server_args validation):
 * SPEC_OK iff topk == 1, num_steps >= 1 and num_draft_tokens ==
 * num_steps + 1.  Host only. */
int tli_check_config(int topk, int num_steps, int num_draft_tokens);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_H */
