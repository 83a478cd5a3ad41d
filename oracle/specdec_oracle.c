/*
 * CPU oracle for the speculative-decoding draft/verify path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * statement of what every step of the path computes.  Only the test suite,
 * the smoke check and the bench's CPU-baseline leg may load it.  The CUDA
 * library never includes, links or calls it, and it shares no header, helper
 * or constant with the CUDA sources.
 *
 * Arithmetic: fp64 throughout, except where the method itself fixes fp32
 * (tree scores are fp32 products of fp32 draft probabilities, so the tree is
 * decided in the precision both sides receive).  Everything runs row by row
 * in index order; no blocking, fusion or reordering.
 *
 * Sources (web pages; cited by title and section):
 *   [HB]  ai-infra-handbooks, "EAGLE speculative decoding in four parts: why
 *         it became a worker", sections "Drafting, verification and slots"
 *         and "Exercises".
 *   [ML]  secrett2633 blog, "[SGLang] Multi-Layer EAGLE", section 2 (draft
 *         step: select_top_k_tokens and tree_info) and section 3 (per-step
 *         softmax then fast_topk).
 *   [ZS]  zero-to-sglang ch.10 "Speculative decoding (code walk-through)",
 *         sections 3.2 (greedy drafting, EOS), 3.3 (row alignment),
 *         4.1-4.2 (greedy commitment, worked rejection), 5.1 (stochastic
 *         acceptance, positive residual, worked example), 5.2 (verify input
 *         and KV restore).
 *   [TLI] SGLang PR #22883 "TLI (Token-Level Intersection)", section
 *         "Modifications" (vocab_mapping.py exports, TLIWorker hooks,
 *         server_args validation).
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes):
 *   - Ties in argmax / top-k go to the lowest index ([ZS] 4.2 asks for
 *     fixed tie handling).  NaN logits are treated as -inf.
 *   - Tree scores are products of draft probabilities along the path; the
 *     candidate pool keeps all k*k expansions of every step; the tree takes
 *     the N-1 best candidates by (score desc, pool id asc) and orders nodes
 *     by ascending pool id.
 *   - Stochastic tree verify is sibling-sequential residual rejection: at a
 *     node, children are tried in sibling order against the current
 *     distribution p_cur, which after each rejection becomes the normalised
 *     positive residual (p_cur - q)+.
 *   - q[y] == 0 accepts iff p_cur[y] > 0 (IEEE: p/0 = +inf, 0/0 = NaN).
 *   - A residual with no positive mass leaves p_cur unchanged (counted).
 *   - Sampling is by inverse CDF over vocabulary order: the smallest v whose
 *     inclusive prefix sum exceeds u times the total; if rounding leaves no
 *     such v, the last v with positive weight (counted).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR -1

#define KIND_NONE 0
#define KIND_CORRECTION 1
#define KIND_BONUS 2

/* ---------------------------------------------------------------- inputs */

/* Element i of a logit buffer as a double.  dtype 0 = fp32, 1 = bf16
 * (upper 16 bits of an fp32; widening is exact). */
static double logit_at(const void* p, int dtype, int64_t i)
{
    if (dtype == 0) return (double)((const float*)p)[i];
    uint32_t w = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Ordering key of a logit: NaN behaves as -inf. */
static double order_key(double x) { return isnan(x) ? -INFINITY : x; }

/* ------------------------------------------------- softmax and top-k (A1) */

/* [ML] section 3: each draft step takes probs = softmax(logits) and then
 * topk_p, topk_index = top-k(probs); those topk_p are the tree scores, so
 * they come from a plain softmax: T_score = 1 in the draft loop.
 * [ZS] 5.1: the draft distribution q that verification reads is the
 * processed one, p_v = exp((l_v - max l)/T) / sum_u exp((l_u - max l)/T),
 * written to probs_or_null at the temperature T.
 * topk_p are the top-k tokens' probabilities under T_score.  Top-k is taken
 * on the logits (same order as on the probabilities at any temperature, no
 * rounding ties), by (logit desc, index asc).  A row whose maximum is not
 * finite gets probability 0 everywhere and row_flag = 1. */
int oracle_softmax_topk(const void* logits, int dtype, int64_t R, int64_t V,
                        double T, double T_score, int k, double* topk_p,
                        int32_t* topk_idx, double* probs_or_null, int32_t* row_flag)
{
    if (R < 0 || V <= 0 || k < 0 || k > V || !(T > 0.0) || !(T_score > 0.0)) return OR_ERR;
    char* taken = (char*)malloc((size_t)V);
    if (!taken) return OR_ERR;
    for (int64_t r = 0; r < R; ++r) {
        int64_t base = r * V;
        double m = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double x = order_key(logit_at(logits, dtype, base + v));
            if (x > m) m = x;
        }
        int finite = isfinite(m);
        double Z = 0.0, Zs = 0.0;  /* normalisers at T and at T_score */
        if (finite)
            for (int64_t v = 0; v < V; ++v) {
                double x = order_key(logit_at(logits, dtype, base + v));
                Z += exp((x - m) / T);
                Zs += exp((x - m) / T_score);
            }
        memset(taken, 0, (size_t)V);
        for (int j = 0; j < k; ++j) {
            int64_t best = -1;
            double bx = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                if (taken[v]) continue;
                double x = order_key(logit_at(logits, dtype, base + v));
                if (best < 0 || x > bx) { best = v; bx = x; }
            }
            taken[best] = 1;
            topk_idx[r * k + j] = (int32_t)best;
            topk_p[r * k + j] = finite ? exp((bx - m) / T_score) / Zs : 0.0;
        }
        if (probs_or_null)
            for (int64_t v = 0; v < V; ++v)
                probs_or_null[base + v] =
                    finite ? exp((order_key(logit_at(logits, dtype, base + v)) - m) / T) / Z : 0.0;
        row_flag[r] = !finite;
    }
    free(taken);
    return OR_OK;
}

/* ------------------------------------------------- inverse-CDF sampling */

/* Sample from non-negative weights w[0..V) with uniform u in [0,1):
 * the smallest v with C_v > u * W, C the inclusive prefix sum and W = C_{V-1}.
 * This is the categorical draw the [ZS] 5.1 fragment makes with multinomial,
 * written as an inverse CDF over vocabulary order.  *margin receives the
 * distance from u to the nearest of the two normalised CDF boundaries around
 * the chosen v.  Returns 1 when rounding or an empty distribution forced the
 * fallback (last index with positive weight, or 0 when there is none). */
static int sample_inverse_cdf(const double* w, int64_t V, double u,
                              int32_t* tok, double* margin)
{
    double W = 0.0;
    for (int64_t v = 0; v < V; ++v) W += w[v];
    *margin = INFINITY;
    if (!(W > 0.0) || !isfinite(W)) {
        *tok = 0;
        for (int64_t v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { *tok = (int32_t)v; break; }
        *margin = 0.0;
        return 1;
    }
    double target = u * W, C = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double before = C;
        C += w[v];
        if (C > target) {
            *tok = (int32_t)v;
            double a = fabs(u - before / W), b = fabs(u - C / W);
            *margin = a < b ? a : b;
            return 0;
        }
    }
    for (int64_t v = V - 1; v >= 0; --v)
        if (w[v] > 0.0) { *tok = (int32_t)v; break; }
    *margin = 0.0;
    return 1;
}

/* Draft-side sampling: a token from softmax(logits/T) of each row, or from
 * the given probability rows, with one uniform per row.  out_prob receives
 * the sampled token's probability (normalised). */
int oracle_sample(const void* logits_or_null, int dtype, const float* probs_or_null,
                  int64_t R, int64_t V, double T, const float* u,
                  int32_t* out_token, double* out_prob, double* margin,
                  int32_t* fallback)
{
    if (R < 0 || V <= 0) return OR_ERR;
    if (!logits_or_null && !probs_or_null) return OR_ERR;
    if (!probs_or_null && !(T > 0.0)) return OR_ERR;
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!w) return OR_ERR;
    for (int64_t r = 0; r < R; ++r) {
        int64_t base = r * V;
        if (probs_or_null) {
            for (int64_t v = 0; v < V; ++v) w[v] = (double)probs_or_null[base + v];
        } else {
            double m = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                double x = order_key(logit_at(logits_or_null, dtype, base + v));
                if (x > m) m = x;
            }
            for (int64_t v = 0; v < V; ++v)
                w[v] = isfinite(m)
                    ? exp((order_key(logit_at(logits_or_null, dtype, base + v)) - m) / T) : 0.0;
        }
        double W = 0.0;
        for (int64_t v = 0; v < V; ++v) W += w[v];
        fallback[r] = sample_inverse_cdf(w, V, (double)u[r], &out_token[r], &margin[r]);
        out_prob[r] = W > 0.0 ? w[out_token[r]] / W : 0.0;
    }
    free(w);
    return OR_OK;
}

/* --------------------------------------------------- tree expansion (A2) */

typedef struct { float score; int32_t id; } scored_t;

/* (score desc, id asc); a NaN score sorts as -inf. */
static int better_first(const void* a, const void* b)
{
    const scored_t* x = (const scored_t*)a;
    const scored_t* y = (const scored_t*)b;
    float sx = isnan(x->score) ? -INFINITY : x->score;
    float sy = isnan(y->score) ? -INFINITY : y->score;
    if (sx > sy) return -1;
    if (sx < sy) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

int64_t oracle_pool_size(int k, int num_steps)
{
    return 1 + (int64_t)k + (int64_t)(num_steps - 1) * k * k;
}

/* One draft step of [ML] section 2's select_top_k_tokens, whose tree_info is
 * (scores, tokens, parents).
 *  step 0: the root's k children, score = topk_p of the root row.
 *  step s >= 1: every frontier node f (k of them) expands into its k
 *  children, score = score_f * topk_p[f][j] (one fp32 multiply), parent f.
 * All expansions enter the candidate pool.  The next frontier is the best k
 * of this step's candidates by (score desc, pool id asc).
 * Pool ids: 0 root; 1..k step 0 by rank; then step s at
 * 1 + k + (s-1)k^2 + f*k + j.
 * pool_qrow records, for each candidate that becomes a frontier node, the
 * row of the step-major draft-row table that holds its draft distribution:
 * step 0 uses rows [0, B) (the roots), step t >= 1 uses rows
 * B + (t-1)Bk + b*k + slot.  Candidates never expanded keep -1. */
int oracle_tree_expand(int step, int num_steps, int B, int k,
                       const float* topk_p, const int32_t* topk_idx,
                       float* pool_score, int32_t* pool_token,
                       int32_t* pool_parent, int32_t* pool_qrow,
                       float* frontier_score, int32_t* frontier_id)
{
    if (B < 0 || k < 1 || num_steps < 1 || step < 0 || step >= num_steps) return OR_ERR;
    int64_t P = oracle_pool_size(k, num_steps);
    int nc = step == 0 ? k : k * k;
    scored_t* cand = (scored_t*)malloc(sizeof(scored_t) * (size_t)nc);
    if (!cand) return OR_ERR;
    for (int b = 0; b < B; ++b) {
        float* sc = pool_score + (int64_t)b * P;
        int32_t* tk = pool_token + (int64_t)b * P;
        int32_t* pa = pool_parent + (int64_t)b * P;
        int32_t* qr = pool_qrow + (int64_t)b * P;
        int64_t base;
        if (step == 0) {
            for (int64_t i = 0; i < P; ++i) { sc[i] = 0.0f; tk[i] = -1; pa[i] = -1; qr[i] = -1; }
            sc[0] = 1.0f;
            qr[0] = b;
            base = 1;
            for (int j = 0; j < k; ++j) {
                sc[base + j] = topk_p[(int64_t)b * k + j];
                tk[base + j] = topk_idx[(int64_t)b * k + j];
                pa[base + j] = 0;
            }
        } else {
            base = 1 + (int64_t)k + (int64_t)(step - 1) * k * k;
            for (int f = 0; f < k; ++f) {
                float parent_score = frontier_score[(int64_t)b * k + f];
                int32_t parent_id = frontier_id[(int64_t)b * k + f];
                for (int j = 0; j < k; ++j) {
                    int64_t row = ((int64_t)b * k + f) * k + j;
                    volatile float prod = parent_score * topk_p[row];
                    sc[base + f * k + j] = prod;
                    tk[base + f * k + j] = topk_idx[row];
                    pa[base + f * k + j] = parent_id;
                }
            }
        }
        for (int c = 0; c < nc; ++c) { cand[c].score = sc[base + c]; cand[c].id = (int32_t)(base + c); }
        qsort(cand, (size_t)nc, sizeof(scored_t), better_first);
        for (int slot = 0; slot < k; ++slot) {
            frontier_score[(int64_t)b * k + slot] = cand[slot].score;
            frontier_id[(int64_t)b * k + slot] = cand[slot].id;
            if (step + 1 < num_steps)
                qr[cand[slot].id] = B + step * B * k + b * k + slot;
        }
    }
    free(cand);
    return OR_OK;
}

/* ------------------------------------------------------- tree build (A3) */

/* [HB] "Drafting, verification and slots": build_eagle_tree turns the
 * candidates into the tree and produces the attention mask and positions;
 * [ZS] 5.2 lists the verify input (draft_token, positions, custom_mask,
 * retrieve_*).  Node 0 is the root (last committed token).  The N-1 best pool
 * candidates by (score desc, pool id asc) become nodes 1..N-1 in ascending
 * pool-id order.
 *   parent[n]          node index of the parent (-1 for the root)
 *   positions[n]       seq_len + depth(n)
 *   tree_mask[n][m]    1 iff m is n or an ancestor of n
 *   retrieve_index[n]  b*N + n
 *   next_token[n]      first child in node order, -1 if none
 *   next_sibling[n]    next node with the same parent, -1 if none
 *   q_row[n]           draft-row table row of n's draft distribution, or -1
 * Returns OR_ERR if the selection is not ancestor-closed. */
int oracle_build_tree(int B, int k, int num_steps, int N,
                      const float* pool_score, const int32_t* pool_token,
                      const int32_t* pool_parent, const int32_t* pool_qrow,
                      const int32_t* root_token, const int32_t* seq_lens,
                      int32_t* draft_token, int32_t* parent, int32_t* positions,
                      uint8_t* tree_mask, int32_t* retrieve_index,
                      int32_t* next_token, int32_t* next_sibling, int32_t* q_row)
{
    int64_t P = oracle_pool_size(k, num_steps);
    if (B < 0 || N < 1 || N > P) return OR_ERR;
    scored_t* cand = (scored_t*)malloc(sizeof(scored_t) * (size_t)P);
    int32_t* node_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
    int32_t* pid_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    char* chosen = (char*)malloc((size_t)P);
    int rc = OR_OK;
    for (int b = 0; b < B && rc == OR_OK; ++b) {
        const float* sc = pool_score + (int64_t)b * P;
        const int32_t* tk = pool_token + (int64_t)b * P;
        const int32_t* pa = pool_parent + (int64_t)b * P;
        const int32_t* qr = pool_qrow + (int64_t)b * P;
        for (int64_t i = 1; i < P; ++i) { cand[i - 1].score = sc[i]; cand[i - 1].id = (int32_t)i; }
        qsort(cand, (size_t)(P - 1), sizeof(scored_t), better_first);
        memset(chosen, 0, (size_t)P);
        chosen[0] = 1;
        for (int i = 0; i < N - 1; ++i) chosen[cand[i].id] = 1;
        int n = 0;
        for (int64_t i = 0; i < P; ++i) {
            node_of[i] = -1;
            if (chosen[i]) { node_of[i] = n; pid_of[n] = (int32_t)i; ++n; }
        }
        int64_t o = (int64_t)b * N;
        for (n = 0; n < N; ++n) {
            int32_t pid = pid_of[n];
            if (n == 0) {
                parent[o] = -1;
                depth[0] = 0;
                draft_token[o] = root_token[b];
            } else {
                int32_t pp = pa[pid];
                if (pp < 0 || pp >= P || node_of[pp] < 0 || node_of[pp] >= n) { rc = OR_ERR; break; }
                parent[o + n] = node_of[pp];
                depth[n] = depth[node_of[pp]] + 1;
                draft_token[o + n] = tk[pid];
            }
            positions[o + n] = seq_lens[b] + depth[n];
            retrieve_index[o + n] = (int32_t)(o + n);
            q_row[o + n] = qr[pid];
        }
        if (rc != OR_OK) break;
        for (n = 0; n < N; ++n) {
            next_token[o + n] = -1;
            next_sibling[o + n] = -1;
            for (int c = n + 1; c < N; ++c)
                if (parent[o + c] == n) { next_token[o + n] = c; break; }
            if (n > 0)
                for (int c = n + 1; c < N; ++c)
                    if (parent[o + c] == parent[o + n]) { next_sibling[o + n] = c; break; }
            uint8_t* row = tree_mask + ((int64_t)b * N + n) * N;
            memset(row, 0, (size_t)N);
            for (int a = n; a >= 0; a = parent[o + a]) row[a] = 1;
        }
    }
    free(cand); free(node_of); free(pid_of); free(depth); free(chosen);
    return rc;
}

/* --------------------------------------------------- greedy verify (A4, A5) */

static int64_t argmax_row(const void* x, int dtype, int64_t base, int64_t V)
{
    int64_t best = 0;
    double bx = order_key(logit_at(x, dtype, base));
    for (int64_t v = 1; v < V; ++v) {
        double y = order_key(logit_at(x, dtype, base + v));
        if (y > bx) { bx = y; best = v; }
    }
    return best;
}

/* First child of node n (in sibling order) whose draft token is t, or -1.
 * *tested receives how many children were looked at without a match. */
static int32_t child_with_token(const int32_t* draft_token, const int32_t* next_token,
                                const int32_t* next_sibling, int64_t o, int32_t n,
                                int32_t t, int* tested)
{
    *tested = 0;
    for (int32_t c = next_token[o + n]; c >= 0; c = next_sibling[o + c]) {
        if (draft_token[o + c] == t) return c;
        ++*tested;
    }
    return -1;
}

/* [ZS] 4.1 greedy_commit, generalised from a chain to a tree.  Target row n
 * holds the next-token logits after root..n, so it verifies n's children
 * ([ZS] 3.3: row L-1+i verifies draft i; the last row gives the bonus).
 *   remaining == 0 -> nothing.
 *   at node n: t = argmax(row n); commit t; if a child carries t it is
 *   accepted; stop if t == eos or the budget is used; stop if no child
 *   matched (t is the correction, or the bonus at a leaf); else descend.
 * budget NULL = unlimited; eos < 0 = none.
 * walk_info[b] = (final node, rejected children over the walk, final kind:
 * 0 accepted draft, 1 correction, 2 bonus). */
int oracle_verify_greedy(int B, int N, int64_t V, int dtype, const void* target,
                         const int32_t* draft_token, const int32_t* next_token,
                         const int32_t* next_sibling, const int32_t* budget_or_null,
                         int32_t eos, int32_t* committed, int32_t* num_committed,
                         int32_t* accept_length, int32_t* accept_path,
                         int32_t* next_root, int32_t* walk_info)
{
    if (B < 0 || N < 1 || V < 1) return OR_ERR;
    for (int b = 0; b < B; ++b) {
        int64_t o = (int64_t)b * N;
        for (int i = 0; i < N; ++i) { committed[o + i] = -1; accept_path[o + i] = -1; }
        int64_t rem = budget_or_null ? budget_or_null[b] : N;
        int len = 0, acc = 0, rejected = 0, kind = KIND_NONE;
        int32_t n = 0;
        accept_path[o] = 0;
        if (rem > 0) {
            for (;;) {
                int32_t t = (int32_t)argmax_row(target, dtype, (o + n) * V, V);
                committed[o + len++] = t;
                int tested;
                int32_t c = child_with_token(draft_token, next_token, next_sibling, o, n, t, &tested);
                rejected += tested;
                if (c >= 0) { accept_path[o + ++acc] = c; }
                if (t == eos || len == rem || c < 0) {
                    if (c >= 0) { kind = KIND_NONE; n = c; }
                    else kind = next_token[o + n] < 0 ? KIND_BONUS : KIND_CORRECTION;
                    break;
                }
                n = c;
            }
        }
        num_committed[b] = len;
        accept_length[b] = acc;
        next_root[b] = len > 0 ? committed[o + len - 1] : -1;
        walk_info[3 * b + 0] = n;
        walk_info[3 * b + 1] = rejected;
        walk_info[3 * b + 2] = kind;
    }
    return OR_OK;
}

/* ------------------------------------------- stochastic verify (A4-A6) */

/* p = softmax(row / T) in fp64; returns 0 when the row max is not finite. */
static int softmax_row(const void* x, int dtype, int64_t base, int64_t V, double T, double* p)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double y = order_key(logit_at(x, dtype, base + v));
        if (y > m) m = y;
    }
    if (!isfinite(m)) {
        for (int64_t v = 0; v < V; ++v) p[v] = 0.0;
        return 0;
    }
    double Z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        p[v] = exp((order_key(logit_at(x, dtype, base + v)) - m) / T);
        Z += p[v];
    }
    for (int64_t v = 0; v < V; ++v) p[v] /= Z;
    return 1;
}

typedef struct { double p; int64_t id; } prob_t;

/* (p desc, id asc) */
static int prob_first(const void* a, const void* b)
{
    const prob_t* x = (const prob_t*)a;
    const prob_t* y = (const prob_t*)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* Target-side filtering of a probability row ([ZS] 5.1: with temperature,
 * top-k or top-p in force the processed probabilities are the ones
 * verification uses), in place.  Order the tokens by (p desc, index asc).
 * top_k > 0 keeps the first top_k of them (top_k <= 0 or >= V: all).
 * top_p < 1 then keeps, in the same order, every kept token whose exclusive
 * prefix of the top-k mass (renormalised) is below top_p; the first token
 * always stays, so the token that crosses top_p is kept.  The kept masses are
 * renormalised; the rest are 0.  A row from which nothing is dropped, and a
 * row of zeros, stay as they are. */
int oracle_filter_probs(int64_t V, double* p, int64_t top_k, double top_p)
{
    if (V < 1) return OR_ERR;
    prob_t* o = (prob_t*)malloc(sizeof(prob_t) * (size_t)V);
    if (!o) return OR_ERR;
    for (int64_t v = 0; v < V; ++v) { o[v].p = p[v]; o[v].id = v; }
    qsort(o, (size_t)V, sizeof(prob_t), prob_first);
    int64_t keep = (top_k > 0 && top_k < V) ? top_k : V;
    double mk = 0.0;
    for (int64_t i = 0; i < keep; ++i) mk += o[i].p;
    if (top_p < 1.0 && mk > 0.0) {
        double prefix = 0.0;
        int64_t n = 0;
        for (int64_t i = 0; i < keep; ++i) {
            if (i > 0 && !(prefix / mk < top_p)) break;
            prefix += o[i].p;
            n = i + 1;
        }
        keep = n;
    }
    if (keep == V) {  /* nothing dropped: the row stays as it is */
        free(o);
        return OR_OK;
    }
    double m = 0.0;
    for (int64_t i = 0; i < keep; ++i) m += o[i].p;
    for (int64_t v = 0; v < V; ++v) p[v] = 0.0;
    if (m > 0.0)
        for (int64_t i = 0; i < keep; ++i) p[o[i].id] = o[i].p / m;
    free(o);
    return OR_OK;
}

/* [ZS] 5.1: a draft y drawn from q is accepted with probability
 * min(1, p[y]/q[y]) (here: coin < p[y]/q[y]); on rejection the token comes
 * from the normalised positive residual (p - q)+; after full acceptance the
 * bonus comes from the target distribution.  On a tree the children of a
 * node are tried in sibling order; each rejection replaces p_cur by
 * (p_cur - q_n)+ / sum (p_cur - q_n)+ and the next sibling is tried against
 * it; if none is accepted the token is drawn from p_cur with u_final.
 * EOS and the budget are checked after every appended token as in greedy.
 * q_row_or_null: row of q for node n (q is then a table of rows); NULL means
 * q is [B, N, V] in node order.
 * margin[b] = smallest |u - boundary| over the request's decisions (accept
 * ratio, or the CDF boundaries around the drawn token): a GPU may disagree
 * only where this is below its tolerance.
 * counters[0] += q[y] == 0 events, counters[1] += residual fallbacks,
 * counters[2] += CDF fallbacks, counters[3] += non-finite target rows.
 * without_replacement != 0: the sibling update for children drawn without
 * replacement -- q_cur starts as the node's q, each rejection of y first
 * replaces p_cur by the residual of p_cur and q_cur, then sets q_cur[y] = 0
 * and renormalises q_cur (all zero once no mass is left); the acceptance
 * ratio of the next sibling is p_cur[y] / q_cur[y].
 * top_k / top_p: target-side filtering (oracle_filter_probs) of every target
 * row after its softmax; top_k <= 0 and top_p >= 1 leave p as it is. */
int oracle_verify_sample(int B, int N, int64_t V, int dtype, const void* target,
                         double T, const float* q, const int32_t* q_row_or_null,
                         const int32_t* draft_token, const int32_t* next_token,
                         const int32_t* next_sibling, const float* coins,
                         const float* u_final, const int32_t* budget_or_null,
                         int32_t eos, int32_t* committed, int32_t* num_committed,
                         int32_t* accept_length, int32_t* accept_path,
                         int32_t* next_root, int32_t* walk_info, double* margin,
                         int64_t* counters, int without_replacement, int64_t top_k, double top_p)
{
    if (B < 0 || N < 1 || V < 1 || !(T > 0.0)) return OR_ERR;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* qw = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p || !r || !qw) { free(p); free(r); free(qw); return OR_ERR; }
    const int filtered = (top_k > 0 && top_k < V) || top_p < 1.0;
    for (int b = 0; b < B; ++b) {
        int64_t o = (int64_t)b * N;
        for (int i = 0; i < N; ++i) { committed[o + i] = -1; accept_path[o + i] = -1; }
        int64_t rem = budget_or_null ? budget_or_null[b] : N;
        int len = 0, acc = 0, rejected = 0, kind = KIND_NONE;
        int32_t n = 0;
        double mg = INFINITY;
        accept_path[o] = 0;
        if (rem > 0) {
            if (!softmax_row(target, dtype, o * V, V, T, p)) counters[3]++;
            if (filtered) oracle_filter_probs(V, p, top_k, top_p);
            for (;;) {
                int32_t accepted = -1;
                const float* qn = NULL;
                if (next_token[o + n] >= 0) {
                    int64_t qrow = q_row_or_null ? q_row_or_null[o + n] : o + n;
                    qn = q + qrow * V;
                    for (int64_t v = 0; v < V; ++v) qw[v] = (double)qn[v];
                }
                for (int32_t c = next_token[o + n]; c >= 0; c = next_sibling[o + c]) {
                    int32_t y = draft_token[o + c];
                    double qy = qw[y], py = p[y];
                    double ratio = py / qy;
                    if (qy == 0.0) counters[0]++;
                    double u = (double)coins[o + c];
                    if (isfinite(ratio)) { double d = fabs(u - ratio); if (d < mg) mg = d; }
                    if (u < ratio) { accepted = c; break; }
                    ++rejected;
                    double R = 0.0;
                    for (int64_t v = 0; v < V; ++v) {
                        double d = p[v] - qw[v];
                        r[v] = d > 0.0 ? d : 0.0;
                        R += r[v];
                    }
                    if (R > 0.0 && isfinite(R))
                        for (int64_t v = 0; v < V; ++v) p[v] = r[v] / R;
                    else
                        counters[1]++;
                    if (without_replacement && y >= 0 && y < V) {
                        double S = 0.0;
                        qw[y] = 0.0;
                        for (int64_t v = 0; v < V; ++v) S += qw[v];
                        for (int64_t v = 0; v < V; ++v) qw[v] = S > 0.0 ? qw[v] / S : 0.0;
                    }
                }
                if (accepted >= 0) {
                    int32_t y = draft_token[o + accepted];
                    committed[o + len++] = y;
                    accept_path[o + ++acc] = accepted;
                    n = accepted;
                    if (y == eos || len == rem) { kind = KIND_NONE; break; }
                    if (!softmax_row(target, dtype, (o + n) * V, V, T, p)) counters[3]++;
                    if (filtered) oracle_filter_probs(V, p, top_k, top_p);
                    continue;
                }
                int32_t t;
                double m2;
                if (sample_inverse_cdf(p, V, (double)u_final[b], &t, &m2)) counters[2]++;
                if (m2 < mg) mg = m2;
                committed[o + len++] = t;
                kind = next_token[o + n] < 0 ? KIND_BONUS : KIND_CORRECTION;
                break;
            }
        }
        num_committed[b] = len;
        accept_length[b] = acc;
        next_root[b] = len > 0 ? committed[o + len - 1] : -1;
        walk_info[3 * b + 0] = n;
        walk_info[3 * b + 1] = rejected;
        walk_info[3 * b + 2] = kind;
        margin[b] = mg;
    }
    free(p);
    free(r);
    free(qw);
    return OR_OK;
}

/* ------------------------------------------------ KV-slot compaction (A7) */

/* [HB] "Drafting, verification and slots": slots for every candidate are
 * allocated before drafting; after verification only the accepted path's
 * slots are kept and the rest freed; with a page size above 1 data has to be
 * copied.  [ZS] 5.2: the cache is restored to the committed path, and the
 * correction/bonus token has no KV yet.
 * Layout (our reading): tree node n sits at logical position seq_len + n,
 * physical slot req_to_token[b][seq_len + n].  Keeping root + accepted path
 * gives new_kv_len = seq_len + 1 + accept_length.
 *   page_size 1: relabel req_to_token[seq_len + i] = old slot of path[i]
 *                (i = 1..a); free the slots of nodes not on the path, in
 *                node order; no data moves.
 *   page_size P > 1: for i = 1..a with path[i] != i emit the move
 *                (src = slot(seq_len + path[i]), dst = slot(seq_len + i)) and,
 *                with a pool, copy bytes_per_slot bytes src -> dst in
 *                increasing i; free the pages first touched by this step
 *                (first position in [seq_len, seq_len + N)) whose first
 *                position is >= new_kv_len, page id = slot / P.
 * freed is compacted across requests in (b, node or page) order.
 * Requests with seq_len < 0, seq_len + N > max_ctx, accept_length outside
 * [0, N) or a path that does not start at 0 and increase are skipped
 * (new_kv_len = -1) and counted in *bad. */
int oracle_compact_slots(int B, int N, int page_size, const int32_t* seq_lens,
                         const int32_t* accept_path, const int32_t* accept_length,
                         int32_t* req_to_token, int64_t max_ctx,
                         int32_t* move_src, int32_t* move_dst, int32_t* num_moves,
                         int32_t* freed, int32_t* num_freed, int32_t* new_kv_len,
                         uint8_t* kv_pool_or_null, int64_t num_slots,
                         int64_t bytes_per_slot, int32_t* bad)
{
    if (B < 0 || N < 1 || page_size < 1) return OR_ERR;
    int32_t nf = 0;
    *bad = 0;
    int32_t* keep = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    char* on_path = (char*)malloc((size_t)N);
    for (int b = 0; b < B; ++b) {
        int64_t o = (int64_t)b * N;
        int32_t* rt = req_to_token + (int64_t)b * max_ctx;
        int64_t sl = seq_lens[b];
        int a = accept_length[b];
        for (int i = 0; i < N; ++i) { move_src[o + i] = -1; move_dst[o + i] = -1; }
        num_moves[b] = 0;
        int ok = sl >= 0 && sl + N <= max_ctx && a >= 0 && a < N && accept_path[o] == 0;
        for (int i = 1; ok && i <= a; ++i)
            ok = accept_path[o + i] > accept_path[o + i - 1] && accept_path[o + i] < N;
        if (!ok) { new_kv_len[b] = -1; ++*bad; continue; }
        new_kv_len[b] = (int32_t)(sl + 1 + a);
        memset(on_path, 0, (size_t)N);
        for (int i = 0; i <= a; ++i) on_path[accept_path[o + i]] = 1;
        if (page_size == 1) {
            for (int i = 1; i <= a; ++i) keep[i] = rt[sl + accept_path[o + i]];
            for (int n = 1; n < N; ++n)
                if (!on_path[n]) freed[nf++] = rt[sl + n];
            for (int i = 1; i <= a; ++i) rt[sl + i] = keep[i];
        } else {
            int m = 0;
            for (int i = 1; i <= a; ++i) {
                int32_t pi = accept_path[o + i];
                if (pi == i) continue;
                int32_t src = rt[sl + pi], dst = rt[sl + i];
                move_src[o + m] = src;
                move_dst[o + m] = dst;
                ++m;
                if (kv_pool_or_null) {
                    if (src < 0 || src >= num_slots || dst < 0 || dst >= num_slots) { ++*bad; continue; }
                    memmove(kv_pool_or_null + (int64_t)dst * bytes_per_slot,
                            kv_pool_or_null + (int64_t)src * bytes_per_slot, (size_t)bytes_per_slot);
                }
            }
            num_moves[b] = m;
            int64_t first_page = (sl + page_size - 1) / page_size;
            for (int64_t lp = first_page; lp * page_size < sl + N; ++lp)
                if (lp * page_size >= new_kv_len[b])
                    freed[nf++] = rt[lp * page_size] / page_size;
        }
    }
    *num_freed = nf;
    free(keep);
    free(on_path);
    return OR_OK;
}

/* ------------------------------------------------------------- TLI (A8) */

/* [TLI] "Modifications": constrain_draft_logits sets every draft logit
 * outside the vocabulary intersection to -inf before the top-k (here top-1,
 * since TLI requires topk == 1); map_draft_to_target_ids maps the chosen id.
 * d2t[v] is the target id of draft id v, or -1 outside the intersection;
 * t2d is its inverse on the intersection.  q_target (optional) is the
 * constrained draft distribution at temperature T written in target-vocab
 * order, zero off the intersection.  A row with no finite intersection logit
 * gets top1 = -1, p = 0, a zero q row and row_flag = 1. */
int oracle_tli_constrain_map(int64_t R, int64_t Vd, int64_t Vt, const void* draft,
                             int dtype, const int32_t* d2t, const int32_t* t2d,
                             double T, int32_t* top1_draft, int32_t* top1_target,
                             double* top1_p, double* q_target_or_null,
                             int32_t* row_flag)
{
    if (R < 0 || Vd < 1 || Vt < 1 || !(T > 0.0)) return OR_ERR;
    for (int64_t r = 0; r < R; ++r) {
        int64_t base = r * Vd;
        int64_t best = -1;
        double m = -INFINITY;
        for (int64_t v = 0; v < Vd; ++v) {
            if (d2t[v] < 0) continue;
            double x = order_key(logit_at(draft, dtype, base + v));
            if (best < 0 || x > m) { best = v; m = x; }
        }
        if (best < 0 || !isfinite(m)) {
            top1_draft[r] = -1;
            top1_target[r] = -1;
            top1_p[r] = 0.0;
            row_flag[r] = 1;
            if (q_target_or_null)
                for (int64_t t = 0; t < Vt; ++t) q_target_or_null[r * Vt + t] = 0.0;
            continue;
        }
        double Z = 0.0;
        for (int64_t v = 0; v < Vd; ++v)
            if (d2t[v] >= 0) Z += exp((order_key(logit_at(draft, dtype, base + v)) - m) / T);
        top1_draft[r] = (int32_t)best;
        top1_target[r] = d2t[best];
        top1_p[r] = 1.0 / Z;
        row_flag[r] = 0;
        if (q_target_or_null)
            for (int64_t t = 0; t < Vt; ++t) {
                int32_t d = t2d[t];
                q_target_or_null[r * Vt + t] =
                    d >= 0 ? exp((order_key(logit_at(draft, dtype, base + d)) - m) / T) / Z : 0.0;
            }
    }
    return OR_OK;
}

/* [TLI] "Modifications", _try_prune_draft_lm_head / _PrunedReindexLMHead:
 * with the vocabulary intersection fixed, the draft LM head keeps only the
 * weight rows of the intersection's draft ids, so each draft row's logits are
 * computed for those K ids alone (O(M K H) instead of O(M V_d H)), in the
 * order of the weight rows (the ascending intersection ids); the constrained
 * top-1, its mapping to the target vocabulary and the constrained draft
 * distribution then follow as in oracle_tli_constrain_map, over those K
 * logits.
 *   hidden [M, H] (hdtype), weight [K, H] (wdtype): logits[m][k] =
 *     sum over h of hidden[m][h] * weight[k][h], in fp64, h in order.
 *   ids [K]: the draft id of weight row k; d2t [V_d] as in
 *     oracle_tli_constrain_map.
 *   top1_rank [M]: the weight row of the largest logit (ties: the lower row,
 *     which is the lower draft id); top1_draft = ids[rank], top1_target =
 *     d2t[ids[rank]]; top1_p: its probability at temperature T;
 *     row_max, row_z: the row's max logit and sum of exp((l - max)/T).
 *   logits_or_null [M, K] fp64.
 * NaN logits count as -inf; a row with no finite logit gets rank -1,
 * probability 0 and row_flag 1. */
int oracle_pruned_head(int64_t M, int64_t H, int64_t K, const void* hidden, int hdtype,
                       const void* weight, int wdtype, const int32_t* ids, const int32_t* d2t,
                       double T, double* logits_or_null, int32_t* top1_rank, int32_t* top1_draft,
                       int32_t* top1_target, double* top1_p, double* row_max, double* row_z,
                       int32_t* row_flag)
{
    if (M < 0 || H < 1 || K < 1 || !(T > 0.0)) return OR_ERR;
    double* l = (double*)malloc(sizeof(double) * (size_t)K);
    if (!l) return OR_ERR;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += logit_at(hidden, hdtype, m * H + h) * logit_at(weight, wdtype, k * H + h);
            l[k] = acc;
            if (logits_or_null) logits_or_null[m * K + k] = acc;
        }
        int64_t best = -1;
        double mx = -INFINITY;
        for (int64_t k = 0; k < K; ++k) {
            double x = order_key(l[k]);
            if (best < 0 || x > mx) { best = k; mx = x; }
        }
        row_max[m] = mx;
        if (!isfinite(mx)) {
            top1_rank[m] = top1_draft[m] = top1_target[m] = -1;
            top1_p[m] = 0.0;
            row_z[m] = 0.0;
            row_flag[m] = 1;
            continue;
        }
        double Z = 0.0;
        for (int64_t k = 0; k < K; ++k) Z += exp((order_key(l[k]) - mx) / T);
        top1_rank[m] = (int32_t)best;
        top1_draft[m] = ids[best];
        top1_target[m] = d2t[ids[best]];
        top1_p[m] = 1.0 / Z;
        row_z[m] = Z;
        row_flag[m] = 0;
    }
    free(l);
    return OR_OK;
}

/* The map plan of a vocabulary pair, written out from its definition (the
 * layout that tli_plan_build fills; [TLI] "Modifications": vocab_mapping.py
 * builds the id maps once per model pair, and the plan restates them):
 * K = number of draft ids with d2t >= 0; for word w of 32 draft ids, bits[w]
 * (bit j set when 32 w + j < Vd and d2t[32 w + j] >= 0) and before[w] (the
 * intersection ids in earlier words); for target id t < Vt4 (Vt rounded up
 * to 4) with d = t2d[t] (-1 past Vt): t2r[t] = the number of intersection
 * ids below d when d is one, -2 - d when 0 <= d < Vd is not one, else -1. */
int oracle_tli_plan(int64_t Vd, int64_t Vt, const int32_t* d2t, const int32_t* t2d,
                    int32_t* K, uint32_t* bits, uint32_t* before, int64_t words,
                    int32_t* t2r, int64_t Vt4)
{
    if (Vd < 1 || Vt < 1 || words * 32 < Vd || Vt4 < Vt) return OR_ERR;
    int32_t* below = (int32_t*)malloc(sizeof(int32_t) * (size_t)Vd);
    if (!below) return OR_ERR;
    int32_t k = 0;
    for (int64_t v = 0; v < Vd; ++v) {
        below[v] = k;
        if (d2t[v] >= 0) ++k;
    }
    *K = k;
    int32_t seen = 0;
    for (int64_t w = 0; w < words; ++w) {
        bits[w] = 0u;
        before[w] = (uint32_t)seen;
        for (int j = 0; j < 32; ++j) {
            int64_t v = 32 * w + j;
            if (v < Vd && d2t[v] >= 0) {
                bits[w] |= 1u << j;
                ++seen;
            }
        }
    }
    for (int64_t t = 0; t < Vt4; ++t) {
        int32_t d = t < Vt ? t2d[t] : -1;
        if (d < 0 || d >= Vd) t2r[t] = -1;
        else if (d2t[d] >= 0) t2r[t] = below[d];
        else t2r[t] = -2 - d;
    }
    free(below);
    return OR_OK;
}

/* [TLI] "Modifications": map_target_to_draft_ids / map_draft_to_target_ids;
 * ids outside the table or without a partner map to the fallback id (the
 * unk id, or eos where a model has no unk). */
int oracle_map_ids(const int32_t* in, int32_t* out, int64_t n, const int32_t* table,
                   int64_t table_len, int32_t fallback)
{
    for (int64_t i = 0; i < n; ++i) {
        int32_t x = in[i];
        out[i] = (x >= 0 && x < table_len && table[x] >= 0) ? table[x] : fallback;
    }
    return OR_OK;
}

/* [TLI] "Modifications", server_args validation: TLI requires topk == 1 and
 * num_draft_tokens == num_steps + 1. */
int oracle_tli_check_config(int topk, int num_steps, int num_draft_tokens)
{
    return (topk == 1 && num_steps >= 1 && num_draft_tokens == num_steps + 1) ? OR_OK : OR_ERR;
}
