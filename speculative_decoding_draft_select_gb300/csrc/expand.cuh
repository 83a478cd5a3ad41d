// One draft step of the candidate-pool expansion for one request, as a CTA
// routine: the standalone tree_expand_kernel runs it with one CTA per
// request, and the draft kernels run it in the CTA that finishes a
// request's last draft row of the step (so that a draft step is one
// launch).
//
// "[SGLang] Multi-Layer EAGLE" (secrett2633 blog), section 2:
// select_top_k_tokens returns tree_info = (scores, tokens, parents) per
// draft step.  Every expansion enters the pool; the next frontier is the
// best k by (score desc, pool id asc).
#pragma once

#include <climits>

#include "common.cuh"

namespace specdec {

// An expansion step's view of the pool (pool_* are [B, P], frontier_* are
// [B, k]); counters [B] are zero between steps.
struct ExpandArgs {
  int step, num_steps, B, k;
  int64_t P;
  float* pool_score;
  int32_t* pool_token;
  int32_t* pool_parent;
  int32_t* pool_qrow;
  float* frontier_score;
  int32_t* frontier_id;
  int32_t* counters;
};

// Sort key for (score desc, pool id asc) as an ascending 64-bit integer.
// NaN sorts as -inf and -0 as +0, matching float comparison.
__device__ __forceinline__ uint64_t rank_key(float s, int32_t id) {
  if (s != s) s = neg_inf();
  if (s == 0.0f) s = 0.0f;
  uint32_t u = __float_as_uint(s);
  uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(~asc) << 32) | static_cast<uint32_t>(id);
}

// Expansion of request b (all threads of the CTA call it; keys holds at
// least k*k entries of shared memory).  topk_p / topk_idx are the step's
// draft outputs: [B, k] at step 0, [B, k, k] after.  Reads them through L2
// (another CTA of the launch may have written them).
__device__ __forceinline__ void expand_request(const ExpandArgs& e, int b, const float* topk_p,
                                               const int32_t* topk_idx, uint64_t* keys) {
  const int k = e.k, step = e.step;
  const int nc = step == 0 ? k : k * k;
  const int64_t base = step == 0 ? 1 : 1 + k + static_cast<int64_t>(step - 1) * k * k;
  const int64_t P = e.P;
  float* sc = e.pool_score + b * P;
  int32_t* tk = e.pool_token + b * P;
  int32_t* pa = e.pool_parent + b * P;
  int32_t* qr = e.pool_qrow + b * P;
  if (step == 0) {
    for (int64_t i = threadIdx.x; i < P; i += blockDim.x) {
      sc[i] = i == 0 ? 1.0f : 0.0f;
      tk[i] = -1;
      pa[i] = -1;
      qr[i] = i == 0 ? b : -1;
    }
    __syncthreads();
  }
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    float score;
    int32_t tok, par;
    if (step == 0) {
      score = __ldcg(topk_p + static_cast<int64_t>(b) * k + c);
      tok = __ldcg(topk_idx + static_cast<int64_t>(b) * k + c);
      par = 0;
    } else {
      const int f = c / k, j = c % k;
      const int64_t row = static_cast<int64_t>(b) * k + f;
      score = __fmul_rn(e.frontier_score[row], __ldcg(topk_p + row * k + j));
      tok = __ldcg(topk_idx + row * k + j);
      par = e.frontier_id[row];
    }
    if (!spec_in(base + c, P, nullptr)) continue;
    sc[base + c] = score;
    tk[base + c] = tok;
    pa[base + c] = par;
    keys[c] = rank_key(score, static_cast<int32_t>(base + c));
  }
  __syncthreads();  // every frontier read above happens before the writes below
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    const uint64_t mine = keys[c];
    int rank = 0;
    for (int o = 0; o < nc; ++o) rank += keys[o] < mine;
    if (rank < k && spec_in(base + c, P, nullptr)) {
      e.frontier_score[static_cast<int64_t>(b) * k + rank] = sc[base + c];
      e.frontier_id[static_cast<int64_t>(b) * k + rank] = static_cast<int32_t>(base + c);
      if (step + 1 < e.num_steps) qr[base + c] = e.B + step * e.B * k + b * k + rank;
    }
  }
}

// A chain's expansion (k = 1) of request b by one thread, from the step's
// top-1 (p, tok) in registers: the same writes as expand_request, without
// a barrier.
__device__ __forceinline__ void expand_chain(const ExpandArgs& e, int b, float p, int32_t tok) {
  const int step = e.step;
  const int64_t P = e.P;
  float* sc = e.pool_score + b * P;
  int32_t* tk = e.pool_token + b * P;
  int32_t* pa = e.pool_parent + b * P;
  int32_t* qr = e.pool_qrow + b * P;
  float score;
  int32_t par;
  int64_t base;
  if (step == 0) {
    for (int64_t i = 0; i < P; ++i) {
      sc[i] = i == 0 ? 1.0f : 0.0f;
      tk[i] = -1;
      pa[i] = -1;
      qr[i] = i == 0 ? b : -1;
    }
    score = p;
    par = 0;
    base = 1;
  } else {
    score = __fmul_rn(e.frontier_score[b], p);
    par = e.frontier_id[b];
    base = 1 + step;
  }
  if (!spec_in(base, P, nullptr)) return;
  sc[base] = score;
  tk[base] = tok;
  pa[base] = par;
  e.frontier_score[b] = score;
  e.frontier_id[b] = static_cast<int32_t>(base);
  if (step + 1 < e.num_steps) qr[base] = e.B + step * e.B + b;
}

// Called by every thread of a draft kernel's CTA after the row's outputs
// are stored (threads that stored them pass wrote = true): the CTA that
// completes request b's rows of this step (1 row at step 0 or with k = 1,
// k rows after) expands request b.  The writers' fences and the counter's
// atomic order their stores before the expanding CTA's reads; the
// expanding CTA resets the counter for the next step.
// e.k == 0 means no expansion.
__device__ __forceinline__ void expand_if_last(const ExpandArgs& e, int64_t row, bool wrote, const float* topk_p,
                                               const int32_t* topk_idx, uint64_t* keys, int* s_last) {
  if (e.k == 0) return;
  const int per = (e.step == 0 || e.k == 1) ? 1 : e.k;
  const int b = static_cast<int>(row / per);
  if (wrote) __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int last = 1;
    if (per > 1) {
      last = atomicAdd(e.counters + b, 1) == per - 1;
      if (last) {
        __threadfence();
        e.counters[b] = 0;
      }
    }
    *s_last = last;
  }
  __syncthreads();
  if (*s_last) expand_request(e, b, topk_p, topk_idx, keys);
}

// Host: the kernels' view of a caller's spec_expand_t for a draft launch of
// R rows with top-k k (SPEC_OK, or the error to return).
inline int expand_args(const spec_expand_t* x, int k, int64_t R, ExpandArgs& e) {
  if (x == nullptr) return SPEC_ERR_INVALID_ARG;
  if (x->k != k || x->B < 1 || x->num_steps < 1 || x->step < 0 || x->step >= x->num_steps)
    return SPEC_ERR_INVALID_ARG;
  if (R != (x->step == 0 ? static_cast<int64_t>(x->B) : static_cast<int64_t>(x->B) * x->k)) return SPEC_ERR_INVALID_ARG;
  if (!x->pool_score || !x->pool_token || !x->pool_parent || !x->pool_qrow || !x->frontier_score ||
      !x->frontier_id || (k > 1 && !x->counters))
    return SPEC_ERR_INVALID_ARG;
  if (k > SPEC_MAX_TOPK || static_cast<int64_t>(x->B) * k * x->num_steps > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  const int64_t P = 1 + k + static_cast<int64_t>(x->num_steps - 1) * k * k;
  e = ExpandArgs{x->step, x->num_steps, x->B, k, P, x->pool_score, x->pool_token, x->pool_parent, x->pool_qrow,
                 x->frontier_score, x->frontier_id, x->counters};
  return SPEC_OK;
}

// No expansion.
inline ExpandArgs no_expand() { return ExpandArgs{0, 0, 0, 0, 0, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr}; }

}  // namespace specdec
