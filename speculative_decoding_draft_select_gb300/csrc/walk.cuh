// Shared pieces of the stochastic verify kernels (the tree walk in
// verify.cu, the chain verify in chain.cu): the walk's launch constants, the
// bounded flag wait, per-thread row statistics, where a node's draft
// distribution q comes from, and the weights of the current distribution
// (target p, or the positive residual of p and q) that the row sweeps and the
// inverse-CDF draw read.
//
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)", 5.1:
// accept y ~ q with min(1, p[y]/q[y]); after a rejection draw from the
// normalised positive residual (p - q)+; after full acceptance draw the bonus
// from p.
#pragma once

#include <climits>

#include "cdf.cuh"
#include "common.cuh"

namespace specdec {
namespace {

#ifndef SPEC_WALK_THREADS
#define SPEC_WALK_THREADS 128
#endif
#ifndef SPEC_WALK_ELEMS
#define SPEC_WALK_ELEMS 16
#endif
// The stochastic walk: a cluster of 1, 2 or 4 CTAs of kWalkThreads threads
// per request.
constexpr int kWalkThreads = SPEC_WALK_THREADS;
constexpr int kWalkElems = SPEC_WALK_ELEMS;  // consecutive elements per thread in a tile
constexpr size_t kMaxDynSmem = 227 * 1024;  // opt-in shared memory of one CTA

// Tiles each walk thread keeps in flight: 2 to 8, the ring at most 32 KB per
// CTA (four CTAs share an SM).
__host__ __device__ constexpr int walk_ring_depth(int chunks) {
  return 32768 / (chunks * kWalkThreads * 16) > 8   ? 8
         : 32768 / (chunks * kWalkThreads * 16) < 2 ? 2
                                                     : 32768 / (chunks * kWalkThreads * 16);
}

// Bound on a wait for another CTA's row (about 50 ms at 2 GHz); past it the
// launch counts SPEC_STAT_WAIT_TIMEOUT and goes on.
constexpr long long kWaitLimitCycles = 100000000LL;

// Waits (one thread) until *flag != 0 or `limit` clock cycles pass; a
// timeout is counted in SPEC_STAT_WAIT_TIMEOUT.  Returns whether the flag
// was seen.
__device__ __forceinline__ bool wait_flag(const int* flag, long long limit, int32_t* stats) {
  const long long t0 = clock64();
  while (!ld_acquire_gpu(flag)) {
    if (clock64() - t0 > limit) {
      bump(stats, SPEC_STAT_WAIT_TIMEOUT);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

__device__ __forceinline__ float prob_of(float key, float c, float mc, float invz) {
  return fminf(fast_exp2(fmaf(key, c, -mc)) * invz, 1.0f);
}

// Per-thread row statistics: running max m (NaN ignored), the first index
// holding it, and for sampling s = sum 2^((x - m) c) in two accumulators
// (shorter dependency chains).  A NaN element turns s into NaN; the kernel
// then recomputes s for that row with NaN as -inf.
template <int DT, bool STOCH>
struct RowStatVisitor {
  float c, m, s0, s1;
  int bi;
  float mc;  // m c
  __device__ __forceinline__ void rescale(float nm) {
    if (STOCH) {
      if (m == neg_inf()) {
        s0 = s1 = 0.0f;
      } else {
        const float f = fast_exp2((m - nm) * c);
        s0 *= f;
        s1 *= f;
      }
      mc = nm * c;
    }
    m = nm;
  }
  __device__ __forceinline__ void visit1(float x, int64_t idx, bool ok) {
    if (!ok) return;
    const float xk = order_key(x);
    if (xk > m) {
      rescale(xk);
      bi = static_cast<int>(idx);
    }
    if (STOCH && m != neg_inf()) s0 += fast_exp2(fmaf(xk, c, -mc));
  }
  __device__ __forceinline__ void visit_vec(const uint4& w, int64_t first, bool) {
    constexpr int kv = Logit<DT>::kVec;
    float x[kv];
    unpack<DT>(w, x);
    float vmax;
    if (DT == SPEC_BF16) {
      vmax = max8_bf16(w);
    } else {
      vmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[kv - 1]));
    }
    if (vmax > m) {
      int j0 = 0;
#pragma unroll
      for (int j = kv - 1; j >= 0; --j)
        if (x[j] == vmax) j0 = j;
      rescale(vmax);
      bi = static_cast<int>(first) + j0;
    }
    if (STOCH && m != neg_inf()) {
      const float2 a = exp2_sum_pairs<kv>(make_float2(s0, s1), x, c, mc);
      s0 = a.x;
      s1 = a.y;
    }
  }
};

// Sum of 2^((key(x) - m) c) over a row with NaN as -inf (the slow path for
// rows that contain NaN).
struct KeyedSum {
  float c, mc, s;
  template <int N>
  __device__ __forceinline__ void visit(const float* x, int64_t) {
#pragma unroll
    for (int j = 0; j < N; ++j) s += fast_exp2(fmaf(order_key(x[j]), c, -mc));
  }
};

// Where a node's draft distribution q comes from.
//   QProbs:     materialised fp32 rows (q[v] read directly).
//   QLogits<D>: the draft logits row and that row's (max, normaliser) as the
//               draft softmax wrote them.  q_at(y), used by the acceptance
//               test, takes the same fp32 operations as the written
//               probabilities, so both forms give bit-identical q[y].
// The residual sweeps need q for a whole row; there (load8, ring_q8,
// sweep_at) the normaliser is folded into the exponent,
// q[v] = 2^(l_v c + nb), nb = -(max c + log2 Z), one operation fewer per
// element.  Rows whose 16-byte chunks start aligned are streamed through the
// walk's shared-memory ring (issue / ring_q8), others with direct loads.

__device__ __forceinline__ bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Exponent offset nb of a row's softmax: p(x) = 2^(x c + nb); -inf when the
// row has no finite max, which makes every probability 0 (a NaN logit gives
// NaN, which the residual's max(0, .) turns into 0).
__device__ __forceinline__ float folded_offset(float m, float c, float z) {
  return (isfinite(m) && z > 0.0f && isfinite(z)) ? -fmaf(m, c, log2f(z)) : neg_inf();
}

// 8 logits [v0, v0 + 8) of a row as floats (NaN kept); past V: -inf.
template <int DT>
__device__ __forceinline__ void raw8_global(const void* row, int64_t V, int64_t v0, float* x) {
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const char* p = static_cast<const char*>(row) + v0 * esz;
  if (v0 + 8 <= V && aligned16(p)) {
    if (DT == SPEC_BF16) {
      unpack<SPEC_BF16>(__ldg(reinterpret_cast<const uint4*>(p)), x);
    } else {
      unpack<SPEC_F32>(__ldg(reinterpret_cast<const uint4*>(p)), x);
      unpack<SPEC_F32>(__ldg(reinterpret_cast<const uint4*>(p) + 1), x + 4);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = v0 + j < V ? Logit<DT>::load1(row, v0 + j) : neg_inf();
  }
}

// Group g (elements [8g, 8g + 8)) of a thread's ring chunks of one row, as
// floats.  DT: logits (bf16 or fp32).
template <int DT>
__device__ __forceinline__ void ring8(const uint4* slot, int stride, int g, float* x) {
  if (DT == SPEC_BF16) {
    unpack<SPEC_BF16>(slot[g * stride], x);
  } else {
    unpack<SPEC_F32>(slot[(2 * g) * stride], x);
    unpack<SPEC_F32>(slot[(2 * g + 1) * stride], x + 4);
  }
}

__device__ __forceinline__ void mask_past(float* x, int64_t v0, int64_t V, float fill) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (v0 + j >= V) x[j] = fill;
}

struct QRowProbs {
  static constexpr int kEsz = 4;
  const float* row;  // nullptr: no row (q = 0)
  int64_t V;
  // elements [e0, e0 + n) as a row of their own
  __device__ __forceinline__ QRowProbs sub(int64_t e0, int64_t n) const { return {row ? row + e0 : nullptr, n}; }
  __device__ __forceinline__ float q_at(int64_t v) const { return row ? __ldg(row + v) : 0.0f; }
  __device__ __forceinline__ float sweep_at(int64_t v) const { return q_at(v); }
  __device__ __forceinline__ void load8(int64_t v0, float* x) const {
    if (row) {
      load8_f32(row, V, v0, x);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
  }
  __device__ __forceinline__ bool ring_ok() const { return row == nullptr || aligned16(row); }
  template <int E>
  __device__ __forceinline__ void issue(uint4* slot, int stride, int64_t v0) const {
    if (row) issue_row<E, 4>(slot, stride, row, V, v0);
  }
  // q of group g from the ring (zero-filled past V)
  __device__ __forceinline__ void ring_q8(const uint4* slot, int stride, int g, int64_t, bool, float* x) const {
    if (row) {
      ring8<SPEC_F32>(slot, stride, g, x);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
  }
};

struct QProbs {
  using Row = QRowProbs;
  const float* q;
  int64_t V;
  __device__ __forceinline__ QRowProbs row(int64_t r) const { return {r >= 0 ? q + r * V : nullptr, V}; }
};

template <int QDT>
struct QRowLogits {
  static constexpr int kEsz = QDT == SPEC_BF16 ? 2 : 4;
  const void* row;  // nullptr: no row, or a row whose max is not finite (q = 0)
  int64_t V;
  float c, mc, invz, nb;
  // elements [e0, e0 + n) as a row of their own (same max and normaliser)
  __device__ __forceinline__ QRowLogits sub(int64_t e0, int64_t n) const {
    return {row ? static_cast<const char*>(row) + e0 * kEsz : nullptr, n, c, mc, invz, nb};
  }
  __device__ __forceinline__ float q_at(int64_t v) const {
    return row ? prob_of(order_key(Logit<QDT>::load1(row, v)), c, mc, invz) : 0.0f;
  }
  __device__ __forceinline__ float sweep_at(int64_t v) const {
    return row ? fast_exp2(fmaf(order_key(Logit<QDT>::load1(row, v)), c, nb)) : 0.0f;
  }
  // 8 q values from 8 logits (NaN as -inf), in the packed form of the sweeps
  __device__ __forceinline__ void probs8(float* x) const {
    const float2 c2 = splat(c), nb2 = splat(nb);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float2 e = exp2_2(fma2(make_float2(order_key(x[j]), order_key(x[j + 1])), c2, nb2));
      x[j] = e.x;
      x[j + 1] = e.y;
    }
  }
  __device__ __forceinline__ void load8(int64_t v0, float* x) const {
    if (row) {
      raw8_global<QDT>(row, V, v0, x);
      probs8(x);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
  }
  __device__ __forceinline__ bool ring_ok() const { return row == nullptr || aligned16(row); }
  template <int E>
  __device__ __forceinline__ void issue(uint4* slot, int stride, int64_t v0) const {
    if (row) issue_row<E, kEsz>(slot, stride, row, V, v0);
  }
  __device__ __forceinline__ void ring_q8(const uint4* slot, int stride, int g, int64_t v0, bool full,
                                          float* x) const {
    if (row) {
      ring8<QDT>(slot, stride, g, x);
      if (!full) mask_past(x, v0, V, neg_inf());
      probs8(x);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
  }
};

template <int QDT>
struct QLogits {
  using Row = QRowLogits<QDT>;
  const void* q;
  const float* stats;  // [rows, 2]: max, normaliser
  int64_t V;
  float c;
  __device__ __forceinline__ QRowLogits<QDT> row(int64_t r) const {
    constexpr int esz = QDT == SPEC_BF16 ? 2 : 4;
    if (r < 0) return {nullptr, V, c, 0.0f, 0.0f, 0.0f};
    const float m = __ldg(stats + 2 * r), z = __ldg(stats + 2 * r + 1);
    if (!isfinite(m)) return {nullptr, V, c, 0.0f, 0.0f, 0.0f};
    return {static_cast<const char*>(q) + r * V * esz, V, c, m * c, 1.0f / z, folded_offset(m, c, z)};
  }
};

// Weights of the current distribution at a node for the sweeps: p (A == 0)
// or the unnormalised residual max(0, p - A q), with p(v) = 2^(l_v c + nb).
// Element values are computed two at a time with the packed fp32
// instructions; load8 (per element, for the draw), ring_sum and load_sum
// (sums for the tile pass) give the same values.
template <int DT, class QRow>
struct ResidualWeights {
  static constexpr int kTargetEsz = DT == SPEC_BF16 ? 2 : 4;
  template <int E>
  __host__ __device__ static constexpr int target_chunks() {
    return E * kTargetEsz / 16;
  }
  template <int E>
  __host__ __device__ static constexpr int chunks() {
    return E * (kTargetEsz + QRow::kEsz) / 16;
  }
  const void* lrow;
  QRow qrow;
  int64_t V;
  float c, nb, A;
  // the weights of elements [e0, e0 + n) as a row of their own
  __device__ __forceinline__ ResidualWeights sub(int64_t e0, int64_t n) const {
    return {static_cast<const char*>(lrow) + e0 * kTargetEsz, qrow.sub(e0, n), n, c, nb, A};
  }
  // x <- weights of 8 elements from logits l (and q values when A != 0)
  __device__ __forceinline__ void values8(float* l, const float* q) const {
    const float2 c2 = splat(c), nb2 = splat(nb), na2 = splat(-A);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float2 r = exp2_2(fma2(make_float2(l[j], l[j + 1]), c2, nb2));
      if (q != nullptr) r = fma2(na2, make_float2(q[j], q[j + 1]), r);
      l[j] = fmaxf(0.0f, r.x);
      l[j + 1] = fmaxf(0.0f, r.y);
    }
  }
  __device__ __forceinline__ static float2 acc8(float2 acc, const float* x) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) acc = add2(acc, make_float2(x[j], x[j + 1]));
    return acc;
  }
  __device__ __forceinline__ void load8(int64_t v0, float* x) const {
    raw8_global<DT>(lrow, V, v0, x);
    if (A != 0.0f) {
      float q[8];
      qrow.load8(v0, q);
      values8(x, q);
    } else {
      values8(x, nullptr);
    }
  }
  __device__ __forceinline__ float at(int64_t v) const {
    const float p = fast_exp2(fmaf(Logit<DT>::load1(lrow, v), c, nb));
    return fmaxf(0.0f, A != 0.0f ? fmaf(-A, qrow.sweep_at(v), p) : p);
  }
  template <int E>
  __device__ __forceinline__ float load_sum(int64_t v0) const {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int g = 0; g < E / 8; ++g) {
      float x[8];
      load8(v0 + 8 * g, x);
      acc = acc8(acc, x);
    }
    return acc.x + acc.y;
  }
  __device__ __forceinline__ bool ring_ok() const { return aligned16(lrow) && (A == 0.0f || qrow.ring_ok()); }
  template <int E>
  __device__ __forceinline__ void issue(uint4* slot, int stride, int64_t v0) const {
    issue_row<E, kTargetEsz>(slot, stride, lrow, V, v0);
    if (A != 0.0f) qrow.template issue<E>(slot + target_chunks<E>() * stride, stride, v0);
  }
  template <int E>
  __device__ __forceinline__ float ring_sum(const uint4* slot, int stride, int64_t v0) const {
    const bool full = v0 + E <= V;
    const uint4* qslot = slot + target_chunks<E>() * stride;
    float2 acc = make_float2(0.0f, 0.0f);
    if (A != 0.0f) {
#pragma unroll
      for (int g = 0; g < E / 8; ++g) {
        float x[8], q[8];
        ring8<DT>(slot, stride, g, x);
        if (!full) mask_past(x, v0 + 8 * g, V, neg_inf());
        qrow.ring_q8(qslot, stride, g, v0 + 8 * g, full, q);
        values8(x, q);
        acc = acc8(acc, x);
      }
    } else {
#pragma unroll
      for (int g = 0; g < E / 8; ++g) {
        float x[8];
        ring8<DT>(slot, stride, g, x);
        if (!full) mask_past(x, v0 + 8 * g, V, neg_inf());
        values8(x, nullptr);
        acc = acc8(acc, x);
      }
    }
    return acc.x + acc.y;
  }
};

}  // namespace
}  // namespace specdec
