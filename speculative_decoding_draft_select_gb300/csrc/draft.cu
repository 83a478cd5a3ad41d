// Draft side: per-step softmax + top-k, and draft sampling.
//
// "[SGLang] Multi-Layer EAGLE" (secrett2633 blog), section 3: every draft
// step computes probs = softmax(logits) and then top-k of them;
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)", 5.1: the
// stored draft distribution is the processed one (temperature applied), and
// drafts are drawn from it.
//
// The tree scores are the top-k probabilities of a plain softmax (the
// Multi-Layer EAGLE page, section 3: no temperature), while the stored q is
// at the temperature T (zero-to-sglang 5.1).  When a launch writes q and the
// two temperatures differ, the pass keeps a normaliser for each.
//
// One CTA streams one logit row with 16-byte loads (8 in flight per thread).
// That pass gives each thread's online softmax partials (max, sum of
// 2^((x - max) * log2e / T)) and its best element.  The K-th best of the
// thread bests bounds the top-K from below, so only the few threads whose
// best reaches it can own a top-K element: the block reads their elements
// again (from L2) and ranks the few that reach the bound.  Block merges are
// fixed-order.  The optional probability row is written by a second sweep
// of the row (served from L2) with streaming stores.
#include <climits>

#include "cdf.cuh"
#include "common.cuh"
#include "expand.cuh"

namespace specdec {
namespace {

#ifndef SPEC_DRAFT_THREADS
#define SPEC_DRAFT_THREADS 128
#endif
constexpr int kDraftThreads = SPEC_DRAFT_THREADS;
#ifndef SPEC_DRAFT_UNROLL
#define SPEC_DRAFT_UNROLL 8
#endif
// 16-byte loads in flight per thread (8 measured faster than 4 for k = 1 at
// R=1024, 53.6 -> 51.1 us, and for the few-rows 512-thread instance; equal
// for k = 8)
constexpr int kDraftUnroll = SPEC_DRAFT_UNROLL;

// Running online-softmax partials of one thread: m = max key seen,
// s = sum 2^((x - m) c).
struct SoftmaxPartial {
  float c, m, s;
  template <int N>
  __device__ __forceinline__ float update(const float* x) {
    float vmax = neg_inf();
#pragma unroll
    for (int j = 0; j < N; ++j) vmax = fmaxf(vmax, x[j]);
    if (vmax > m) {
      s = (m == neg_inf()) ? 0.0f : s * fast_exp2((m - vmax) * c);
      m = vmax;
    }
    if (m != neg_inf()) {
      const float mc = m * c;
#pragma unroll
      for (int j = 0; j < N; ++j) s += fast_exp2(fmaf(x[j], c, -mc));
    }
    return vmax;
  }
};

// Register top-K of one thread, sorted by (value desc, index asc).
template <int K>
struct TopK {
  float v[K];
  int i[K];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      v[j] = neg_inf();
      i[j] = INT_MAX;
    }
  }
  __device__ __forceinline__ void push(float x, int idx) {
    if (!before(x, idx, v[K - 1], i[K - 1])) return;
    v[K - 1] = x;
    i[K - 1] = idx;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
      if (before(v[j], i[j], v[j - 1], i[j - 1])) {
        const float tv = v[j];
        v[j] = v[j - 1];
        v[j - 1] = tv;
        const int ti = i[j];
        i[j] = i[j - 1];
        i[j - 1] = ti;
      }
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      v[j] = v[j + 1];
      i[j] = i[j + 1];
    }
    v[K - 1] = neg_inf();
    i[K - 1] = INT_MAX;
  }
};

// Pass A of a draft row: each thread's online softmax and its best element
// (key desc, index asc; NaN as -inf).  A thread visits its elements in
// increasing index order, so only a strictly larger key replaces its best;
// a thread whose keys are all -inf ends with bi = INT_MAX and takes its
// first element afterwards (own_first).  For K == 1 the block's best is the
// top-1; for K > 1 the thread bests give the pass-B threshold.
//
// TWO: a second normaliser at another temperature, c1 = log2(e) / T_score:
// s0 then sums 2^((x - m) c) and s1 sums 2^((x - m) c1); without it s0 and s1
// are two halves of the one sum at c.
template <int DT, bool SECOND = false, bool TWO = false>
struct ArgmaxVisitor {
  float c, c1, m, mc, mc1, s0, s1;  // mc = m c, mc1 = m c1
  int bi;
  float m2v;  // SECOND: the largest key of the thread's other elements (NaN skipped)
  __device__ __forceinline__ void reset() {
    m = neg_inf();
    mc = mc1 = 0.0f;
    s0 = s1 = 0.0f;
    bi = INT_MAX;
    m2v = neg_inf();
  }
  __device__ __forceinline__ void rescale(float nm) {
    if (m == neg_inf()) {
      s0 = s1 = 0.0f;
    } else if (TWO) {
      s0 *= fast_exp2((m - nm) * c);
      s1 *= fast_exp2((m - nm) * c1);
    } else {
      const float f = fast_exp2((m - nm) * c);
      s0 *= f;
      s1 *= f;
    }
    m = nm;
    mc = nm * c;
    if (TWO) mc1 = nm * c1;
  }
  __device__ __forceinline__ void visit1(float x, int64_t idx, bool ok) {
    if (!ok) return;
    const float xk = order_key(x);
    if (xk > m) {
      if (SECOND) m2v = m;
      rescale(xk);
      bi = static_cast<int>(idx);
    } else if (SECOND) {
      m2v = fmaxf(m2v, xk);
    }
    if (m != neg_inf()) {
      s0 += fast_exp2(fmaf(xk, c, -mc));
      if (TWO) s1 += fast_exp2(fmaf(xk, c1, -mc1));
    }
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int64_t first, bool ok) {
    constexpr int kv = Logit<DT>::kVec;
    float x[kv];
    unpack<DT>(raw, x);
    float vmax;
    if (DT == SPEC_BF16) {
      vmax = max8_bf16(raw);
    } else {
      vmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[kv - 1]));
    }
    if (ok && vmax > m) {
      int j0 = 0;
#pragma unroll
      for (int j = kv - 1; j >= 0; --j)
        if (x[j] == vmax) j0 = j;
      if (SECOND) {
        // the old best and the vector's other elements
        float sec = m;
#pragma unroll
        for (int j = 0; j < kv; ++j)
          if (j != j0) sec = fmaxf(sec, x[j]);
        m2v = sec;
      }
      rescale(vmax);
      bi = static_cast<int>(first) + j0;
    } else if (SECOND && ok) {
      m2v = fmaxf(m2v, vmax);
    }
    if (m != neg_inf()) {
      const float2 a = TWO ? exp2_sum_two<kv>(make_float2(s0, s1), x, make_float2(c, c1), make_float2(mc, mc1))
                           : exp2_sum_pairs<kv>(make_float2(s0, s1), x, c, mc);
      s0 = a.x;
      s1 = a.y;
    }
  }
  // the thread's first element in the visiting order, if its best is unset
  __device__ __forceinline__ void own_first(const void* row, int64_t V, int tid) {
    if (bi != INT_MAX) return;
    constexpr int kv = Logit<DT>::kVec;
    const RowSpan sp = row_span<DT>(row, V);
    if (tid < sp.head) {
      bi = tid;
    } else if (tid < sp.nvec) {
      bi = static_cast<int>(sp.head + static_cast<int64_t>(tid) * kv);
    } else if (sp.head + sp.nvec * kv + tid < V) {
      bi = static_cast<int>(sp.head + sp.nvec * kv + tid);
    }
  }
};

// Pass B of a draft row (K > 1): collect every element that comes before or
// at the threshold pair (tv, ti) in the (value desc, index asc) order.  The
// threshold is the K-th best of the thread bests of pass A, so at least K
// elements qualify and no element after it can be in the top-K.  Appends use
// a shared counter; their order does not matter (the final selection is by
// the total order).
constexpr int kCandCap = 1024;
// Up to this many candidates are placed by ranking (n^2 / threads compares
// per thread); more (long runs of equal keys) go to the warp select.
constexpr int kRankCands = 256;

template <int DT>
struct CandVisitor {
  float tv;
  int ti;
  float* bv;
  int* bi;
  int* cnt;
  __device__ __forceinline__ bool qualifies(float x, int idx) const {
    return x > tv || (x == tv && idx <= ti);
  }
  __device__ __forceinline__ void add(float x, int idx) {
    const int pos = atomicAdd(cnt, 1);
    if (pos < kCandCap) {
      bv[pos] = x;
      bi[pos] = idx;
    }
  }
  __device__ __forceinline__ void visit1(float x, int64_t idx, bool ok) {
    const float xk = order_key(x);
    if (ok && qualifies(xk, static_cast<int>(idx))) add(xk, static_cast<int>(idx));
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int64_t first, bool ok) {
    constexpr int kv = Logit<DT>::kVec;
    float vmax;
    float x[kv];
    unpack<DT>(raw, x);
    if (DT == SPEC_BF16) {
      vmax = max8_bf16(raw);
    } else {
      vmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[kv - 1]));
    }
    // a -inf threshold (fewer than K finite keys) must still see -inf keys
    if (!ok || !(vmax > tv || (vmax == tv && first <= ti) || tv == neg_inf())) return;
#pragma unroll
    for (int j = 0; j < kv; ++j) {
      const float xk = order_key(x[j]);
      if (qualifies(xk, static_cast<int>(first) + j)) add(xk, static_cast<int>(first) + j);
    }
  }
};

constexpr int kRescanUnroll = 4;  // loads in flight per thread (8 measured slower)

// The elements owned by the threads listed in owner[0..n_owner) (owner t
// holds, in the layout of for_row_raw, the scalars t, t + nthreads, ... of
// the head and tail and the 16-byte vectors t, t + nthreads, ...), visited
// by the whole block: each block thread takes every nthreads-th (owner,
// vector) pair, kRescanUnroll loads in flight.
template <int DT, class F>
__device__ __forceinline__ void rescan_owners(const void* row, int64_t V, F& f, const int* owner, int n_owner,
                                              int nthreads) {
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const RowSpan sp = row_span<DT>(row, V);
  const int tid = threadIdx.x;
  const int64_t tail0 = sp.head + sp.nvec * kv;
  for (int e = tid; e < n_owner; e += nthreads) {
    const int t = owner[e];
    for (int64_t i = t; i < sp.head; i += nthreads) f.visit1(Logit<DT>::load1(row, i), i, true);
    for (int64_t i = tail0 + t; i < V; i += nthreads) f.visit1(Logit<DT>::load1(row, i), i, true);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  const int nvec = static_cast<int>(sp.nvec);  // V < 2^31
  // kRescanUnroll owners at a time; thread tid takes vector j of each, j =
  // tid, tid + nthreads, ... (owner t's j-th vector is t + j nthreads)
  for (int o0 = 0; o0 < n_owner; o0 += kRescanUnroll) {
    for (int j = tid; j * nthreads < nvec; j += nthreads) {
      uint4 v[kRescanUnroll];
      int vi[kRescanUnroll];
#pragma unroll
      for (int u = 0; u < kRescanUnroll; ++u) {
        vi[u] = o0 + u < n_owner ? owner[o0 + u] + j * nthreads : nvec;
        if (vi[u] < nvec) v[u] = __ldg(vp + vi[u]);
      }
#pragma unroll
      for (int u = 0; u < kRescanUnroll; ++u)
        if (vi[u] < nvec) f.visit_vec(v[u], sp.head + static_cast<int64_t>(vi[u]) * kv, true);
    }
  }
}

// Number of the n pairs (v, idx) in shared memory that come before (x, i)
// in the (value desc, index asc) order.
__device__ __forceinline__ int rank_among(float x, int i, const float* v, const int* idx, int n) {
  int r = 0;
  for (int e = 0; e < n; ++e) r += before(v[e], idx[e], x, i) ? 1 : 0;
  return r;
}

// The K best (value desc, index asc) of n pairs in shared memory, by warp 0:
// K rounds of a warp-wide argmax, the winner's owner removing it.  Results
// in out_v / out_i [K].
template <int K>
__device__ __forceinline__ void warp_select_k(float* v, int* idx, int n, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < K; ++r) {
    float bv = neg_inf();
    int bi = INT_MAX, bpos = -1;
    for (int e = lane; e < n; e += 32)
      if (before(v[e], idx[e], bv, bi)) {
        bv = v[e];
        bi = idx[e];
        bpos = e;
      }
    float wv = bv;
    int wi = bi;
    warp_best(wv, wi);
    if (bpos >= 0 && wi != INT_MAX && bv == wv && bi == wi) {
      v[bpos] = neg_inf();
      idx[bpos] = INT_MAX;
    }
    __syncwarp();
    if (lane == 0) {
      out_v[r] = wv;
      out_i[r] = wi;
    }
  }
  __syncwarp();
}

// Sum of 2^((key(x) - m) c) over a row with NaN as -inf.
struct KeyedSum {
  float c, mc, s;
  template <int N>
  __device__ __forceinline__ void visit(const float* x, int64_t) {
#pragma unroll
    for (int j = 0; j < N; ++j) s += fast_exp2(fmaf(order_key(x[j]), c, -mc));
  }
};

// Block merge of (m, s) partials; every thread receives the row's (m, s).
template <int UNUSED>
__device__ __forceinline__ void block_ms(float& m, float& s, float c, float* sm, float* ss) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_merge_ms(m, s, c);
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    float mm = lane < nw ? sm[lane] : neg_inf();
    float s2 = lane < nw ? ss[lane] : 0.0f;
    warp_merge_ms(mm, s2, c);
    if (lane == 0) {
      sm[32] = mm;
      ss[32] = s2;
    }
  }
  __syncthreads();
  m = sm[32];
  s = ss[32];
}

// Per-thread stats-only visitor (draft sampling from logits).
struct StatsVisitor {
  SoftmaxPartial sp;
  template <int N>
  __device__ __forceinline__ void visit(const float* xin, int64_t) {
    float x[N];
#pragma unroll
    for (int j = 0; j < N; ++j) x[j] = order_key(xin[j]);
    sp.template update<N>(x);
  }
};

// Writes p = 2^((x - m) c) / Z for every element of a row.
template <int DT>
struct ProbWriter {
  float c, mc, invz;
  float* out;
  bool vec_ok;
  template <int N>
  __device__ __forceinline__ void visit(const float* xin, int64_t first) {
    float p[N];
#pragma unroll
    for (int j = 0; j < N; ++j) p[j] = fminf(fast_exp2(fmaf(order_key(xin[j]), c, -mc)) * invz, 1.0f);
    if (N >= 4 && vec_ok) {
#pragma unroll
      for (int j = 0; j + 3 < N; j += 4)
        st_stream(out + first + j, make_float4(p[j], p[j + 1], p[j + 2], p[j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < N; ++j) out[first + j] = p[j];
    }
  }
};

struct ZeroWriter {
  float* out;
  template <int N>
  __device__ __forceinline__ void visit(const float*, int64_t first) {
#pragma unroll
    for (int j = 0; j < N; ++j) out[first + j] = 0.0f;
  }
};

// The n best of a row by (key desc, index asc; NaN as -inf), by one warp:
// each pick is the best element after the previous pick in that order,
// starting after (+inf, -1), which every element follows (rows with long
// runs of equal keys, and the fewer-than-k fallback).
template <int DT>
__device__ void warp_rank_row(const void* row, int64_t V, int n, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  float pv = __int_as_float(0x7f800000);
  int pi = -1;
  for (int rr = 0; rr < n; ++rr) {
    float bv = neg_inf();
    int bi = INT_MAX;
    for (int64_t v = lane; v < V; v += 32) {
      const float x = order_key(Logit<DT>::load1(row, v));
      if (before(pv, pi, x, static_cast<int>(v)) && before(x, static_cast<int>(v), bv, bi)) {
        bv = x;
        bi = static_cast<int>(v);
      }
    }
    warp_best(bv, bi);
    if (lane == 0) {
      out_v[rr] = bv;
      out_i[rr] = bi;
    }
    pv = bv;
    pi = bi;
    __syncwarp();
  }
}

// p = min(2^((key(x) - m) c) / Z, 1) for the V elements of a row, written
// to out (zeros when the row has no finite max), streaming stores.
template <int DT>
__device__ __forceinline__ void write_probs(const void* row, int64_t V, bool finite, float mc, float c, float invz,
                                            float* out) {
  if (finite) {
    const RowSpan sp = row_span<DT>(row, V);
    ProbWriter<DT> pw{c, mc, invz, out, (reinterpret_cast<uintptr_t>(out + sp.head) & 15) == 0};
    for_row<DT, 2>(row, V, pw);
  } else {
    ZeroWriter z{out};
    for_row<DT, 2>(row, V, z);
  }
}

template <int K>
__host__ __device__ constexpr size_t draft_smem_bytes() {
  return K == 1 ? 16 : kCandCap * (sizeof(float) + sizeof(int));
}

// One CTA per row, 16-byte loads (8 in flight per thread).  Pass A: the
// online softmax and every thread's best element; the K-th best of those
// bests is a threshold with at least K elements before or at it.  Pass B
// (K > 1): the block reads again (from L2) the elements of the threads
// whose best reaches the threshold (about K of them), collecting the
// elements before or at it; the exact top-K is ranked among them.  All
// reductions are fixed-order.
//
// c = log2(e) / T is the temperature of probs and row_stats (q); with TWO,
// topk_p are at c1 = log2(e) / T_score (the tree scores), else at c.
template <int DT, int K, int THREADS, bool TWO>
__global__ void __launch_bounds__(THREADS, 1024 / THREADS)
    softmax_topk_kernel(const void* __restrict__ logits, int64_t V, float c, float c1, int k,
                        float* __restrict__ topk_p, int32_t* __restrict__ topk_idx,
                        float* __restrict__ probs, float* __restrict__ row_stats,
                        int32_t* __restrict__ stats, ExpandArgs ex) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kWarps = THREADS / 32;
  extern __shared__ __align__(16) unsigned char dsm[];  // K > 1: candidate buffer
  __shared__ float lv[THREADS];
  __shared__ int li[THREADS];
  __shared__ float fv[K];
  __shared__ int fi[K];
  __shared__ float sm[33], ss[33];
  __shared__ int s_owner[K > 1 ? THREADS : 1];
  __shared__ int s_cnt, s_nown, s_ti;
  __shared__ float s_tv;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t r = blockIdx.x;
  const void* row = static_cast<const char*>(logits) + r * V * esz;
  if (!spec_smem_ok(draft_smem_bytes<K>(), stats)) return;
  // pass A: online softmax and every thread's best element (and for K > 1
  // the largest key among its other elements)
  ArgmaxVisitor<DT, (K > 1), TWO> st{c, c1};
  st.reset();
  for_row_fast<DT, kDraftUnroll>(row, V, st, threadIdx.x, THREADS);
  st.own_first(row, V, threadIdx.x);
  lv[threadIdx.x] = st.m;
  li[threadIdx.x] = st.bi;
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_nown = 0;
    s_tv = neg_inf();  // no thread best ranked K-1 (equal empty pairs): all qualify
    s_ti = INT_MAX;
  }
  if (threadIdx.x < K) {
    fv[threadIdx.x] = neg_inf();
    fi[threadIdx.x] = INT_MAX;
  }
  float m = st.m, s = TWO ? st.s0 : st.s0 + st.s1;
  float m1 = st.m, s1 = st.s1;  // TWO: the score temperature's normaliser
  block_ms<0>(m, s, c, sm, ss);  // its barriers also publish lv / li
  if (TWO) block_ms<0>(m1, s1, c1, sm, ss);  // m1 == m: the same keys
  if (isfinite(m) && !(isfinite(s) && (!TWO || isfinite(s1)))) {
    // the row holds a NaN: recompute the normalisers with NaN as -inf
    KeyedSum ks{c, m * c, 0.0f};
    for_row<DT, 2>(row, V, ks);
    const float part = warp_sum(ks.s);
    __syncthreads();
    if (lane == 0) ss[warp] = part;
    __syncthreads();
    float tot = 0.0f;
    for (int w2 = 0; w2 < kWarps; ++w2) tot += ss[w2];
    s = tot;
    if (TWO) {
      KeyedSum ks1{c1, m * c1, 0.0f};
      for_row<DT, 2>(row, V, ks1);
      const float part1 = warp_sum(ks1.s);
      __syncthreads();
      if (lane == 0) ss[warp] = part1;
      __syncthreads();
      float tot1 = 0.0f;
      for (int w2 = 0; w2 < kWarps; ++w2) tot1 += ss[w2];
      s1 = tot1;
    }
  }
  if (!TWO) s1 = s;
  if constexpr (K == 1) {
    if (warp == 0) warp_select_k<1>(lv, li, THREADS, fv, fi);
  } else {
    // threshold: the K-th best of the thread bests (K distinct elements
    // come before or at it).  With 128 threads every thread ranks its own
    // best among them (pairs are distinct but for empty (-inf, INT_MAX)
    // ones; with fewer than K real bests no thread ranks K-1 and everything
    // qualifies); with more threads (few rows, 512-thread CTAs) the ranking
    // costs more than K rounds of a warp argmax in warp 0, measured.
    if constexpr (THREADS > 128) {
      if (warp == 0) {
        warp_select_k<K>(lv, li, THREADS, fv, fi);
        if (lane == 0) {
          s_tv = fv[K - 1];
          s_ti = fi[K - 1];
        }
      }
    } else {
      const float mv = lv[threadIdx.x];
      const int mi = li[threadIdx.x];
      int rk = 0;
#pragma unroll 8
      for (int e = 0; e < THREADS; ++e) rk += before(lv[e], li[e], mv, mi) ? 1 : 0;
      if (rk == K - 1 && mi != INT_MAX) {
        s_tv = mv;
        s_ti = mi;
      }
    }
    __syncthreads();
    const float tv = s_tv;
    const int ti = s_ti;
    // pass B: an element can only qualify if its thread's best does; the
    // block reads the few qualifying threads' elements again (from L2)
    float* cv = reinterpret_cast<float*>(dsm);
    int* ci = reinterpret_cast<int*>(cv + kCandCap);
    CandVisitor<DT> cand{tv, ti, cv, ci, &s_cnt};
    if (cand.qualifies(st.m, st.bi)) {
      // a thread whose other elements are all below the threshold's key
      // contributes its best alone; the others are read again
      if (st.m2v >= tv) {
        s_owner[atomicAdd(&s_nown, 1)] = threadIdx.x;
      } else {
        cand.add(st.m, st.bi);
      }
    }
    __syncthreads();
    rescan_owners<DT>(row, V, cand, s_owner, s_nown, THREADS);
    __syncthreads();
    const int n = s_cnt;
    if (n <= kRankCands) {
      // the candidates' pairs are distinct: their ranks place them
      for (int e = threadIdx.x; e < n; e += THREADS) {
        const int rk = rank_among(cv[e], ci[e], cv, ci, n);
        if (rk < K) {
          fv[rk] = cv[e];
          fi[rk] = ci[e];
        }
      }
    } else if (warp == 0) {
      if (n <= kCandCap) {
        warp_select_k<K>(cv, ci, n, fv, fi);
      } else {
        // more candidates than the buffer holds (a long run of equal
        // keys): rank the whole row
        warp_rank_row<DT>(row, V, K, fv, fi);
      }
    }
    __syncthreads();
  }
  if (warp == 0) {
    __syncwarp();
    // fewer than k non-NaN logits: rank the row again with NaN as -inf
    if (fi[k - 1] == INT_MAX && k <= V) warp_rank_row<DT>(row, V, k, fv, fi);
  }
  __syncthreads();

  const bool finite = isfinite(m);
  const float mc = m * c;
  const float invz = 1.0f / s;
  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    // the score: at c1 with TWO, else at c (c1 == c or no q written)
    const float cs = TWO ? c1 : c;
    const float pj = finite ? fminf(fast_exp2(fmaf(fv[j], cs, -(m * cs))) * (TWO ? 1.0f / s1 : invz), 1.0f) : 0.0f;
    topk_idx[r * k + j] = fi[j];
    topk_p[r * k + j] = pj;
    // a chain's pool expansion (k = 1) by thread 0 from its own outputs
    if (ex.k == 1) expand_chain(ex, static_cast<int>(r), pj, fi[j]);
  }
  if (threadIdx.x == 0) {
    if (!finite) bump(stats, SPEC_STAT_NONFINITE_ROW);
    if (row_stats != nullptr) {
      row_stats[2 * r] = m;
      row_stats[2 * r + 1] = s;
    }
  }
  if (probs != nullptr) write_probs<DT>(row, V, finite, mc, c, invz, probs + r * V);
  // a tree's pool expansion (k > 1), by the CTA that completes the
  // request's rows (dsm holds at least k*k keys: 8 KB for K > 1)
  if (ex.k > 1) {
    __shared__ int s_last;
    expand_if_last(ex, r, threadIdx.x < k, topk_p, topk_idx, reinterpret_cast<uint64_t*>(dsm), &s_last);
  }
}

// ---------------------------------------------------------------- sampling

constexpr int kSampleThreads = 512;

// Weights of one row for the inverse-CDF draw: given fp32 weights, or
// 2^((x - m) c) of logits (m the row max).
struct ProbWeights {
  const float* row;
  int64_t V;
  __device__ __forceinline__ void load8(int64_t v0, float* x) const { load8_f32(row, V, v0, x); }
  __device__ __forceinline__ float at(int64_t v) const { return __ldg(row + v); }
};

template <int DT>
struct LogitWeights {
  const void* row;
  int64_t V;
  float c, mc;
  __device__ __forceinline__ void load8(int64_t v0, float* x) const {
    load8_logits<DT>(row, V, v0, x);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = fast_exp2(fmaf(x[j], c, -mc));
  }
  __device__ __forceinline__ float at(int64_t v) const {
    return fast_exp2(fmaf(order_key(Logit<DT>::load1(row, v)), c, -mc));
  }
};

template <class W>
__device__ __forceinline__ void sample_row(const W& w, int64_t V, float u, float* red, float* tile_sum,
                                           float* scan_sh, int32_t* stats, int32_t* out_token,
                                           float* out_prob) {
  const float total = cdf_tile_pass<kSampleThreads>(w, V, red, tile_sum);
  const int32_t tok = cdf_search<kSampleThreads>(w, V, u, tile_sum, total, scan_sh, stats);
  if (threadIdx.x == 0) {
    *out_token = tok;
    if (out_prob) *out_prob = total > 0.0f ? w.at(tok) / total : 0.0f;
  }
}

template <int DT, bool FROM_PROBS>
__global__ void __launch_bounds__(kSampleThreads)
    sample_kernel(const void* __restrict__ logits, const float* __restrict__ probs, int64_t V,
                  float c, const float* __restrict__ u, int32_t* __restrict__ out_token,
                  float* __restrict__ out_prob, const float* __restrict__ row_stats, int32_t* __restrict__ stats) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  extern __shared__ float dyn[];
  __shared__ float scan_sh[33];
  __shared__ float sm[33], ss[33];
  const int64_t ntiles = (V + kSampleThreads * 8 - 1) / (kSampleThreads * 8);
  float* tile_sum = dyn;
  float* red = dyn + ntiles;
  if (!spec_smem_ok(sizeof(float) * cdf_smem_floats<kSampleThreads>(V), stats)) return;
  const int64_t r = blockIdx.x;
  float* op = out_prob ? out_prob + r : nullptr;
  if (FROM_PROBS) {
    ProbWeights w{probs + r * V, V};
    sample_row(w, V, __ldg(u + r), red, tile_sum, scan_sh, stats, out_token + r, op);
    return;
  }
  const void* row = static_cast<const char*>(logits) + r * V * esz;
  float m;
  if (row_stats != nullptr) {
    m = __ldg(row_stats + 2 * r);  // the row's max from the caller's softmax pass
  } else {
    StatsVisitor st{{c, neg_inf(), 0.0f}};
    for_row<DT, 4>(row, V, st);
    float s = st.sp.s;
    m = st.sp.m;
    block_ms<0>(m, s, c, sm, ss);
  }
  if (!isfinite(m)) {
    if (threadIdx.x == 0) {
      bump(stats, SPEC_STAT_NONFINITE_ROW);
      out_token[r] = 0;
      if (op) *op = 0.0f;
    }
    return;
  }
  LogitWeights<DT> w{row, V, c, m * c};
  sample_row(w, V, __ldg(u + r), red, tile_sum, scan_sh, stats, out_token + r, op);
}

// ------------------------------------------------ fused softmax + sampling
//
// Sampled chains (one token per draft row, [ZS] 5.1: "a candidate y drawn
// from the draft distribution q") need the row's softmax statistics, which
// verification reads, and an inverse-CDF draw from the same distribution.
// One CTA per row streams the row once with the lean loop's layout.  Tile i
// is kFusedRounds rounds of 16-byte vectors (round u: vectors i U T + u T +
// [0, T), contiguous in the vocabulary).  Each thread keeps its running max
// key and its sums relative to it: its partial of every finished tile in
// shared memory, as log2(partial) + max c, and its total.  After the pass one
// block max, 2^(stored - M c) and fixed-order reductions give Z and the tile
// sums; the draw walks
// the tile sums and rescans only the crossing tile, round by round with a
// block scan.  Head and tail scalars (rows not 16-byte aligned) form a tile
// of their own before and after the vectors.
constexpr int kFusedThreads = 128;  // all rows of a 1024-row step resident at once
constexpr int kFusedRounds = 4;
constexpr int kFusedMaxTiles = 128;  // partials: tiles x threads floats of shared memory

template <int DT>
__host__ __device__ constexpr int64_t fused_max_vocab() {
  return static_cast<int64_t>(kFusedMaxTiles) * kFusedRounds * kFusedThreads * Logit<DT>::kVec;
}

template <int DT>
__global__ void __launch_bounds__(kFusedThreads, 1024 / kFusedThreads)
    softmax_sample_kernel(const void* __restrict__ logits, int64_t V64, float c, const float* __restrict__ u,
                          int32_t* __restrict__ out_token, float* __restrict__ out_prob,
                          float* __restrict__ row_stats, float* __restrict__ probs, int32_t* __restrict__ stats,
                          ExpandArgs ex) {
  pdl_enter();
  constexpr int T = kFusedThreads, U = kFusedRounds, kv = Logit<DT>::kVec, kWarps = T / 32;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  extern __shared__ float part[];  // [ntiles][T]: log2 of the partials plus the max they are relative to
  __shared__ float tsum[kFusedMaxTiles + 2];
  __shared__ float red[33], scan_sh[33], rtot[U * kWarps];
  __shared__ int s_tok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const void* row = static_cast<const char*>(logits) + r * V64 * esz;
  const RowSpan sp = row_span<DT>(row, V64);
  const int V = static_cast<int>(V64), head = static_cast<int>(sp.head), nvec = static_cast<int>(sp.nvec);
  const int tail0 = head + nvec * kv, ntiles = (nvec + U * T - 1) / (U * T);
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  if (!spec_smem_ok(sizeof(float) * ntiles * T, stats) || !spec_in(ntiles + 1, kFusedMaxTiles + 2, stats)) return;

  float m = neg_inf(), mc = 0.0f, s = 0.0f, hs = 0.0f, tl = 0.0f;
  if (tid < head) {  // head < kv <= T
    const float x = order_key(Logit<DT>::load1(row, tid));
    if (x != neg_inf()) {
      m = x;
      mc = x * c;
      hs = s = 1.0f;
    }
  }
  // tile i's partial is stored as log2(partial) + m c, m the thread's max at
  // the tile's end; 2^(stored - M c) brings it to the row max after the pass
  auto vec_step = [&](const uint4& raw, float2& acc) {
    float x[kv];
    unpack<DT>(raw, x);
    // NaN-ignoring max; a NaN element makes the sums NaN (repaired below)
    const float vmax = DT == SPEC_BF16 ? max8_bf16(raw) : fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[kv - 1]));
    if (vmax > m) {
      const float f = m == neg_inf() ? 0.0f : fast_exp2((m - vmax) * c);
      s *= f;
      hs *= f;
      acc.x *= f;
      acc.y *= f;
      m = vmax;
      mc = vmax * c;
    }
    if (m != neg_inf()) acc = exp2_sum_pairs<kv>(acc, x, c, mc);
  };
  const int nfull = nvec / (U * T);
  for (int i = 0; i < nfull; ++i) {  // full tiles: no bounds tests
    const int base = i * U * T + tid;
    uint4 v[U];
#pragma unroll
    for (int q = 0; q < U; ++q) v[q] = ld_stream(vp + base + q * T);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < U; ++q) vec_step(v[q], acc);
    const float pt = acc.x + acc.y;
    part[i * T + tid] = fast_log2(pt) + mc;
    s += pt;
  }
  if (nfull < ntiles) {  // the last, partial tile
    const int base = nfull * U * T + tid;
    uint4 v[U];
#pragma unroll
    for (int q = 0; q < U; ++q)
      if (base + q * T < nvec) v[q] = ld_stream(vp + base + q * T);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < U; ++q)
      if (base + q * T < nvec) vec_step(v[q], acc);
    const float pt = acc.x + acc.y;
    part[nfull * T + tid] = fast_log2(pt) + mc;
    s += pt;
  }
  if (tail0 + tid < V) {  // fewer than kv tail elements
    const float x = order_key(Logit<DT>::load1(row, tail0 + tid));
    if (x > m) {
      const float f = m == neg_inf() ? 0.0f : fast_exp2((m - x) * c);
      s *= f;
      hs *= f;
      m = x;
      mc = x * c;
    }
    if (m != neg_inf()) {
      tl = fast_exp2(fmaf(x, c, -mc));
      s += tl;
    }
  }
  // a NaN in this thread's elements: recompute its partials with NaN as -inf
  // (the max is already NaN-free)
  if (!isfinite(s) && m != neg_inf() && isfinite(m)) {
    s = 0.0f;
    for (int i = 0; i < ntiles; ++i) {
      const int base = i * U * T + tid;
      float pt = 0.0f;
      for (int q = 0; q < U; ++q) {
        if (base + q * T >= nvec) continue;
        float x[kv];
        unpack<DT>(__ldg(vp + base + q * T), x);
#pragma unroll
        for (int j = 0; j < kv; ++j) pt += fast_exp2(fmaf(order_key(x[j]), c, -mc));
      }
      part[i * T + tid] = fast_log2(pt) + mc;
      s += pt;
    }
    s += hs + tl;
  }
  // row max, per-thread scale, normaliser (fixed order)
  float mb = warp_max(m);
  if (lane == 0) red[warp] = mb;
  __syncthreads();
  if (warp == 0) {
    float x = lane < kWarps ? red[lane] : neg_inf();
    x = warp_max(x);
    if (lane == 0) red[32] = x;
  }
  __syncthreads();
  const float M = red[32];
  const bool finite = isfinite(M);
  const float f = (finite && m != neg_inf()) ? fast_exp2((m - M) * c) : 0.0f;
  const float zw = warp_sum(s * f);
  __syncthreads();
  if (lane == 0) red[warp] = zw;
  const float Mc_ = M * c;
  for (int j = 0; j < ntiles; ++j) part[j * T + tid] = finite ? fast_exp2(part[j * T + tid] - Mc_) : 0.0f;
  hs *= f;
  tl *= f;
  __syncthreads();
  float Z = 0.0f;
  for (int w2 = 0; w2 < kWarps; ++w2) Z += red[w2];
  for (int j = warp; j < ntiles; j += kWarps) {
    float a = 0.0f;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) a += part[j * T + q * 32 + lane];
    a = warp_sum(a);
    if (lane == 0) tsum[1 + j] = a;
  }
  if (warp == 0) {  // head and tail threads are all in warp 0
    const float h = warp_sum(hs), t = warp_sum(tl);
    if (lane == 0) {
      tsum[0] = h;
      tsum[ntiles + 1] = t;
      s_tok = INT_MAX;
    }
  }
  __syncthreads();
  if (!finite) {
    if (tid == 0) {
      bump(stats, SPEC_STAT_NONFINITE_ROW);
      out_token[r] = 0;
      if (out_prob) out_prob[r] = 0.0f;
      if (row_stats) {
        row_stats[2 * r] = M;
        row_stats[2 * r + 1] = Z;
      }
      if (ex.k != 0) expand_chain(ex, static_cast<int>(r), 0.0f, 0);  // the step's pool expansion
    }
    if (probs) write_probs<DT>(row, V64, false, 0.0f, c, 0.0f, probs + r * V64);
    return;
  }
  float W = 0.0f;
  for (int j = 0; j < ntiles + 2; ++j) W += tsum[j];
  const float Mc = M * c;
  const float target = __ldg(u + r) * W;
  float prefix = 0.0f;
  if (W > 0.0f && isfinite(W)) {
    for (int j = 0; j < ntiles + 2; ++j) {
      const float after = prefix + tsum[j];
      if (after > target) {
        if (j == 0 || j == ntiles + 1) {  // a scalar tile, scanned by thread 0
          if (tid == 0) {
            const int lo = j == 0 ? 0 : tail0, hi = j == 0 ? head : V;
            float C = prefix;
            for (int e = lo; e < hi; ++e) {
              C += fast_exp2(fmaf(order_key(Logit<DT>::load1(row, e)), c, -Mc));
              if (C > target) {
                s_tok = e;
                break;
              }
            }
          }
        } else {
          // the tile's rounds: all loads at once, the rounds' totals, then
          // a block scan of the crossing round only (later rounds if
          // rounding moves the crossing)
          float w[U][kv], ws[U];
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const int vi = (j - 1) * U * T + q * T + tid;
            ws[q] = 0.0f;
            if (vi < nvec) {
              unpack<DT>(__ldg(vp + vi), w[q]);
            } else {
#pragma unroll
              for (int k = 0; k < kv; ++k) w[q][k] = neg_inf();
            }
          }
#pragma unroll
          for (int q = 0; q < U; ++q) {
#pragma unroll
            for (int k = 0; k < kv; ++k) {
              w[q][k] = fast_exp2(fmaf(order_key(w[q][k]), c, -Mc));
              ws[q] += w[q][k];
            }
          }
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const float t = warp_sum(ws[q]);
            if (lane == 0) rtot[q * kWarps + warp] = t;
          }
          __syncthreads();
          float C0 = prefix;
#pragma unroll
          for (int q = 0; q < U; ++q) {
            float rt = 0.0f;
            for (int w2 = 0; w2 < kWarps; ++w2) rt += rtot[q * kWarps + w2];
            if (C0 + rt > target || q == U - 1) {
              const int vi = (j - 1) * U * T + q * T + tid;
              float tot;
              const float incl = block_inclusive_scan(ws[q], scan_sh, tot);
              float C = C0 + (incl - ws[q]);
              int fnd = -1;
#pragma unroll
              for (int k = 0; k < kv; ++k) {
                C += w[q][k];
                if (fnd < 0 && C > target && vi < nvec) fnd = k;
              }
              if (fnd >= 0) atomicMin(&s_tok, head + vi * kv + fnd);
              __syncthreads();
              if (s_tok != INT_MAX) break;
            }
            C0 += rt;
          }
        }
        __syncthreads();
        if (s_tok != INT_MAX) break;
      }
      prefix = after;
    }
  }
  __syncthreads();
  if (s_tok == INT_MAX) {
    // rounding left no crossing: the last index of positive weight
    __syncthreads();
    if (tid == 0) s_tok = -1;
    __syncthreads();
    for (int v = tid; v < V; v += T)
      if (fast_exp2(fmaf(order_key(Logit<DT>::load1(row, v)), c, -Mc)) > 0.0f) atomicMax(&s_tok, v);
    __syncthreads();
    if (tid == 0) {
      if (s_tok < 0) s_tok = 0;
      bump(stats, SPEC_STAT_CDF_FALLBACK);
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int tok = s_tok;
    out_token[r] = tok;
    const float pr = W > 0.0f ? fast_exp2(fmaf(order_key(Logit<DT>::load1(row, tok)), c, -Mc)) / W : 0.0f;
    if (out_prob) out_prob[r] = pr;
    if (row_stats) {
      row_stats[2 * r] = M;
      row_stats[2 * r + 1] = Z;
    }
    if (ex.k != 0) expand_chain(ex, static_cast<int>(r), pr, tok);  // the step's pool expansion
  }
  if (probs) write_probs<DT>(row, V64, true, Mc, c, 1.0f / Z, probs + r * V64);
}

template <int DT, int K, int THREADS, bool TWO>
int launch_softmax_topk_t2(const void* logits, int64_t R, int64_t V, float c, float c1, int k, float* topk_p,
                           int32_t* topk_idx, float* probs, float* row_stats, int32_t* stats, const ExpandArgs& ex,
                           cudaStream_t s) {
  constexpr size_t smem = draft_smem_bytes<K>();
  if (smem > 48 * 1024 && cudaFuncSetAttribute(softmax_topk_kernel<DT, K, THREADS, TWO>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  launch_k(softmax_topk_kernel<DT, K, THREADS, TWO>, static_cast<unsigned>(R), THREADS, smem, s, logits, V, c, c1, k,
           topk_p, topk_idx, probs, row_stats, stats, ex);
  return launch_status();
}

// c: the temperature of q (probs, row_stats); c1: that of topk_p.  The
// two-normaliser instance runs only when q is written at another
// temperature than the scores.
template <int DT, int K, int THREADS>
int launch_softmax_topk_t(const void* logits, int64_t R, int64_t V, float c, float c1, int k, float* topk_p,
                          int32_t* topk_idx, float* probs, float* row_stats, int32_t* stats, const ExpandArgs& ex,
                          cudaStream_t s) {
  const bool want_q = probs != nullptr || row_stats != nullptr;
  if (want_q && c != c1)
    return launch_softmax_topk_t2<DT, K, THREADS, true>(logits, R, V, c, c1, k, topk_p, topk_idx, probs, row_stats,
                                                        stats, ex, s);
  const float cc = want_q ? c : c1;
  return launch_softmax_topk_t2<DT, K, THREADS, false>(logits, R, V, cc, cc, k, topk_p, topk_idx, probs, row_stats,
                                                       stats, ex, s);
}

// One CTA per row.  With few rows (at most two per SM of a 152-SM GB300)
// a row gets 512 threads, so that each SM still keeps enough loads in
// flight; otherwise kDraftThreads.
constexpr int64_t kFewRows = 2 * 152;

template <int DT, int K>
int launch_softmax_topk(const void* logits, int64_t R, int64_t V, float c, float c1, int k, float* topk_p,
                        int32_t* topk_idx, float* probs, float* row_stats, int32_t* stats, const ExpandArgs& ex,
                        cudaStream_t s) {
  if (R <= kFewRows)
    return launch_softmax_topk_t<DT, K, 512>(logits, R, V, c, c1, k, topk_p, topk_idx, probs, row_stats, stats, ex,
                                             s);
  return launch_softmax_topk_t<DT, K, kDraftThreads>(logits, R, V, c, c1, k, topk_p, topk_idx, probs, row_stats,
                                                     stats, ex, s);
}

template <int DT>
int dispatch_softmax_topk(const void* logits, int64_t R, int64_t V, float c, float c1, int k, float* topk_p,
                          int32_t* topk_idx, float* probs, float* row_stats, int32_t* stats, const ExpandArgs& ex,
                          cudaStream_t s) {
#define SPEC_TOPK_CASE(KK)                                                                                   \
  return launch_softmax_topk<DT, KK>(logits, R, V, c, c1, k, topk_p, topk_idx, probs, row_stats, stats, ex, s)
  if (k <= 1) SPEC_TOPK_CASE(1);
  if (k <= 2) SPEC_TOPK_CASE(2);
  if (k <= 4) SPEC_TOPK_CASE(4);
  if (k <= 8) SPEC_TOPK_CASE(8);
  if (k <= 16) SPEC_TOPK_CASE(16);
  SPEC_TOPK_CASE(32);
#undef SPEC_TOPK_CASE
}

}  // namespace
}  // namespace specdec

using namespace specdec;

namespace {
int softmax_topk_impl(const void* logits, int dtype, int64_t R, int64_t V, float T, float T_score, int k,
                      float* topk_p, int32_t* topk_idx, float* probs_or_null, float* row_stats_or_null,
                      int32_t* stats_or_null, const spec_expand_t* expand, spec_stream_t stream) {
  if (R < 0 || V < 1 || k < 1 || k > V || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (!(T_score > 0.0f) || !isfinite(T_score)) return SPEC_ERR_INVALID_ARG;
  if (R > 0 && (logits == nullptr || topk_p == nullptr || topk_idx == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (k > SPEC_MAX_TOPK || V > SPEC_MAX_VOCAB || R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  ExpandArgs ex = no_expand();
  if (expand != nullptr) {
    const int e = expand_args(expand, k, R, ex);
    if (e != SPEC_OK) return e;
  }
  if (R == 0) return SPEC_OK;
  const float c = kLog2e / T, c1 = T_score == T ? c : kLog2e / T_score;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SPEC_BF16
             ? dispatch_softmax_topk<SPEC_BF16>(logits, R, V, c, c1, k, topk_p, topk_idx, probs_or_null,
                                                row_stats_or_null, stats_or_null, ex, s)
             : dispatch_softmax_topk<SPEC_F32>(logits, R, V, c, c1, k, topk_p, topk_idx, probs_or_null,
                                               row_stats_or_null, stats_or_null, ex, s);
}
}  // namespace

extern "C" int spec_softmax_topk(const void* logits, int dtype, int64_t R, int64_t V, float T, float T_score, int k,
                                 float* topk_p, int32_t* topk_idx, float* probs_or_null,
                                 float* row_stats_or_null, int32_t* stats_or_null, spec_stream_t stream) {
  return softmax_topk_impl(logits, dtype, R, V, T, T_score, k, topk_p, topk_idx, probs_or_null, row_stats_or_null,
                           stats_or_null, nullptr, stream);
}

extern "C" int spec_softmax_topk_expand(const void* logits, int dtype, int64_t R, int64_t V, float T, float T_score,
                                        int k, float* topk_p, int32_t* topk_idx, float* probs_or_null,
                                        float* row_stats_or_null, int32_t* stats_or_null,
                                        const spec_expand_t* expand, spec_stream_t stream) {
  if (expand == nullptr) return SPEC_ERR_INVALID_ARG;
  return softmax_topk_impl(logits, dtype, R, V, T, T_score, k, topk_p, topk_idx, probs_or_null, row_stats_or_null,
                           stats_or_null, expand, stream);
}

namespace {
int softmax_sample_impl(const void* logits, int dtype, int64_t R, int64_t V, float T, const float* u,
                        int32_t* out_token, float* out_prob_or_null, float* row_stats_or_null, float* probs_or_null,
                        int32_t* stats_or_null, const spec_expand_t* expand, spec_stream_t stream) {
  if (R < 0 || V < 1 || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (R > 0 && (logits == nullptr || u == nullptr || out_token == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  if (V > (dtype == SPEC_BF16 ? fused_max_vocab<SPEC_BF16>() : fused_max_vocab<SPEC_F32>()))
    return SPEC_ERR_UNSUPPORTED;
  ExpandArgs ex = no_expand();
  if (expand != nullptr) {
    if (out_prob_or_null == nullptr) return SPEC_ERR_INVALID_ARG;
    const int e = expand_args(expand, 1, R, ex);
    if (e != SPEC_OK) return e;
  }
  if (R == 0) return SPEC_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  const int kv = dtype == SPEC_BF16 ? 8 : 4;
  const int64_t ntiles = (V / kv + kFusedRounds * kFusedThreads - 1) / (kFusedRounds * kFusedThreads);
  const size_t smem = sizeof(float) * static_cast<size_t>(ntiles > 0 ? ntiles : 1) * kFusedThreads;
  const unsigned grid = static_cast<unsigned>(R);
  if (dtype == SPEC_BF16) {
    if (smem > 48 * 1024 && cudaFuncSetAttribute(softmax_sample_kernel<SPEC_BF16>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem)) != cudaSuccess)
      return SPEC_ERR_CUDA;
    launch_k(softmax_sample_kernel<SPEC_BF16>, grid, kFusedThreads, smem, s, logits, V, c, u, out_token,
             out_prob_or_null, row_stats_or_null, probs_or_null, stats_or_null, ex);
  } else {
    if (smem > 48 * 1024 && cudaFuncSetAttribute(softmax_sample_kernel<SPEC_F32>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem)) != cudaSuccess)
      return SPEC_ERR_CUDA;
    launch_k(softmax_sample_kernel<SPEC_F32>, grid, kFusedThreads, smem, s, logits, V, c, u, out_token,
             out_prob_or_null, row_stats_or_null, probs_or_null, stats_or_null, ex);
  }
  return launch_status();
}
}  // namespace

extern "C" int spec_softmax_sample(const void* logits, int dtype, int64_t R, int64_t V, float T, const float* u,
                                   int32_t* out_token, float* out_prob_or_null, float* row_stats_or_null,
                                   float* probs_or_null, int32_t* stats_or_null, spec_stream_t stream) {
  return softmax_sample_impl(logits, dtype, R, V, T, u, out_token, out_prob_or_null, row_stats_or_null,
                             probs_or_null, stats_or_null, nullptr, stream);
}

extern "C" int spec_softmax_sample_expand(const void* logits, int dtype, int64_t R, int64_t V, float T,
                                          const float* u, int32_t* out_token, float* out_prob,
                                          float* row_stats_or_null, float* probs_or_null, int32_t* stats_or_null,
                                          const spec_expand_t* expand, spec_stream_t stream) {
  if (expand == nullptr) return SPEC_ERR_INVALID_ARG;
  return softmax_sample_impl(logits, dtype, R, V, T, u, out_token, out_prob, row_stats_or_null, probs_or_null,
                             stats_or_null, expand, stream);
}

extern "C" int spec_sample(const void* logits_or_null, int dtype, const float* probs_or_null, int64_t R,
                           int64_t V, float T, const float* u, int32_t* out_token, float* out_prob_or_null,
                           const float* row_stats_or_null, int32_t* stats_or_null, spec_stream_t stream) {
  if (R < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (R > 0 && (u == nullptr || out_token == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (R > 0 && logits_or_null == nullptr && probs_or_null == nullptr) return SPEC_ERR_INVALID_ARG;
  if (probs_or_null == nullptr && (!(T > 0.0f) || !isfinite(T))) return SPEC_ERR_INVALID_ARG;
  if (probs_or_null == nullptr && dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (V > SPEC_MAX_VOCAB || R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  if (R == 0) return SPEC_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t smem = sizeof(float) * static_cast<size_t>(cdf_smem_floats<kSampleThreads>(V));
  const float c = probs_or_null ? 0.0f : kLog2e / T;
  const unsigned grid = static_cast<unsigned>(R);
  if (smem > 48 * 1024) {
    cudaFuncSetAttribute(sample_kernel<SPEC_F32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(sample_kernel<SPEC_F32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(sample_kernel<SPEC_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  }
  if (probs_or_null)
    launch_k(sample_kernel<SPEC_F32, true>, grid, kSampleThreads, smem, s, nullptr, probs_or_null, V, c, u, out_token,
             out_prob_or_null, nullptr, stats_or_null);
  else if (dtype == SPEC_BF16)
    launch_k(sample_kernel<SPEC_BF16, false>, grid, kSampleThreads, smem, s, logits_or_null, nullptr, V, c, u,
             out_token, out_prob_or_null, row_stats_or_null, stats_or_null);
  else
    launch_k(sample_kernel<SPEC_F32, false>, grid, kSampleThreads, smem, s, logits_or_null, nullptr, V, c, u,
             out_token, out_prob_or_null, row_stats_or_null, stats_or_null);
  return launch_status();
}
