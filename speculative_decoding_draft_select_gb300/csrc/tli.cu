// TLI (Token-Level Intersection): heterogeneous-vocabulary drafting.
//
// SGLang PR #22883 "TLI (Token-Level Intersection)", section Modifications:
// vocab_mapping.py exposes constrain_draft_logits (non-intersection draft
// logits set to -inf before the top-k), map_target_to_draft_ids and
// map_draft_to_target_ids, and intersection_draft_ids; the TLIWorker hook
// capture_for_decode constrains the draft logits before top-k sampling; the
// server arguments require topk == 1 and num_draft_tokens == num_steps + 1.
// The rejection sampler of the target is unchanged, so verification reads
// the constrained draft distribution written in target-vocabulary order.
//
// Two kernels compute the same outputs:
// tli_constrain_kernel (tli_constrain_map): one CTA per draft row.  Pass 1
// streams the row with 16-byte loads together with the matching 16-byte
// loads of d2t (the table is shared by every row and stays in L2), masks
// ids outside the intersection (d2t[v] < 0) to -inf and keeps the masked
// top-1 and online-softmax partials.  Pass 2 (optional) writes q in target
// order: q_t[t] = p(t2d[t]) or 0, with coalesced 16-byte stores and gathers
// from the draft row (L2-resident), 8 in flight per thread.
// tli_planned_kernel (tli_constrain_map_planned): persistent CTAs with a
// plan of the two maps (built once by tli_plan_build) that keep the
// intersection bitmap and the row's intersection logits in shared memory,
// so that pass 2's gathers are shared-memory reads (described below).
#include <climits>

#include "common.cuh"
#include "expand.cuh"

namespace specdec {
namespace {

constexpr int kTliThreads = 512;

// Pass 1 of a draft row: the online softmax and the best element over the
// intersection only (ids with d2t < 0 count as -inf, as do NaN logits).
// Each thread visits its elements in increasing index order, so only a
// strictly larger key replaces its best.  The mask comes with the logits:
// two 16-byte loads of d2t per 8 bf16 logits (one per 4 fp32 ones).
template <int DT>
struct MaskedVisitor {
  const int32_t* d2t;
  float c, m, mc, s0, s1;
  int bi;
  __device__ __forceinline__ void rescale(float nm) {
    if (m == neg_inf()) {
      s0 = s1 = 0.0f;
    } else {
      const float f = fast_exp2((m - nm) * c);
      s0 *= f;
      s1 *= f;
    }
    m = nm;
    mc = nm * c;
  }
  __device__ __forceinline__ void visit1(float x, int64_t idx, bool ok) {
    if (!ok || __ldg(d2t + idx) < 0) return;
    const float xk = order_key(x);
    if (xk > m) {
      rescale(xk);
      bi = static_cast<int>(idx);
    }
    if (m != neg_inf()) s0 += fast_exp2(fmaf(xk, c, -mc));
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int64_t first, bool) {
    constexpr int kv = Logit<DT>::kVec;
    float x[kv];
    unpack<DT>(raw, x);
    int d[kv];
    if ((reinterpret_cast<uintptr_t>(d2t + first) & 15) == 0) {
#pragma unroll
      for (int h = 0; h < kv / 4; ++h) {
        const int4 t = __ldg(reinterpret_cast<const int4*>(d2t + first) + h);
        d[4 * h] = t.x;
        d[4 * h + 1] = t.y;
        d[4 * h + 2] = t.z;
        d[4 * h + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kv; ++j) d[j] = __ldg(d2t + first + j);
    }
    float vmax = neg_inf();
#pragma unroll
    for (int j = 0; j < kv; ++j) {
      x[j] = d[j] >= 0 ? order_key(x[j]) : neg_inf();
      vmax = fmaxf(vmax, x[j]);
    }
    if (vmax > m) {
      int j0 = 0;
#pragma unroll
      for (int j = kv - 1; j >= 0; --j)
        if (x[j] == vmax) j0 = j;
      rescale(vmax);
      bi = static_cast<int>(first) + j0;
    }
    if (m != neg_inf()) {
      const float2 a = exp2_sum_pairs<kv>(make_float2(s0, s1), x, c, mc);
      s0 = a.x;
      s1 = a.y;
    }
  }
};

// q_t = min(2^((key - m) c) / Z, 1) of draft logit d of the row, or 0 off
// the intersection (d < 0) or when the row has no intersection logit.
template <int DT>
__device__ __forceinline__ float q_of(const void* row, int32_t d, int64_t Vd, bool ok, float c, float mc,
                                      float invz) {
  return (ok && d >= 0 && d < Vd) ? fminf(fast_exp2(fmaf(order_key(Logit<DT>::load1(row, d)), c, -mc)) * invz, 1.0f)
                                  : 0.0f;
}

template <int DT>
struct Elem;
template <>
struct Elem<SPEC_BF16> {
  using T = uint16_t;
  __device__ __forceinline__ static T at(const uint4& raw, int j) {
    const uint32_t w = j < 2 ? raw.x : j < 4 ? raw.y : j < 6 ? raw.z : raw.w;
    return static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xffffu));
  }
  // x as loaded by Logit<SPEC_BF16>::load1 (a bf16 value widened exactly)
  __device__ __forceinline__ static T of_value(float x) { return static_cast<uint16_t>(__float_as_uint(x) >> 16); }
  __device__ __forceinline__ static float value(T e) { return __uint_as_float(static_cast<uint32_t>(e) << 16); }
};
template <>
struct Elem<SPEC_F32> {
  using T = float;
  __device__ __forceinline__ static T at(const uint4& raw, int j) {
    return __uint_as_float(j == 0 ? raw.x : j == 1 ? raw.y : j == 2 ? raw.z : raw.w);
  }
  __device__ __forceinline__ static T of_value(float x) { return x; }
  __device__ __forceinline__ static float value(T e) { return e; }
};

// Where pass 2 writes the constrained draft distribution in target order
// (each output optional).  q: fp32 probabilities.  ql and qs: the same
// distribution in logit form -- ql[t] the draft logit (raw bits) of t's
// partner t2d[t], -inf without one, and qs = (m, Z), the row's largest
// intersection key and its normaliser sum 2^((key - m) c); the stochastic
// verify recomputes q[t] = min(2^((key - m) c) / Z, 1) from them with the
// operations of the written probabilities, bit for bit.
struct QOut {
  float* q;
  void* ql;
  float* qs;
};

// 4 consecutive elements with one streaming 8- or 16-byte store
__device__ __forceinline__ void st_stream4(uint16_t* p, uint16_t a, uint16_t b, uint16_t c, uint16_t d) {
  asm volatile("st.global.cs.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16)),
               "r"(static_cast<uint32_t>(c) | (static_cast<uint32_t>(d) << 16))
               : "memory");
}
__device__ __forceinline__ void st_stream4(float* p, float a, float b, float c, float d) {
  st_stream(p, make_float4(a, b, c, d));
}

template <int DT>
__global__ void __launch_bounds__(kTliThreads)
    tli_constrain_kernel(int64_t Vd, int64_t Vt, const void* __restrict__ draft, const int32_t* __restrict__ d2t,
                         const int32_t* __restrict__ t2d, float c, int32_t* __restrict__ top1_draft,
                         int32_t* __restrict__ top1_target, float* __restrict__ top1_p, QOut qo,
                         int32_t* __restrict__ stats) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kWarps = kTliThreads / 32;
  __shared__ float wm[kWarps], ws[kWarps], wv[kWarps];
  __shared__ int wi[kWarps];
  __shared__ float s_m, s_invz;
  __shared__ int s_best;
  const int64_t r = blockIdx.x;
  const void* row = static_cast<const char*>(draft) + r * Vd * esz;
  MaskedVisitor<DT> st{d2t, c, neg_inf(), 0.0f, 0.0f, 0.0f, INT_MAX};
  for_row_fast<DT, 4>(row, Vd, st, threadIdx.x, kTliThreads);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float bv = st.m;
  int bi = st.bi;
  warp_best(bv, bi);
  float m = st.m, s = st.s0 + st.s1;
  warp_merge_ms(m, s, c);
  if (lane == 0) {
    wv[warp] = bv;
    wi[warp] = bi;
    wm[warp] = m;
    ws[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kWarps ? wv[lane] : neg_inf();
    bi = lane < kWarps ? wi[lane] : INT_MAX;
    warp_best(bv, bi);
    m = lane < kWarps ? wm[lane] : neg_inf();
    s = lane < kWarps ? ws[lane] : 0.0f;
    warp_merge_ms(m, s, c);
    if (lane == 0) {
      const bool ok = bi != INT_MAX && isfinite(bv);
      s_best = ok ? bi : -1;
      s_m = m;
      s_invz = 1.0f / s;
      top1_draft[r] = ok ? bi : -1;
      top1_target[r] = ok ? __ldg(d2t + bi) : -1;
      top1_p[r] = ok ? fminf(fast_exp2(fmaf(bv, c, -m * c)) * (1.0f / s), 1.0f) : 0.0f;
      if (!ok) bump(stats, SPEC_STAT_EMPTY_INTERSECTION);
      if (qo.qs != nullptr) {
        qo.qs[2 * r] = ok ? m : neg_inf();
        qo.qs[2 * r + 1] = s;
      }
    }
  }
  __syncthreads();
  if (qo.ql != nullptr) {
    // logit form: the partners' logits gathered from the row, -inf without one
    using E = typename Elem<DT>::T;
    E* lo = static_cast<E*>(qo.ql) + r * Vt;
    auto l_of = [&](int32_t d) -> E {
      return Elem<DT>::of_value(d >= 0 && d < Vd ? Logit<DT>::load1(row, d) : neg_inf());
    };
    const bool vl =
        (reinterpret_cast<uintptr_t>(lo) & (4 * esz - 1)) == 0 && (reinterpret_cast<uintptr_t>(t2d) & 15) == 0;
    const int nl = vl ? static_cast<int>(Vt / 4) : 0;
    for (int i = threadIdx.x; i < nl; i += kTliThreads) {
      const int4 d = __ldg(reinterpret_cast<const int4*>(t2d) + i);
      st_stream4(lo + 4 * i, l_of(d.x), l_of(d.y), l_of(d.z), l_of(d.w));
    }
    for (int64_t t = static_cast<int64_t>(nl) * 4 + threadIdx.x; t < Vt; t += kTliThreads) lo[t] = l_of(__ldg(t2d + t));
  }
  if (qo.q == nullptr) return;
  float* out = qo.q + r * Vt;
  const bool ok = s_best >= 0;
  const float mc = s_m * c, invz = s_invz;
  const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0 && (reinterpret_cast<uintptr_t>(t2d) & 15) == 0;
  const int nv = vec ? static_cast<int>(Vt / 4) : 0;
  // two groups of 4 targets per thread and step: 8 gathers from the draft
  // row (just read, in L2) in flight
  int i = threadIdx.x;
  for (; i + kTliThreads < nv; i += 2 * kTliThreads) {
    const int4 d0 = __ldg(reinterpret_cast<const int4*>(t2d) + i);
    const int4 d1 = __ldg(reinterpret_cast<const int4*>(t2d) + i + kTliThreads);
    float4 p0, p1;
    p0.x = q_of<DT>(row, d0.x, Vd, ok, c, mc, invz);
    p0.y = q_of<DT>(row, d0.y, Vd, ok, c, mc, invz);
    p0.z = q_of<DT>(row, d0.z, Vd, ok, c, mc, invz);
    p0.w = q_of<DT>(row, d0.w, Vd, ok, c, mc, invz);
    p1.x = q_of<DT>(row, d1.x, Vd, ok, c, mc, invz);
    p1.y = q_of<DT>(row, d1.y, Vd, ok, c, mc, invz);
    p1.z = q_of<DT>(row, d1.z, Vd, ok, c, mc, invz);
    p1.w = q_of<DT>(row, d1.w, Vd, ok, c, mc, invz);
    st_stream(out + 4 * i, p0);
    st_stream(out + 4 * (i + kTliThreads), p1);
  }
  for (; i < nv; i += kTliThreads) {
    const int4 d = __ldg(reinterpret_cast<const int4*>(t2d) + i);
    st_stream(out + 4 * i,
              make_float4(q_of<DT>(row, d.x, Vd, ok, c, mc, invz), q_of<DT>(row, d.y, Vd, ok, c, mc, invz),
                          q_of<DT>(row, d.z, Vd, ok, c, mc, invz), q_of<DT>(row, d.w, Vd, ok, c, mc, invz)));
  }
  for (int64_t t = static_cast<int64_t>(nv) * 4 + threadIdx.x; t < Vt; t += kTliThreads)
    out[t] = q_of<DT>(row, __ldg(t2d + t), Vd, ok, c, mc, invz);
}

// ------------------------------------------------------------ map plan
//
// The two vocabulary maps are fixed for a model pair, so the per-row work
// leans on a plan built from them (tli_plan_build):
//   K           the number of intersection ids (d2t >= 0);
//   mw[w]       bitmap word w of the draft vocabulary (bit j set when
//               d2t[32 w + j] >= 0) and the number of set bits in the words
//               before it, so that the rank of an intersection id among
//               the intersection ids (in id order) is a popcount away;
//   t2r[t]      for every target id, the rank of its draft partner d =
//               t2d[t] (t2r >= 0), -1 when it has none (t2d < 0 or d past
//               V_d), or -2 - d when d lies outside the intersection.
// Layout (16-byte aligned): int32 K and 3 pad words, uint2 mw[Wp] (W =
// ceil(V_d / 32) rounded up to even), int32 t2r[V_t rounded up to 4].
__host__ __device__ inline int64_t plan_words(int64_t Vd) { return ((Vd + 31) / 32 + 1) & ~int64_t(1); }
__host__ __device__ inline int64_t plan_bytes(int64_t Vd, int64_t Vt) {
  return 16 + 8 * plan_words(Vd) + 4 * ((Vt + 3) & ~int64_t(3));
}
struct PlanView {
  int32_t* K;
  uint2* mw;
  int32_t* t2r;
};
__host__ __device__ inline PlanView plan_view(void* plan, int64_t Vd) {
  char* p = static_cast<char*>(plan);
  return {reinterpret_cast<int32_t*>(p), reinterpret_cast<uint2*>(p + 16),
          reinterpret_cast<int32_t*>(p + 16 + 8 * plan_words(Vd))};
}

// Exclusive scan of one int per thread across the block (thread order);
// `sh` holds at least 33 ints.  Returns the thread's exclusive prefix and
// the block total in `total`.
__device__ __forceinline__ int block_exclusive_scan_int(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) sh[lane] = w;
  }
  __syncthreads();
  total = sh[nw - 1];
  const int r = x - v + (warp > 0 ? sh[warp - 1] : 0);
  __syncthreads();  // sh may be reused
  return r;
}

// Bitmap words, one warp-wide ballot over 32 consecutive d2t entries each.
__global__ void plan_bits_kernel(const int32_t* __restrict__ d2t, int64_t Vd, uint2* __restrict__ mw) {
  pdl_enter();
  const int Wp = static_cast<int>(plan_words(Vd));
  const int lane = threadIdx.x & 31;
  const int gw = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  for (int w = gw; w < Wp; w += nwarps) {  // warp-uniform bound
    const int64_t v = 32 * static_cast<int64_t>(w) + lane;
    const uint32_t b = __ballot_sync(0xffffffffu, v < Vd && __ldg(d2t + v) >= 0);
    if (lane == 0) mw[w] = make_uint2(b, 0u);
  }
}

constexpr int kPlanScanThreads = 1024;

// Set bits before each word (exclusive scan of the popcounts) and K.
__global__ void __launch_bounds__(kPlanScanThreads) plan_scan_kernel(int64_t Vd, uint2* __restrict__ mw,
                                                                     int32_t* __restrict__ K_out) {
  pdl_enter();
  __shared__ int sh[33];
  const int Wp = static_cast<int>(plan_words(Vd));
  const int per = (Wp + kPlanScanThreads - 1) / kPlanScanThreads;
  const int w0 = static_cast<int>(threadIdx.x) * per;
  int cnt = 0;
  for (int j = 0; j < per; ++j)
    if (w0 + j < Wp) cnt += __popc(mw[w0 + j].x);
  int K;
  int run = block_exclusive_scan_int(cnt, sh, K);
  for (int j = 0; j < per; ++j)
    if (w0 + j < Wp) {
      mw[w0 + j].y = static_cast<uint32_t>(run);
      run += __popc(mw[w0 + j].x);
    }
  if (threadIdx.x == 0) *K_out = K;
}

// Rank of every target's draft partner (see the plan layout).
__global__ void plan_t2r_kernel(const int32_t* __restrict__ t2d, int64_t Vd, int64_t Vt,
                                const uint2* __restrict__ mw, int32_t* __restrict__ t2r) {
  pdl_enter();
  const int64_t Vt4 = (Vt + 3) & ~int64_t(3);
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < Vt4;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int32_t r = -1;
    const int32_t d = t < Vt ? __ldg(t2d + t) : -1;
    if (d >= 0 && d < Vd) {
      const uint2 e = __ldg(mw + (d >> 5));
      const uint32_t bit = 1u << (d & 31);
      r = (e.x & bit) ? static_cast<int32_t>(e.y) + __popc(e.x & (bit - 1u)) : -2 - d;
    }
    t2r[t] = r;
  }
}

// ------------------------------------------------- planned (resident) kernel
//
// tli_planned_kernel: persistent CTAs (one per SM at the c4 vocabulary
// sizes) walking rows blockIdx.x, blockIdx.x + gridDim.x, ...; the bitmap
// is copied into shared memory once.  Per row, when the K intersection
// logits fit in shared memory:
//   pass 1   streams the row through a per-thread cp.async ring, copies
//            every intersection logit to its rank (id order) and keeps the
//            masked online softmax and best element of those logits;
//   pass 2   streams t2r and writes q in target order, each gather a
//            shared-memory read (logit form: warps 1.. only, while thread 0
//            writes the top-1 outputs).
// Otherwise (no q wanted, or more intersection logits than fit) pass 1
// masks with the bitmap and pass 2 gathers from the row in global memory
// (L2), t2d streamed through the ring.  Results are those of tli_constrain_kernel.
// 1024 threads with a 3-deep cp.async ring measured faster at the c4 sizes
// than 512 threads, and than 16-byte loads into registers (2 or 4 in
// flight per thread): the row and the t2r stream stay in flight without
// registers, which the per-element work needs.
constexpr int kResThreads = 1024;
// 16-byte copies in flight per thread (16 KB of shared memory each): 4 measured
// slightly faster than 3 per row (the row stream is bound by bytes in flight),
// and at V_d = 151936 still leaves room for 63952 intersection logits
constexpr int kResRing = 4;
// warps left out of the logit-form pass 2: warp 0 writes the row's top-1
// outputs meanwhile (global loads and stores, about 3 us), so that latency no
// longer holds up the row's end (row span of a c4 launch 54 -> 47 us)
constexpr int kP2Skip = 1;
// 16-byte loads of the rank table in flight per thread in the logit-form
// pass 2 (register loads: the shared-memory port is busy with the gathers)
constexpr int kP2Unroll = 4;

// f(v, i) for the n 16-byte items src[i], each thread taking i = tid + j
// THREADS in increasing j, U loads in flight per thread.
template <int THREADS, int U, class F>
__device__ __forceinline__ void direct_stream(const uint4* __restrict__ src, int n, F&& f, int tid) {
  int i = tid;
  for (; i + (U - 1) * THREADS < n; i += U * THREADS) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = __ldg(src + i + u * THREADS);
#pragma unroll
    for (int u = 0; u < U; ++u) f(v[u], i + u * THREADS);
  }
  for (; i < n; i += THREADS) f(__ldg(src + i), i);
}

// Bits of ids [first, first + N) from the bitmap (N <= 8).
template <int N>
__device__ __forceinline__ uint32_t bits_at(const uint2* mw, int first) {
  const int w = first >> 5, sh = first & 31;
  uint32_t b = mw[w].x >> sh;
  if (sh > 32 - N) b |= mw[w + 1].x << (32 - sh);  // the run crosses into word w + 1
  return b & ((1u << N) - 1u);
}
// Intersection ids before id (its rank when it is one).
__device__ __forceinline__ int rank_before(const uint2* mw, int id) {
  const uint2 e = mw[id >> 5];
  return static_cast<int>(e.y) + __popc(e.x & ((1u << (id & 31)) - 1u));
}
// Pass 1 (compacting) with the row's statistics: every intersection logit
// of the row to cpt[rank] (id order) and, over the same logits, the masked
// online softmax and best element (value desc, id asc) of the thread's
// elements in increasing index order (NaN as -inf).  The stream is bound by
// the bytes in flight, so the statistics ride along instead of taking a
// pass over the compacted logits of their own (4.8 us per c4 row).
template <int DT>
struct CompactStatWriter {
  const uint2* mw;
  typename Elem<DT>::T* cpt;
  int K;  // entries of cpt (the debug build's bounds)
  float c, m, mc, s0, s1;
  int bi;
  __device__ __forceinline__ void rescale(float nm) {
    if (m == neg_inf()) {
      s0 = s1 = 0.0f;
    } else {
      const float f = fast_exp2((m - nm) * c);
      s0 *= f;
      s1 *= f;
    }
    m = nm;
    mc = nm * c;
  }
  __device__ __forceinline__ void visit1(float x, int64_t idx, bool) {
    const int id = static_cast<int>(idx);
    if (!((mw[id >> 5].x >> (id & 31)) & 1u)) return;
    const int r = rank_before(mw, id);
    if (spec_in(r, K, nullptr)) cpt[r] = Elem<DT>::of_value(x);
    const float xk = order_key(x);
    if (xk > m) {
      rescale(xk);
      bi = id;
    }
    if (m != neg_inf()) s0 += fast_exp2(fmaf(xk, c, -mc));
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int first) {
    constexpr int kv = Logit<DT>::kVec;
    const int w = first >> 5, sh = first & 31;
    const uint2 e = mw[w];
    uint32_t b = e.x >> sh;
    if (sh > 32 - kv) b |= mw[w + 1].x << (32 - sh);  // the vector crosses into word w + 1
    b &= (1u << kv) - 1u;
    if (b == 0u) return;
    int r = static_cast<int>(e.y) + __popc(e.x & ((1u << sh) - 1u));
#pragma unroll
    for (int j = 0; j < kv; ++j)
      if (((b >> j) & 1u) && spec_in(r, K, nullptr)) cpt[r++] = Elem<DT>::at(raw, j);
    float x[kv];
    unpack<DT>(raw, x);
    float vmax = neg_inf();
#pragma unroll
    for (int j = 0; j < kv; ++j) {
      x[j] = ((b >> j) & 1u) ? order_key(x[j]) : neg_inf();
      vmax = fmaxf(vmax, x[j]);
    }
    if (vmax > m) {
      int j0 = 0;
#pragma unroll
      for (int j = kv - 1; j >= 0; --j)
        if (x[j] == vmax) j0 = j;
      rescale(vmax);
      bi = first + j0;
    }
    if (m != neg_inf()) {
      const float2 a = exp2_sum_pairs<kv>(make_float2(s0, s1), x, c, mc);
      s0 = a.x;
      s1 = a.y;
    }
  }
};

// Masked pass 1 (no room for the intersection logits): the masked online
// softmax and best element with the mask from the bitmap.
template <int DT>
struct BitmapMaskedVisitor {
  const uint2* mw;
  float c, m, mc, s0, s1;
  int bi;
  __device__ __forceinline__ void rescale(float nm) {
    if (m == neg_inf()) {
      s0 = s1 = 0.0f;
    } else {
      const float f = fast_exp2((m - nm) * c);
      s0 *= f;
      s1 *= f;
    }
    m = nm;
    mc = nm * c;
  }
  __device__ __forceinline__ void visit1(float x, int64_t idx, bool) {
    const int id = static_cast<int>(idx);
    if (!((mw[id >> 5].x >> (id & 31)) & 1u)) return;
    const float xk = order_key(x);
    if (xk > m) {
      rescale(xk);
      bi = id;
    }
    if (m != neg_inf()) s0 += fast_exp2(fmaf(xk, c, -mc));
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int first) {
    constexpr int kv = Logit<DT>::kVec;
    const uint32_t b = bits_at<kv>(mw, first);
    float x[kv];
    unpack<DT>(raw, x);
    float vmax = neg_inf();
#pragma unroll
    for (int j = 0; j < kv; ++j) {
      x[j] = ((b >> j) & 1u) ? order_key(x[j]) : neg_inf();
      vmax = fmaxf(vmax, x[j]);
    }
    if (vmax > m) {
      int j0 = 0;
#pragma unroll
      for (int j = kv - 1; j >= 0; --j)
        if (x[j] == vmax) j0 = j;
      rescale(vmax);
      bi = first + j0;
    }
    if (m != neg_inf()) {
      const float2 a = exp2_sum_pairs<kv>(make_float2(s0, s1), x, c, mc);
      s0 = a.x;
      s1 = a.y;
    }
  }
};

// Visits the elements of a row (leading scalars, 16-byte vectors through
// the ring, trailing scalars): f.visit1(x, idx, true), f.visit_vec(raw,
// first); each thread in increasing index order.
template <int DT, class F>
__device__ __forceinline__ void ring_row(const void* row, int64_t Vd, uint4* ring, F& f) {
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kv = Logit<DT>::kVec;
  const int tid = threadIdx.x;
  const RowSpan sp = row_span<DT>(row, Vd);
  const int head = static_cast<int>(sp.head), nvec = static_cast<int>(sp.nvec);
  if (tid < head) f.visit1(Logit<DT>::load1(row, tid), tid, true);
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  ring_stream<kResThreads, kResRing>(vp, nvec, ring, [&](const uint4& v, int i) { f.visit_vec(v, head + i * kv); });
  const int64_t t = head + static_cast<int64_t>(nvec) * kv + tid;
  if (t < Vd) f.visit1(Logit<DT>::load1(row, t), t, true);
}

template <int DT>
__global__ void __launch_bounds__(kResThreads, 1)
    tli_planned_kernel(int64_t R, int64_t Vd, int64_t Vt, const void* __restrict__ draft,
                       const int32_t* __restrict__ d2t, const int32_t* __restrict__ t2d,
                       const void* __restrict__ plan, float c, int cap, int32_t* __restrict__ top1_draft,
                       int32_t* __restrict__ top1_target, float* __restrict__ top1_p, QOut qo,
                       int32_t* __restrict__ stats, ExpandArgs ex) {
  pdl_enter();
  using E = typename Elem<DT>::T;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kWarps = kResThreads / 32;
  extern __shared__ __align__(16) unsigned char res_dsm[];
  __shared__ float wm[kWarps], ws[kWarps], wv[kWarps];
  __shared__ int wi[kWarps];
  __shared__ float s_m, s_s, s_bv;
  __shared__ int s_bi;
  const int Wp = static_cast<int>(plan_words(Vd));
  const PlanView pv = plan_view(const_cast<void*>(plan), Vd);
  uint4* ring = reinterpret_cast<uint4*>(res_dsm);  // kResRing slots per thread
  uint2* mw = reinterpret_cast<uint2*>(ring + kResRing * kResThreads);
  E* cpt_buf = reinterpret_cast<E*>(mw + Wp);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < Wp / 2; i += kResThreads)
    reinterpret_cast<uint4*>(mw)[i] = __ldg(reinterpret_cast<const uint4*>(pv.mw) + i);
  const int K = __ldg(pv.K);
  __syncthreads();
  if (!spec_smem_ok(reinterpret_cast<unsigned char*>(cpt_buf) - res_dsm, stats) || !spec_in(K, Vd + 1, stats)) return;
  E* const cpt = ((qo.q != nullptr || qo.ql != nullptr) && K <= cap &&
                  spec_smem_ok(reinterpret_cast<unsigned char*>(cpt_buf + K) - res_dsm, stats))
                     ? cpt_buf
                     : nullptr;
  const int32_t* t2r = pv.t2r;

  // block merge of the per-thread partials into s_m, s_s, s_bv, s_bi
  auto merge = [&](float m, float s, float bv, int bi) {
    warp_best(bv, bi);
    warp_merge_ms(m, s, c);
    if (lane == 0) {
      wv[warp] = bv;
      wi[warp] = bi;
      wm[warp] = m;
      ws[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
      bv = lane < kWarps ? wv[lane] : neg_inf();
      bi = lane < kWarps ? wi[lane] : INT_MAX;
      warp_best(bv, bi);
      m = lane < kWarps ? wm[lane] : neg_inf();
      s = lane < kWarps ? ws[lane] : 0.0f;
      warp_merge_ms(m, s, c);
      if (lane == 0) {
        s_m = m;
        s_s = s;
        s_bv = bv;
        s_bi = bi;
      }
    }
    __syncthreads();
  };

  for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
    const void* row = static_cast<const char*>(draft) + r * Vd * esz;
    if (cpt != nullptr) {
      CompactStatWriter<DT> cw{mw, cpt, K, c, neg_inf(), 0.0f, 0.0f, 0.0f, INT_MAX};
      ring_row<DT>(row, Vd, ring, cw);
      // (the merge's barriers also complete the compacted logits)
      merge(cw.m, cw.s0 + cw.s1, cw.m, cw.bi);
    } else {
      BitmapMaskedVisitor<DT> st{mw, c, neg_inf(), 0.0f, 0.0f, 0.0f, INT_MAX};
      ring_row<DT>(row, Vd, ring, st);
      merge(st.m, st.s0 + st.s1, st.m, st.bi);
    }
    // the row's statistics for every thread; s_bi is the best draft id
    const bool ok = s_bi != INT_MAX && isfinite(s_bv);
    const float mc = s_m * c, invz = 1.0f / s_s;
    if (tid == 0) {
      // the top-1 outputs (thread 0 alone; the other warps go on) and the
      // step's pool expansion for this row's request (a chain: one row each)
      const int best = ok ? s_bi : -1;
      const int32_t tgt = ok && spec_in(best, Vd, stats) ? __ldg(d2t + best) : -1;
      const float pr = ok ? fminf(fast_exp2(fmaf(s_bv, c, -mc)) * invz, 1.0f) : 0.0f;
      top1_draft[r] = best;
      top1_target[r] = tgt;
      top1_p[r] = pr;
      if (!ok) bump(stats, SPEC_STAT_EMPTY_INTERSECTION);
      if (qo.qs != nullptr) {
        qo.qs[2 * r] = ok ? s_m : neg_inf();
        qo.qs[2 * r + 1] = s_s;
      }
      if (ex.k != 0) expand_chain(ex, static_cast<int>(r), pr, tgt);
    }
    if (qo.q != nullptr) {
      float* out = qo.q + r * Vt;
      const bool vec_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
      if (!ok) {
        // no finite intersection logit: a zero row
        for (int64_t t = tid; t < Vt; t += kResThreads) out[t] = 0.0f;
      } else if (cpt != nullptr) {
        // pass 2: target order, the partners' ranks streamed through the
        // ring; a ranked partner's logit is at most the row max, so its
        // probability needs no clamp (a partner outside the intersection,
        // read from the row, does)
        auto q_far = [&](int32_t k) -> float {
          if (!spec_in(-2 - k, Vd, stats)) return 0.0f;
          return fminf(fast_exp2(fmaf(order_key(Logit<DT>::load1(row, -2 - k)), c, -mc)) * invz, 1.0f);
        };
        auto q_pair = [&](int32_t k0, int32_t k1) -> float2 {
          const float2 x = make_float2(order_key(Elem<DT>::value(cpt[k0 > 0 && spec_in(k0, K, stats) ? k0 : 0])),
                                       order_key(Elem<DT>::value(cpt[k1 > 0 && spec_in(k1, K, stats) ? k1 : 0])));
          const float2 y = fma2(x, splat(c), splat(-mc));
          const float2 p = fma2(exp2_2(y), splat(invz), splat(0.0f));
          return make_float2(k0 >= 0 ? p.x : 0.0f, k1 >= 0 ? p.y : 0.0f);
        };
        const int nv = vec_out ? static_cast<int>(Vt / 4) : 0;
        ring_stream<kResThreads, kResRing>(reinterpret_cast<const uint4*>(t2r), nv, ring,
                                           [&](const uint4& kk, int i) {
                                             const int32_t k0 = static_cast<int32_t>(kk.x);
                                             const int32_t k1 = static_cast<int32_t>(kk.y);
                                             const int32_t k2 = static_cast<int32_t>(kk.z);
                                             const int32_t k3 = static_cast<int32_t>(kk.w);
                                             const float2 a = q_pair(k0, k1), b = q_pair(k2, k3);
                                             float4 o = make_float4(a.x, a.y, b.x, b.y);
                                             if (min(min(k0, k1), min(k2, k3)) < -1) {
                                               if (k0 < -1) o.x = q_far(k0);
                                               if (k1 < -1) o.y = q_far(k1);
                                               if (k2 < -1) o.z = q_far(k2);
                                               if (k3 < -1) o.w = q_far(k3);
                                             }
                                             st_stream(out + 4 * i, o);
                                           });
        for (int64_t t = static_cast<int64_t>(nv) * 4 + tid; t < Vt; t += kResThreads) {
          const int32_t k = __ldg(t2r + t);
          out[t] = k >= 0 ? fast_exp2(fmaf(order_key(Elem<DT>::value(cpt[spec_in(k, K, stats) ? k : 0])), c, -mc)) * invz
                          : (k == -1 ? 0.0f : q_far(k));
        }
      } else {
        // pass 2: target order, gathers from the row in global memory
        auto q_at = [&](int32_t d) -> float {
          if (d < 0 || d >= Vd) return 0.0f;
          return fminf(fast_exp2(fmaf(order_key(Logit<DT>::load1(row, d)), c, -mc)) * invz, 1.0f);
        };
        const bool vec = vec_out && (reinterpret_cast<uintptr_t>(t2d) & 15) == 0;
        const int nv = vec ? static_cast<int>(Vt / 4) : 0;
        ring_stream<kResThreads, kResRing>(reinterpret_cast<const uint4*>(t2d), nv, ring,
                                           [&](const uint4& d, int i) {
                                             st_stream(out + 4 * i,
                                                       make_float4(q_at(static_cast<int32_t>(d.x)),
                                                                   q_at(static_cast<int32_t>(d.y)),
                                                                   q_at(static_cast<int32_t>(d.z)),
                                                                   q_at(static_cast<int32_t>(d.w))));
                                           });
        for (int64_t t = static_cast<int64_t>(nv) * 4 + tid; t < Vt; t += kResThreads) out[t] = q_at(__ldg(t2d + t));
      }
    }
    if (qo.ql != nullptr) {
      // logit form: the partners' logits in target order (raw bits, -inf
      // without a partner), from the shared intersection logits by rank
      // or gathered from the row
      E* lo = static_cast<E*>(qo.ql) + r * Vt;
      const E ninf = Elem<DT>::of_value(neg_inf());
      const bool vl = (reinterpret_cast<uintptr_t>(lo) & (4 * esz - 1)) == 0;
      if (cpt != nullptr) {
        // branch-free for ranked partners and none (-1); a partner outside
        // the intersection (-2 - d, rare) is read from the row
        auto near = [&](int32_t k) -> E {
          const E v = cpt[k > 0 && spec_in(k, K, stats) ? k : 0];
          return k >= 0 ? v : ninf;
        };
        auto far = [&](int32_t k) -> E {
          return spec_in(-2 - k, Vd, stats) ? Elem<DT>::of_value(Logit<DT>::load1(row, -2 - k)) : ninf;
        };
        auto l_of = [&](int32_t k) -> E { return k < -1 ? far(k) : near(k); };
        const int nl = vl ? static_cast<int>(Vt / 4) : 0;
        constexpr int kP2T = kResThreads - 32 * kP2Skip;
        const int p2 = tid - 32 * kP2Skip;
        if (p2 >= 0) {
        direct_stream<kP2T, kP2Unroll>(reinterpret_cast<const uint4*>(t2r), nl, [&](const uint4& kk, int i) {
          const int32_t k0 = static_cast<int32_t>(kk.x), k1 = static_cast<int32_t>(kk.y);
          const int32_t k2 = static_cast<int32_t>(kk.z), k3 = static_cast<int32_t>(kk.w);
          E e0 = near(k0), e1 = near(k1), e2 = near(k2), e3 = near(k3);
          if (min(min(k0, k1), min(k2, k3)) < -1) {
            if (k0 < -1) e0 = far(k0);
            if (k1 < -1) e1 = far(k1);
            if (k2 < -1) e2 = far(k2);
            if (k3 < -1) e3 = far(k3);
          }
          st_stream4(lo + 4 * i, e0, e1, e2, e3);
        }, p2);
        for (int64_t t = static_cast<int64_t>(nl) * 4 + p2; t < Vt; t += kP2T) lo[t] = l_of(__ldg(t2r + t));
        }
      } else {
        auto l_of = [&](int32_t d) -> E {
          return (d >= 0 && d < Vd) ? Elem<DT>::of_value(Logit<DT>::load1(row, d)) : ninf;
        };
        const int nl = (vl && (reinterpret_cast<uintptr_t>(t2d) & 15) == 0) ? static_cast<int>(Vt / 4) : 0;
        ring_stream<kResThreads, kResRing>(reinterpret_cast<const uint4*>(t2d), nl, ring,
                                           [&](const uint4& d, int i) {
                                             st_stream4(lo + 4 * i, l_of(static_cast<int32_t>(d.x)),
                                                        l_of(static_cast<int32_t>(d.y)),
                                                        l_of(static_cast<int32_t>(d.z)),
                                                        l_of(static_cast<int32_t>(d.w)));
                                           });
        for (int64_t t = static_cast<int64_t>(nl) * 4 + tid; t < Vt; t += kResThreads) lo[t] = l_of(__ldg(t2d + t));
      }
    }
    __syncthreads();  // before the next row overwrites the shared logits and statistics
  }
}

__global__ void map_ids_kernel(const int32_t* __restrict__ in, int32_t* __restrict__ out, int64_t n,
                               const int32_t* __restrict__ table, int64_t table_len, int32_t fallback) {
  pdl_enter();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t x = __ldg(in + i);
    int32_t y = fallback;
    if (x >= 0 && x < table_len) {
      const int32_t t = __ldg(table + x);
      if (t >= 0) y = t;
    }
    out[i] = y;
  }
}

// Launches tli_planned_kernel when the copy ring and the bitmap (8 bytes per
// 32 draft ids) fit in the CTA's opt-in shared memory; the rest of it holds
// up to `cap` intersection logits.  Returns false (nothing launched)
// otherwise.
template <int DT>
bool launch_planned(int64_t R, int64_t Vd, int64_t Vt, const void* draft, const int32_t* d2t, const int32_t* t2d,
                    const void* plan, float c, int32_t* top1_draft, int32_t* top1_target, float* top1_p, QOut qo,
                    int32_t* stats, const ExpandArgs& ex, cudaStream_t s) {
  constexpr int64_t esz = DT == SPEC_BF16 ? 2 : 4;
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int64_t fixed = static_cast<int64_t>(sizeof(uint4)) * kResRing * kResThreads + 8 * plan_words(Vd);
  const int64_t budget = static_cast<int64_t>(optin) - 1024;  // the kernel's static shared memory is below 1 KB
  if (fixed + 16 > budget) return false;
  int64_t cap = (budget - fixed) / esz;
  if (cap > Vd) cap = Vd;
  cap &= ~int64_t(7);
  if (cap < 8) return false;
  const size_t smem = static_cast<size_t>((fixed + cap * esz + 15) & ~int64_t(15));
  if (smem > 48 * 1024 && cudaFuncSetAttribute(tli_planned_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tli_planned_kernel<DT>, kResThreads, smem) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return false;
  }
  const int64_t slots = static_cast<int64_t>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(R < slots ? R : slots);
  launch_k(tli_planned_kernel<DT>, grid, kResThreads, smem, s, R, Vd, Vt, draft, d2t, t2d, plan, c,
           static_cast<int>(cap), top1_draft, top1_target, top1_p, qo, stats, ex);
  return true;
}

}  // namespace
}  // namespace specdec

using namespace specdec;

namespace {
// The per-row kernel (no plan).
int constrain_rows(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype, const int32_t* d2t,
                   const int32_t* t2d_or_null, float T, int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                   QOut qo, int32_t* stats_or_null, spec_stream_t stream) {
  if (R < 0 || V_d < 1 || V_t < 1 || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (V_d > SPEC_MAX_VOCAB || V_t > SPEC_MAX_VOCAB || R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  if (R == 0) return SPEC_OK;
  if (!draft_logits || !d2t || !top1_draft || !top1_target || !top1_p) return SPEC_ERR_INVALID_ARG;
  if ((qo.q || qo.ql) && !t2d_or_null) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  const unsigned grid = static_cast<unsigned>(R);
  if (dtype == SPEC_BF16)
    launch_k(tli_constrain_kernel<SPEC_BF16>, grid, kTliThreads, 0, s, V_d, V_t, draft_logits, d2t, t2d_or_null, c,
             top1_draft, top1_target, top1_p, qo, stats_or_null);
  else
    launch_k(tli_constrain_kernel<SPEC_F32>, grid, kTliThreads, 0, s, V_d, V_t, draft_logits, d2t, t2d_or_null, c,
             top1_draft, top1_target, top1_p, qo, stats_or_null);
  return launch_status();
}
}  // namespace

extern "C" int tli_constrain_map(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                                 const int32_t* d2t, const int32_t* t2d_or_null, float T, int32_t* top1_draft,
                                 int32_t* top1_target, float* top1_p, float* q_target_or_null,
                                 int32_t* stats_or_null, spec_stream_t stream) {
  return constrain_rows(R, V_d, V_t, draft_logits, dtype, d2t, t2d_or_null, T, top1_draft, top1_target, top1_p,
                        QOut{q_target_or_null, nullptr, nullptr}, stats_or_null, stream);
}

extern "C" int64_t tli_plan_bytes(int64_t V_d, int64_t V_t) {
  if (V_d < 1 || V_t < 1 || V_d > SPEC_MAX_VOCAB || V_t > SPEC_MAX_VOCAB) return -1;
  return plan_bytes(V_d, V_t);
}

extern "C" int tli_plan_build(int64_t V_d, int64_t V_t, const int32_t* d2t, const int32_t* t2d, void* plan,
                              spec_stream_t stream) {
  if (V_d < 1 || V_t < 1) return SPEC_ERR_INVALID_ARG;
  if (V_d > SPEC_MAX_VOCAB || V_t > SPEC_MAX_VOCAB) return SPEC_ERR_UNSUPPORTED;
  if (!d2t || !t2d || !plan || (reinterpret_cast<uintptr_t>(plan) & 15) != 0) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const PlanView pv = plan_view(plan, V_d);
  const int64_t Wp = plan_words(V_d);
  const int64_t bits_blocks = (Wp + 7) / 8;  // 8 warps, one word each per round
  launch_k(plan_bits_kernel, static_cast<unsigned>(bits_blocks < 1024 ? bits_blocks : 1024), 256, 0, s, d2t, V_d,
           pv.mw);
  launch_k(plan_scan_kernel, 1, kPlanScanThreads, 0, s, V_d, pv.mw, pv.K);
  const int64_t t_blocks = ((V_t + 3) / 4 * 4 + 255) / 256;
  launch_k(plan_t2r_kernel, static_cast<unsigned>(t_blocks < 4096 ? t_blocks : 4096), 256, 0, s, t2d, V_d, V_t,
           static_cast<const uint2*>(pv.mw), pv.t2r);
  return launch_status();
}

namespace {
int constrain_planned_impl(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                           const int32_t* d2t, const int32_t* t2d_or_null, const void* plan, float T,
                           int32_t* top1_draft, int32_t* top1_target, float* top1_p, QOut qo,
                           int32_t* stats_or_null, const spec_expand_t* expand, spec_stream_t stream) {
  if (R < 0 || V_d < 1 || V_t < 1 || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (V_d > SPEC_MAX_VOCAB || V_t > SPEC_MAX_VOCAB || R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  ExpandArgs ex = no_expand();
  if (expand != nullptr) {
    const int e = expand_args(expand, 1, R, ex);
    if (e != SPEC_OK) return e;
  }
  if (R == 0) return SPEC_OK;
  if (!draft_logits || !d2t || !plan || !top1_draft || !top1_target || !top1_p) return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(plan) & 15) != 0) return SPEC_ERR_INVALID_ARG;
  if ((qo.q || qo.ql) && !t2d_or_null) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  if (dtype == SPEC_BF16 ? launch_planned<SPEC_BF16>(R, V_d, V_t, draft_logits, d2t, t2d_or_null, plan, c,
                                                     top1_draft, top1_target, top1_p, qo, stats_or_null, ex, s)
                         : launch_planned<SPEC_F32>(R, V_d, V_t, draft_logits, d2t, t2d_or_null, plan, c, top1_draft,
                                                    top1_target, top1_p, qo, stats_or_null, ex, s))
    return launch_status();
  // the bitmap does not fit in shared memory: the per-row kernel, and the
  // expansion as its own launch
  const int e = constrain_rows(R, V_d, V_t, draft_logits, dtype, d2t, t2d_or_null, T, top1_draft, top1_target,
                               top1_p, qo, stats_or_null, stream);
  if (e != SPEC_OK || expand == nullptr) return e;
  return spec_tree_expand(expand->step, expand->num_steps, expand->B, 1, top1_p, top1_target, expand->pool_score,
                          expand->pool_token, expand->pool_parent, expand->pool_qrow, expand->frontier_score,
                          expand->frontier_id, stream);
}
}  // namespace

extern "C" int tli_constrain_map_planned(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                                         const int32_t* d2t, const int32_t* t2d_or_null, const void* plan, float T,
                                         int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                                         float* q_target_or_null, int32_t* stats_or_null, spec_stream_t stream) {
  return constrain_planned_impl(R, V_d, V_t, draft_logits, dtype, d2t, t2d_or_null, plan, T, top1_draft, top1_target,
                                top1_p, QOut{q_target_or_null, nullptr, nullptr}, stats_or_null, nullptr, stream);
}

extern "C" int tli_constrain_map_planned_expand(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits,
                                                int dtype, const int32_t* d2t, const int32_t* t2d_or_null,
                                                const void* plan, float T, int32_t* top1_draft,
                                                int32_t* top1_target, float* top1_p, float* q_target_or_null,
                                                int32_t* stats_or_null, const spec_expand_t* expand,
                                                spec_stream_t stream) {
  if (expand == nullptr) return SPEC_ERR_INVALID_ARG;
  return constrain_planned_impl(R, V_d, V_t, draft_logits, dtype, d2t, t2d_or_null, plan, T, top1_draft, top1_target,
                                top1_p, QOut{q_target_or_null, nullptr, nullptr}, stats_or_null, expand, stream);
}

extern "C" int tli_constrain_map_qlogits(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                                         const int32_t* d2t, const int32_t* t2d, const void* plan_or_null, float T,
                                         int32_t* top1_draft, int32_t* top1_target, float* top1_p,
                                         void* q_logits_target, float* q_stats, int32_t* stats_or_null,
                                         const spec_expand_t* expand_or_null, spec_stream_t stream) {
  if (R > 0) {
    const uintptr_t esz = dtype == SPEC_BF16 ? 2 : 4;
    if (!t2d || !q_logits_target || !q_stats) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_logits_target) & (esz - 1)) != 0 ||
        (reinterpret_cast<uintptr_t>(q_stats) & 3) != 0)
      return SPEC_ERR_INVALID_ARG;
  }
  const QOut qo{nullptr, q_logits_target, q_stats};
  if (plan_or_null != nullptr)
    return constrain_planned_impl(R, V_d, V_t, draft_logits, dtype, d2t, t2d, plan_or_null, T, top1_draft,
                                  top1_target, top1_p, qo, stats_or_null, expand_or_null, stream);
  if (expand_or_null != nullptr) {
    ExpandArgs ex = no_expand();
    const int e = expand_args(expand_or_null, 1, R, ex);
    if (e != SPEC_OK) return e;
  }
  const int e = constrain_rows(R, V_d, V_t, draft_logits, dtype, d2t, t2d, T, top1_draft, top1_target, top1_p, qo,
                               stats_or_null, stream);
  if (e != SPEC_OK || expand_or_null == nullptr || R == 0) return e;
  return spec_tree_expand(expand_or_null->step, expand_or_null->num_steps, expand_or_null->B, 1, top1_p, top1_target,
                          expand_or_null->pool_score, expand_or_null->pool_token, expand_or_null->pool_parent,
                          expand_or_null->pool_qrow, expand_or_null->frontier_score, expand_or_null->frontier_id,
                          stream);
}

extern "C" int tli_map_ids(const int32_t* in, int32_t* out, int64_t n, const int32_t* table, int64_t table_len,
                           int32_t fallback_id, spec_stream_t stream) {
  if (n < 0 || table_len < 0) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  if (!in || !out || (!table && table_len > 0)) return SPEC_ERR_INVALID_ARG;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  const unsigned grid = static_cast<unsigned>(blocks < 4096 ? blocks : 4096);
  launch_k(map_ids_kernel, grid, threads, 0, reinterpret_cast<cudaStream_t>(stream), in, out, n, table, table_len,
           fallback_id);
  return launch_status();
}

extern "C" int tli_check_config(int topk, int num_steps, int num_draft_tokens) {
  return (topk == 1 && num_steps >= 1 && num_draft_tokens == num_steps + 1) ? SPEC_OK : SPEC_ERR_INVALID_ARG;
}
