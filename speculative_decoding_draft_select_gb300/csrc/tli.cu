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
// tli_constrain_kernel: one CTA per draft row.  Pass 1 streams the row with
// 16-byte loads together with the matching 16-byte loads of d2t (the table
// is shared by every row and stays in L2), masks ids outside the
// intersection (d2t[v] < 0) to -inf and keeps the masked top-1 and
// online-softmax partials.  Pass 2 (optional) writes q in target order:
// q_t[t] = p(t2d[t]) or 0, with coalesced 16-byte stores and gathers from
// the draft row (L2-resident), 8 in flight per thread.
#include <climits>

#include "common.cuh"

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
__global__ void __launch_bounds__(kTliThreads)
    tli_constrain_kernel(int64_t Vd, int64_t Vt, const void* __restrict__ draft, const int32_t* __restrict__ d2t,
                         const int32_t* __restrict__ t2d, float c, int32_t* __restrict__ top1_draft,
                         int32_t* __restrict__ top1_target, float* __restrict__ top1_p, float* __restrict__ q,
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
    }
  }
  __syncthreads();
  if (q == nullptr) return;
  float* out = q + r * Vt;
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

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" int tli_constrain_map(int64_t R, int64_t V_d, int64_t V_t, const void* draft_logits, int dtype,
                                 const int32_t* d2t, const int32_t* t2d_or_null, float T, int32_t* top1_draft,
                                 int32_t* top1_target, float* top1_p, float* q_target_or_null,
                                 int32_t* stats_or_null, spec_stream_t stream) {
  if (R < 0 || V_d < 1 || V_t < 1 || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (V_d > SPEC_MAX_VOCAB || V_t > SPEC_MAX_VOCAB || R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  if (R == 0) return SPEC_OK;
  if (!draft_logits || !d2t || !top1_draft || !top1_target || !top1_p) return SPEC_ERR_INVALID_ARG;
  if (q_target_or_null && !t2d_or_null) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  const unsigned grid = static_cast<unsigned>(R);
  if (dtype == SPEC_BF16)
    launch_k(tli_constrain_kernel<SPEC_BF16>, grid, kTliThreads, 0, s, V_d, V_t, draft_logits, d2t, t2d_or_null, c,
             top1_draft, top1_target, top1_p, q_target_or_null, stats_or_null);
  else
    launch_k(tli_constrain_kernel<SPEC_F32>, grid, kTliThreads, 0, s, V_d, V_t, draft_logits, d2t, t2d_or_null, c,
             top1_draft, top1_target, top1_p, q_target_or_null, stats_or_null);
  return launch_status();
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
