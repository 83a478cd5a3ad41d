// Draft side: per-step softmax + top-k, and draft sampling.
//
// "[SGLang] Multi-Layer EAGLE" (secrett2633 blog), section 3: every draft
// step computes probs = softmax(logits) and then top-k of them;
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)", 5.1: the
// stored draft distribution is the processed one (temperature applied), and
// drafts are drawn from it.
//
// One CTA streams one logit row with 16-byte loads (UNROLL in flight per
// thread).  A single pass gives the online softmax partials (max, sum of
// 2^((x - max) * log2e / T)) and each thread's top-K list; block merges are
// fixed-order.  The optional probability row is written by a second sweep
// of the row (served from L2) with streaming stores.
#include <climits>

#include "cdf.cuh"
#include "common.cuh"

namespace specdec {
namespace {

constexpr int kDraftThreads = 512;

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
  // Insert (x, idx) if it beats the K-th entry; keeps (value desc, index asc).
  __device__ __forceinline__ void push(float x, int idx) {
    if (!before(x, idx, v[K - 1], i[K - 1])) return;
    v[K - 1] = x;
    i[K - 1] = idx;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
      if (before(v[j], i[j], v[j - 1], i[j - 1])) {
        float tv = v[j];
        v[j] = v[j - 1];
        v[j - 1] = tv;
        int ti = i[j];
        i[j] = i[j - 1];
        i[j - 1] = ti;
      }
    }
  }
  // Remove the head (the caller has consumed it).
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

// Per-thread state of the softmax + top-k sweep.
template <int K, bool WANT_TOPK>
struct SoftmaxTopKVisitor {
  float c;  // log2(e) / T
  float m;  // running max (ordering keys)
  float s;  // sum of 2^((x - m) c)
  TopK<K> top;

  template <int N>
  __device__ __forceinline__ void visit(const float* xin, int64_t first) {
    float x[N];
    float vmax = neg_inf();
#pragma unroll
    for (int j = 0; j < N; ++j) {
      x[j] = order_key(xin[j]);
      vmax = fmaxf(vmax, x[j]);
    }
    if (vmax > m) {
      s = (m == neg_inf()) ? 0.0f : s * fast_exp2((m - vmax) * c);
      m = vmax;
    }
    if (m != neg_inf()) {
      const float mc = m * c;
#pragma unroll
      for (int j = 0; j < N; ++j) s += fast_exp2(fmaf(x[j], c, -mc));
    }
    if (WANT_TOPK && vmax >= top.v[K - 1]) {
#pragma unroll
      for (int j = 0; j < N; ++j) top.push(x[j], static_cast<int>(first + j));
    }
  }
};

// Block merge of per-thread top-K lists: each warp pops its best K into
// shared memory, then warp 0 merges the warps' lists the same way.
// Result in out_v / out_i [K] (shared).  All threads call it.
template <int K>
__device__ void block_topk(TopK<K>& t, float* wv, int* wi, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int r = 0; r < K; ++r) {
    float bv = t.v[0];
    int bi = t.i[0];
    warp_best(bv, bi);
    if (t.v[0] == bv && t.i[0] == bi && bi != INT_MAX) t.pop();
    if (lane == 0) {
      wv[warp * K + r] = bv;
      wi[warp * K + r] = bi;
    }
  }
  __syncthreads();
  if (warp == 0) {
    TopK<K> u;
    u.init();
    for (int e = lane; e < nw * K; e += 32) u.push(wv[e], wi[e]);
    for (int r = 0; r < K; ++r) {
      float bv = u.v[0];
      int bi = u.i[0];
      warp_best(bv, bi);
      if (u.v[0] == bv && u.i[0] == bi && bi != INT_MAX) u.pop();
      if (lane == 0) {
        out_v[r] = bv;
        out_i[r] = bi;
      }
    }
  }
  __syncthreads();
}

// Block merge of (m, s) partials; every thread receives the row's (m, s).
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

template <int DT, int K>
__global__ void __launch_bounds__(kDraftThreads)
    softmax_topk_kernel(const void* __restrict__ logits, int64_t V, float c, int k,
                        float* __restrict__ topk_p, int32_t* __restrict__ topk_idx,
                        float* __restrict__ probs, int32_t* __restrict__ stats) {
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  __shared__ float wv[(kDraftThreads / 32) * K];
  __shared__ int wi[(kDraftThreads / 32) * K];
  __shared__ float fv[K];
  __shared__ int fi[K];
  __shared__ float sm[33], ss[33];

  const int64_t r = blockIdx.x;
  const void* row = static_cast<const char*>(logits) + r * V * esz;

  SoftmaxTopKVisitor<K, true> st;
  st.c = c;
  st.m = neg_inf();
  st.s = 0.0f;
  st.top.init();
  for_row<DT, 4>(row, V, st);

  float m = st.m, s = st.s;
  block_ms(m, s, c, sm, ss);
  block_topk<K>(st.top, wv, wi, fv, fi);

  const bool finite = isfinite(m);
  const float mc = m * c;
  const float invz = 1.0f / s;
  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    topk_idx[r * k + j] = fi[j];
    topk_p[r * k + j] = finite ? fminf(fast_exp2(fmaf(fv[j], c, -mc)) * invz, 1.0f) : 0.0f;
  }
  if (threadIdx.x == 0 && !finite) bump(stats, SPEC_STAT_NONFINITE_ROW);
  if (probs != nullptr) {
    float* out = probs + r * V;
    if (finite) {
      const RowSpan sp = row_span<DT>(row, V);
      ProbWriter<DT> w{c, mc, invz, out,
                       (reinterpret_cast<uintptr_t>(out + sp.head) & 15) == 0};
      for_row<DT, 2>(row, V, w);
    } else {
      ZeroWriter z{out};
      for_row<DT, 2>(row, V, z);
    }
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
                  float* __restrict__ out_prob, int32_t* __restrict__ stats) {
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  extern __shared__ float dyn[];
  __shared__ float scan_sh[33];
  __shared__ float sm[33], ss[33];
  const int64_t ntiles = (V + kSampleThreads * 8 - 1) / (kSampleThreads * 8);
  float* tile_sum = dyn;
  float* red = dyn + ntiles;
  const int64_t r = blockIdx.x;
  float* op = out_prob ? out_prob + r : nullptr;
  if (FROM_PROBS) {
    ProbWeights w{probs + r * V, V};
    sample_row(w, V, __ldg(u + r), red, tile_sum, scan_sh, stats, out_token + r, op);
    return;
  }
  const void* row = static_cast<const char*>(logits) + r * V * esz;
  SoftmaxTopKVisitor<1, false> st;
  st.c = c;
  st.m = neg_inf();
  st.s = 0.0f;
  st.top.init();
  for_row<DT, 4>(row, V, st);
  float m = st.m, s = st.s;
  block_ms(m, s, c, sm, ss);
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

template <int DT, int K>
int launch_softmax_topk(const void* logits, int64_t R, int64_t V, float c, int k, float* topk_p,
                        int32_t* topk_idx, float* probs, int32_t* stats, cudaStream_t s) {
  softmax_topk_kernel<DT, K><<<static_cast<unsigned>(R), kDraftThreads, 0, s>>>(
      logits, V, c, k, topk_p, topk_idx, probs, stats);
  return launch_status();
}

template <int DT>
int dispatch_softmax_topk(const void* logits, int64_t R, int64_t V, float c, int k, float* topk_p,
                          int32_t* topk_idx, float* probs, int32_t* stats, cudaStream_t s) {
  if (k <= 1) return launch_softmax_topk<DT, 1>(logits, R, V, c, k, topk_p, topk_idx, probs, stats, s);
  if (k <= 2) return launch_softmax_topk<DT, 2>(logits, R, V, c, k, topk_p, topk_idx, probs, stats, s);
  if (k <= 4) return launch_softmax_topk<DT, 4>(logits, R, V, c, k, topk_p, topk_idx, probs, stats, s);
  if (k <= 8) return launch_softmax_topk<DT, 8>(logits, R, V, c, k, topk_p, topk_idx, probs, stats, s);
  if (k <= 16) return launch_softmax_topk<DT, 16>(logits, R, V, c, k, topk_p, topk_idx, probs, stats, s);
  return launch_softmax_topk<DT, 32>(logits, R, V, c, k, topk_p, topk_idx, probs, stats, s);
}

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" int spec_softmax_topk(const void* logits, int dtype, int64_t R, int64_t V, float T, int k,
                                 float* topk_p, int32_t* topk_idx, float* probs_or_null,
                                 int32_t* stats_or_null, spec_stream_t stream) {
  if (R < 0 || V < 1 || k < 1 || k > V || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (R > 0 && (logits == nullptr || topk_p == nullptr || topk_idx == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (k > SPEC_MAX_TOPK || V > SPEC_MAX_VOCAB || R > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  if (R == 0) return SPEC_OK;
  const float c = kLog2e / T;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SPEC_BF16
             ? dispatch_softmax_topk<SPEC_BF16>(logits, R, V, c, k, topk_p, topk_idx, probs_or_null, stats_or_null, s)
             : dispatch_softmax_topk<SPEC_F32>(logits, R, V, c, k, topk_p, topk_idx, probs_or_null, stats_or_null, s);
}

extern "C" int spec_sample(const void* logits_or_null, int dtype, const float* probs_or_null, int64_t R,
                           int64_t V, float T, const float* u, int32_t* out_token, float* out_prob_or_null,
                           int32_t* stats_or_null, spec_stream_t stream) {
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
    sample_kernel<SPEC_F32, true><<<grid, kSampleThreads, smem, s>>>(nullptr, probs_or_null, V, c, u, out_token,
                                                                     out_prob_or_null, stats_or_null);
  else if (dtype == SPEC_BF16)
    sample_kernel<SPEC_BF16, false><<<grid, kSampleThreads, smem, s>>>(logits_or_null, nullptr, V, c, u, out_token,
                                                                       out_prob_or_null, stats_or_null);
  else
    sample_kernel<SPEC_F32, false><<<grid, kSampleThreads, smem, s>>>(logits_or_null, nullptr, V, c, u, out_token,
                                                                      out_prob_or_null, stats_or_null);
  return launch_status();
}
