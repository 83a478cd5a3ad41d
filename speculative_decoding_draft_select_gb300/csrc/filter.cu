// Target-side top-k / top-p filtering of logit rows, in place.
//
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)", 5.1: when
// temperature, top-k or top-p are in force, verification uses the processed
// target probabilities.  The rule (the oracle's): order a row's tokens by
// (p desc, index asc), p = softmax(row / T); top_k keeps the first top_k;
// top_p then keeps, in that order, every token whose exclusive prefix of the
// top-k mass is below top_p times that mass (the first token always stays);
// the kept probabilities are renormalised.
//
// Keeping a set S and renormalising is the softmax of the row with every
// logit outside S set to -inf: the maximum is in S (the first token always
// stays) and the normaliser runs over S.  So this kernel writes -inf outside
// S, and the stochastic verify run on the filtered rows reads exactly the
// filtered distribution.  The order by p is the order by logit (exp is
// increasing), so S is a prefix of the order (key desc, index asc) on the
// logits, cut at one element: kept iff key > cut key, or key == cut key and
// index <= cut index.
//
// One CTA per row.  Keys are the logits mapped to unsigned integers in the
// same order (NaN as -inf); bf16 logits need their upper 16 bits only.  The
// cut is found by radix selection, 8 bits per level: a histogram of the next
// byte over the elements matching the bytes chosen so far -- counts for
// top-k (the element of rank top_k - 1), masses for top-p (the first element
// whose inclusive prefix mass reaches top_p times the top-k mass).  Masses
// are 2^((x - max) log2(e) / T) in 2^-40 fixed point, summed with integer
// atomics: exact and independent of the order of the additions, so the cut
// is deterministic; only the ratios matter, so no normaliser is needed.
// Among equal keys the cut goes by index: a pass over the row in index order
// (one contiguous range per thread) finds the n-th element of the cut key.
#include <climits>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kFT = 512;            // threads per CTA
constexpr double kFix = 1099511627776.0;  // 2^40

template <int DT>
struct FKey {
  // bits of the order-preserving key of a logit; bf16 keys use 16
  static constexpr int kBits = DT == SPEC_BF16 ? 16 : 32;
  __device__ __forceinline__ static uint32_t of(float x) {
    uint32_t u = isnan(x) ? 0xFF800000u : __float_as_uint(x);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return DT == SPEC_BF16 ? (u >> 16) : u;
  }
};

template <int DT>
__device__ __forceinline__ float logit_at(const void* row, int64_t v) {
  return Logit<DT>::load1(row, v);
}

// Radix selection over the elements of a row (block-wide, all threads).
// mode 0: the element of rank `rank` (0-based) in key-descending order;
// mode 1: the first element, in that order, whose inclusive prefix mass
// reaches `target` (fixed point).  Returns the key and, through the
// references, the number (mode 0) or mass (mode 1) of the elements with a
// larger key.
template <int DT>
__device__ uint32_t radix_select(const void* row, int64_t V, float c, float mc, int mode, int64_t rank,
                                 unsigned long long target, int64_t& above_cnt, unsigned long long& above_mass,
                                 int* cnt_sh, unsigned long long* mass_sh,
                                 uint32_t* s_sel, int64_t* s_acnt, unsigned long long* s_amass) {
  constexpr int kBits = FKey<DT>::kBits;
  uint32_t prefix = 0;
  int64_t acnt = 0;
  unsigned long long amass = 0;
  for (int shift = kBits - 8; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kFT) {
      cnt_sh[i] = 0;
      mass_sh[i] = 0;
    }
    __syncthreads();
    const uint32_t hi_mask = shift + 8 >= kBits ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int64_t v = threadIdx.x; v < V; v += kFT) {
      const float x = logit_at<DT>(row, v);
      const uint32_t k = FKey<DT>::of(x);
      if ((k & hi_mask) != (prefix & hi_mask)) continue;
      const int bin = (k >> shift) & 255;
      if (mode == 0) {
        atomicAdd(cnt_sh + bin, 1);
      } else {
        const float w = fast_exp2(fmaf(order_key(x), c, -mc));
        atomicAdd(mass_sh + bin, static_cast<unsigned long long>(__float2ull_rn(w * static_cast<float>(kFix))));
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int bin = 0;
      for (int b = 255; b >= 0; --b) {
        if (mode == 0) {
          if (acnt + cnt_sh[b] > rank) {
            bin = b;
            break;
          }
          acnt += cnt_sh[b];
        } else {
          if (amass + mass_sh[b] >= target) {
            bin = b;
            break;
          }
          amass += mass_sh[b];
        }
      }
      *s_sel = prefix | (static_cast<uint32_t>(bin) << shift);
      *s_acnt = acnt;
      *s_amass = amass;
    }
    __syncthreads();
    prefix = *s_sel;
    acnt = *s_acnt;
    amass = *s_amass;
    __syncthreads();
  }
  above_cnt = acnt;
  above_mass = amass;
  return prefix;
}

// The index of the n-th (0-based) element of key `key` in index order
// (block-wide); each thread scans one contiguous range.
template <int DT>
__device__ int64_t nth_of_key(const void* row, int64_t V, uint32_t key, int64_t n, float* scan_sh, int64_t* s_idx) {
  const int64_t per = (V + kFT - 1) / kFT;
  const int64_t a = threadIdx.x * per, b = a + per < V ? a + per : V;
  int cnt = 0;
  for (int64_t v = a; v < b; ++v) cnt += FKey<DT>::of(logit_at<DT>(row, v)) == key ? 1 : 0;
  float tot;
  const float incl = block_inclusive_scan(static_cast<float>(cnt), scan_sh, tot);  // counts < 2^24: exact
  const int64_t before_me = static_cast<int64_t>(incl) - cnt;
  if (threadIdx.x == 0) *s_idx = -1;
  __syncthreads();
  if (n >= before_me && n < before_me + cnt) {
    int64_t seen = before_me;
    for (int64_t v = a; v < b; ++v)
      if (FKey<DT>::of(logit_at<DT>(row, v)) == key) {
        if (seen == n) {
          *s_idx = v;
          break;
        }
        ++seen;
      }
  }
  __syncthreads();
  return *s_idx;
}

template <int DT>
__global__ void __launch_bounds__(kFT) filter_kernel(void* __restrict__ logits, int64_t R, int64_t V, float c,
                                                    int64_t top_k, float top_p, int32_t* __restrict__ stats) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  __shared__ int cnt_sh[256];
  __shared__ unsigned long long mass_sh[256];
  __shared__ float red[33], scan_sh[33];
  __shared__ uint32_t s_sel;
  __shared__ int64_t s_acnt, s_idx;
  __shared__ unsigned long long s_amass;
  for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
    void* row = static_cast<char*>(logits) + r * V * esz;
    // the row's maximum (NaN as -inf)
    float m = neg_inf();
    for (int64_t v = threadIdx.x; v < V; v += kFT) m = fmaxf(m, order_key(logit_at<DT>(row, v)));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
      float x = threadIdx.x < kFT / 32 ? red[threadIdx.x] : neg_inf();
      x = warp_max(x);
      if (threadIdx.x == 0) red[32] = x;
    }
    __syncthreads();
    m = red[32];
    __syncthreads();
    if (!isfinite(m)) {  // no distribution: the row stays as it is
      if (threadIdx.x == 0) bump(stats, SPEC_STAT_NONFINITE_ROW);
      continue;
    }
    const float mc = m * c;
    const bool use_k = top_k > 0 && top_k < V, use_p = top_p < 1.0f;
    // cut = the last kept element, (key, index)
    uint32_t cut_key = 0;
    int64_t cut_idx = V;  // everything kept
    int64_t acnt;
    unsigned long long amass, mk = 0;
    if (use_k) {
      const uint32_t kk = radix_select<DT>(row, V, c, mc, 0, top_k - 1, 0ull, acnt, amass, cnt_sh, mass_sh,
                                           &s_sel, &s_acnt, &s_amass);
      cut_key = kk;
      cut_idx = nth_of_key<DT>(row, V, kk, top_k - 1 - acnt, scan_sh, &s_idx);
    }
    if (use_p) {
      // the top-k mass: every element up to the top-k cut
      unsigned long long part = 0;
      for (int64_t v = threadIdx.x; v < V; v += kFT) {
        const float x = logit_at<DT>(row, v);
        const uint32_t k = FKey<DT>::of(x);
        if (!use_k || k > cut_key || (k == cut_key && v <= cut_idx))
          part += __float2ull_rn(fast_exp2(fmaf(order_key(x), c, -mc)) * static_cast<float>(kFix));
      }
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if ((threadIdx.x & 31) == 0) mass_sh[threadIdx.x >> 5] = part;
      __syncthreads();
      if (threadIdx.x == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < kFT / 32; ++w) t += mass_sh[w];
        s_amass = t;
      }
      __syncthreads();
      mk = s_amass;
      __syncthreads();
      // the first element whose inclusive prefix mass reaches top_p * mk;
      // top_p <= 0 keeps the first element only
      const unsigned long long target =
          top_p > 0.0f ? static_cast<unsigned long long>(static_cast<double>(top_p) * static_cast<double>(mk)) : 0ull;
      if (target == 0ull) {
        // the first element: rank 0
        const uint32_t kp = radix_select<DT>(row, V, c, mc, 0, 0, 0ull, acnt, amass, cnt_sh, mass_sh, &s_sel,
                                             &s_acnt, &s_amass);
        const int64_t ip = nth_of_key<DT>(row, V, kp, 0, scan_sh, &s_idx);
        if (!use_k || kp > cut_key || (kp == cut_key && ip < cut_idx)) {
          cut_key = kp;
          cut_idx = ip;
        }
      } else {
        const uint32_t kp = radix_select<DT>(row, V, c, mc, 1, 0, target, acnt, amass, cnt_sh, mass_sh, &s_sel,
                                             &s_acnt, &s_amass);
        // one element of key kp weighs what any of them does: find it
        if (threadIdx.x == 0) s_amass = 0;
        __syncthreads();
        for (int64_t v = threadIdx.x; v < V; v += kFT) {
          const float x = logit_at<DT>(row, v);
          if (FKey<DT>::of(x) == kp) {
            s_amass = __float2ull_rn(fast_exp2(fmaf(order_key(x), c, -mc)) * static_cast<float>(kFix));
            break;
          }
        }
        __syncthreads();
        const unsigned long long w1 = s_amass;
        __syncthreads();
        // elements of key kp needed: the smallest j >= 1 with amass + j w1 >= target
        const int64_t j = w1 > 0 ? static_cast<int64_t>((target - amass + w1 - 1) / w1) : 1;
        const int64_t ip = nth_of_key<DT>(row, V, kp, (j < 1 ? 1 : j) - 1, scan_sh, &s_idx);
        const bool earlier = !use_k || kp > cut_key || (kp == cut_key && ip < cut_idx);
        if (ip >= 0 && earlier) {
          cut_key = kp;
          cut_idx = ip;
        }
      }
    }
    if (!spec_in(cut_idx, V + 1, stats) || cut_idx >= V) continue;  // nothing dropped
    // every element after the cut becomes -inf
    for (int64_t v = threadIdx.x; v < V; v += kFT) {
      const uint32_t k = FKey<DT>::of(logit_at<DT>(row, v));
      if (k < cut_key || (k == cut_key && v > cut_idx)) {
        if (DT == SPEC_BF16)
          static_cast<uint16_t*>(row)[v] = 0xFF80u;
        else
          static_cast<float*>(row)[v] = neg_inf();
      }
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" int spec_filter_logits(void* logits, int dtype, int64_t R, int64_t V, float T, int64_t top_k, float top_p,
                                  int32_t* stats_or_null, spec_stream_t stream) {
  if (R < 0 || V < 1 || !(T > 0.0f) || !isfinite(T) || isnan(top_p)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (V > SPEC_MAX_VOCAB) return SPEC_ERR_UNSUPPORTED;
  if (R == 0 || ((top_k <= 0 || top_k >= V) && top_p >= 1.0f)) return SPEC_OK;  // nothing to filter
  if (logits == nullptr) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  // rows stay in L2 for their passes: at most a few rows per SM at a time
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  const int64_t grid = std::min<int64_t>(R, static_cast<int64_t>(sms) * 2);
  if (dtype == SPEC_BF16)
    launch_k(filter_kernel<SPEC_BF16>, static_cast<unsigned>(grid), kFT, 0, s, logits, R, V, c, top_k, top_p,
             stats_or_null);
  else
    launch_k(filter_kernel<SPEC_F32>, static_cast<unsigned>(grid), kFT, 0, s, logits, R, V, c, top_k, top_p,
             stats_or_null);
  return launch_status();
}
