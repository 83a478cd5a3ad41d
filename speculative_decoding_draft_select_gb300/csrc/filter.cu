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
// One CTA per row at a time (rows stay in L2 across the passes).  Keys are
// the logits mapped to unsigned integers in the same order (NaN as -inf);
// bf16 logits need their upper 16 bits only.  Masses are
// 2^((x - max) log2(e) / T) in 2^-40 fixed point, summed as integers: exact
// and independent of the order of the additions, so every cut is
// deterministic; only ratios matter, so no normaliser is needed.
//   top-k: radix selection of the element of rank top_k - 1, 8 bits per
//          level, on count histograms kept per warp (a row's keys crowd
//          into a few high bytes: one shared histogram serialised its
//          atomics) with the lanes of a warp that share a bin adding once;
//          among equal keys the cut goes by index (the n-th element of the
//          cut key in index order: a count per contiguous range, a block
//          scan, one range rescanned).
//   top-p after a top-k of at most kCandMax tokens: the kept tokens are
//          gathered into shared memory, sorted by (key desc, index asc) and
//          the cut is the first whose inclusive prefix mass reaches top_p
//          times their mass.
//   top-p otherwise: radix selection on mass histograms (per warp) for the
//          key where the prefix mass crosses, then the element of that key
//          by index.
// A last pass writes -inf over every element after the cut.
#include <climits>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kFT = 512;            // threads per CTA
constexpr int kFW = kFT / 32;       // warps per CTA
constexpr int kCandMax = 4096;      // candidates sorted in shared memory
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

// Fixed-point mass of a logit (NaN as -inf: 0).
__device__ __forceinline__ unsigned long long fmass(float x, float c, float mc) {
  return __float2ull_rn(fast_exp2(fmaf(order_key(x), c, -mc)) * static_cast<float>(kFix));
}

// Dynamic shared memory of the kernel: the radix histograms or the sorted
// candidates (never both at once), and the threads' row maxima.
struct FShared {
  union {
    struct {
      int cnt[kFW][256];
      unsigned long long mass[kFW][256];
    };
    struct {
      uint32_t ckey[kCandMax];
      int32_t cidx[kCandMax];
      unsigned long long cw[kCandMax];
    };
  };
  float tmax[kFT];
};

// Largest logit of a 16-byte vector, NaN as -inf.
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& raw) {
  if (DT == SPEC_BF16) return order_key(max8_bf16(raw));
  float x[4];
  unpack<SPEC_F32>(raw, x);
  return order_key(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));  // four NaNs give NaN
}

// This thread's maximum (NaN as -inf), a vector at a time.
template <int DT>
struct MaxV {
  float m;
  __device__ __forceinline__ void visit_vec(const uint4& raw, int64_t, bool) { m = fmaxf(m, vec_max<DT>(raw)); }
  __device__ __forceinline__ void visit1(float x, int64_t, bool) { m = fmaxf(m, order_key(x)); }
};

// One level of the radix selection: each element whose key matches the
// bytes chosen so far adds to its warp's histogram of the next byte (count,
// or mass).  Warp-uniform (for_row_raw): lanes that share a bin add their
// count once.
template <int DT, bool MASS>
struct HistV {
  uint32_t hi_mask, prefix;
  int shift;
  float c, mc;
  int* cnt;                  // this warp's count histogram
  unsigned long long* mass;  // this warp's mass histogram
  __device__ __forceinline__ void add(float x, bool ok) {
    const uint32_t k = FKey<DT>::of(x);
    const bool in = ok && (k & hi_mask) == prefix;
    const int bin = in ? static_cast<int>((k >> shift) & 255u) : -1;
    if (!MASS) {
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (in && static_cast<int>(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(cnt + bin, __popc(peers));
    } else if (in) {
      atomicAdd(mass + bin, fmass(x, c, mc));
    }
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int64_t, bool ok) {
    constexpr int kv = Logit<DT>::kVec;
    float x[kv];
    unpack<DT>(raw, x);
#pragma unroll
    for (int j = 0; j < kv; ++j) add(x[j], ok);
  }
  __device__ __forceinline__ void visit1(float x, int64_t, bool ok) { add(x, ok); }
};

// Radix selection over the elements of a row (block-wide, all threads).
// MASS false: the element of rank `rank` (0-based) in key-descending order;
// MASS true: the first element, in that order, whose inclusive prefix mass
// reaches `target` (fixed point).  Returns its key and, through the
// references, the number (count mode) or mass (mass mode) of the elements
// with a larger key.
template <int DT, bool MASS>
__device__ uint32_t radix_select(const void* row, int64_t V, float c, float mc, int64_t rank,
                                 unsigned long long target, int64_t& above_cnt, unsigned long long& above_mass,
                                 FShared& sh, uint32_t* s_sel, int64_t* s_acnt, unsigned long long* s_amass) {
  constexpr int kBits = FKey<DT>::kBits;
  const int warp = threadIdx.x >> 5;
  uint32_t prefix = 0;
  int64_t acnt = 0;
  unsigned long long amass = 0;
  for (int shift = kBits - 8; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < kFW * 256; i += kFT) {
      if (MASS) (&sh.mass[0][0])[i] = 0;
      else (&sh.cnt[0][0])[i] = 0;
    }
    __syncthreads();
    const uint32_t hi_mask = shift + 8 >= kBits ? 0u : (0xFFFFFFFFu << (shift + 8));
    HistV<DT, MASS> hv{hi_mask, prefix & hi_mask, shift, c, mc, sh.cnt[warp], sh.mass[warp]};
    for_row_raw<DT, 4>(row, V, hv, threadIdx.x, kFT);
    __syncthreads();
    // the warps' histograms into row 0 (one bin per thread)
    for (int b = threadIdx.x; b < 256; b += kFT) {
      if (MASS) {
        unsigned long long t = 0;
#pragma unroll
        for (int w = 0; w < kFW; ++w) t += sh.mass[w][b];
        sh.mass[0][b] = t;
      } else {
        int t = 0;
#pragma unroll
        for (int w = 0; w < kFW; ++w) t += sh.cnt[w][b];
        sh.cnt[0][b] = t;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int bin = 0;
      for (int b = 255; b >= 0; --b) {
        if (!MASS) {
          if (acnt + sh.cnt[0][b] > rank) {
            bin = b;
            break;
          }
          acnt += sh.cnt[0][b];
        } else {
          if (amass + sh.mass[0][b] >= target) {
            bin = b;
            break;
          }
          amass += sh.mass[0][b];
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

// Elements [a, b) of thread t's contiguous range of a row in index order:
// the head scalars go to thread 0, the 16-byte vectors are split evenly, the
// tail scalars go to the last thread.  f(x, index) per element, in order.
template <int DT, class F>
__device__ __forceinline__ void range_visit(const void* row, int64_t V, F&& f) {
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const RowSpan sp = row_span<DT>(row, V);
  const int t = threadIdx.x;
  if (t == 0)
    for (int64_t i = 0; i < sp.head; ++i) f(Logit<DT>::load1(row, i), i);
  const int64_t per = (sp.nvec + kFT - 1) / kFT;
  const int64_t a = t * per, b = a + per < sp.nvec ? a + per : sp.nvec;
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  for (int64_t i = a; i < b; ++i) {
    float x[kv];
    unpack<DT>(__ldg(vp + i), x);
#pragma unroll
    for (int j = 0; j < kv; ++j) f(x[j], sp.head + i * kv + j);
  }
  if (t == kFT - 1)
    for (int64_t i = sp.head + sp.nvec * kv; i < V; ++i) f(Logit<DT>::load1(row, i), i);
}

// The index of the n-th (0-based) element of key `key` in index order
// (block-wide): a count per contiguous range, a block scan, and the range
// that holds it scanned again.
template <int DT>
__device__ int64_t nth_of_key(const void* row, int64_t V, uint32_t key, int64_t n, float* scan_sh, int64_t* s_idx) {
  int cnt = 0;
  range_visit<DT>(row, V, [&](float x, int64_t) { cnt += FKey<DT>::of(x) == key ? 1 : 0; });
  float tot;
  const float incl = block_inclusive_scan(static_cast<float>(cnt), scan_sh, tot);  // counts < 2^24: exact
  const int64_t before_me = static_cast<int64_t>(incl) - cnt;
  if (threadIdx.x == 0) *s_idx = -1;
  __syncthreads();
  if (n >= before_me && n < before_me + cnt) {
    int64_t seen = before_me, found = -1;
    range_visit<DT>(row, V, [&](float x, int64_t v) {
      if (found < 0 && FKey<DT>::of(x) == key) {
        if (seen == n) found = v;
        ++seen;
      }
    });
    *s_idx = found;
  }
  __syncthreads();
  const int64_t r = *s_idx;
  __syncthreads();
  return r;
}

// Whether candidate a comes before candidate b: key desc, index asc.
__device__ __forceinline__ bool cand_before(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// The block's sum of one u64 per thread (every thread gets it).
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kFW; ++w) t += red[w];
  __syncthreads();
  return t;
}

// Candidates into the arrays: with TAU, every element whose key is at
// least tau's; else the kept tokens of a top-k cut (key > ck, or key == ck
// and index <= ci).  The count goes on past kCandMax (the caller then takes
// another path); entries past it are not stored.
template <int DT, bool TAU>
struct GatherV {
  FShared* sh;
  int* nc;
  uint32_t ck;
  int64_t ci;
  float c, mc;
  __device__ __forceinline__ void one(float x, int64_t v) {
    const uint32_t k = FKey<DT>::of(x);
    if (TAU ? k >= ck : (k > ck || (k == ck && v <= ci))) {
      const int slot = atomicAdd(nc, 1);
      if (slot < kCandMax) {
        sh->ckey[slot] = k;
        sh->cidx[slot] = static_cast<int32_t>(v);
        sh->cw[slot] = fmass(x, c, mc);
      }
    }
  }
  __device__ __forceinline__ void visit_vec(const uint4& raw, int64_t first, bool) {
    if (FKey<DT>::of(vec_max<DT>(raw)) < ck) return;  // no element of the vector qualifies (most of them)
    constexpr int kv = Logit<DT>::kVec;
    float x[kv];
    unpack<DT>(raw, x);
#pragma unroll
    for (int j = 0; j < kv; ++j) one(x[j], first + j);
  }
  __device__ __forceinline__ void visit1(float x, int64_t v, bool) { one(x, v); }
};

// Sorts the first nc (<= kCandMax) candidates into (key desc, index asc):
// a bitonic network over the next power of two, padded with entries that
// sort last (block-wide).
__device__ void sort_cands(FShared& sh, int nc) {
  int n2 = 1;
  while (n2 < nc) n2 <<= 1;
  for (int i = nc + threadIdx.x; i < n2; i += kFT) {
    sh.ckey[i] = 0;
    sh.cidx[i] = INT_MAX;
    sh.cw[i] = 0;
  }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n2; i += kFT) {
        const int j = i ^ stride;
        if (j > i) {
          const bool first_half = (i & size) == 0;
          const bool jb = cand_before(sh.ckey[j], sh.cidx[j], sh.ckey[i], sh.cidx[i]);
          if (jb == first_half) {
            const uint32_t tk = sh.ckey[i];
            const int32_t ti = sh.cidx[i];
            const unsigned long long tw = sh.cw[i];
            sh.ckey[i] = sh.ckey[j];
            sh.cidx[i] = sh.cidx[j];
            sh.cw[i] = sh.cw[j];
            sh.ckey[j] = tk;
            sh.cidx[j] = ti;
            sh.cw[j] = tw;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Among the first n sorted candidates, the first position whose inclusive
// prefix mass reaches top_p times their mass (top_p <= 0: position 0)
// (block-wide).
__device__ int p_cut(const FShared& sh, int n, float top_p, unsigned long long* red64, int* s_pos) {
  constexpr int kPer = kCandMax / kFT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long part = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int i = threadIdx.x * kPer + e;
    part += i < n ? sh.cw[i] : 0ull;
  }
  const unsigned long long mk = block_sum_u64(part, red64);
  const unsigned long long target =
      top_p > 0.0f ? static_cast<unsigned long long>(static_cast<double>(top_p) * static_cast<double>(mk)) : 0ull;
  // exclusive prefix of this thread's entries: a warp scan, then the warps
  unsigned long long x = part;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red64[warp] = x;
  if (threadIdx.x == 0) *s_pos = INT_MAX;
  __syncthreads();
  unsigned long long pre = x - part;
  for (int w = 0; w < warp; ++w) pre += red64[w];
  for (int e = 0; e < kPer; ++e) {
    const int i = threadIdx.x * kPer + e;
    if (i >= n) break;
    pre += sh.cw[i];
    if (pre >= target) {
      atomicMin(s_pos, i);
      break;
    }
  }
  __syncthreads();
  const int pos = *s_pos == INT_MAX ? n - 1 : *s_pos;
  __syncthreads();
  return pos;
}

// This thread's part of the mass of the elements up to the top-k cut (all
// elements without one).
template <int DT>
struct KMassV {
  uint32_t ck;
  int64_t ci;
  bool use_k;
  float c, mc;
  unsigned long long s;
  template <int N>
  __device__ __forceinline__ void visit(const float* x, int64_t first) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const uint32_t k = FKey<DT>::of(x[j]);
      if (!use_k || k > ck || (k == ck && first + j <= ci)) s += fmass(x[j], c, mc);
    }
  }
};

// The mass of one element of key kp (every element of that key has it).
template <int DT>
struct OneOfV {
  uint32_t kp;
  float c, mc;
  unsigned long long* out;
  template <int N>
  __device__ __forceinline__ void visit(const float* x, int64_t) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (FKey<DT>::of(x[j]) == kp) *out = fmass(x[j], c, mc);  // every writer writes the same value
  }
};

template <int DT>
__global__ void __launch_bounds__(kFT, 2) filter_kernel(void* __restrict__ logits, int64_t R, int64_t V, float c,
                                                    int64_t top_k, float top_p, int32_t* __restrict__ stats) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kv = Logit<DT>::kVec;
  extern __shared__ __align__(16) unsigned char f_dsm[];
  FShared& sh = *reinterpret_cast<FShared*>(f_dsm);
  if (!spec_smem_ok(sizeof(FShared), stats)) return;
  __shared__ float red[33], scan_sh[33];
  __shared__ unsigned long long red64[kFW];
  __shared__ uint32_t s_sel;
  __shared__ int64_t s_acnt, s_idx;
  __shared__ unsigned long long s_amass;
  __shared__ int s_nc, s_pos;
  __shared__ uint32_t s_tau;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
    void* row = static_cast<char*>(logits) + r * V * esz;
    // the row's maximum (NaN as -inf)
    MaxV<DT> mv{neg_inf()};
    for_row_fast<DT, 4>(row, V, mv, tid, kFT);
    sh.tmax[tid] = mv.m;
    float m = warp_max(mv.m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (tid < 32) {
      float x = tid < kFW ? red[tid] : neg_inf();
      x = warp_max(x);
      if (tid == 0) red[32] = x;
    }
    __syncthreads();
    m = red[32];
    __syncthreads();
    if (!isfinite(m)) {  // no distribution: the row stays as it is
      if (tid == 0) bump(stats, SPEC_STAT_NONFINITE_ROW);
      continue;
    }
    const float mc = m * c;
    const bool use_k = top_k > 0 && top_k < V, use_p = top_p < 1.0f;
    // cut = the last kept element, (key, index)
    uint32_t cut_key = 0;
    int64_t cut_idx = V;  // everything kept
    int64_t acnt;
    unsigned long long amass;
    bool done = false;
    if (use_k && top_k <= kFT) {
      // a lower bound of the top-k cut: the top_k-th largest of the
      // threads' maxima (top_k threads each hold an element at least as
      // large); every element at or above it is a candidate, sorted exactly
      // (the maxima sorted in descending order by a bitonic network)
      for (int size = 2; size <= kFT; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const int j = tid ^ stride;
          if (j > tid) {
            const float a = sh.tmax[tid], b = sh.tmax[j];
            if ((b > a) == ((tid & size) == 0)) {
              sh.tmax[tid] = b;
              sh.tmax[j] = a;
            }
          }
          __syncthreads();
        }
      }
      if (tid == 0) {
        s_tau = FKey<DT>::of(sh.tmax[top_k - 1]);
        s_nc = 0;
      }
      __syncthreads();
      GatherV<DT, true> gv{&sh, &s_nc, s_tau, 0, c, mc};
      for_row_fast<DT, 4>(row, V, gv, tid, kFT);
      __syncthreads();
      const int nc = s_nc;
      if (nc <= kCandMax) {
        sort_cands(sh, nc);
        const int pos = use_p ? p_cut(sh, static_cast<int>(top_k), top_p, red64, &s_pos) : static_cast<int>(top_k) - 1;
        cut_key = sh.ckey[pos];
        cut_idx = sh.cidx[pos];
        done = true;
      }
      __syncthreads();
    }
    if (done) {
    } else if (use_k) {
      const uint32_t kk = radix_select<DT, false>(row, V, c, mc, top_k - 1, 0ull, acnt, amass, sh, &s_sel, &s_acnt,
                                                  &s_amass);
      cut_key = kk;
      cut_idx = nth_of_key<DT>(row, V, kk, top_k - 1 - acnt, scan_sh, &s_idx);
    }
    if (done || !use_p) {
    } else if (use_k && top_k <= kCandMax) {
      // the top-k tokens, sorted by (key desc, index asc) in shared memory
      if (tid == 0) s_nc = 0;
      __syncthreads();
      GatherV<DT, false> gv{&sh, &s_nc, cut_key, cut_idx, c, mc};
      for_row_fast<DT, 4>(row, V, gv, tid, kFT);
      __syncthreads();
      const int nc = min(s_nc, kCandMax);
      sort_cands(sh, nc);
      const int pos = p_cut(sh, nc, top_p, red64, &s_pos);
      cut_key = sh.ckey[pos];
      cut_idx = sh.cidx[pos];
      __syncthreads();
    } else if (use_p) {
      // the top-k mass: every element up to the top-k cut
      KMassV<DT> km{cut_key, cut_idx, use_k, c, mc, 0ull};
      for_row<DT, 4>(row, V, km, tid, kFT);
      const unsigned long long mk = block_sum_u64(km.s, red64);
      // the first element whose inclusive prefix mass reaches top_p * mk;
      // top_p <= 0 keeps the first element only
      const unsigned long long target =
          top_p > 0.0f ? static_cast<unsigned long long>(static_cast<double>(top_p) * static_cast<double>(mk)) : 0ull;
      if (target == 0ull) {
        const uint32_t kp = radix_select<DT, false>(row, V, c, mc, 0, 0ull, acnt, amass, sh, &s_sel, &s_acnt,
                                                    &s_amass);
        const int64_t ip = nth_of_key<DT>(row, V, kp, 0, scan_sh, &s_idx);
        if (!use_k || kp > cut_key || (kp == cut_key && ip < cut_idx)) {
          cut_key = kp;
          cut_idx = ip;
        }
      } else {
        const uint32_t kp = radix_select<DT, true>(row, V, c, mc, 0, target, acnt, amass, sh, &s_sel, &s_acnt,
                                                   &s_amass);
        // one element of key kp weighs what any of them does: find it
        if (tid == 0) s_amass = 0;
        __syncthreads();
        OneOfV<DT> oo{kp, c, mc, &s_amass};
        for_row<DT, 4>(row, V, oo, tid, kFT);
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
    // every element after the cut becomes -inf (vectors rewritten only where
    // something drops)
    const RowSpan sp = row_span<DT>(row, V);
    auto dropped = [&](float x, int64_t v) {
      const uint32_t k = FKey<DT>::of(x);
      return k < cut_key || (k == cut_key && v > cut_idx);
    };
    for (int64_t v = tid; v < sp.head; v += kFT)
      if (dropped(Logit<DT>::load1(row, v), v)) {
        if (DT == SPEC_BF16) static_cast<uint16_t*>(row)[v] = 0xFF80u;
        else static_cast<float*>(row)[v] = neg_inf();
      }
    uint4* vp = reinterpret_cast<uint4*>(static_cast<char*>(row) + sp.head * esz);
    const uint4 all_ninf = DT == SPEC_BF16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                           : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    for (int64_t i = tid; i < sp.nvec; i += kFT) {
      uint4 raw = vp[i];
      if (FKey<DT>::of(vec_max<DT>(raw)) < cut_key) {  // every element drops
        vp[i] = all_ninf;
        continue;
      }
      float x[kv];
      unpack<DT>(raw, x);
      uint32_t* w = reinterpret_cast<uint32_t*>(&raw);
      bool any = false;
#pragma unroll
      for (int j = 0; j < kv; ++j) {
        if (!dropped(x[j], sp.head + i * kv + j)) continue;
        any = true;
        if (DT == SPEC_BF16) {
          w[j >> 1] = (j & 1) ? ((w[j >> 1] & 0x0000FFFFu) | 0xFF800000u) : ((w[j >> 1] & 0xFFFF0000u) | 0xFF80u);
        } else {
          w[j] = 0xFF800000u;
        }
      }
      if (any) vp[i] = raw;
    }
    for (int64_t v = sp.head + sp.nvec * kv + tid; v < V; v += kFT)
      if (dropped(Logit<DT>::load1(row, v), v)) {
        if (DT == SPEC_BF16) static_cast<uint16_t*>(row)[v] = 0xFF80u;
        else static_cast<float*>(row)[v] = neg_inf();
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
  constexpr size_t smem = sizeof(FShared);
  auto kernel = dtype == SPEC_BF16 ? filter_kernel<SPEC_BF16> : filter_kernel<SPEC_F32>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  launch_k(kernel, static_cast<unsigned>(grid), kFT, smem, s, logits, R, V, c, top_k, top_p, stats_or_null);
  return launch_status();
}
