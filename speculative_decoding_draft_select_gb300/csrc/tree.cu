// Draft tree: per-step expansion into the candidate pool, and the tree build
// (node selection, parents, positions, tree attention mask, retrieve links).
//
// "[SGLang] Multi-Layer EAGLE" (secrett2633 blog), section 2:
// select_top_k_tokens returns tree_info = (scores, tokens, parents) per draft
// step.  "EAGLE speculative decoding in four parts" (ai-infra-handbooks),
// "Drafting, verification and slots": build_eagle_tree expands the
// candidates into a tree and produces the attention mask and positions for
// verification.  zero-to-sglang ch.10 "Speculative decoding (code
// walk-through)" 5.2 lists the verify input (draft_token, positions,
// custom_mask, retrieve_*).
//
// Both kernels run one CTA per request; the work is a few hundred elements,
// so they are latency kernels: everything is staged in shared memory.
#include <climits>

#include "common.cuh"
#include "expand.cuh"

namespace specdec {
namespace {

__global__ void tree_expand_kernel(ExpandArgs e, const float* __restrict__ topk_p,
                                   const int32_t* __restrict__ topk_idx) {
  pdl_enter();
  extern __shared__ uint64_t keys[];
  if (!spec_smem_ok(sizeof(uint64_t) * (e.step == 0 ? e.k : e.k * e.k), nullptr)) return;
  expand_request(e, blockIdx.x, topk_p, topk_idx, keys);
}

// Exclusive scan of one int per thread (thread order); returns the total.
__device__ __forceinline__ int block_exclusive_scan_int(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) sh[lane] = w;
  }
  __syncthreads();
  total = sh[nw - 1];
  return x - v + (warp > 0 ? sh[warp - 1] : 0);
}

constexpr int kBuildThreads = 512;
constexpr int64_t kRankPool = 1024;  // selection by rank counting up to this many candidates
constexpr int kParallelLinks = 256;  // first child / next sibling one thread per node up to N

__global__ void __launch_bounds__(kBuildThreads)
    build_tree_kernel(int N, int64_t P, int64_t L, const float* __restrict__ pool_score,
                      const int32_t* __restrict__ pool_token, const int32_t* __restrict__ pool_parent,
                      const int32_t* __restrict__ pool_qrow, const int32_t* __restrict__ root_token,
                      const int32_t* __restrict__ seq_lens, int32_t* draft_token, int32_t* parent,
                      int32_t* positions, uint8_t* tree_mask, int32_t* retrieve_index,
                      int32_t* next_token, int32_t* next_sibling, int32_t* q_row) {
  pdl_enter();
  extern __shared__ uint64_t dyn[];
  uint64_t* keys = dyn;                                       // [L]
  int32_t* node_of = reinterpret_cast<int32_t*>(keys + L);    // [P]
  int32_t* npid = node_of + P;                                // [N]
  int32_t* npar = npid + N;                                   // [N]
  int32_t* nxt = npar + N;                                    // [N]
  if (!spec_smem_ok(reinterpret_cast<char*>(nxt + N) - reinterpret_cast<char*>(dyn), nullptr)) return;
  __shared__ int scan_sh[33];
  const int b = blockIdx.x;
  const int nt = blockDim.x;
  const float* sc = pool_score + b * P;
  const int32_t* tk = pool_token + b * P;
  const int32_t* pa = pool_parent + b * P;
  const int32_t* qr = pool_qrow + b * P;

  // 1. the N-1 best non-root candidates by (score desc, pool id asc): keys
  // are distinct, so a candidate's rank is the number of smaller keys
  // (small pools); larger pools are sorted (bitonic)
  for (int64_t i = threadIdx.x; i < L; i += nt)
    keys[i] = i < P - 1 ? rank_key(__ldg(sc + i + 1), static_cast<int32_t>(i + 1)) : ~0ull;
  for (int64_t i = threadIdx.x; i < P; i += nt) node_of[i] = i == 0 ? 1 : 0;
  __syncthreads();
  if (P - 1 <= kRankPool) {
    for (int64_t i = threadIdx.x; i < P - 1; i += nt) {
      const uint64_t ki = keys[i];
      int rank = 0;
      for (int64_t j = 0; j < P - 1; ++j) rank += keys[j] < ki ? 1 : 0;
      if (rank < N - 1) node_of[i + 1] = 1;
    }
  } else {
    for (int64_t size = 2; size <= L; size <<= 1) {
      for (int64_t stride = size >> 1; stride > 0; stride >>= 1) {
        for (int64_t i = threadIdx.x; i < L; i += nt) {
          const int64_t j = i ^ stride;
          if (j > i) {
            const bool asc = (i & size) == 0;
            const uint64_t a = keys[i], c = keys[j];
            if ((a > c) == asc) {
              keys[i] = c;
              keys[j] = a;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int64_t r = threadIdx.x; r < N - 1; r += nt)
      if (spec_in(static_cast<uint32_t>(keys[r]), P, nullptr)) node_of[static_cast<uint32_t>(keys[r])] = 1;
  }
  __syncthreads();
  // 2. the root and the selected candidates, numbered in pool-id order
  const int64_t chunk = (P + nt - 1) / nt;
  const int64_t lo = threadIdx.x * chunk, hi = min(P, lo + chunk);
  int cnt = 0;
  for (int64_t i = lo; i < hi; ++i) cnt += node_of[i];
  int total;
  int idx = block_exclusive_scan_int(cnt, scan_sh, total);
  for (int64_t i = lo; i < hi; ++i) {
    if (node_of[i] && spec_in(idx, N, nullptr)) {
      npid[idx] = static_cast<int32_t>(i);
      node_of[i] = idx++;
    } else {
      node_of[i] = -1;
    }
  }
  __syncthreads();
  // 3. per-node fields
  const int64_t o = static_cast<int64_t>(b) * N;
  for (int n = threadIdx.x; n < N; n += nt) {
    const int32_t pid = npid[n];
    if (!spec_in(pid, P, nullptr)) continue;
    int32_t par = -1;
    if (n > 0) {
      const int32_t pp = __ldg(pa + pid);
      par = (pp >= 0 && pp < P) ? node_of[pp] : -1;
      if (par >= n) par = -1;  // only possible when a child outscores its parent
    }
    npar[n] = par;
    draft_token[o + n] = n == 0 ? __ldg(root_token + b) : __ldg(tk + pid);
    parent[o + n] = par;
    retrieve_index[o + n] = static_cast<int32_t>(o + n);
    q_row[o + n] = __ldg(qr + pid);
  }
  __syncthreads();
  const int32_t sl = __ldg(seq_lens + b);
  for (int n = threadIdx.x; n < N; n += nt) {
    int d = 0;
    for (int a = n; a > 0 && d <= N; a = npar[a]) ++d;
    positions[o + n] = sl + d;
  }
  // mask[n][m] = 1 iff m is n or an ancestor of n (ancestors have smaller ids)
  uint8_t* mask = tree_mask + o * N;
  for (int64_t e = threadIdx.x; e < static_cast<int64_t>(N) * N; e += nt) {
    const int n = static_cast<int>(e / N), m = static_cast<int>(e % N);
    int a = n;
    while (a > m) a = npar[a];
    mask[e] = a == m ? 1 : 0;
  }
  // 4. first child and next sibling, in node order (the smallest later node
  // with parent n, or with n's parent)
  if (N <= kParallelLinks) {
    for (int n = threadIdx.x; n < N; n += nt) {
      const int p = n > 0 ? npar[n] : -1;
      int fc = -1, ns = -1;
      for (int m2 = n + 1; m2 < N && (fc < 0 || (p >= 0 && ns < 0)); ++m2) {
        const int q = npar[m2];
        if (fc < 0 && q == n) fc = m2;
        if (p >= 0 && ns < 0 && q == p) ns = m2;
      }
      next_token[o + n] = fc;
      next_sibling[o + n] = ns;
    }
  } else {
    if (threadIdx.x == 0) {
      for (int n = 0; n < N; ++n) nxt[n] = -1;
      for (int n = N - 1; n >= 1; --n) {
        const int p = npar[n];
        next_sibling[o + n] = p >= 0 ? nxt[p] : -1;
        if (p >= 0) nxt[p] = n;
      }
      next_sibling[o] = -1;
    }
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += nt) next_token[o + n] = nxt[n];
  }
}

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" int64_t spec_tree_pool_size(int k, int num_steps) {
  if (k < 1 || num_steps < 1) return -1;
  return 1 + static_cast<int64_t>(k) + static_cast<int64_t>(num_steps - 1) * k * k;
}

extern "C" int spec_tree_expand(int step, int num_steps, int B, int k, const float* topk_p,
                                const int32_t* topk_idx, float* pool_score, int32_t* pool_token,
                                int32_t* pool_parent, int32_t* pool_qrow, float* frontier_score,
                                int32_t* frontier_id, spec_stream_t stream) {
  if (B < 0 || k < 1 || num_steps < 1 || step < 0 || step >= num_steps) return SPEC_ERR_INVALID_ARG;
  if (k > SPEC_MAX_TOPK) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!topk_p || !topk_idx || !pool_score || !pool_token || !pool_parent || !pool_qrow || !frontier_score ||
      !frontier_id)
    return SPEC_ERR_INVALID_ARG;
  const int64_t P = spec_tree_pool_size(k, num_steps);
  if (static_cast<int64_t>(B) * k * num_steps > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  const int nc = step == 0 ? k : k * k;
  const int threads = ((nc + 31) / 32) * 32;
  const ExpandArgs e{step, num_steps, B, k, P, pool_score, pool_token, pool_parent, pool_qrow, frontier_score,
                     frontier_id, nullptr};
  launch_k(tree_expand_kernel, B, threads, sizeof(uint64_t) * nc, reinterpret_cast<cudaStream_t>(stream), e, topk_p,
           topk_idx);
  return launch_status();
}

extern "C" int spec_build_tree(int B, int k, int num_steps, int N, const float* pool_score,
                               const int32_t* pool_token, const int32_t* pool_parent,
                               const int32_t* pool_qrow, const int32_t* root_token, const int32_t* seq_lens,
                               int32_t* draft_token, int32_t* parent, int32_t* positions, uint8_t* tree_mask,
                               int32_t* retrieve_index, int32_t* retrieve_next_token,
                               int32_t* retrieve_next_sibling, int32_t* q_row, spec_stream_t stream) {
  if (B < 0 || k < 1 || num_steps < 1 || N < 1) return SPEC_ERR_INVALID_ARG;
  const int64_t P = spec_tree_pool_size(k, num_steps);
  if (N > P) return SPEC_ERR_INVALID_ARG;
  if (P > SPEC_MAX_POOL || N > SPEC_MAX_NODES || k > SPEC_MAX_TOPK) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!pool_score || !pool_token || !pool_parent || !pool_qrow || !root_token || !seq_lens || !draft_token ||
      !parent || !positions || !tree_mask || !retrieve_index || !retrieve_next_token || !retrieve_next_sibling ||
      !q_row)
    return SPEC_ERR_INVALID_ARG;
  int64_t L = 1;
  while (L < P - 1) L <<= 1;
  const size_t smem = sizeof(uint64_t) * L + sizeof(int32_t) * (P + 3 * static_cast<int64_t>(N));
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  launch_k(build_tree_kernel, B, kBuildThreads, smem, reinterpret_cast<cudaStream_t>(stream), N, P, L, pool_score,
           pool_token, pool_parent, pool_qrow, root_token, seq_lens, draft_token, parent, positions, tree_mask,
           retrieve_index, retrieve_next_token, retrieve_next_sibling, q_row);
  return launch_status();
}
