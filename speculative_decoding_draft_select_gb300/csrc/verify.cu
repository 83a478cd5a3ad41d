// Batched verification over the target logits of every tree node.
//
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)":
//   3.3  row L-1+i of the target output verifies draft i, row L+k-1 gives the
//        bonus -- here row (b, n) verifies node n's children;
//   4.1  greedy_commit: commit the target's choice, stop at the first
//        mismatch, at EOS or when the budget is used; bonus on full accept;
//   5.1  stochastic acceptance: accept y ~ q with min(1, p[y]/q[y]); after a
//        rejection draw from the normalised positive residual (p - q)+; after
//        full acceptance draw the bonus from p.
// "EAGLE speculative decoding in four parts" (ai-infra-handbooks),
// "Drafting, verification and slots": one target pass verifies every tree
// candidate; the verify kernels walk the tree to each request's longest
// accepted path.
//
// Greedy: row_argmax_kernel streams every target row once with 16-byte
// loads (one CTA per row) for its argmax; greedy_walk_kernel then walks
// each request's tree (one warp per request).  Stochastic:
// sample_verify_kernel, one persistent launch, computes the online-softmax
// max and normaliser of every target row (the batched pass, each row read
// once) and walks each request's tree as soon as the rows on its path are
// done (a cluster of CTAs per request).  The walk gathers p[y] and q[y] of
// every child of the current node at once, and after each rejection streams
// the node's target and q rows to get the residual's mass.
// The residual after j rejections is kept in closed form,
//   p_j(v) = max(0, p(v) - A_j q(v)) / c_j,  A_{j+1} = A_j + c_j,
//   c_{j+1} = sum_v max(0, p(v) - A_{j+1} q(v)),  A_0 = 0, c_0 = 1,
// which equals the repeated normalised update (p_j - q)+ / sum (p_j - q)+.
// The last residual pass also leaves the per-tile sums the inverse-CDF draw
// needs, so a correction token costs one row sweep plus one tile rescan.
#include <climits>
#include <vector>

#include "cdf.cuh"
#include "chain.h"
#include "common.cuh"
#include "walk.cuh"

namespace specdec {
namespace {

__global__ void wait_probe_kernel(const int* flag, long long limit, int32_t* stats, int32_t* seen) {
  pdl_enter();
  if (threadIdx.x == 0) *seen = wait_flag(flag, limit, stats) ? 1 : 0;
}

constexpr int kStatThreads = 256;
constexpr int kStatUnroll = 8;  // 16-byte loads in flight per thread

// Greedy pass 1: one CTA per target row streams it with 16-byte loads (8 in
// flight per thread) and reduces it to its argmax (value desc, index asc,
// NaN skipped).  Measured on GB300 this plain load loop keeps HBM at the
// copy rate; staging through shared memory with bulk copies was slower for
// this access pattern.  (The stochastic verify computes its row statistics
// inside sample_verify_kernel.)
template <int DT>
__global__ void __launch_bounds__(kStatThreads, 1024 / kStatThreads)
    row_argmax_kernel(const void* __restrict__ logits, int64_t V, int32_t* __restrict__ amax,
                      int32_t* __restrict__ stats) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kWarps = kStatThreads / 32;
  __shared__ float wv[kWarps];
  __shared__ int wi[kWarps];
  const int64_t r = blockIdx.x;
  const void* row = static_cast<const char*>(logits) + r * V * esz;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  RowStatVisitor<DT, false> v{0.0f, neg_inf(), 0.0f, 0.0f, INT_MAX, 0.0f};
  for_row_fast<DT, kStatUnroll>(row, V, v, threadIdx.x, kStatThreads);
  float bv = v.m;
  int bi = v.bi;
  warp_best(bv, bi);
  if (lane == 0) {
    wv[warp] = bv;
    wi[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kWarps ? wv[lane] : neg_inf();
    bi = lane < kWarps ? wi[lane] : INT_MAX;
    warp_best(bv, bi);
    if (lane == 0 && spec_in(r, gridDim.x, stats)) {
      amax[r] = bi == INT_MAX ? 0 : bi;
      if (!isfinite(bv)) bump(stats, SPEC_STAT_NONFINITE_ROW);
    }
  }
}

template <int DT>
int launch_row_argmax(const void* logits, int64_t V, int64_t R, int32_t* amax, int32_t* stats, cudaStream_t s) {
  launch_k(row_argmax_kernel<DT>, static_cast<unsigned>(R), kStatThreads, 0, s, logits, V, amax, stats);
  return launch_status();
}

// ------------------------------------------------------------ greedy walk

__global__ void greedy_walk_kernel(int N, const int32_t* __restrict__ amax, const int32_t* __restrict__ dtok,
                                   const int32_t* __restrict__ ntok, const int32_t* __restrict__ nsib,
                                   const int32_t* __restrict__ budget, int32_t eos, int32_t* committed,
                                   int32_t* num_committed, int32_t* accept_length, int32_t* accept_path,
                                   int32_t* next_root, int32_t* walk_info, int32_t* stats) {
  pdl_enter();
  extern __shared__ int32_t sh[];
  int32_t *s_am = sh, *s_dt = sh + N, *s_nt = sh + 2 * N, *s_ns = sh + 3 * N, *s_com = sh + 4 * N,
          *s_path = sh + 5 * N;
  const int b = blockIdx.x, lane = threadIdx.x;
  const int64_t o = static_cast<int64_t>(b) * N;
  for (int i = lane; i < N; i += 32) {
    s_am[i] = __ldg(amax + o + i);
    s_dt[i] = __ldg(dtok + o + i);
    s_nt[i] = __ldg(ntok + o + i);
    s_ns[i] = __ldg(nsib + o + i);
    s_com[i] = -1;
    s_path[i] = -1;
  }
  __syncwarp();
  if (lane == 0) {
    const int rem = budget ? __ldg(budget + b) : INT_MAX;
    int len = 0, acc = 0, rej = 0, kind = SPEC_FINAL_ACCEPTED, n = 0;
    s_path[0] = 0;
    while (rem > 0 && len < N) {
      const int32_t t = s_am[n];
      s_com[len++] = t;
      int found = -1, hops = 0;
      for (int c = s_nt[n]; c > 0 && c < N && hops < N; c = s_ns[c], ++hops) {
        if (s_dt[c] == t) {
          found = c;
          break;
        }
        ++rej;
      }
      // (links that loop cannot push the path past N entries)
      if (found >= 0 && acc + 1 < N) s_path[++acc] = found;
      if (t == eos || len == rem || found < 0) {
        if (found >= 0) {
          kind = SPEC_FINAL_ACCEPTED;
          n = found;
        } else {
          kind = s_nt[n] > 0 ? SPEC_FINAL_CORRECTION : SPEC_FINAL_BONUS;
        }
        break;
      }
      n = found;
    }
    num_committed[b] = len;
    accept_length[b] = acc;
    next_root[b] = len > 0 ? s_com[len - 1] : -1;
    if (walk_info) {
      walk_info[3 * b] = n;
      walk_info[3 * b + 1] = rej;
      walk_info[3 * b + 2] = kind;
    }
  }
  __syncwarp();
  for (int i = lane; i < N; i += 32) {
    if (!spec_in(o + i, static_cast<int64_t>(gridDim.x) * N, stats)) continue;
    committed[o + i] = s_com[i];
    accept_path[o + i] = s_path[i];
  }
}

// -------------------------------------------------------- stochastic walk

// The residual weights of a node after rejections without replacement:
// those of W except at the ny rejected tokens ys, whose weights stay frozen
// at fs (the draw's rescan and fallback read element values through here).
template <class W>
struct FrozenWeights {
  W w;
  const int32_t* ys;
  const float* fs;
  int ny;
  __device__ __forceinline__ void load8(int64_t v0, float* x) const {
    w.load8(v0, x);
    for (int i = 0; i < ny; ++i) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (v0 + j == ys[i]) x[j] = fs[i];
    }
  }
  __device__ __forceinline__ float at(int64_t v) const {
    for (int i = 0; i < ny; ++i)
      if (v == ys[i]) return fs[i];
    return w.at(v);
  }
};

// Stochastic verify in one persistent launch: the row statistics of every
// target row (the batched pass) and the walk of every request.  Work is
// taken from two queues in the workspace (zeroed before the launch): rows
// in node-major order (every request's root first, then node 1, ...; a
// child always has a larger node index than its parent, so the rows a walk
// reaches come in the order it reaches them) and requests.  A cluster walks
// one request at a time; on entering a node whose row is not done yet, one
// CTA of the cluster claims and computes that row itself if no CTA has, and
// the others compute queued rows until it is done (a waiting CTA always has
// work or waits on a row another running CTA is computing, which never
// waits, so the launch cannot deadlock; the wait is bounded all the same).  Clusters without a request left compute the
// remaining rows.  A row's statistics are published with a release store
// of its flag and read after an acquire load of it.
template <int DT, class QSrc, int C, bool WOR>
__global__ void __launch_bounds__(kWalkThreads, 512 / kWalkThreads)
    sample_verify_kernel(int B, int N, int64_t V, float c, const void* __restrict__ target,
                       float* __restrict__ m_row, float* __restrict__ z_row, int32_t* __restrict__ ready,
                       int32_t* __restrict__ queues, int32_t* __restrict__ claim, QSrc qsrc,
                       const int32_t* __restrict__ q_row, const int32_t* __restrict__ dtok,
                       const int32_t* __restrict__ ntok, const int32_t* __restrict__ nsib,
                       const float* __restrict__ coins, const float* __restrict__ u_final,
                       const int32_t* __restrict__ budget, int32_t eos, int32_t* committed,
                       int32_t* num_committed, int32_t* accept_length, int32_t* accept_path,
                       int32_t* next_root, int32_t* walk_info, int32_t* stats) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kTileW = kWalkThreads * kWalkElems;  // tile of the passes and of the draw
  using Weights = ResidualWeights<DT, typename QSrc::Row>;
  constexpr int kChunks = Weights::template chunks<kWalkElems>();
  constexpr int kRing = walk_ring_depth(kChunks);
  extern __shared__ uint4 dyn_ring[];
  uint4* ring = dyn_ring;
  float* dyn = reinterpret_cast<float*>(ring + kRing * kChunks * kWalkThreads);
  const int64_t ntiles = (V + kWalkThreads * kWalkElems - 1) / (kWalkThreads * kWalkElems);
  float* tile_sums = dyn;  // two buffers of ntiles, used by alternate passes
  float* part = tile_sums + 2 * ntiles;
  float* g_l = part + static_cast<int64_t>(cdf_part_tiles<kWalkThreads, kWalkElems, C>(V)) * kWalkThreads;
  float* g_q = g_l + N;
  float* g_u = g_q + N;
  int32_t* s_dt = reinterpret_cast<int32_t*>(g_u + N);
  int32_t* s_nt = s_dt + N;
  int32_t* s_ns = s_nt + N;
  int32_t* s_com = s_ns + N;
  int32_t* s_path = s_com + N;
  int32_t* s_ch = s_path + N;
  // without replacement: the node's rejected tokens, their frozen residual
  // weights, and per-token corrections of a pass
  int32_t* s_ry = s_ch + N;
  float* s_rf = reinterpret_cast<float*>(s_ry + N);
  float* s_rd = s_rf + N;
  // (the rejected-token arrays exist only without replacement)
  if (!spec_smem_ok(reinterpret_cast<char*>(WOR ? reinterpret_cast<int32_t*>(s_rd + N) : s_ch + N) -
                        reinterpret_cast<char*>(dyn_ring),
                    stats))
    return;
  __shared__ float scan_sh[33];
  __shared__ int s_nry, s_newy;
  __shared__ float s_S, s_wsum;
  __shared__ int s_n, s_len, s_acc, s_rej, s_kind, s_done, s_nch, s_accept, s_tiles_ok, s_rem;
  __shared__ int64_t s_qrow;
  __shared__ float s_m, s_invz, s_nb, s_A, s_cj, s_total;

  __shared__ int s_b, s_item, s_flag;
  __shared__ float sw_m[kWalkThreads / 32], sw_s[kWalkThreads / 32];

  // the C CTAs of a cluster walk request b together: each pass
  // over a row is split between them, everything else is done by each CTA
  // on the same data, so all of them take the same decisions; rank 0 alone
  // counts anomalies and writes the outputs
  const unsigned rank = C > 1 ? cluster_rank() : 0u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* const cstats = rank == 0 ? stats : nullptr;
  const int64_t rows = static_cast<int64_t>(B) * N;
  int32_t* const next_row = queues;
  int32_t* const next_req = queues + 1;
  int par = 0;  // tile-sum buffer of the next pass
  auto pass = [&](const Weights& w) -> float {
    float* ts = tile_sums + par * ntiles;
    par ^= 1;
    return cdf_tile_pass_split<kWalkThreads, kWalkElems, kRing, C>(w, V, part, ts, ring, rank);
  };
  // without replacement: the mass of the pass just made (its total `all`)
  // and its tile sums with the node's rejected tokens at their frozen
  // weights (warp 0, in list order); every CTA of a cluster does the same
  auto frozen_fix = [&](const Weights& w, float all) -> float {
    if (warp == 0) {
      float* ts = tile_sums + (par ^ 1) * ntiles;
      const int ny = s_nry;
      for (int e = lane; e < ny; e += 32) s_rd[e] = s_rf[e] - w.at(s_ry[e]);
      __syncwarp();
      if (lane == 0) {
        float W = all;
        for (int e = 0; e < ny; ++e) {
          W += s_rd[e];
          ts[s_ry[e] / kTileW] += s_rd[e];
        }
        s_wsum = W;
      }
    }
    __syncthreads();
    return s_wsum;
  };
  // queued row i (node-major): its max and normaliser, then its flag
  // row r: its max and normaliser, then its flag (the caller holds its claim)
  auto stats_row = [&](int64_t r) {
    const void* row = static_cast<const char*>(target) + r * V * esz;
    RowStatVisitor<DT, true> v{c, neg_inf(), 0.0f, 0.0f, INT_MAX, 0.0f};
    {
      // the walk's copy ring (idle here): kRing * kChunks 16-byte copies in
      // flight per thread, in the visiting order of for_row_fast
      constexpr int kv = Logit<DT>::kVec;
      const RowSpan sp = row_span<DT>(row, V);
      const int head = static_cast<int>(sp.head), nvec = static_cast<int>(sp.nvec);
      if (tid < head) v.visit1(Logit<DT>::load1(row, tid), tid, true);
      const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
      ring_stream<kWalkThreads, kRing * kChunks>(
          vp, nvec, ring, [&](const uint4& x, int i) { v.visit_vec(x, head + static_cast<int64_t>(i) * kv, true); });
      const int64_t t = head + static_cast<int64_t>(nvec) * kv + tid;
      if (t < V) v.visit1(Logit<DT>::load1(row, t), t, true);
    }
    float m = v.m, sum = v.s0 + v.s1;
    warp_merge_ms(m, sum, c);
    if (lane == 0) {
      sw_m[warp] = m;
      sw_s[warp] = sum;
    }
    __syncthreads();
    m = sw_m[0];
    sum = sw_s[0];
#pragma unroll
    for (int w2 = 1; w2 < kWalkThreads / 32; ++w2) merge_ms(m, sum, sw_m[w2], sw_s[w2], c);
    if (isfinite(m) && !isfinite(sum)) {
      // the row holds a NaN: the normaliser again with NaN as -inf
      KeyedSum ks{c, m * c, 0.0f};
      for_row<DT, 2>(row, V, ks, tid, kWalkThreads);
      const float part_s = warp_sum(ks.s);
      __syncthreads();
      if (lane == 0) sw_s[warp] = part_s;
      __syncthreads();
      sum = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < kWalkThreads / 32; ++w2) sum += sw_s[w2];
    }
    if (tid == 0) {
      if (!isfinite(m)) bump(stats, SPEC_STAT_NONFINITE_ROW);
      if (spec_in(r, rows, stats)) {
        m_row[r] = m;
        z_row[r] = sum;
        st_release_gpu(ready + r, 1);
      }
    }
    __syncthreads();  // sw_* reused by the next row
  };
  // this CTA computes queued rows until row r is done (or, with the queue
  // empty, waits for the CTA computing it).  Taking other rows while row r
  // is in flight keeps the HBM stream going; measured at the c3 sizes it
  // beats waiting idle for r.
  // Rows are claimed (an exchange on claim[r]) by the CTA that computes
  // them: queued rows in node-major order, or a row a walk needs, claimed
  // by one of the walking CTAs out of order so that the walk does not wait
  // for the queue to reach it (the others take queued rows meanwhile).
  // A claimed row is always being computed, so a wait on it ends.
  auto wait_row = [&](int64_t r) {
    for (;;) {
      if (tid == 0) {
        s_flag = ld_acquire_gpu(ready + r);
        if (s_flag) {
          s_item = 0;
        } else if (atomicExch(claim + r, 1) == 0) {
          s_item = -1;  // this CTA computes row r now
        } else {
          const int64_t i = atomicAdd(next_row, 1);
          const int64_t ri = (i % B) * N + i / B;
          s_item = i >= rows ? rows : (atomicExch(claim + ri, 1) == 0 ? ri : -2);
        }
      }
      __syncthreads();
      if (s_flag) break;
      const int64_t item = s_item;
      __syncthreads();
      if (item == -2) continue;  // that queued row was claimed by a walk
      if (item < rows) {
        stats_row(item < 0 ? r : item);
        continue;
      }
      // every row is taken: row r is in flight on a running CTA
      if (tid == 0) wait_flag(ready + r, kWaitLimitCycles, stats);
      __syncthreads();
      break;
    }
  };
  for (;;) {
  // next request of this cluster, from rank 0 to every CTA of it
  if (rank == 0 && tid == 0) {
    const int nb = atomicAdd(next_req, 1);
    if (C > 1) {
#pragma unroll
      for (int q = 0; q < C; ++q) st_cluster_i32(&s_b, q, nb);
    } else {
      s_b = nb;
    }
  }
  if (C > 1) cluster_barrier(); else __syncthreads();
  const int b = s_b;
  if (b >= B) break;
  const int64_t o = static_cast<int64_t>(b) * N;
  for (int i = tid; i < N; i += kWalkThreads) {
    s_dt[i] = __ldg(dtok + o + i);
    s_nt[i] = __ldg(ntok + o + i);
    s_ns[i] = __ldg(nsib + o + i);
    s_com[i] = -1;
    s_path[i] = -1;
  }
  if (tid == 0) {
    s_rem = budget ? __ldg(budget + b) : INT_MAX;
    s_n = 0;
    s_len = 0;
    s_acc = 0;
    s_rej = 0;
    s_kind = SPEC_FINAL_ACCEPTED;
    s_done = s_rem <= 0;
    s_path[0] = 0;
  }
  __syncthreads();
  const float cT = c;
  while (!s_done) {
    // enter node n: children in sibling order, row statistics, q row
    wait_row(o + s_n);
    if (tid == 0) {
      const int n = s_n;
      int nch = 0;
      for (int ch = s_nt[n]; ch > 0 && ch < N && nch < N; ch = s_ns[ch]) s_ch[nch++] = ch;
      s_nch = nch;
      const float z = __ldcg(z_row + o + n);
      s_m = __ldcg(m_row + o + n);
      s_invz = 1.0f / z;
      s_nb = folded_offset(s_m, c, z);
      s_qrow = q_row ? static_cast<int64_t>(__ldg(q_row + o + n)) : o + n;
      // a node with children needs its draft row (the table's row count is
      // not an argument: only the sign is checked)
      if (nch > 0 && !spec_in(s_qrow, INT64_MAX, stats)) s_qrow = -1;
      s_A = 0.0f;
      s_cj = 1.0f;
      s_tiles_ok = 0;
      s_nry = 0;
      s_S = 1.0f;
    }
    __syncthreads();
    const int n = s_n, nch = s_nch;
    const void* lrow = static_cast<const char*>(target) + (o + n) * V * esz;
    const auto qrow = qsrc.row(nch > 0 ? s_qrow : -1);
    const float mc = s_m * cT, invz = s_invz, nb = s_nb;
    const bool p_finite = isfinite(s_m);  // else p = 0 on the whole row
    for (int t = tid; t < nch; t += kWalkThreads) {
      const int ch = s_ch[t];
      const int32_t y = s_dt[ch];
      const bool ok = y >= 0 && y < V;
      g_l[t] = ok ? order_key(Logit<DT>::load1(lrow, y)) : neg_inf();
      g_q[t] = ok ? qrow.q_at(y) : 0.0f;
      g_u[t] = __ldg(coins + o + ch);
    }
    __syncthreads();
    int accepted = -1;
    for (int i = 0; i < nch; ++i) {
      if (tid == 0) {
        const float p = p_finite ? prob_of(g_l[i], cT, mc, invz) : 0.0f;
        float pc, qi = g_q[i];
        if constexpr (!WOR) {
          pc = s_A == 0.0f ? p : fmaxf(0.0f, fmaf(-s_A, g_q[i], p)) / s_cj;
        } else {
          // a token rejected before keeps its frozen weight and has no q
          // left; the others: the closed form against q renormalised over
          // the tokens not rejected (the q row taken as summing to 1)
          const int32_t y = s_dt[s_ch[i]];
          int f = -1;
          for (int e = 0; e < s_nry; ++e)
            if (s_ry[e] == y) f = e;
          const float r = f >= 0 ? s_rf[f] : (s_A == 0.0f ? p : fmaxf(0.0f, fmaf(-s_A, g_q[i], p)));
          pc = (s_A == 0.0f && s_nry == 0) ? p : r / s_cj;
          qi = (f >= 0 || !(s_S > 0.0f)) ? 0.0f : g_q[i] / s_S;
        }
        const float ratio = pc / qi;
        if (qi == 0.0f) bump(cstats, SPEC_STAT_Q_ZERO);
        s_accept = g_u[i] < ratio;
      }
      __syncthreads();
      if (s_accept) {
        accepted = s_ch[i];
        break;
      }
      // rejected: mass of the next residual
      if constexpr (!WOR) {
        const Weights w{lrow, qrow, V, cT, nb, s_A + s_cj};
        const float total = pass(w);
        if (tid == 0) {
          if (total > 0.0f && isfinite(total)) {
            s_A = s_A + s_cj;
            s_cj = total;
            s_tiles_ok = 1;
            s_total = total;
          } else {
            bump(cstats, SPEC_STAT_RESIDUAL_FALLBACK);
            s_tiles_ok = 0;
          }
          ++s_rej;
        }
        __syncthreads();
      } else {
        // without replacement: A_{j+1} = A_j + W_j / S_j (S_j the q mass not
        // yet rejected); the rejected token joins the list with its weight
        // under A_{j+1}, and q loses its mass
        const float An = s_S > 0.0f ? s_A + s_cj / s_S : s_A;
        const Weights w{lrow, qrow, V, cT, nb, An};
        const float all = pass(w);
        if (tid == 0) {
          const int32_t y = s_dt[s_ch[i]];
          bool seen = false;
          for (int e = 0; e < s_nry; ++e) seen = seen || s_ry[e] == y;
          s_newy = -1;
          if (!seen && y >= 0 && y < V && spec_in(s_nry, N, cstats)) {
            s_ry[s_nry] = y;
            s_rf[s_nry] = w.at(y);
            s_newy = s_nry++;
            s_S -= g_q[i];
          }
        }
        __syncthreads();
        const float W = frozen_fix(w, all);
        if (tid == 0) {
          if (W > 0.0f && isfinite(W)) {
            s_A = An;
            s_cj = W;
            s_tiles_ok = 1;
            s_total = W;
          } else {
            // no residual mass: p_cur stays, and so does the new token's weight
            bump(cstats, SPEC_STAT_RESIDUAL_FALLBACK);
            s_tiles_ok = 0;
            if (s_newy >= 0) s_rf[s_newy] = Weights{lrow, qrow, V, cT, nb, s_A}.at(s_ry[s_newy]);
          }
          ++s_rej;
        }
        __syncthreads();
      }
    }
    if (accepted >= 0) {
      if (tid == 0) {
        const int32_t y = s_dt[accepted];
        s_com[s_len++] = y;
        if (s_acc + 1 < N) s_path[++s_acc] = accepted;  // (links that loop cannot push the path past N)
        s_n = accepted;
        if (y == eos || s_len == s_rem || s_len >= N) {
          s_kind = SPEC_FINAL_ACCEPTED;
          s_done = 1;
        }
      }
      __syncthreads();
      continue;
    }
    // no child accepted (or a leaf): draw from the current distribution
    const Weights w{lrow, qrow, V, cT, nb, s_A};
    float total;
    if (s_tiles_ok) {
      total = s_total;  // the last pass's tile sums are in buffer par ^ 1
    } else {
      total = pass(w);
      if constexpr (WOR) total = frozen_fix(w, total);
    }
    int32_t tok = -1;
    bool drawn = false;
    if constexpr (WOR) {
      if (s_nry > 0) {
        const FrozenWeights<Weights> fw{w, s_ry, s_rf, s_nry};
        tok = cdf_search<kWalkThreads, FrozenWeights<Weights>, kWalkElems>(
            fw, V, __ldg(u_final + b), tile_sums + (par ^ 1) * ntiles, total, scan_sh, cstats);
        drawn = true;
      }
    }
    if (!drawn)
      tok = cdf_search<kWalkThreads, Weights, kWalkElems>(w, V, __ldg(u_final + b), tile_sums + (par ^ 1) * ntiles,
                                                          total, scan_sh, cstats);
    if (tid == 0) {
      s_com[s_len++] = tok;
      s_kind = nch > 0 ? SPEC_FINAL_CORRECTION : SPEC_FINAL_BONUS;
      s_done = 1;
    }
    __syncthreads();
  }
  if (rank == 0) {
    if (tid == 0) {
      num_committed[b] = s_len;
      accept_length[b] = s_acc;
      next_root[b] = s_len > 0 ? s_com[s_len - 1] : -1;
      if (walk_info) {
        walk_info[3 * b] = s_n;
        walk_info[3 * b + 1] = s_rej;
        walk_info[3 * b + 2] = s_kind;
      }
    }
    for (int i = tid; i < N; i += kWalkThreads) {
      if (!spec_in(o + i, static_cast<int64_t>(B) * N, stats)) continue;
      committed[o + i] = s_com[i];
      accept_path[o + i] = s_path[i];
    }
  }
  // every CTA of the cluster is done with this request (its shared state
  // and its stores into the others) before rank 0 hands out the next one
  if (C > 1) cluster_barrier(); else __syncthreads();
  }
  // no request left: the remaining rows
  for (;;) {
    if (tid == 0) {
      const int64_t i = atomicAdd(next_row, 1);
      const int64_t ri = (i % B) * N + i / B;
      s_item = i >= rows ? rows : (atomicExch(claim + ri, 1) == 0 ? ri : -2);
    }
    __syncthreads();
    const int64_t item = s_item;
    __syncthreads();
    if (item >= rows) break;
    if (item >= 0) stats_row(item);
  }
  if (C > 1) cluster_barrier();  // no CTA leaves while another may store into it
}

// Workspace: per-row argmax (greedy) or ready flags (stochastic, followed
// by the two work-queue counters), max and normaliser.
struct VerifyWs {
  int32_t* amax;   // greedy: argmax per row
  int32_t* ready;  // stochastic: flag per row, then next_row, next_req (same memory as amax)
  float* m;
  float* z;
  void* req;       // chain verify: per-request state (chain_ws_bytes)
};

VerifyWs carve(void* ws, int B, int N) {
  const size_t rows = static_cast<size_t>(B) * N;
  char* p = static_cast<char*>(ws);
  VerifyWs w;
  w.amax = reinterpret_cast<int32_t*>(p);
  w.ready = w.amax;
  p += align256((2 * rows + 2) * sizeof(int32_t));  // flags, the two queue counters, row claims
  w.m = reinterpret_cast<float*>(p);
  p += align256(rows * sizeof(float));
  w.z = reinterpret_cast<float*>(p);
  p += align256(rows * sizeof(float));
  w.req = p;
  return w;
}

int check_common(int B, int N, int64_t V, int dtype, const void* target, const int32_t* dtok,
                 const int32_t* ntok, const int32_t* nsib, int32_t* committed, int32_t* num_committed,
                 int32_t* accept_length, int32_t* accept_path, int32_t* next_root, void* ws, size_t ws_bytes) {
  if (B < 0 || N < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (N > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB || static_cast<int64_t>(B) * N > INT_MAX)
    return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!target || !dtok || !ntok || !nsib || !committed || !num_committed || !accept_length || !accept_path ||
      !next_root || !ws)
    return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPEC_ERR_INVALID_ARG;
  if (ws_bytes < spec_verify_ws_size(B, N)) return SPEC_ERR_WORKSPACE;
  return 1;
}

}  // namespace
}  // namespace specdec

using namespace specdec;

#ifdef SPEC_DEBUG
namespace specdec {
namespace {
std::vector<BoundsReader>& bounds_readers() {
  static std::vector<BoundsReader> r;
  return r;
}
}  // namespace
void register_bounds_reader(BoundsReader r) { bounds_readers().push_back(r); }
}  // namespace specdec
#endif

extern "C" int spec_debug_bounds(int64_t* count, int reset) {
#ifdef SPEC_DEBUG
  if (count == nullptr) return SPEC_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPEC_ERR_CUDA;
  int64_t total = 0;
  for (auto r : specdec::bounds_readers()) {
    const int rc = r(&total, reset);
    if (rc != SPEC_OK) return rc;
  }
  *count = total;
  return SPEC_OK;
#else
  (void)count;
  (void)reset;
  return SPEC_ERR_UNSUPPORTED;
#endif
}

extern "C" int spec_wait_probe(const int32_t* flag, int64_t limit_cycles, int32_t* stats, int32_t* seen,
                               spec_stream_t stream) {
  if (!flag || !seen || limit_cycles < 0) return SPEC_ERR_INVALID_ARG;
  launch_k(wait_probe_kernel, 1, 32, 0, reinterpret_cast<cudaStream_t>(stream), flag,
           static_cast<long long>(limit_cycles), stats, seen);
  return launch_status();
}

extern "C" size_t spec_verify_ws_size(int B, int N) {
  if (B < 0 || N < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * N;
  return align256((2 * rows + 2) * sizeof(int32_t)) + 2 * align256(rows * sizeof(float)) + chain_ws_bytes(B, N);
}

extern "C" int spec_verify_greedy(int B, int N, int64_t V, int dtype, const void* target_logits,
                                  const int32_t* draft_token, const int32_t* retrieve_next_token,
                                  const int32_t* retrieve_next_sibling, const int32_t* budget_or_null,
                                  int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                  int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                  int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                  size_t ws_bytes, spec_stream_t stream) {
  const int rc = check_common(B, N, V, dtype, target_logits, draft_token, retrieve_next_token,
                              retrieve_next_sibling, committed, num_committed, accept_length, accept_path,
                              next_root, ws, ws_bytes);
  if (rc <= 0) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  VerifyWs w = carve(ws, B, N);
  const int64_t rows = static_cast<int64_t>(B) * N;
  int e = dtype == SPEC_BF16
              ? launch_row_argmax<SPEC_BF16>(target_logits, V, rows, w.amax, stats_or_null, s)
              : launch_row_argmax<SPEC_F32>(target_logits, V, rows, w.amax, stats_or_null, s);
  if (e != SPEC_OK) return e;
  launch_k(greedy_walk_kernel, B, 32, sizeof(int32_t) * 6 * N, s, N, w.amax, draft_token, retrieve_next_token,
           retrieve_next_sibling, budget_or_null, eos_id, committed, num_committed, accept_length, accept_path,
           next_root, walk_info_or_null, stats_or_null);
  return launch_status();
}

namespace specdec {
namespace {

// Shared memory of the walk kernel with C CTAs per request.
// Shared memory of the verify kernel with C CTAs per request.
template <int DT, class QSrc, int C, bool WOR>
size_t walk_smem(int N, int64_t V) {
  using Weights = ResidualWeights<DT, typename QSrc::Row>;
  constexpr int kChunks = Weights::template chunks<kWalkElems>();
  const int64_t ntiles = (V + kWalkThreads * kWalkElems - 1) / (kWalkThreads * kWalkElems);
  const size_t ring = sizeof(uint4) * walk_ring_depth(kChunks) * kChunks * kWalkThreads;
  const int64_t parts = static_cast<int64_t>(cdf_part_tiles<kWalkThreads, kWalkElems, C>(V)) * kWalkThreads;
  // without replacement: the rejected-token list (ints) and two float arrays
  return ring + sizeof(float) * (2 * ntiles + parts + (WOR ? 5 : 3) * static_cast<int64_t>(N)) +
         sizeof(int32_t) * (WOR ? 7 : 6) * static_cast<int64_t>(N);
}

// Clusters of C CTAs the GPU holds at once with this shared memory, or 0
// when the kernel cannot be configured.
template <int DT, class QSrc, int C, bool WOR>
int64_t walk_capacity(size_t smem) {
  auto kernel = sample_verify_kernel<DT, QSrc, C, WOR>;
  if (smem > kMaxDynSmem) return 0;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (C == 1) {
    int dev = 0, sms = 0, per = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kWalkThreads, smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return static_cast<int64_t>(sms) * per;
  }
  LaunchCfg lc(dim3(C), dim3(kWalkThreads), smem, nullptr, C);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &lc.cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int DT, class QSrc, int C, bool WOR>
void launch_verify(int64_t clusters, size_t smem, cudaStream_t s, int B, int N, int64_t V, const void* target,
                   float c, QSrc qsrc, const int32_t* q_row, const int32_t* dtok, const int32_t* ntok,
                   const int32_t* nsib, const float* coins, const float* u_final, const int32_t* budget, int32_t eos,
                   int32_t* committed, int32_t* num_committed, int32_t* accept_length, int32_t* accept_path,
                   int32_t* next_root, int32_t* walk_info, int32_t* stats, const VerifyWs& w) {
  const int64_t rows = static_cast<int64_t>(B) * N;
  launch_kc(sample_verify_kernel<DT, QSrc, C, WOR>, static_cast<unsigned>(clusters * C), kWalkThreads, smem, s, C, B,
            N, V, c, target, w.m, w.z, w.ready, w.ready + rows, w.ready + rows + 2, qsrc, q_row, dtok, ntok, nsib, coins, u_final, budget,
            eos, committed, num_committed, accept_length, accept_path, next_root, walk_info, stats);
}

// One persistent launch (after zeroing the row flags and queue counters):
// as many clusters as the GPU holds, C CTAs each, the largest C of 4, 2, 1
// for which every request can have its cluster at once (a request's
// passes run one after another), else 1.
template <int DT, class QSrc, bool WOR>
int launch_sample_verify_t(int B, int N, int64_t V, const void* target, float c, QSrc qsrc, const int32_t* q_row,
                           const int32_t* dtok, const int32_t* ntok, const int32_t* nsib, const float* coins,
                           const float* u_final, const int32_t* budget, int32_t eos, int32_t* committed,
                           int32_t* num_committed, int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                           int32_t* walk_info, int32_t* stats, VerifyWs w, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(B) * N;
  const size_t smem4 = walk_smem<DT, QSrc, 4, WOR>(N, V), smem2 = walk_smem<DT, QSrc, 2, WOR>(N, V),
               smem1 = walk_smem<DT, QSrc, 1, WOR>(N, V);
  if (smem1 > kMaxDynSmem) return SPEC_ERR_UNSUPPORTED;  // V in the millions
  const int64_t cap4 = walk_capacity<DT, QSrc, 4, WOR>(smem4), cap2 = walk_capacity<DT, QSrc, 2, WOR>(smem2),
                cap1 = walk_capacity<DT, QSrc, 1, WOR>(smem1);
  if (cap1 < 1) return SPEC_ERR_CUDA;
  if (cudaMemsetAsync(w.ready, 0, sizeof(int32_t) * static_cast<size_t>(2 * rows + 2), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cap4 >= B)
    launch_verify<DT, QSrc, 4, WOR>(cap4, smem4, s, B, N, V, target, c, qsrc, q_row, dtok, ntok, nsib, coins, u_final,
                               budget, eos, committed, num_committed, accept_length, accept_path, next_root,
                               walk_info, stats, w);
  else if (cap2 >= 1)  // pairs also when they take several requests each (B=1024 x 16: 708 vs 730 us alone)
    launch_verify<DT, QSrc, 2, WOR>(cap2, smem2, s, B, N, V, target, c, qsrc, q_row, dtok, ntok, nsib, coins, u_final,
                               budget, eos, committed, num_committed, accept_length, accept_path, next_root,
                               walk_info, stats, w);
  else
    launch_verify<DT, QSrc, 1, WOR>(cap1, smem1, s, B, N, V, target, c, qsrc, q_row, dtok, ntok, nsib, coins, u_final,
                               budget, eos, committed, num_committed, accept_length, accept_path, next_root,
                               walk_info, stats, w);
  return launch_status();
}

template <int DT, class QSrc>
int launch_sample_verify(int B, int N, int64_t V, const void* target, float c, QSrc qsrc, const int32_t* q_row,
                         const int32_t* dtok, const int32_t* ntok, const int32_t* nsib, const float* coins,
                         const float* u_final, const int32_t* budget, int32_t eos, int32_t* committed,
                         int32_t* num_committed, int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                         int32_t* walk_info, int32_t* stats, VerifyWs w, int wor, cudaStream_t s) {
  return wor ? launch_sample_verify_t<DT, QSrc, true>(B, N, V, target, c, qsrc, q_row, dtok, ntok, nsib, coins,
                                                      u_final, budget, eos, committed, num_committed, accept_length,
                                                      accept_path, next_root, walk_info, stats, w, s)
             : launch_sample_verify_t<DT, QSrc, false>(B, N, V, target, c, qsrc, q_row, dtok, ntok, nsib, coins,
                                                       u_final, budget, eos, committed, num_committed,
                                                       accept_length, accept_path, next_root, walk_info, stats, w,
                                                       s);
}

}  // namespace
}  // namespace specdec

namespace {
int verify_sample_impl(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                  const float* q, const int32_t* q_row_or_null, const int32_t* draft_token,
                                  const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                  const float* coins, const float* u_final, const int32_t* budget_or_null,
                                  int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                  int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                  int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                  size_t ws_bytes, int flags, spec_stream_t stream) {
  if (!(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if ((flags & ~(SPEC_VERIFY_WITHOUT_REPLACEMENT | SPEC_VERIFY_CHAIN)) != 0) return SPEC_ERR_INVALID_ARG;
  const int wor = (flags & SPEC_VERIFY_WITHOUT_REPLACEMENT) ? 1 : 0;
  const int rc = check_common(B, N, V, dtype, target_logits, draft_token, retrieve_next_token,
                              retrieve_next_sibling, committed, num_committed, accept_length, accept_path,
                              next_root, ws, ws_bytes);
  if (rc <= 0) return rc;
  if (!q || !coins || !u_final) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  if (flags & SPEC_VERIFY_CHAIN) {
    // one child per node: without replacement is the same rule
    const VerifyWs w = carve(ws, B, N);
    const ChainIO io{q_row_or_null, draft_token, retrieve_next_token, retrieve_next_sibling, coins, u_final,
                     budget_or_null, eos_id, committed, num_committed, accept_length, accept_path, next_root,
                     walk_info_or_null, stats_or_null, nullptr, 0, -1, nullptr};
    return chain_verify(dtype, B, N, V, target_logits, c, ChainQ{0, q, nullptr, 0.0f}, io, w.ready, w.m, w.z, w.req,
                        s);
  }
  const QProbs qs{q, V};
  if (dtype == SPEC_BF16)
    return launch_sample_verify<SPEC_BF16>(B, N, V, target_logits, c, qs, q_row_or_null, draft_token,
                                           retrieve_next_token, retrieve_next_sibling, coins, u_final,
                                           budget_or_null, eos_id, committed, num_committed, accept_length,
                                           accept_path, next_root, walk_info_or_null, stats_or_null,
                                           carve(ws, B, N), wor, s);
  return launch_sample_verify<SPEC_F32>(B, N, V, target_logits, c, qs, q_row_or_null, draft_token,
                                        retrieve_next_token, retrieve_next_sibling, coins, u_final, budget_or_null,
                                        eos_id, committed, num_committed, accept_length, accept_path, next_root,
                                        walk_info_or_null, stats_or_null, carve(ws, B, N), wor, s);
}
}  // namespace

extern "C" int spec_verify_sample(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                  const float* q, const int32_t* q_row_or_null, const int32_t* draft_token,
                                  const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                  const float* coins, const float* u_final, const int32_t* budget_or_null,
                                  int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                  int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                  int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                  size_t ws_bytes, spec_stream_t stream) {
  return verify_sample_impl(B, N, V, dtype, target_logits, T, q, q_row_or_null, draft_token, retrieve_next_token,
                            retrieve_next_sibling, coins, u_final, budget_or_null, eos_id, committed, num_committed,
                            accept_length, accept_path, next_root, walk_info_or_null, stats_or_null, ws, ws_bytes, 0,
                            stream);
}

extern "C" int spec_verify_sample_flags(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                        const float* q, const int32_t* q_row_or_null, const int32_t* draft_token,
                                        const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                        const float* coins, const float* u_final, const int32_t* budget_or_null,
                                        int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                        int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                        int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                        size_t ws_bytes, int flags, spec_stream_t stream) {
  return verify_sample_impl(B, N, V, dtype, target_logits, T, q, q_row_or_null, draft_token, retrieve_next_token,
                            retrieve_next_sibling, coins, u_final, budget_or_null, eos_id, committed, num_committed,
                            accept_length, accept_path, next_root, walk_info_or_null, stats_or_null, ws, ws_bytes,
                            flags, stream);
}

namespace specdec {
namespace {

template <int DT, int QDT>
int sample_verify_qlogits(int B, int N, int64_t V, const void* target, float c, const void* q_logits,
                          const float* q_stats, float cq, const int32_t* q_row, const int32_t* dtok,
                          const int32_t* ntok, const int32_t* nsib, const float* coins, const float* u_final,
                          const int32_t* budget, int32_t eos, int32_t* committed, int32_t* num_committed,
                          int32_t* accept_length, int32_t* accept_path, int32_t* next_root, int32_t* walk_info,
                          int32_t* stats, VerifyWs w, int wor, cudaStream_t s) {
  const QLogits<QDT> qs{q_logits, q_stats, V, cq};
  return launch_sample_verify<DT>(B, N, V, target, c, qs, q_row, dtok, ntok, nsib, coins, u_final, budget, eos,
                                  committed, num_committed, accept_length, accept_path, next_root, walk_info, stats,
                                  w, wor, s);
}

}  // namespace
}  // namespace specdec

namespace {
int verify_sample_qlogits_impl(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                          const void* q_logits, int q_dtype, const float* q_stats, float T_q,
                                          const int32_t* q_row_or_null, const int32_t* draft_token,
                                          const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                          const float* coins, const float* u_final, const int32_t* budget_or_null,
                                          int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                          int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                          int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                          size_t ws_bytes, int flags, const spec_id_map_t* map,
                                          spec_stream_t stream) {
  if (!(T > 0.0f) || !isfinite(T) || !(T_q > 0.0f) || !isfinite(T_q)) return SPEC_ERR_INVALID_ARG;
  if ((flags & ~(SPEC_VERIFY_WITHOUT_REPLACEMENT | SPEC_VERIFY_CHAIN)) != 0) return SPEC_ERR_INVALID_ARG;
  if (map != nullptr && (!(flags & SPEC_VERIFY_CHAIN) || map->table == nullptr || map->table_len < 1 ||
                         map->out == nullptr))
    return SPEC_ERR_INVALID_ARG;
  const int wor = (flags & SPEC_VERIFY_WITHOUT_REPLACEMENT) ? 1 : 0;
  const int rc = check_common(B, N, V, dtype, target_logits, draft_token, retrieve_next_token,
                              retrieve_next_sibling, committed, num_committed, accept_length, accept_path,
                              next_root, ws, ws_bytes);
  if (rc <= 0) return rc;
  if (!q_logits || !q_stats || !coins || !u_final) return SPEC_ERR_INVALID_ARG;
  if (q_dtype != SPEC_F32 && q_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T, cq = kLog2e / T_q;
  const VerifyWs w = carve(ws, B, N);
  if (flags & SPEC_VERIFY_CHAIN) {
    const ChainIO io{q_row_or_null, draft_token, retrieve_next_token, retrieve_next_sibling, coins, u_final,
                     budget_or_null, eos_id, committed, num_committed, accept_length, accept_path, next_root,
                     walk_info_or_null, stats_or_null,
                     map ? map->table : nullptr, map ? map->table_len : 0, map ? map->fallback_id : -1,
                     map ? map->out : nullptr};
    return chain_verify(dtype, B, N, V, target_logits, c, ChainQ{q_dtype == SPEC_BF16 ? 1 : 2, q_logits, q_stats, cq},
                        io, w.ready, w.m, w.z, w.req, s);
  }
#define SPEC_QL(DT, QDT)                                                                                         \
  return sample_verify_qlogits<DT, QDT>(B, N, V, target_logits, c, q_logits, q_stats, cq, q_row_or_null,        \
                                        draft_token, retrieve_next_token, retrieve_next_sibling, coins, u_final, \
                                        budget_or_null, eos_id, committed, num_committed, accept_length,         \
                                        accept_path, next_root, walk_info_or_null, stats_or_null, w, wor, s)
  if (dtype == SPEC_BF16) {
    if (q_dtype == SPEC_BF16) SPEC_QL(SPEC_BF16, SPEC_BF16);
    SPEC_QL(SPEC_BF16, SPEC_F32);
  }
  if (q_dtype == SPEC_BF16) SPEC_QL(SPEC_F32, SPEC_BF16);
  SPEC_QL(SPEC_F32, SPEC_F32);
#undef SPEC_QL
}
}  // namespace

extern "C" int spec_verify_sample_qlogits(int B, int N, int64_t V, int dtype, const void* target_logits, float T,
                                          const void* q_logits, int q_dtype, const float* q_stats, float T_q,
                                          const int32_t* q_row_or_null, const int32_t* draft_token,
                                          const int32_t* retrieve_next_token, const int32_t* retrieve_next_sibling,
                                          const float* coins, const float* u_final, const int32_t* budget_or_null,
                                          int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                          int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                          int32_t* walk_info_or_null, int32_t* stats_or_null, void* ws,
                                          size_t ws_bytes, spec_stream_t stream) {
  return verify_sample_qlogits_impl(B, N, V, dtype, target_logits, T, q_logits, q_dtype, q_stats, T_q, q_row_or_null,
                                    draft_token, retrieve_next_token, retrieve_next_sibling, coins, u_final,
                                    budget_or_null, eos_id, committed, num_committed, accept_length, accept_path,
                                    next_root, walk_info_or_null, stats_or_null, ws, ws_bytes, 0, nullptr, stream);
}

extern "C" int spec_verify_sample_qlogits_flags(int B, int N, int64_t V, int dtype, const void* target_logits,
                                                float T, const void* q_logits, int q_dtype, const float* q_stats,
                                                float T_q, const int32_t* q_row_or_null, const int32_t* draft_token,
                                                const int32_t* retrieve_next_token,
                                                const int32_t* retrieve_next_sibling, const float* coins,
                                                const float* u_final, const int32_t* budget_or_null, int32_t eos_id,
                                                int32_t* committed, int32_t* num_committed, int32_t* accept_length,
                                                int32_t* accept_path, int32_t* next_root, int32_t* walk_info_or_null,
                                                int32_t* stats_or_null, void* ws, size_t ws_bytes, int flags,
                                                spec_stream_t stream) {
  return verify_sample_qlogits_impl(B, N, V, dtype, target_logits, T, q_logits, q_dtype, q_stats, T_q, q_row_or_null,
                                    draft_token, retrieve_next_token, retrieve_next_sibling, coins, u_final,
                                    budget_or_null, eos_id, committed, num_committed, accept_length, accept_path,
                                    next_root, walk_info_or_null, stats_or_null, ws, ws_bytes, flags, nullptr,
                                    stream);
}

extern "C" int spec_verify_sample_qlogits_mapped(int B, int N, int64_t V, int dtype, const void* target_logits,
                                                 float T, const void* q_logits, int q_dtype, const float* q_stats,
                                                 float T_q, const int32_t* q_row_or_null, const int32_t* draft_token,
                                                 const int32_t* retrieve_next_token,
                                                 const int32_t* retrieve_next_sibling, const float* coins,
                                                 const float* u_final, const int32_t* budget_or_null, int32_t eos_id,
                                                 int32_t* committed, int32_t* num_committed, int32_t* accept_length,
                                                 int32_t* accept_path, int32_t* next_root, int32_t* walk_info_or_null,
                                                 int32_t* stats_or_null, void* ws, size_t ws_bytes, int flags,
                                                 const spec_id_map_t* map, spec_stream_t stream) {
  if (map == nullptr) return SPEC_ERR_INVALID_ARG;
  return verify_sample_qlogits_impl(B, N, V, dtype, target_logits, T, q_logits, q_dtype, q_stats, T_q, q_row_or_null,
                                    draft_token, retrieve_next_token, retrieve_next_sibling, coins, u_final,
                                    budget_or_null, eos_id, committed, num_committed, accept_length, accept_path,
                                    next_root, walk_info_or_null, stats_or_null, ws, ws_bytes, flags, map, stream);
}

// ------------------------------------------------- greedy verify, no scratch
//
// For callers that cannot allocate: the per-row argmax lives in this fixed
// array (SPEC_NOALLOC_MAX_ROWS entries) instead of caller scratch.  Host code
// may not use the array's name as a device pointer; its device address is
// looked up once per device with cudaGetSymbolAddress and cached.
#include <atomic>
#include <mutex>

namespace specdec {
namespace {

__device__ __align__(256) int32_t g_noalloc_argmax[SPEC_NOALLOC_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::atomic<int32_t*> g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of g_noalloc_argmax on the current device (nullptr on error).
int32_t* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int32_t* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_argmax) != cudaSuccess || addr == nullptr) return nullptr;
    p = static_cast<int32_t*>(addr);
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace
}  // namespace specdec

extern "C" int spec_verify_greedy_noalloc(int B, int N, int64_t V, int dtype, const void* target_logits,
                                          const int32_t* draft_token, const int32_t* retrieve_next_token,
                                          const int32_t* retrieve_next_sibling, const int32_t* budget_or_null,
                                          int32_t eos_id, int32_t* committed, int32_t* num_committed,
                                          int32_t* accept_length, int32_t* accept_path, int32_t* next_root,
                                          int32_t* walk_info_or_null, int32_t* stats_or_null,
                                          spec_stream_t stream) {
  if (B < 0 || N < 1 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (N > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB || static_cast<int64_t>(B) * N > SPEC_NOALLOC_MAX_ROWS)
    return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !draft_token || !retrieve_next_token || !retrieve_next_sibling || !committed ||
      !num_committed || !accept_length || !accept_path || !next_root)
    return SPEC_ERR_INVALID_ARG;
  int32_t* amax = noalloc_scratch();
  if (amax == nullptr) return SPEC_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t rows = static_cast<int64_t>(B) * N;
  int e = dtype == SPEC_BF16
              ? launch_row_argmax<SPEC_BF16>(target_logits, V, rows, amax, stats_or_null, s)
              : launch_row_argmax<SPEC_F32>(target_logits, V, rows, amax, stats_or_null, s);
  if (e != SPEC_OK) return e;
  launch_k(greedy_walk_kernel, B, 32, sizeof(int32_t) * 6 * N, s, N, amax, draft_token, retrieve_next_token,
           retrieve_next_sibling, budget_or_null, eos_id, committed, num_committed, accept_length, accept_path,
           next_root, walk_info_or_null, stats_or_null);
  return launch_status();
}
