// Stochastic verification of chains in one persistent launch.
//
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)":
//   3.3  row L-1+i of the target output verifies draft i -- here target row
//        (b, n) verifies node n's child, and a leaf's row gives the bonus;
//   5.1  a draft y drawn from q is accepted with min(1, p[y]/q[y]); at the
//        first rejection the token is drawn from the normalised positive
//        residual (p - q)+; after full acceptance the bonus is drawn from p.
//
// In a chain every node has one child, so the acceptance test at node n
// needs only row n's statistics, q row n and the child's coin: it does not
// depend on the walk.  The launch takes target rows from a node-major queue
// (each row streamed once through the CTA's copy ring) and computes, with
// the row's max and normaliser, the test of its child at once.  A request
// is resolved as soon as the rows on its path are done: at its first
// rejected node, at its leaf, or at a stop (EOS, budget).  Its one draw --
// the residual after the rejection, or p at the leaf -- is a pass over the
// row cut into chunks of whole tiles; each chunk is a work item any CTA may
// take, and the CTA that completes a request's last chunk searches its
// inverse CDF (chunk totals, then the crossing chunk's tiles, then one tile
// with a block scan).  CTAs take draw items before rows, so requests finish
// while the batched pass is still streaming.
//
// Every decision takes the same fp32 operations as the tree walk of
// verify.cu (acceptance ratio, residual weights, inverse CDF over tile
// sums); only the order in which tile sums are added differs (by chunk).
#include "chain.h"

#include <climits>

#include "walk.cuh"

namespace specdec {
namespace {

constexpr int kCT = kWalkThreads;  // threads of a CTA
constexpr int kCE = kWalkElems;    // consecutive elements per thread in a tile
constexpr int kTile = kCT * kCE;
constexpr int kRingItems = 16;     // 16-byte copies in flight per thread (row statistics)
constexpr int kMaxChunks = 64;     // draw items per request, at most
constexpr int kMinChunkTiles = 4;
constexpr int kMaxChunkTiles = 32;  // (SPEC_MAX_VOCAB / kTile) / kMaxChunks
constexpr int kBatch = 4;           // tiles whose loads a chunk pass issues together
constexpr int kCounters = 8;

// row flag bits (a row's flag is published with them after its statistics)
constexpr int kRowDone = 1, kRowAccept = 2, kRowQZero = 4, kRowLeaf = 8, kRowMulti = 16;

__host__ __device__ inline int chunk_tiles(int64_t ntiles) {
  const int64_t t = (ntiles + kMaxChunks - 1) / kMaxChunks;
  return t < kMinChunkTiles ? kMinChunkTiles : static_cast<int>(t);
}

struct ChainParams {
  int B, N;
  int64_t V;
  float c;
  const void* target;
  ChainIO io;
  int32_t* ready;
  float* m_row;
  float* z_row;
  // per-request workspace
  int32_t* cnt;  // [0] next row, [1] draw items claimed, [2] slots reserved, [3] requests resolved
  int32_t *state, *done, *slot_req, *slot_ready, *node, *len, *kind, *rows_done;
  int32_t* front;  // per request: len * 4096 + node of the deepest accepted node seen with every row before it done
  float* A;     // 0: draw from p (bonus), 1: from the residual after one rejection
  float* ctot;  // [B][kMaxChunks] chunk totals of the draw
  int ntiles, tpc, nchunks;
};

__device__ __forceinline__ int ld_volatile(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }

// Read-modify-writes at GPU scope.  acq_rel: the update is ordered after
// this thread's earlier writes and before its later reads; two threads'
// updates of one word are ordered, so the later one sees what the earlier
// one published.  release: ordered after this thread's earlier writes.
__device__ __forceinline__ int atom_add_acq_rel(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void atom_add_release(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Draw items are numbered slot * nchunks + chunk in the order slots are
// reserved, and claimed with one atomic add on a single counter (no
// retries).  A claim may run ahead of the reservations; the claimer then
// holds it until its slot is reserved, or drops it once every request is
// resolved without that slot.

// The committed id y through the caller's map ([TLI] Modifications,
// map_target_to_draft_ids: unmapped ids take the fallback id).
__device__ __forceinline__ int32_t mapped_id(const ChainIO& io, int32_t y) {
  return (y >= 0 && y < io.map_len && __ldg(io.map_table + y) >= 0) ? __ldg(io.map_table + y) : io.map_fallback;
}

// Returns true when the caller (the CTA that finished row `row_node` of b,
// allowed by `here_ok`) is to draw the request itself: it resolved here, at
// that very row.
__device__ bool try_resolve(const ChainParams& p, int b, int row_node, bool here_ok) {
  if (ld_acquire_gpu(p.state + b) != 0) return false;
  const ChainIO& io = p.io;
  const int N = p.N;
  const int64_t o = static_cast<int64_t>(b) * N;
  const int rem = io.budget ? __ldg(io.budget + b) : INT_MAX;
  // resume from the deepest accepted node an earlier attempt reached
  const int fr = ld_volatile(p.front + b);
  int n = fr & 4095, len = fr >> 12, kind = SPEC_FINAL_ACCEPTED, multi = 0;
  float A = -1.0f;  // no draw
  if (rem > 0 && !(len > 0 && len >= rem)) {
    for (;;) {
      const int f = ld_acquire_gpu(p.ready + o + n);
      if (!(f & kRowDone)) {
        // a row on the path is not done: its CTA resolves later
        if (len > (fr >> 12)) atomicMax(p.front + b, len * 4096 + n);
        return false;
      }
      multi |= f & kRowMulti;
      if (f & kRowLeaf) {
        A = 0.0f;
        kind = SPEC_FINAL_BONUS;
        break;
      }
      // a chain of N nodes reaches its leaf after N - 1 accepted drafts; a
      // longer walk (links that loop) stops here, so every index stays below N
      if (len >= N - 1) break;
      if (!(f & kRowAccept)) {
        A = 1.0f;
        kind = SPEC_FINAL_CORRECTION;
        break;
      }
      const int ch = __ldg(io.ntok + o + n);
      const int32_t y = __ldg(io.dtok + o + ch);
      ++len;
      n = ch;
      if (y == io.eos || len == rem) break;
    }
  }
  if (atomicCAS(p.state + b, 0, 1) != 0) return false;  // another CTA resolved it
  // the owner walks the path once more for the outputs and the q[y] = 0
  // tests on it (the rows on it are done and visible)
  int node = 0, qz = 0, multi2 = 0;
  io.accept_path[o] = 0;
  for (int i = 0; i < N; ++i) {
    if (i < len) {
      const int f = ld_acquire_gpu(p.ready + o + node);
      qz += (f & kRowQZero) ? 1 : 0;
      multi2 |= f & kRowMulti;
      const int ch = __ldg(io.ntok + o + node);
      const int32_t y = __ldg(io.dtok + o + ch);
      io.committed[o + i] = y;
      if (io.committed_mapped) io.committed_mapped[o + i] = mapped_id(io, y);
      io.accept_path[o + i + 1] = ch;
      node = ch;
    } else {
      io.committed[o + i] = -1;
      if (io.committed_mapped) io.committed_mapped[o + i] = -1;
      if (i + 1 < N) io.accept_path[o + i + 1] = -1;
    }
  }
  if (kind == SPEC_FINAL_CORRECTION && (ld_acquire_gpu(p.ready + o + n) & kRowQZero)) ++qz;  // the rejected test
  if (qz) bump(io.stats, SPEC_STAT_Q_ZERO, qz);
  if (multi | multi2) bump(io.stats, SPEC_STAT_BAD_REQUEST);
  if (A < 0.0f) {
    io.num_committed[b] = len;
    io.accept_length[b] = len;
    io.next_root[b] = len > 0 ? io.committed[o + len - 1] : -1;
    if (io.walk_info) {
      io.walk_info[3 * b] = n;
      io.walk_info[3 * b + 1] = 0;
      io.walk_info[3 * b + 2] = SPEC_FINAL_ACCEPTED;
    }
    atom_add_release(p.cnt + 3, 1);
    return false;
  }
  p.node[b] = n;
  p.len[b] = len;
  p.kind[b] = kind;
  p.A[b] = A;
  if (here_ok && n == row_node) {
    atom_add_release(p.cnt + 3, 1);  // resolved; this CTA draws it
    return true;
  }
  const int k = atomicAdd(p.cnt + 2, 1);  // a draw slot; its items become takeable now
  p.slot_req[k] = b;
  st_release_gpu(p.slot_ready + k, 1);     // publishes node, len, kind, A and the slot
  atom_add_release(p.cnt + 3, 1);          // after the reservation: whoever sees every request resolved sees the slot
  return false;
}

template <int DT, class QSrc>
__global__ void __launch_bounds__(kCT, 4) chain_verify_kernel(const ChainParams p, const QSrc qsrc) {
  pdl_enter();
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4, kWarps = kCT / 32;
  using Weights = ResidualWeights<DT, typename QSrc::Row>;
  extern __shared__ uint4 ring[];  // kRingItems * kCT slots, then the in-place draw's partials and tile sums
  float* part = reinterpret_cast<float*>(ring + kRingItems * kCT);
  float* tsum = part + cdf_part_tiles<kCT, kCE, 1>(p.V) * kCT;
  __shared__ float sw_m[kWarps], sw_s[kWarps];
  __shared__ float red[kBatch][kWarps];  // tile sums of a chunk pass, by warp
  __shared__ float tile_sh[kMaxChunkTiles];
  __shared__ float ctot_sh[kMaxChunks];
  __shared__ float scan_sh[33];
  __shared__ float s_tot, s_A;
  __shared__ int s_what, s_item, s_last, s_tok, s_b, s_n, s_here;
  const ChainIO& io = p.io;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B, N = p.N;
  const int64_t V = p.V, rows = static_cast<int64_t>(B) * N;
  const float c = p.c;
  long long idle0 = 0;
  bool idle = false;
  int pend = -1;  // thread 0: a claimed draw item whose slot is not reserved yet

  // tile sums of chunk j of a draw row into tile_sh (thread 0), their total
  // in tile order to every thread.  Each thread copies its elements of D
  // tiles at once into its slots of the copy ring (D = what the ring holds
  // at this operand width), then sums them; rows that are not 16-byte
  // aligned take direct loads.
  constexpr int K = Weights::template chunks<kCE>();
  constexpr int D = kRingItems / K < 1 ? 1 : (kRingItems / K > kBatch ? kBatch : kRingItems / K);
  auto chunk_pass = [&](const Weights& w, int j) -> float {
    const int t0 = j * p.tpc, t1 = min(p.ntiles, t0 + p.tpc);
    const bool rg = w.ring_ok();
    uint4* mine = ring + tid;
    float tot = 0.0f;
    for (int t = t0; t < t1; t += D) {
      float ps[D];
      if (rg) {
#pragma unroll
        for (int u = 0; u < D; ++u)
          if (t + u < t1) w.template issue<kCE>(mine + u * K * kCT, kCT, static_cast<int64_t>(t + u) * kTile + tid * kCE);
        cp_async_commit();
        cp_async_wait<0>();
#pragma unroll
        for (int u = 0; u < D; ++u)
          ps[u] = t + u < t1 ? w.template ring_sum<kCE>(mine + u * K * kCT, kCT,
                                                         static_cast<int64_t>(t + u) * kTile + tid * kCE)
                             : 0.0f;
      } else {
#pragma unroll
        for (int u = 0; u < D; ++u)
          ps[u] = t + u < t1 ? w.template load_sum<kCE>(static_cast<int64_t>(t + u) * kTile + tid * kCE) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < D; ++u) {
        const float s = warp_sum(ps[u]);
        if (lane == 0) red[u][warp] = s;
      }
      __syncthreads();
      if (tid == 0) {
        for (int u = 0; u < D && t + u < t1; ++u) {
          float ts = 0.0f;
#pragma unroll
          for (int w2 = 0; w2 < kWarps; ++w2) ts += red[u][w2];
          tile_sh[t + u - t0] = ts;
          tot += ts;
        }
      }
      __syncthreads();
    }
    if (tid == 0) s_tot = tot;
    __syncthreads();
    const float r = s_tot;
    __syncthreads();
    return r;
  };

  // the first element of tile t whose running prefix (from `prefix`)
  // exceeds target, into s_tok by atomicMin (INT_MAX stays if none)
  auto rescan_tile = [&](const Weights& w, int t, float prefix, float target) {
    const int64_t v0 = static_cast<int64_t>(t) * kTile + tid * kCE;
    float x[kCE];
#pragma unroll
    for (int g = 0; g < kCE / 8; ++g) w.load8(v0 + 8 * g, x + 8 * g);
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < kCE; ++j) sum += x[j];
    float tot;
    const float incl = block_inclusive_scan(sum, scan_sh, tot);
    float C = prefix + (incl - sum);
    int found = -1;
#pragma unroll
    for (int j = 0; j < kCE; ++j) {
      C += x[j];
      if (found < 0 && C > target && v0 + j < V) found = j;
    }
    if (found >= 0) atomicMin(&s_tok, static_cast<int>(v0 + found));
    __syncthreads();
  };

  // the last outputs of request b, drawn token tok at node n (thread 0)
  auto write_draw = [&](int b, int n, int tok) {
    const int64_t o = static_cast<int64_t>(b) * N;
    const int len = __ldcg(p.len + b), kind = __ldcg(p.kind + b);
    io.committed[o + len] = tok;
    if (io.committed_mapped) io.committed_mapped[o + len] = mapped_id(io, tok);
    io.num_committed[b] = len + 1;
    io.accept_length[b] = len;
    io.next_root[b] = tok;
    if (io.walk_info) {
      io.walk_info[3 * b] = n;
      io.walk_info[3 * b + 1] = kind == SPEC_FINAL_CORRECTION ? 1 : 0;
      io.walk_info[3 * b + 2] = kind;
    }
  };

  // the inverse-CDF draw of request b at node n from the chunk totals in
  // ctot_sh (every CTA takes the same operations in the same order), then
  // the request's last outputs
  auto finish_draw = [&](int b, int n, Weights w) {
    if (tid == 0) s_tok = INT_MAX;
    __syncthreads();
    float W = 0.0f;
    for (int q = 0; q < p.nchunks; ++q) W += ctot_sh[q];
    if (w.A != 0.0f && !(W > 0.0f && isfinite(W))) {
      // no residual mass: the draw is from p itself (counted)
      if (tid == 0) bump(io.stats, SPEC_STAT_RESIDUAL_FALLBACK);
      w.A = 0.0f;
      for (int q = 0; q < p.nchunks; ++q) {
        const float t = chunk_pass(w, q);
        if (tid == 0) ctot_sh[q] = t;
      }
      __syncthreads();
      W = 0.0f;
      for (int q = 0; q < p.nchunks; ++q) W += ctot_sh[q];
    }
    const float target = __ldg(io.u_final + b) * W;
    if (W > 0.0f && isfinite(W)) {
      float prefix = 0.0f;
      for (int q = 0; q < p.nchunks; ++q) {
        const float after = prefix + ctot_sh[q];
        if (!(after > target)) {
          prefix = after;
          continue;
        }
        chunk_pass(w, q);  // the chunk's tile sums again, as its pass made them
        const int t0 = q * p.tpc, nt = min(p.ntiles, t0 + p.tpc) - t0;
        for (int i = 0; i < nt; ++i) {
          const float a2 = prefix + tile_sh[i];
          if (a2 > target) {
            rescan_tile(w, t0 + i, prefix, target);
            if (s_tok != INT_MAX) break;
          }
          prefix = a2;
        }
        if (s_tok != INT_MAX) break;
      }
    }
    __syncthreads();
    if (s_tok == INT_MAX) {
      // rounding left no crossing (or no mass): the last index of positive weight
      __syncthreads();
      if (tid == 0) s_tok = -1;
      __syncthreads();
      for (int64_t v = tid; v < V; v += kCT)
        if (w.at(v) > 0.0f) atomicMax(&s_tok, static_cast<int>(v));
      __syncthreads();
      if (tid == 0) {
        if (s_tok < 0) s_tok = 0;
        bump(io.stats, SPEC_STAT_CDF_FALLBACK);
      }
    }
    __syncthreads();
    if (tid == 0) write_draw(b, n, s_tok);
    __syncthreads();
  };

  // the weights a request's draw reads: the residual at a rejected node
  // (A = 1), or p at a leaf (A = 0)
  auto draw_weights = [&](int b, int n, float A) -> Weights {
    const int64_t rr = static_cast<int64_t>(b) * N + n;
    const void* row = static_cast<const char*>(p.target) + rr * V * esz;
    const float m = __ldcg(p.m_row + rr), z = __ldcg(p.z_row + rr);
    const auto qrow = qsrc.row(A != 0.0f ? (io.q_row ? static_cast<int64_t>(__ldg(io.q_row + rr)) : rr) : -1);
    return Weights{row, qrow, V, c, folded_offset(m, c, z), A};
  };

  for (;;) {
    if (tid == 0) {
      // rows first: the batched pass is the critical path; then draw items
      int what = 3, item = 0;
      const int r = ld_volatile(p.cnt) < rows ? atomicAdd(p.cnt, 1) : static_cast<int>(rows);
      if (r < rows) {
        what = 2;
        item = r;
      } else {
        // read first: if every request was resolved by then, the reserved
        // slots are final
        const bool all_resolved = ld_acquire_gpu(p.cnt + 3) >= B;
        const int reserved = ld_acquire_gpu(p.cnt + 2);
        if (pend < 0 && ld_volatile(p.cnt + 1) < reserved * p.nchunks) pend = atomicAdd(p.cnt + 1, 1);
        if (pend >= 0 && pend / p.nchunks < reserved) {
          what = 1;
          item = pend;
          pend = -1;
        } else if (all_resolved) {
          pend = -1;  // its slot will never be reserved
          if (ld_volatile(p.cnt + 1) >= reserved * p.nchunks) what = 0;
        }
        if (what == 3) {
          // nothing to take yet: rows or resolutions are in flight on
          // running CTAs, which never wait; bounded all the same
          if (!idle) {
            idle = true;
            idle0 = clock64();
          } else if (clock64() - idle0 > kWaitLimitCycles) {
            bump(io.stats, SPEC_STAT_WAIT_TIMEOUT);
            what = 0;
          }
          if (what != 0) __nanosleep(256);
        }
      }
      if (what == 1 || what == 2) idle = false;
      s_what = what;
      s_item = item;
    }
    __syncthreads();
    const int what = s_what, item = s_item;
    __syncthreads();
    if (what == 0) break;
    if (what == 3) continue;

    if (what == 2) {
      // ---------------------------------------------------------- a row
      const int b = item % B, n = item / B;
      const int64_t o = static_cast<int64_t>(b) * N, rr = o + n;
      const void* row = static_cast<const char*>(p.target) + rr * V * esz;
      RowStatVisitor<DT, true> v{c, neg_inf(), 0.0f, 0.0f, INT_MAX, 0.0f};
      {
        constexpr int kv = Logit<DT>::kVec;
        const RowSpan sp = row_span<DT>(row, V);
        const int head = static_cast<int>(sp.head), nvec = static_cast<int>(sp.nvec);
        if (tid < head) v.visit1(Logit<DT>::load1(row, tid), tid, true);
        const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
        ring_stream<kCT, kRingItems>(vp, nvec, ring,
                                     [&](const uint4& x, int i) { v.visit_vec(x, head + static_cast<int64_t>(i) * kv, true); });
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
      for (int w2 = 1; w2 < kWarps; ++w2) merge_ms(m, sum, sw_m[w2], sw_s[w2], c);
      if (isfinite(m) && !isfinite(sum)) {
        // the row holds a NaN: the normaliser again with NaN as -inf
        KeyedSum ks{c, m * c, 0.0f};
        for_row<DT, 2>(row, V, ks, tid, kCT);
        const float part_s = warp_sum(ks.s);
        __syncthreads();
        if (lane == 0) sw_s[warp] = part_s;
        __syncthreads();
        sum = 0.0f;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) sum += sw_s[w2];
      }
      if (tid == 0) {
        if (!isfinite(m)) bump(io.stats, SPEC_STAT_NONFINITE_ROW);
        p.m_row[rr] = m;
        p.z_row[rr] = sum;
        // the test of the node's child, with the walk's operations
        int bits = kRowDone;
        const int ch = __ldg(io.ntok + rr);
        if (ch <= 0 || ch >= N) {
          bits |= kRowLeaf;
        } else {
          if (__ldg(io.nsib + o + ch) >= 0) bits |= kRowMulti;  // only the first child is tested
          const int32_t y = __ldg(io.dtok + o + ch);
          const bool ok = y >= 0 && y < V;
          const auto qrow = qsrc.row(io.q_row ? static_cast<int64_t>(__ldg(io.q_row + rr)) : rr);
          const float l = ok ? order_key(Logit<DT>::load1(row, y)) : neg_inf();
          const float qi = ok ? qrow.q_at(y) : 0.0f;
          const float pr = isfinite(m) ? prob_of(l, c, m * c, 1.0f / sum) : 0.0f;
          const float ratio = pr / qi;
          if (qi == 0.0f) bits |= kRowQZero;
          if (__ldg(io.coins + o + ch) < ratio) bits |= kRowAccept;
        }
        st_release_gpu(p.ready + rr, bits);
        // the request's rows are counted on one word: of two CTAs finishing
        // rows of request b, the one counting later sees the other's flag
        atom_add_acq_rel(p.rows_done + b, 1);
        // while many rows remain, a request resolved at this very row is
        // drawn here at once (its target row is still in L2); near the end of
        // the batched pass its draw is cut into chunks for every CTA
        const bool here_ok = rows - ld_volatile(p.cnt) >= 2 * static_cast<int64_t>(gridDim.x);
        s_here = try_resolve(p, b, n, here_ok) ? 1 : 0;
        if (s_here) s_A = __ldcg(p.A + b);
      }
      __syncthreads();  // sw_* reused by the next row
      if (s_here) {
        // the tree walk's own pass and draw (one CTA): the row streamed
        // through the copy ring, tile sums in tile order, then the search
        Weights w = draw_weights(b, n, s_A);
        float total = cdf_tile_pass_split<kCT, kCE, walk_ring_depth(K), 1>(w, V, part, tsum, ring, 0u);
        if (w.A != 0.0f && !(total > 0.0f && isfinite(total))) {
          if (tid == 0) bump(io.stats, SPEC_STAT_RESIDUAL_FALLBACK);
          w.A = 0.0f;
          total = cdf_tile_pass_split<kCT, kCE, walk_ring_depth(K), 1>(w, V, part, tsum, ring, 0u);
        }
        const int32_t tok = cdf_search<kCT, Weights, kCE>(w, V, __ldg(io.u_final + b), tsum, total, scan_sh, io.stats);
        if (tid == 0) write_draw(b, n, tok);
        __syncthreads();
      }
      continue;
    }

    // ------------------------------------------------- a draw chunk
    if (tid == 0) {
      const int k = item / p.nchunks;
      // the slot was reserved by a resolving thread that publishes it next
      const int b = wait_flag(p.slot_ready + k, kWaitLimitCycles, io.stats) ? __ldcg(p.slot_req + k) : -1;
      s_b = (b >= 0 && b < B) ? b : -1;  // a wait that ran out (counted): the item is dropped
      if (s_b >= 0) {
        s_n = __ldcg(p.node + b);
        s_A = __ldcg(p.A + b);
      }
    }
    __syncthreads();
    if (s_b < 0) continue;
    const int b = s_b, n = s_n, j = item % p.nchunks;
    const Weights w = draw_weights(b, n, s_A);
    const float tot = chunk_pass(w, j);
    if (tid == 0) {
      p.ctot[static_cast<int64_t>(b) * kMaxChunks + j] = tot;
      // acq_rel: the last chunk's CTA sees every other chunk's total
      s_last = atom_add_acq_rel(p.done + b, 1) == p.nchunks - 1;
    }
    __syncthreads();
    if (!s_last) continue;
    // the last chunk of request b: the inverse-CDF draw
    if (tid < p.nchunks) ctot_sh[tid] = __ldcg(p.ctot + static_cast<int64_t>(b) * kMaxChunks + tid);
    __syncthreads();
    finish_draw(b, n, w);
  }
}

struct ReqWs {
  int32_t* ints;  // counters, then 9 arrays of B
  size_t int_bytes;
  float* A;
  float* ctot;
};

ReqWs carve_req(void* ws, int B) {
  char* q = static_cast<char*>(ws);
  ReqWs r;
  r.ints = reinterpret_cast<int32_t*>(q);
  r.int_bytes = sizeof(int32_t) * (kCounters + 9 * static_cast<size_t>(B));
  q += align256(r.int_bytes);
  r.A = reinterpret_cast<float*>(q);
  q += align256(sizeof(float) * static_cast<size_t>(B));
  r.ctot = reinterpret_cast<float*>(q);
  return r;
}

template <int DT, class QSrc>
int launch_chain(ChainParams& p, const QSrc& qsrc, cudaStream_t s) {
  auto kernel = chain_verify_kernel<DT, QSrc>;
  const size_t smem = sizeof(uint4) * kRingItems * kCT +
                      sizeof(float) * (static_cast<size_t>(cdf_part_tiles<kCT, kCE, 1>(p.V)) * kCT + p.ntiles);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  int dev = 0, sms = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kCT, smem) != cudaSuccess || per < 1) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  // persistent: every CTA resident at once (no CTA ever waits on one that
  // has not started); no more CTAs than there are rows and draw items
  const int64_t items = static_cast<int64_t>(p.B) * p.N + static_cast<int64_t>(p.B) * p.nchunks;
  const int64_t grid = std::min<int64_t>(static_cast<int64_t>(sms) * per, items);
  launch_k(kernel, static_cast<unsigned>(grid), kCT, smem, s, p, qsrc);
  return launch_status();
}

}  // namespace

size_t chain_ws_bytes(int B) {
  if (B < 0) return 0;
  const size_t b = static_cast<size_t>(B);
  return align256(sizeof(int32_t) * (kCounters + 9 * b)) + align256(sizeof(float) * b) +
         align256(sizeof(float) * kMaxChunks * b);
}

int chain_verify(int dtype, int B, int N, int64_t V, const void* target, float c, const ChainQ& q,
                 const ChainIO& io, int32_t* ready, float* m_row, float* z_row, void* req_ws, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(B) * N;
  ChainParams p;
  p.B = B;
  p.N = N;
  p.V = V;
  p.c = c;
  p.target = target;
  p.io = io;
  p.ready = ready;
  p.m_row = m_row;
  p.z_row = z_row;
  const ReqWs r = carve_req(req_ws, B);
  p.cnt = r.ints;
  p.state = p.cnt + kCounters;
  p.done = p.state + B;
  p.slot_req = p.done + B;
  p.slot_ready = p.slot_req + B;
  p.node = p.slot_ready + B;
  p.len = p.node + B;
  p.kind = p.len + B;
  p.rows_done = p.kind + B;
  p.front = p.rows_done + B;
  p.A = r.A;
  p.ctot = r.ctot;
  const int64_t ntiles = (V + kTile - 1) / kTile;
  p.ntiles = static_cast<int>(ntiles);
  p.tpc = chunk_tiles(ntiles);
  p.nchunks = static_cast<int>((ntiles + p.tpc - 1) / p.tpc);
  if (p.tpc > kMaxChunkTiles || p.nchunks > kMaxChunks) return SPEC_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(ready, 0, sizeof(int32_t) * static_cast<size_t>(rows), s) != cudaSuccess ||
      cudaMemsetAsync(r.ints, 0, r.int_bytes, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (q.kind == 0) {
    const QProbs qs{static_cast<const float*>(q.q), V};
    return dtype == SPEC_BF16 ? launch_chain<SPEC_BF16>(p, qs, s) : launch_chain<SPEC_F32>(p, qs, s);
  }
  if (q.kind == 1) {
    const QLogits<SPEC_BF16> qs{q.q, q.q_stats, V, q.cq};
    return dtype == SPEC_BF16 ? launch_chain<SPEC_BF16>(p, qs, s) : launch_chain<SPEC_F32>(p, qs, s);
  }
  const QLogits<SPEC_F32> qs{q.q, q.q_stats, V, q.cq};
  return dtype == SPEC_BF16 ? launch_chain<SPEC_BF16>(p, qs, s) : launch_chain<SPEC_F32>(p, qs, s);
}

}  // namespace specdec
