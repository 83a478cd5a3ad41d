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
// Tuning knobs (compile-time; the defaults are the fastest of the settings
// measured at B=256 x 5 and B=1024 x 16 nodes): copy-ring depth, pieces per
// row, CTAs per SM, and draws started in place by the CTA that finishes a
// request's rows (1: 833 against 798 us at B=1024 x 16, 134 against 128 us
// at B=256 x 5).
#ifndef SPEC_CHAIN_RING
#define SPEC_CHAIN_RING 16
#endif
#ifndef SPEC_CHAIN_SPLIT
#define SPEC_CHAIN_SPLIT 1
#endif
#ifndef SPEC_CHAIN_CTAS_PER_SM
#define SPEC_CHAIN_CTAS_PER_SM 5
#endif
#ifndef SPEC_CHAIN_HERE
#define SPEC_CHAIN_HERE 0
#endif
constexpr int kRingItems = SPEC_CHAIN_RING;  // 16-byte copies in flight per thread (row statistics)
// pieces a row's statistics are cut into (each a work item; the CTA that
// finishes a row's last piece merges them in piece order)
constexpr int kSplit = SPEC_CHAIN_SPLIT;
static_assert(kSplit == 1 || kSplit == 2, "a row is one or two pieces");
constexpr int kMaxChunks = 64;     // draw items per request, at most
constexpr int kMinChunkTiles = 8;  // a draw item streams at least 8 tiles (the fixed cost of an item amortised)
constexpr int kMaxChunkTiles = 32;  // (SPEC_MAX_VOCAB / kTile) / kMaxChunks
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
  int32_t* half_done;  // [B N] halves of the row done
  float* half_ms;      // [B N][2][2] each half's (max, sum)
  int ntiles, tpc, nchunks;
  int64_t half;  // elements of a row's first half (a multiple of 8)
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
// draft-table row of target row rr (the table's row count is not an
// argument: the debug build checks the sign only)
__device__ __forceinline__ int64_t q_row_of(const ChainIO& io, int64_t rr) {
  const int64_t r = io.q_row ? static_cast<int64_t>(__ldg(io.q_row + rr)) : rr;
  return spec_in(r, INT64_MAX, io.stats) ? r : -1;
}

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
    if (!spec_in(o + i, static_cast<int64_t>(p.B) * N, io.stats)) break;
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
  if (!spec_in(k, p.B, io.stats)) return false;
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
  if (!spec_smem_ok(reinterpret_cast<char*>(tsum + (p.V + kTile - 1) / kTile) - reinterpret_cast<char*>(ring),
                    p.io.stats))
    return;
  __shared__ float sw_m[kWarps], sw_s[kWarps];
  __shared__ float tile_sh[kMaxChunkTiles];  // tile sums of one chunk
  __shared__ float ctot_sh[kMaxChunks];
  __shared__ float scan_sh[33];
  __shared__ float s_A;
  __shared__ int s_what, s_item, s_last, s_tok, s_b, s_n, s_here;
  const ChainIO& io = p.io;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B, N = p.N;
  const int64_t V = p.V, rows = static_cast<int64_t>(B) * N;
  const float c = p.c;
  long long idle0 = 0;
  bool idle = false;
  int pend = -1;  // thread 0: a claimed draw item whose slot is not reserved yet

  // tile sums of chunk j of a draw row into tile_sh, their total (in tile
  // order) to every thread: the chunk's tiles, a tile-aligned piece of the
  // row, streamed by the walk's own pass through the copy ring
  constexpr int K = Weights::template chunks<kCE>();
  // tiles in flight per thread in the draw passes: what the ring holds
  constexpr int kDR = walk_ring_depth(K) < kRingItems / K ? walk_ring_depth(K) : (kRingItems / K < 1 ? 1 : kRingItems / K);
  auto chunk_pass = [&](const Weights& w, int j) -> float {
    const int64_t e0 = static_cast<int64_t>(j) * p.tpc * kTile;
    const int64_t n = min(V, e0 + static_cast<int64_t>(p.tpc) * kTile) - e0;
    return cdf_tile_pass_split<kCT, kCE, kDR, 1>(w.sub(e0, n), n, part, tile_sh, ring, 0u);
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
    if (!spec_in(len, N, io.stats)) return;
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
    const auto qrow = qsrc.row(A != 0.0f ? q_row_of(io, rr) : -1);
    return Weights{row, qrow, V, c, folded_offset(m, c, z), A};
  };

  for (;;) {
    if (tid == 0) {
      // rows first: the batched pass is the critical path; then draw items
      int what = 3, item = 0;
      const int r = ld_volatile(p.cnt) < kSplit * rows ? atomicAdd(p.cnt, 1) : static_cast<int>(kSplit * rows);
      if (r < kSplit * rows) {
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
      // ------------------------------------------------ a row (or a piece)
      // item = kSplit * (node-major row) + piece; the CTA finishing a row's
      // last piece merges the pieces in order and tests the node's child
      const int ri = kSplit == 2 ? item >> 1 : item, hf = kSplit == 2 ? item & 1 : 0;
      const int b = ri % B, n = ri / B;
      const int64_t o = static_cast<int64_t>(b) * N, rr = o + n;
      const void* row = static_cast<const char*>(p.target) + rr * V * esz;
      const int64_t h0 = hf * p.half, hlen = (hf ? V : p.half) - h0;
      const void* hrow = static_cast<const char*>(row) + h0 * esz;
      RowStatVisitor<DT, true> v{c, neg_inf(), 0.0f, 0.0f, INT_MAX, 0.0f};
      {
        constexpr int kv = Logit<DT>::kVec;
        const RowSpan sp = row_span<DT>(hrow, hlen);
        const int head = static_cast<int>(sp.head), nvec = static_cast<int>(sp.nvec);
        if (tid < head) v.visit1(Logit<DT>::load1(hrow, tid), tid, true);
        const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(hrow) + sp.head * esz);
        ring_stream<kCT, kRingItems>(vp, nvec, ring,
                                     [&](const uint4& x, int i) { v.visit_vec(x, head + static_cast<int64_t>(i) * kv, true); });
        const int64_t t = head + static_cast<int64_t>(nvec) * kv + tid;
        if (t < hlen) v.visit1(Logit<DT>::load1(hrow, t), t, true);
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
      if (kSplit == 2) {
        if (tid == 0) {
          p.half_ms[4 * rr + 2 * hf] = m;
          p.half_ms[4 * rr + 2 * hf + 1] = sum;
          // acq_rel: the second half's CTA sees the first half's partials
          s_last = atom_add_acq_rel(p.half_done + rr, 1) == 1;
        }
        __syncthreads();
        if (!s_last) continue;
        // both halves: (max, sum) of half 0 merged with half 1's, in that order
        m = __ldcg(p.half_ms + 4 * rr);
        sum = __ldcg(p.half_ms + 4 * rr + 1);
        merge_ms(m, sum, __ldcg(p.half_ms + 4 * rr + 2), __ldcg(p.half_ms + 4 * rr + 3), c);
      }
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
          const auto qrow = qsrc.row(q_row_of(io, rr));
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
        const bool here_ok = SPEC_CHAIN_HERE && kSplit * rows - ld_volatile(p.cnt) >= static_cast<int64_t>(gridDim.x);
        s_here = try_resolve(p, b, n, here_ok) ? 1 : 0;
        if (s_here) s_A = __ldcg(p.A + b);
      }
      __syncthreads();  // sw_* reused by the next row
      if (s_here) {
        // the tree walk's own pass and draw (one CTA): the row streamed
        // through the copy ring, tile sums in tile order, then the search
        Weights w = draw_weights(b, n, s_A);
        float total = cdf_tile_pass_split<kCT, kCE, kDR, 1>(w, V, part, tsum, ring, 0u);
        if (w.A != 0.0f && !(total > 0.0f && isfinite(total))) {
          if (tid == 0) bump(io.stats, SPEC_STAT_RESIDUAL_FALLBACK);
          w.A = 0.0f;
          total = cdf_tile_pass_split<kCT, kCE, kDR, 1>(w, V, part, tsum, ring, 0u);
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
    if (tid == 0 && spec_in(j, kMaxChunks, io.stats)) {
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
  int32_t* ints;  // counters, then 9 arrays of B, then B N half counters
  size_t int_bytes;
  float* A;
  float* ctot;
  float* half_ms;
};

ReqWs carve_req(void* ws, int B, int N) {
  char* q = static_cast<char*>(ws);
  const size_t rows = static_cast<size_t>(B) * N;
  ReqWs r;
  r.ints = reinterpret_cast<int32_t*>(q);
  r.int_bytes = sizeof(int32_t) * (kCounters + 9 * static_cast<size_t>(B) + rows);
  q += align256(r.int_bytes);
  r.A = reinterpret_cast<float*>(q);
  q += align256(sizeof(float) * static_cast<size_t>(B));
  r.ctot = reinterpret_cast<float*>(q);
  q += align256(sizeof(float) * kMaxChunks * static_cast<size_t>(B));
  r.half_ms = reinterpret_cast<float*>(q);
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
  // as much shared memory as the SM has (more CTAs resident: more rows in flight)
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
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
  // (a grid larger than what is resident at once is safe too: a CTA waits
  // only on work running CTAs have taken)
  if (SPEC_CHAIN_CTAS_PER_SM > per) per = SPEC_CHAIN_CTAS_PER_SM;
  const int64_t items = kSplit * static_cast<int64_t>(p.B) * p.N + static_cast<int64_t>(p.B) * p.nchunks;
  const int64_t grid = std::min<int64_t>(static_cast<int64_t>(sms) * per, items);
  launch_k(kernel, static_cast<unsigned>(grid), kCT, smem, s, p, qsrc);
  return launch_status();
}

}  // namespace

size_t chain_ws_bytes(int B, int N) {
  if (B < 0 || N < 1) return 0;
  const size_t b = static_cast<size_t>(B), rows = b * static_cast<size_t>(N);
  return align256(sizeof(int32_t) * (kCounters + 9 * b + rows)) + align256(sizeof(float) * b) +
         align256(sizeof(float) * kMaxChunks * b) + align256(sizeof(float) * 4 * rows);
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
  const ReqWs r = carve_req(req_ws, B, N);
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
  p.half_done = p.front + B;
  p.half_ms = r.half_ms;
  p.half = kSplit == 2 ? ((V + 1) / 2 + 7) / 8 * 8 : V;
  if (p.half > V) p.half = V;
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
