// Accepted-path KV-slot compaction.
//
// "EAGLE speculative decoding in four parts" (ai-infra-handbooks),
// "Drafting, verification and slots": slots for every candidate are
// allocated before drafting; after verification only the slots on the
// accepted path are kept and the rest freed; with a page size above 1 the
// data has to be copied.  zero-to-sglang ch.10 "Speculative decoding (code
// walk-through)" 5.2: the cache is restored to the committed path, and the
// correction / bonus token has no KV of its own yet.
//
// Two launches.  The index kernel (one CTA; a group of 8 lanes per request)
// does the relabelling or emits the moves, and compacts the freed list
// across requests with a block scan.  The payload kernel (one CTA per request)
// copies each move's bytes in increasing path order with a barrier between
// moves, so a source is always read before a later move overwrites it (the
// path [0, 2, 3] case: node 3 lands where node 2 was).
#include <climits>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kIndexThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan_i(int v, int* sh, int& total) {
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

// A group of kLanes lanes per request (kIndexThreads / kLanes requests per
// round of the one CTA): the lanes split the request's nodes, pages and path
// entries, and ballots within the group keep every list in its order.
constexpr int kLanes = 8;
constexpr int kGroups = kIndexThreads / kLanes;

__global__ void __launch_bounds__(kIndexThreads)
    compact_index_kernel(int B, int N, int ps, const int32_t* __restrict__ seq_lens,
                         const int32_t* __restrict__ path, const int32_t* __restrict__ acc_len,
                         int32_t* req_to_token, int64_t max_ctx, int32_t* move_src, int32_t* move_dst,
                         int32_t* num_moves, int32_t* freed, int64_t freed_cap, int32_t* num_freed,
                         int32_t* new_kv_len, int32_t* stats) {
  pdl_enter();
  __shared__ int scan_sh[33];
  __shared__ int running;
  const int lane = threadIdx.x & 31, g = threadIdx.x / kLanes, gl = threadIdx.x % kLanes;
  // this group's lanes: every collective below names only them, since the
  // groups of a warp run different trip counts
  const unsigned gmask = ((1u << kLanes) - 1u) << (lane & ~(kLanes - 1));
  const unsigned below = (1u << gl) - 1u;
  auto group_bits = [&](bool p) -> unsigned {  // bit j: lane j of the group
    return __ballot_sync(gmask, p) >> (lane & ~(kLanes - 1));
  };
  auto group_all = [&](bool p) { return group_bits(!p) == 0u; };
  if (threadIdx.x == 0) running = 0;
  __syncthreads();
  for (int base = 0; base < B; base += kGroups) {
    const int b = base + g;
    const bool in = b < B;
    const int64_t o = static_cast<int64_t>(in ? b : 0) * N;
    const int32_t* pb = path + o;
    int32_t* rt = req_to_token + static_cast<int64_t>(in ? b : 0) * max_ctx;
    const int64_t sl = in ? __ldg(seq_lens + b) : 0;
    const int a = in ? __ldg(acc_len + b) : 0;
    // validity: a seq_len and accept length in range, a path that starts at
    // 0 and increases within [0, N)
    bool valid = in && sl >= 0 && sl + N <= max_ctx && a >= 0 && a < N;
    if (valid) valid = __ldg(pb) == 0;
    for (int i0 = 1; i0 <= (in ? a : 0) && i0 < N; i0 += kLanes) {
      const int i = i0 + gl;
      bool ok = true;
      if (valid && i <= a) {
        const int32_t pi = __ldg(pb + i);
        ok = pi > __ldg(pb + i - 1) && pi < N;
      }
      valid = group_all(ok) && valid;
    }
    const int64_t nk = sl + 1 + a;
    int cnt = 0;
    if (in && valid) {
      if (ps == 1) {
        cnt = N - 1 - a;
      } else {
        for (int64_t lp = (sl + ps - 1) / ps + gl; lp * ps < sl + N; lp += kLanes) cnt += lp * ps >= nk;
        for (int off = kLanes / 2; off > 0; off >>= 1) cnt += __shfl_xor_sync(gmask, cnt, off);
      }
    }
    if (in) {
      for (int i = gl; i < N; i += kLanes) {
        move_src[o + i] = -1;
        move_dst[o + i] = -1;
      }
      if (gl == 0) {
        new_kv_len[b] = valid ? static_cast<int32_t>(nk) : -1;
        if (!valid) {
          num_moves[b] = 0;
          bump(stats, SPEC_STAT_BAD_REQUEST);
        }
      }
    }
    // freed-list offsets: exclusive scan of the groups' counts
    int total;
    const int mine = gl == 0 ? cnt : 0;
    const int off0 = running + block_exclusive_scan_i(mine, scan_sh, total);
    int w = __shfl_sync(gmask, off0, lane & ~(kLanes - 1));
    if (in && valid) {
      if (ps == 1) {
        // freed: slots of the nodes off the path, in node order (old
        // mapping); the path is increasing, so node n is on it iff the
        // merge pointer meets it
        int j = 1;  // next path entry not below the chunk
        for (int n0 = 1; n0 < N; n0 += kLanes) {
          const int n = n0 + gl;
          while (j <= a && __ldg(pb + j) < n0) ++j;
          bool on = false;
          for (int jj = j; jj <= a; ++jj) {
            const int32_t pj = __ldg(pb + jj);
            if (pj >= n0 + kLanes) break;
            on = on || pj == n;
          }
          const bool off = n < N && !on;
          const unsigned bits = group_bits(off);
          const int32_t slot = off ? rt[sl + n] : 0;
          if (off && spec_in(w + __popc(bits & below), freed_cap, stats)) freed[w + __popc(bits & below)] = slot;
          w += __popc(bits);
        }
        __syncwarp(gmask);
        // relabel: position sl + i takes the slot of sl + path[i]; every
        // read position path[i] >= i is past every write of earlier chunks,
        // and a chunk reads all before it writes
        for (int i0 = 1; i0 <= a; i0 += kLanes) {
          const int i = i0 + gl;
          const int32_t v = i <= a ? rt[sl + __ldg(pb + i)] : 0;
          __syncwarp(gmask);
          if (i <= a) rt[sl + i] = v;
        }
        if (gl == 0) num_moves[b] = 0;
      } else {
        // moves in increasing i for the path entries not in place
        int m = 0;
        for (int i0 = 1; i0 <= a; i0 += kLanes) {
          const int i = i0 + gl;
          const int32_t pi = i <= a ? __ldg(pb + i) : i;
          const bool mv = i <= a && pi != i;
          const unsigned bits = group_bits(mv);
          if (mv && spec_in(m + __popc(bits & below), N, stats)) {
            move_src[o + m + __popc(bits & below)] = rt[sl + pi];
            move_dst[o + m + __popc(bits & below)] = rt[sl + i];
          }
          m += __popc(bits);
        }
        if (gl == 0) num_moves[b] = m;
        // pages first touched by this step at or past the new length
        for (int64_t lp0 = (sl + ps - 1) / ps; lp0 * ps < sl + N; lp0 += kLanes) {
          const int64_t lp = lp0 + gl;
          const bool fr = lp * ps < sl + N && lp * ps >= nk;
          const unsigned bits = group_bits(fr);
          if (fr && spec_in(w + __popc(bits & below), freed_cap, stats)) freed[w + __popc(bits & below)] = rt[lp * ps] / ps;
          w += __popc(bits);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) running += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) *num_freed = running;
}

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
    compact_payload_kernel(int N, const int32_t* __restrict__ move_src, const int32_t* __restrict__ move_dst,
                           const int32_t* __restrict__ num_moves, uint8_t* kv, int64_t num_slots,
                           int64_t bps, int32_t* stats) {
  pdl_enter();
  const int b = blockIdx.x;
  const int nm = num_moves[b];
  if (!spec_in(nm, N + 1, stats)) return;
  const bool vec = (bps & 15) == 0 && (reinterpret_cast<uintptr_t>(kv) & 15) == 0;
  for (int m = 0; m < nm; ++m) {
    const int32_t src = move_src[static_cast<int64_t>(b) * N + m];
    const int32_t dst = move_dst[static_cast<int64_t>(b) * N + m];
    if (src < 0 || src >= num_slots || dst < 0 || dst >= num_slots) {
      if (threadIdx.x == 0) bump(stats, SPEC_STAT_BAD_REQUEST);
      continue;
    }
    const uint8_t* s = kv + src * bps;
    uint8_t* d = kv + dst * bps;
    if (vec) {
      const uint4* s4 = reinterpret_cast<const uint4*>(s);
      uint4* d4 = reinterpret_cast<uint4*>(d);
      for (int64_t i = threadIdx.x; i < bps / 16; i += kCopyThreads) d4[i] = s4[i];
    } else {
      for (int64_t i = threadIdx.x; i < bps; i += kCopyThreads) d[i] = s[i];
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" int64_t spec_compact_freed_capacity(int B, int N, int page_size) {
  if (B < 0 || N < 1 || page_size < 1) return -1;
  if (page_size == 1) return static_cast<int64_t>(B) * (N - 1);
  return static_cast<int64_t>(B) * ((N + page_size - 1) / page_size + 1);
}

extern "C" int spec_compact_slots(int B, int N, int page_size, const int32_t* seq_lens,
                                  const int32_t* accept_path, const int32_t* accept_length,
                                  int32_t* req_to_token, int64_t max_ctx, int32_t* move_src, int32_t* move_dst,
                                  int32_t* num_moves, int32_t* freed, int64_t freed_capacity, int32_t* num_freed,
                                  int32_t* new_kv_len, void* kv_pool_or_null, int64_t num_slots,
                                  int64_t bytes_per_slot, int32_t* stats_or_null, spec_stream_t stream) {
  if (B < 0 || N < 1 || page_size < 1 || max_ctx < N) return SPEC_ERR_INVALID_ARG;
  if (N > SPEC_MAX_NODES || max_ctx > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  if (!num_freed) return SPEC_ERR_INVALID_ARG;
  if (freed_capacity < spec_compact_freed_capacity(B, N, page_size)) return SPEC_ERR_INVALID_ARG;
  if (B > 0 && (!seq_lens || !accept_path || !accept_length || !req_to_token || !move_src || !move_dst ||
                !num_moves || !new_kv_len || (!freed && freed_capacity > 0)))
    return SPEC_ERR_INVALID_ARG;
  if (kv_pool_or_null && (num_slots < 1 || bytes_per_slot < 1)) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  launch_k(compact_index_kernel, 1, kIndexThreads, 0, s, B, N, page_size, seq_lens, accept_path, accept_length,
           req_to_token, max_ctx, move_src, move_dst, num_moves, freed, freed_capacity, num_freed, new_kv_len,
           stats_or_null);
  int e = launch_status();
  if (e != SPEC_OK || B == 0 || !kv_pool_or_null || page_size == 1) return e;
  launch_k(compact_payload_kernel, B, kCopyThreads, 0, s, N, move_src, move_dst, num_moves,
           static_cast<uint8_t*>(kv_pool_or_null), num_slots, bytes_per_slot, stats_or_null);
  return launch_status();
}
