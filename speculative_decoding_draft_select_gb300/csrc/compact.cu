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
// Two launches.  The index kernel (one CTA; one thread per request) does the
// relabelling or emits the moves, and compacts the freed list across
// requests with a block scan.  The payload kernel (one CTA per request)
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

__global__ void __launch_bounds__(kIndexThreads)
    compact_index_kernel(int B, int N, int ps, const int32_t* __restrict__ seq_lens,
                         const int32_t* __restrict__ path, const int32_t* __restrict__ acc_len,
                         int32_t* req_to_token, int64_t max_ctx, int32_t* move_src, int32_t* move_dst,
                         int32_t* num_moves, int32_t* freed, int32_t* num_freed, int32_t* new_kv_len,
                         int32_t* stats) {
  pdl_enter();
  __shared__ int scan_sh[33];
  __shared__ int running;
  if (threadIdx.x == 0) running = 0;
  __syncthreads();
  for (int base = 0; base < B; base += kIndexThreads) {
    const int b = base + threadIdx.x;
    int cnt = 0;
    bool valid = false;
    int64_t sl = 0, nk = 0;
    int a = 0;
    const int32_t* pb = path + static_cast<int64_t>(b) * N;
    int32_t* rt = req_to_token + static_cast<int64_t>(b) * max_ctx;
    if (b < B) {
      sl = __ldg(seq_lens + b);
      a = __ldg(acc_len + b);
      valid = sl >= 0 && sl + N <= max_ctx && a >= 0 && a < N && __ldg(pb) == 0;
      for (int i = 1; valid && i <= a; ++i) {
        const int32_t pi = __ldg(pb + i);
        valid = pi > __ldg(pb + i - 1) && pi < N;
      }
      if (!valid) {
        new_kv_len[b] = -1;
        num_moves[b] = 0;
        bump(stats, SPEC_STAT_BAD_REQUEST);
      } else {
        nk = sl + 1 + a;
        new_kv_len[b] = static_cast<int32_t>(nk);
        if (ps == 1) {
          cnt = N - 1 - a;
        } else {
          for (int64_t lp = (sl + ps - 1) / ps; lp * ps < sl + N; ++lp) cnt += lp * ps >= nk;
        }
      }
      for (int i = 0; i < N; ++i) {
        move_src[static_cast<int64_t>(b) * N + i] = -1;
        move_dst[static_cast<int64_t>(b) * N + i] = -1;
      }
    }
    int total;
    const int off = running + block_exclusive_scan_i(cnt, scan_sh, total);
    if (valid) {
      int w = off;
      if (ps == 1) {
        // freed: slots of the nodes off the path, node order (old mapping)
        int j = 1;
        for (int n = 1; n < N; ++n) {
          if (j <= a && __ldg(pb + j) == n) {
            ++j;
            continue;
          }
          freed[w++] = rt[sl + n];
        }
        // relabel in increasing i: position sl+path[i] is read before
        // position sl+i is written, and path[i] >= i
        for (int i = 1; i <= a; ++i) rt[sl + i] = rt[sl + __ldg(pb + i)];
        num_moves[b] = 0;
      } else {
        int m = 0;
        for (int i = 1; i <= a; ++i) {
          const int32_t pi = __ldg(pb + i);
          if (pi == i) continue;
          move_src[static_cast<int64_t>(b) * N + m] = rt[sl + pi];
          move_dst[static_cast<int64_t>(b) * N + m] = rt[sl + i];
          ++m;
        }
        num_moves[b] = m;
        for (int64_t lp = (sl + ps - 1) / ps; lp * ps < sl + N; ++lp)
          if (lp * ps >= nk) freed[w++] = rt[lp * ps] / ps;
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
           req_to_token, max_ctx, move_src, move_dst, num_moves, freed, num_freed, new_kv_len, stats_or_null);
  int e = launch_status();
  if (e != SPEC_OK || B == 0 || !kv_pool_or_null || page_size == 1) return e;
  launch_k(compact_payload_kernel, B, kCopyThreads, 0, s, N, move_src, move_dst, num_moves,
           static_cast<uint8_t*>(kv_pool_or_null), num_slots, bytes_per_slot, stats_or_null);
  return launch_status();
}
