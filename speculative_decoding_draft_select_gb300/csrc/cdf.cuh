// Block-wide inverse-CDF draw over a row of non-negative weights.
//
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)", 5.1 draws
// the correction token from the normalised positive residual and the bonus
// from the target distribution (a categorical draw).  With a caller uniform
// u the draw is the smallest v whose inclusive prefix sum of the weights
// exceeds u * W, W the total.
//
// The row is cut into tiles of THREADS * E elements; thread j of a tile
// owns its E consecutive elements (E = 8 for the one-CTA-per-row draft
// sampler, larger for the walk).  cdf_tile_pass / cdf_tile_pass_split stream
// the row once and record every tile's sum in a fixed order, no atomics.
// cdf_search walks the tile sums in order to the first tile whose running
// prefix exceeds u * W and rescans only that tile with a block scan; if
// rounding leaves no crossing inside it, the following tiles are scanned;
// with none at all the last index of positive weight is taken and counted.
#pragma once

#include <climits>

#include "common.cuh"

namespace specdec {

// W provides:  void load8(int64_t v0, float* x) const   (0 beyond V)
//              float at(int64_t v) const
template <int THREADS, class W, int kUnroll = 4>
__device__ float cdf_tile_pass(const W& w, int64_t V, float* red, float* tile_sum) {
  constexpr int kTile = THREADS * 8, kWarps = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ntiles = (V + kTile - 1) / kTile;
  // kUnroll tiles per iteration: all their loads are issued before the sums
  for (int64_t t = 0; t < ntiles; t += kUnroll) {
    float x[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (t + u < ntiles) {
        w.load8((t + u) * kTile + threadIdx.x * 8, x[u]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[u][j] = 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float s0 = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) s0 += x[u][j];
      s0 = warp_sum(s0);
      if (lane == 0 && t + u < ntiles) red[(t + u) * kWarps + warp] = s0;
    }
  }
  __syncthreads();
  for (int64_t i = threadIdx.x; i < ntiles; i += THREADS) {
    float s = 0.0f;
    for (int k = 0; k < kWarps; ++k) s += red[i * kWarps + k];
    tile_sum[i] = s;
  }
  __syncthreads();
  // total in tile order (every thread computes the same value)
  float total = 0.0f;
  for (int64_t i = 0; i < ntiles; ++i) total += tile_sum[i];
  return total;
}

// cdf_tile_pass split over the C CTAs of a thread-block cluster that walk
// one row together (a latency-bound walk; C = 1 is a lone CTA).  Tiles are
// THREADS * E elements.  CTA `rank` sums the tiles rank, rank + C, ... (its
// local tiles i = 0, 1, ...): every thread stores the sum of its E elements
// of local tile i in part[i % P][thread], and every P local tiles (and at
// the end) each warp reduces whole tiles (lanes over the partials in thread
// order, then a butterfly), so the stream itself carries no reduction.
// Each tile sum is stored into tile_sum of every CTA of the cluster; after
// the cluster barrier all of them hold the same tile sums and the same total
// (tile order).
//
// Loads: where w.ring_ok(), each thread keeps its next D tiles in flight
// with asynchronous copies into its own slots of a shared-memory ring, so
// loading overlaps the arithmetic without block barriers (a thread reads
// only what it copied); otherwise direct 16-byte loads.  W provides
//   template <int E> static constexpr int chunks()   16-byte chunks per thread and tile
//   bool ring_ok() const                             rows 16-byte aligned
//   template <int E> void issue(uint4* slot, int stride, int64_t v0) const
//   template <int E> float ring_sum(const uint4* slot, int stride, int64_t v0) const
//   template <int E> float load_sum(int64_t v0) const
// where ring_sum and load_sum add the same values in the same order.  ring:
// D * chunks<E>() * THREADS 16-byte slots, chunk c of slot s of thread t at
// ring[(s * chunks + c) * THREADS + t].  part: cdf_part_tiles * THREADS
// floats.  V + THREADS * E < 2^31.
constexpr int kPartTiles = 16;  // P

template <int THREADS, int E, int C>
__host__ __device__ inline int cdf_part_tiles(int64_t V) {
  const int64_t ntiles = (V + THREADS * E - 1) / (THREADS * E);
  const int64_t nloc = (ntiles + C - 1) / C;
  return static_cast<int>(nloc < kPartTiles ? nloc : kPartTiles);
}

template <int THREADS, int E, int D, int C, class W>
__device__ float cdf_tile_pass_split(const W& w, int64_t V64, float* part, float* tile_sum, uint4* ring,
                                     unsigned rank) {
  constexpr int kTile = THREADS * E, kWarps = THREADS / 32, K = W::template chunks<E>(), P = kPartTiles;
  const int V = static_cast<int>(V64);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int ntiles = (V + kTile - 1) / kTile;
  const int r = static_cast<int>(rank);
  const int nloc = ntiles > r ? (ntiles - r + C - 1) / C : 0;
  const int off = tid * E;
  auto first = [&](int i) { return (r + C * i) * kTile + off; };  // thread's first element of local tile i
  // reduce local tiles [i0, i1) (at most P) and store their sums everywhere
  auto flush = [&](int i0, int i1) {
    __syncthreads();
    for (int i = i0 + warp; i < i1; i += kWarps) {
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < kWarps; ++j) s += part[(i % P) * THREADS + j * 32 + lane];
      s = warp_sum(s);
      if (lane == 0 && spec_in(r + C * i, ntiles, nullptr)) {
        const int t = r + C * i;
        if (C == 1) {
          tile_sum[t] = s;
        } else {
#pragma unroll
          for (int q = 0; q < C; ++q) st_cluster_f32(tile_sum + t, q, s);
        }
      }
    }
    __syncthreads();
  };
  int done = 0;  // local tiles reduced so far
  if (w.ring_ok()) {
    uint4* mine = ring + tid;
#pragma unroll
    for (int s = 0; s < D; ++s) {
      if (s < nloc) w.template issue<E>(mine + s * K * THREADS, THREADS, first(s));
      cp_async_commit();  // one group per local tile (empty ones keep the count)
    }
    int s = 0;
    for (int i = 0; i < nloc; ++i) {
      cp_async_wait<D - 1>();  // tile i has landed
      const float ps = w.template ring_sum<E>(mine + s * K * THREADS, THREADS, first(i));
      part[(i % P) * THREADS + tid] = ps;  // the slot has been read
      if (i + D < nloc) w.template issue<E>(mine + s * K * THREADS, THREADS, first(i + D));
      cp_async_commit();
      s = s + 1 == D ? 0 : s + 1;
      if (i + 1 - done == P && i + 1 < nloc) {
        flush(done, i + 1);
        done = i + 1;
      }
    }
    cp_async_wait<0>();
  } else {
    for (int i = 0; i < nloc; ++i) {
      part[(i % P) * THREADS + tid] = w.template load_sum<E>(first(i));
      if (i + 1 - done == P && i + 1 < nloc) {
        flush(done, i + 1);
        done = i + 1;
      }
    }
  }
  flush(done, nloc);
  if (C > 1) cluster_barrier();
  float total = 0.0f;
  for (int t = 0; t < ntiles; ++t) total += tile_sum[t];
  return total;
}

template <int THREADS, class W, int E = 8>
__device__ int32_t cdf_search(const W& w, int64_t V, float u, const float* tile_sum, float total,
                              float* scan_sh, int32_t* stats) {
  static_assert(E % 8 == 0, "elements per thread come in groups of 8");
  constexpr int kTile = THREADS * E;
  __shared__ int32_t s_tok;
  const int64_t ntiles = (V + kTile - 1) / kTile;
  if (threadIdx.x == 0) s_tok = INT_MAX;
  __syncthreads();
  const float target = u * total;
  float prefix = 0.0f;
  if (total > 0.0f && isfinite(total)) {
    for (int64_t t = 0; t < ntiles; ++t) {
      const float after = prefix + tile_sum[t];
      if (after > target) {
        const int64_t v0 = t * kTile + threadIdx.x * E;
        float x[E];
#pragma unroll
        for (int g = 0; g < E / 8; ++g) w.load8(v0 + 8 * g, x + 8 * g);
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < E; ++j) sum += x[j];
        float tot;
        const float incl = block_inclusive_scan(sum, scan_sh, tot);
        float C = prefix + (incl - sum);
        int found = -1;
#pragma unroll
        for (int j = 0; j < E; ++j) {
          C += x[j];
          if (found < 0 && C > target && v0 + j < V) found = j;
        }
        if (found >= 0) atomicMin(&s_tok, static_cast<int32_t>(v0 + found));
        __syncthreads();
        if (s_tok != INT_MAX) break;
      }
      prefix = after;
    }
  }
  __syncthreads();
  if (s_tok == INT_MAX) {
    __syncthreads();
    if (threadIdx.x == 0) s_tok = -1;
    __syncthreads();
    for (int64_t v = threadIdx.x; v < V; v += THREADS)
      if (w.at(v) > 0.0f) atomicMax(&s_tok, static_cast<int32_t>(v));
    __syncthreads();
    if (threadIdx.x == 0) {
      if (s_tok < 0) s_tok = 0;
      bump(stats, SPEC_STAT_CDF_FALLBACK);
    }
  }
  __syncthreads();
  const int32_t tok = s_tok;
  __syncthreads();
  return tok;
}

// Shared-memory floats cdf_tile_pass needs for a row of V elements.
template <int THREADS>
__host__ __device__ inline int64_t cdf_smem_floats(int64_t V) {
  const int64_t ntiles = (V + THREADS * 8 - 1) / (THREADS * 8);
  return ntiles * (THREADS / 32) + ntiles;
}

// 8 consecutive elements of an fp32 row (vector loads where aligned).
__device__ __forceinline__ void load8_f32(const float* row, int64_t V, int64_t v0, float* x) {
  if (v0 + 8 <= V && (reinterpret_cast<uintptr_t>(row + v0) & 15) == 0) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(row + v0));
    const float4 b = __ldg(reinterpret_cast<const float4*>(row + v0 + 4));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (v0 + j < V) ? __ldg(row + v0 + j) : 0.0f;
  }
}

// 8 consecutive logits of a row as ordering keys; beyond V: -inf.
template <int DT>
__device__ __forceinline__ void load8_logits(const void* row, int64_t V, int64_t v0, float* x) {
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const char* p = static_cast<const char*>(row) + v0 * esz;
  if (v0 + 8 <= V && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    if (DT == SPEC_BF16) {
      unpack<SPEC_BF16>(__ldg(reinterpret_cast<const uint4*>(p)), x);
    } else {
      unpack<SPEC_F32>(__ldg(reinterpret_cast<const uint4*>(p)), x);
      unpack<SPEC_F32>(__ldg(reinterpret_cast<const uint4*>(p) + 1), x + 4);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = order_key(x[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (v0 + j < V) ? order_key(Logit<DT>::load1(row, v0 + j)) : neg_inf();
  }
}

}  // namespace specdec
