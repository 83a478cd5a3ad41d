// Block-wide inverse-CDF draw over a row of non-negative weights.
//
// zero-to-sglang ch.10 "Speculative decoding (code walk-through)", 5.1 draws
// the correction token from the normalised positive residual and the bonus
// from the target distribution (a categorical draw).  With a caller uniform
// u the draw is the smallest v whose inclusive prefix sum of the weights
// exceeds u * W, W the total.
//
// The row is cut into tiles of THREADS * 8 elements; thread j of a tile owns
// its 8 consecutive elements.  cdf_tile_pass streams the row once and
// records every tile's sum (warp sums in a fixed order, no atomics).
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

template <int THREADS, class W>
__device__ int32_t cdf_search(const W& w, int64_t V, float u, const float* tile_sum, float total,
                              float* scan_sh, int32_t* stats) {
  constexpr int kTile = THREADS * 8;
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
        const int64_t v0 = t * kTile + threadIdx.x * 8;
        float x[8];
        w.load8(v0, x);
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) sum += x[j];
        float tot;
        const float incl = block_inclusive_scan(sum, scan_sh, tot);
        float C = prefix + (incl - sum);
        int found = -1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
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
