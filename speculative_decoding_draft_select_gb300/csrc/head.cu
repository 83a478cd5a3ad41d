// Pruned draft LM head on the fifth-generation tensor cores (tcgen05).
//
// SGLang PR #22883 "TLI (Token-Level Intersection)", Modifications:
// _try_prune_draft_lm_head / _PrunedReindexLMHead keep only the LM-head
// weight rows of the vocabulary intersection's draft ids, so the draft
// logits are computed for those K ids alone -- O(M K H) instead of
// O(M V_d H) -- and the constrained top-1 (constrain_draft_logits, then
// map_draft_to_target_ids) is taken over them.
//
// logits[m][k] = sum over h of hidden[m][h] * weight[k][h], hidden [M, H] and
// weight [K, H] in bf16, both rows contiguous along H.  One CTA per tile of
// 128 weight rows and up to 256 hidden rows (two 128-row halves), so the
// weight tile -- the bulk of the bytes -- is read once:
//   warp 0, one thread: TMA copies of 64-column slabs of hidden and weight
//     (128-byte swizzle) into a 4-stage shared-memory ring, each stage
//     guarded by a "full" and an "empty" mbarrier;
//   warp 1, one thread: tcgen05.mma (kind::f16: bf16 operands, fp32
//     accumulation; M = 128, N = 128, K = 16 per instruction) into one
//     128 x 128 fp32 accumulator in tensor memory per half, each stage
//     released with tcgen05.commit on its "empty" barrier;
//   warp 2: allocates, and at the end frees, the 256 tensor-memory columns;
//   warps 4-7: the epilogue -- each thread takes one row of an accumulator
//     (its warp's 32 lanes) with tcgen05.ld and reduces its 128 logits to an
//     online-softmax partial (max, sum of 2^((x - max) c)) and the first
//     largest column; optionally it stores the fp32 logits.
// Every mbarrier wait is bounded; a wait that runs out is counted in
// SPEC_STAT_WAIT_TIMEOUT and the CTA drains its copies, frees its tensor
// memory and returns.  A second kernel merges each row's partials over the
// tiles in a fixed order into the top-1 (ties: the lower weight row, which is
// the lower draft id), the row's (max, normaliser) and the probability, and
// maps the top-1's rank to its draft and target ids.
#include <cuda.h>

#include <climits>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kHeadThreads = 384;  // warps: 0 TMA, 1 MMA, 2 tensor memory, 3 idle, 4-11 epilogue
constexpr int kEpiWarps = 8;
constexpr int kSubRows = 16;  // rows of the boxes a trimmed tile is loaded in
constexpr int kBM = 128;  // rows of an accumulator (hidden rows)
constexpr int kBN = 128;  // weight rows of a tile
constexpr int kBK = 64;   // H columns per stage: 128 bytes, one swizzle row
constexpr int kStages = 4;
constexpr int kSlab = kBM * kBK * 2;  // bytes of one 128-row slab (16 KB)
constexpr int kStageBytes = 3 * kSlab;
constexpr int kUmmaK = 16;  // K of one bf16 MMA instruction (32 bytes)
constexpr uint32_t kTmemCols = 512;  // two buffers x two 128-row halves x 128 columns
constexpr size_t kHeadSmem = static_cast<size_t>(kStages) * kStageBytes + 1024;  // + alignment slack
constexpr long long kHeadWaitCycles = 20000000LL;  // about 10 ms at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase of `parity` has completed, at most `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

// 2-D tiled TMA load of box (x, y) of `map` into shared memory, completing
// on `bar` (x: the innermost coordinate, a multiple of 64 elements here).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand slab written by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes
// apart.  Fields: start address >> 4 (bits 0-13), leading offset (unused for
// this layout, 1), stride offset 1024 >> 4 (bits 32-45), the descriptor
// version 1 (bits 46-47), swizzle mode 2 = 128 bytes (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both
// operands K-major, no negation: D format (bits 4-5) 1 = fp32, A and B
// formats (bits 7-9, 10-12) 1 = bf16, N >> 3 (bits 17-22), M >> 4 (bits
// 24-28).
// (N is added per tile: the rows of a trimmed last tile.)
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kBM >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued before
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Persistent: CTA i owns weight rows [i R, min(K, (i + 1) R)), R a multiple
// of 16 chosen so that every SM gets one slice (the MMA work is balanced),
// processed in tiles of up to 128 rows; a trimmed last tile (a multiple of 16
// rows) is loaded in 16-row boxes and multiplied with N = its rows.  The two
// accumulator buffers in tensor memory (columns [0, 256) and [256, 512), each
// two 128-row halves of 128 columns) let the epilogue of tile t run while the
// MMAs of tile t + 1 fill the other buffer ("tmem full" / "tmem empty"
// mbarriers).  The epilogue is 8 warps: warp 4 + e reads the lane quarter e %
// 4 and the columns [64 (e / 4), 64 (e / 4) + 64) of the tile, and writes
// one partial per (row, tile, column half); slots without columns get the
// neutral partial, so the merge reads every slot.
__global__ void __launch_bounds__(kHeadThreads, 1)
    pruned_head_kernel(const __grid_constant__ CUtensorMap tm_hidden, const __grid_constant__ CUtensorMap tm_w128,
                       const __grid_constant__ CUtensorMap tm_w16, int M, int K, int H, float c, int rows_per_cta,
                       int tiles_per_cta, float4* __restrict__ partial, float* __restrict__ logits,
                       int32_t* __restrict__ stats) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  // stage s: hidden rows [0, 128) at s * kStageBytes, rows [128, 256) after
  // it, the weight slab last; every slab 1024-byte aligned (swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (!spec_smem_ok((smem - smem_raw) + static_cast<size_t>(kStages) * kStageBytes, stats)) return;
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * rows_per_cta, r1 = min(K, r0 + rows_per_cta);
  const int ntile = r1 > r0 ? (r1 - r0 + kBN - 1) / kBN : 0;
  const int m_base = blockIdx.y * 2 * kBM;
  const int nM = M - m_base > kBM ? 2 : 1;
  const int nkb = (H + kBK - 1) / kBK;
  const int nslots = gridDim.x * 2;  // one partial per (row, CTA, column half)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&tfull_bar[j], 1);
      mbar_init(&tempty_bar[j], kEpiWarps);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0 && lane == 0) {
    // producer: the stage ring runs on across the tiles
    int g = 0, issued = 0, consumed_hint = 0;
    for (int t = 0; t < ntile && !*reinterpret_cast<volatile int*>(&s_abort); ++t) {
      const int n0 = r0 + t * kBN, nr16 = (min(kBN, r1 - n0) + 15) & ~15;
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        const int s = g % kStages;
        if (!mbar_wait(&empty_bar[s], (static_cast<uint32_t>(g / kStages) & 1u) ^ 1u, kHeadWaitCycles)) {
          atomicExch(&s_abort, 1);
          break;
        }
        consumed_hint = g - kStages + 1;
        uint8_t* st = smem + static_cast<size_t>(s) * kStageBytes;
        mbar_expect_tx(&full_bar[s], static_cast<uint32_t>(nM * kSlab + nr16 * kBK * 2));
        tma_load_2d(st, &tm_hidden, &full_bar[s], kb * kBK, m_base);
        if (nM == 2) tma_load_2d(st + kSlab, &tm_hidden, &full_bar[s], kb * kBK, m_base + kBM);
        if (nr16 == kBN) {
          tma_load_2d(st + 2 * kSlab, &tm_w128, &full_bar[s], kb * kBK, n0);
        } else {
          for (int i = 0; i < nr16 / kSubRows; ++i)
            tma_load_2d(st + 2 * kSlab + i * kSubRows * kBK * 2, &tm_w16, &full_bar[s], kb * kBK, n0 + i * kSubRows);
        }
        issued = g + 1;
      }
    }
    // after an abort: copies issued but possibly never consumed land before exit
    if (*reinterpret_cast<volatile int*>(&s_abort))
      for (int q = consumed_hint > 0 ? consumed_hint : 0; q < issued; ++q)
        mbar_wait(&full_bar[q % kStages], static_cast<uint32_t>(q / kStages) & 1u, kHeadWaitCycles);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    int g = 0;
    for (int t = 0; t < ntile && !*reinterpret_cast<volatile int*>(&s_abort); ++t) {
      const int j = t & 1;
      const int n0 = r0 + t * kBN, nr16 = (min(kBN, r1 - n0) + 15) & ~15;
      if (!mbar_wait(&tempty_bar[j], (static_cast<uint32_t>(t >> 1) & 1u) ^ 1u, kHeadWaitCycles)) {
        atomicExch(&s_abort, 1);
        break;
      }
      tc_fence_after();
      const uint32_t idesc = kIdescBase | (static_cast<uint32_t>(nr16 >> 3) << 17);
      const uint32_t acc0 = tmem + static_cast<uint32_t>(j * 2 * kBN);
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        const int s = g % kStages;
        if (!mbar_wait(&full_bar[s], static_cast<uint32_t>(g / kStages) & 1u, kHeadWaitCycles)) {
          atomicExch(&s_abort, 1);
          break;
        }
        tc_fence_after();
        const uint32_t st = smem_u32(smem + static_cast<size_t>(s) * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
          const uint64_t bdesc = sw128_desc(st + 2 * kSlab + kk * kUmmaK * 2);
          const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
          tc_mma(acc0, sw128_desc(st + kk * kUmmaK * 2), bdesc, idesc, acc);
          if (nM == 2) tc_mma(acc0 + kBN, sw128_desc(st + kSlab + kk * kUmmaK * 2), bdesc, idesc, acc);
        }
        tc_commit(&empty_bar[s]);  // the stage is free once these MMAs have read it
      }
      tc_commit(&tfull_bar[j]);  // buffer j holds tile t
    }
  } else if (warp >= 4) {
    // epilogue: each thread keeps its rows' partials over the CTA's tiles and
    // writes them once
    const int e = warp - 4, q = warp & 3, grp = e >> 2;
    const int slot = blockIdx.x * 2 + grp;
    float mx[2] = {neg_inf(), neg_inf()}, sum[2] = {0.0f, 0.0f}, bv[2] = {neg_inf(), neg_inf()};
    int bi[2] = {INT_MAX, INT_MAX};
    for (int t = 0; t < ntile; ++t) {
      const int n0 = r0 + t * kBN, nr = min(kBN, r1 - n0);
      const int c_begin = grp * 64, c_end = min(nr, c_begin + 64);
      const int j = t & 1;
      bool ok = mbar_wait(&tfull_bar[j], static_cast<uint32_t>(t >> 1) & 1u, kHeadWaitCycles) &&
                !*reinterpret_cast<volatile int*>(&s_abort);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-wide: the whole warp reads or none
      if (!ok && lane == 0) atomicExch(&s_abort, 1);
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h >= nM || !ok) continue;
        const int row = m_base + h * kBM + q * 32 + lane;
#pragma unroll 1
        for (int c0 = c_begin; c0 < c_end; c0 += 16) {
          uint32_t r[16];
          tc_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(j * 2 * kBN + h * kBN + c0), r);
          const int col0 = n0 + c0;
          float x[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) x[jj] = c0 + jj < c_end ? order_key(__uint_as_float(r[jj])) : neg_inf();
          if (logits != nullptr && row < M && spec_in(n0 + c_end - 1, K, stats)) {
            float* out = logits + static_cast<int64_t>(row) * K + col0;
            if (c0 + 16 <= c_end && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
#pragma unroll
              for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4*>(out + jj) =
                    make_float4(__uint_as_float(r[jj]), __uint_as_float(r[jj + 1]), __uint_as_float(r[jj + 2]),
                                __uint_as_float(r[jj + 3]));
            } else {
              for (int jj = 0; jj < 16 && c0 + jj < c_end; ++jj) out[jj] = __uint_as_float(r[jj]);
            }
          }
          float cm = neg_inf();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            cm = fmaxf(cm, x[jj]);
            if (x[jj] > bv[h]) {  // columns in increasing order: the first largest stays
              bv[h] = x[jj];
              bi[h] = col0 + jj;
            }
          }
          if (cm > mx[h]) {
            sum[h] = mx[h] == neg_inf() ? 0.0f : sum[h] * fast_exp2((mx[h] - cm) * c);
            mx[h] = cm;
          }
          if (mx[h] != neg_inf()) {
            const float mc = mx[h] * c;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) sum[h] += fast_exp2(fmaf(x[jj], c, -mc));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[j]);  // buffer j may be refilled
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = m_base + h * kBM + q * 32 + lane;
      if (h < nM && row < M && spec_in(slot, nslots, stats)) partial[static_cast<int64_t>(row) * nslots + slot] = make_float4(mx[h], sum[h], bv[h], __int_as_float(bi[h]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (threadIdx.x == 0 && s_abort) bump(stats, SPEC_STAT_WAIT_TIMEOUT);
}

// One CTA per row: the row's partials merged in slot order (thread t takes
// slots t, t + 256, ...; then warps, then the CTA, in fixed orders), then
// its top-1 mapped to draft and target ids.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
    head_merge_kernel(int M, int K, int nslots, float c, const float4* __restrict__ partial,
                      const int32_t* __restrict__ ids,
                      const int32_t* __restrict__ d2t, int64_t Vd, int32_t* __restrict__ top1_rank,
                      int32_t* __restrict__ top1_draft, int32_t* __restrict__ top1_target, float* __restrict__ top1_p,
                      float* __restrict__ row_stats, int32_t* __restrict__ stats) {
  pdl_enter();
  constexpr int kWarps = kMergeThreads / 32;
  __shared__ float sm[kWarps], ss[kWarps], sv[kWarps];
  __shared__ int si[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;
  float m = neg_inf(), s = 0.0f, bv = neg_inf();
  int bi = INT_MAX;
  for (int t = threadIdx.x; t < nslots; t += kMergeThreads) {
    const float4 p = __ldg(partial + static_cast<int64_t>(row) * nslots + t);
    merge_ms(m, s, p.x, p.y, c);
    const int pi = __float_as_int(p.w);
    if (before(p.z, pi, bv, bi)) {
      bv = p.z;
      bi = pi;
    }
  }
  warp_merge_ms(m, s, c);
  warp_best(bv, bi);
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  m = sm[0];
  s = ss[0];
  bv = sv[0];
  bi = si[0];
  for (int w = 1; w < kWarps; ++w) {
    merge_ms(m, s, sm[w], ss[w], c);
    if (before(sv[w], si[w], bv, bi)) {
      bv = sv[w];
      bi = si[w];
    }
  }
  const bool finite = isfinite(m) && bi != INT_MAX;
  if (!finite) bump(stats, SPEC_STAT_EMPTY_INTERSECTION);
  const int32_t d = finite && spec_in(bi, K, stats) ? __ldg(ids + bi) : -1;
  if (top1_rank) top1_rank[row] = finite ? bi : -1;
  top1_draft[row] = d;
  top1_target[row] = (d >= 0 && d < Vd) ? __ldg(d2t + d) : -1;
  top1_p[row] = finite ? fminf(fast_exp2(fmaf(bv, c, -(m * c))) / s, 1.0f) : 0.0f;
  if (row_stats) {
    row_stats[2 * row] = m;
    row_stats[2 * row + 1] = s;
  }
}

// cuTensorMapEncodeTiled from the driver, looked up once.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<EncodeTiledFn>(nullptr);
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Tensor map of a row-major bf16 matrix [rows, cols]: boxes of box_rows
// rows x 64 columns (128 bytes), 128-byte swizzle, zero fill out of bounds.
bool bf16_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split of the K weight rows over the CTAs: one slice of R rows (a
// multiple of 16) per SM of the current device.
struct HeadSplit {
  int rows_per_cta, grid, tiles_per_cta, nslots;
};

bool head_split(int64_t K, HeadSplit& h) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || sms < 1) {
    cudaGetLastError();
    return false;
  }
  const int64_t per = ((K + sms - 1) / sms + kSubRows - 1) / kSubRows * kSubRows;
  h.rows_per_cta = static_cast<int>(per);
  h.grid = static_cast<int>((K + per - 1) / per);
  h.tiles_per_cta = static_cast<int>((per + kBN - 1) / kBN);
  h.nslots = h.grid * 2;
  return true;
}

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" size_t tli_pruned_head_ws_size(int64_t M, int64_t K) {
  HeadSplit h;
  if (M < 0 || K < 1 || !head_split(K, h)) return 0;
  return align256(static_cast<size_t>(M) * static_cast<size_t>(h.nslots) * sizeof(float4));
}

extern "C" int tli_pruned_head(int64_t M, int64_t H, int64_t K, const void* hidden, const void* weight,
                               const int32_t* ids, const int32_t* d2t, int64_t V_d, float T, int32_t* top1_draft,
                               int32_t* top1_target, float* top1_p, int32_t* top1_rank_or_null,
                               float* row_stats_or_null, float* logits_or_null, int32_t* stats_or_null, void* ws,
                               size_t ws_bytes, spec_stream_t stream) {
  if (M < 0 || H < 1 || K < 1 || V_d < 1 || !(T > 0.0f) || !isfinite(T)) return SPEC_ERR_INVALID_ARG;
  if (M == 0) return SPEC_OK;
  if (!hidden || !weight || !ids || !d2t || !top1_draft || !top1_target || !top1_p || !ws)
    return SPEC_ERR_INVALID_ARG;
  // TMA: 16-byte aligned bases and row strides (H a multiple of 8 bf16)
  if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(weight) & 15) || (H % 8) != 0)
    return SPEC_ERR_UNSUPPORTED;
  if (K > INT_MAX - kBN || H > INT_MAX || M > 65535LL * 2 * kBM) return SPEC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPEC_ERR_INVALID_ARG;
  HeadSplit hs;
  if (!head_split(K, hs)) return SPEC_ERR_CUDA;
  if (ws_bytes < static_cast<size_t>(M) * static_cast<size_t>(hs.nslots) * sizeof(float4)) return SPEC_ERR_WORKSPACE;
  CUtensorMap tm_h, tm_w128, tm_w16;
  if (!bf16_map(&tm_h, hidden, M, H, kBM) || !bf16_map(&tm_w128, weight, K, H, kBN) ||
      !bf16_map(&tm_w16, weight, K, H, kSubRows))
    return SPEC_ERR_CUDA;
  static const bool smem_ok =
      cudaFuncSetAttribute(pruned_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kHeadSmem)) == cudaSuccess;
  if (!smem_ok) return SPEC_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float c = kLog2e / T;
  float4* partial = static_cast<float4*>(ws);
  launch_k(pruned_head_kernel, dim3(hs.grid, static_cast<unsigned>((M + 2 * kBM - 1) / (2 * kBM))), kHeadThreads,
           kHeadSmem, s, tm_h, tm_w128, tm_w16, static_cast<int>(M), static_cast<int>(K), static_cast<int>(H), c,
           hs.rows_per_cta, hs.tiles_per_cta, partial, logits_or_null, stats_or_null);
  if (launch_status() != SPEC_OK) return SPEC_ERR_CUDA;
  launch_k(head_merge_kernel, static_cast<unsigned>(M), kMergeThreads, 0, s, static_cast<int>(M), static_cast<int>(K),
           hs.nslots,
           c, static_cast<const float4*>(partial), ids, d2t, V_d, top1_rank_or_null, top1_draft, top1_target, top1_p,
           row_stats_or_null, stats_or_null);
  return launch_status();
}
