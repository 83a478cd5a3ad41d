// Shared device helpers of the sm_103a kernels: logit decoding, streaming
// vector loads, the (value desc, index asc) order, warp/block reductions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "specdec.h"

namespace specdec {

constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ inline float neg_inf() { return -__builtin_huge_valf(); }

// Ordering key of a logit: NaN becomes -inf (max.f32 returns the non-NaN
// operand), every other value is kept.
__device__ __forceinline__ float order_key(float x) { return fmaxf(x, neg_inf()); }

// 2^x with the hardware approximation (relative error about 2^-22; inputs
// below -126 flush to 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) with the hardware approximation (log2(0) = -inf).
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int DT>
struct Logit;

// fp32 logits: a 16-byte vector holds 4 elements.
template <>
struct Logit<SPEC_F32> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
};

// bf16 logits: a 16-byte vector holds 8 elements.
template <>
struct Logit<SPEC_BF16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t*>(p) + i)) << 16);
  }
};

// Read-only 16-byte load that does not allocate in L1 (streamed data).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Streaming 16-byte store (evict-first).
__device__ __forceinline__ void st_stream(void* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// 16-byte asynchronous copy global -> shared (cp.async, cached in L2
// only); bytes past src_bytes (0..16) are zero-filled.  The source must be
// 16-byte aligned.  Completion is awaited with cp_async_wait by the issuing
// thread, which alone may then read the destination.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// cp.async of 16 bytes to a shared-memory address given as a 32-bit
// shared-window offset.
__device__ __forceinline__ void cp_async16_s(unsigned smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}

// Streams the 16-byte items src[i], i = tid, tid + THREADS, ... < n, through
// this thread's D slots of a cp.async ring (slot s at ring[s * THREADS +
// tid]), D items in flight; calls f(item, i) in increasing i.  Only the
// issuing thread reads its slots, so no barrier is needed.  The loop runs
// in rounds of D items (item j uses slot j mod D), so slot addresses are
// constants; one commit group per item keeps "item j landed" equal to
// "at most D - 1 groups pending".
template <int THREADS, int D, class F>
__device__ __forceinline__ void ring_stream(const uint4* src, int n, uint4* ring, F&& f) {
  const int tid = threadIdx.x;
  uint4* mine = ring + tid;
  const unsigned sb = static_cast<unsigned>(__cvta_generic_to_shared(mine));
  const uint4* g = src + tid;
  const int cnt = n > tid ? (n - tid + THREADS - 1) / THREADS : 0;  // this thread's items
#pragma unroll
  for (int s = 0; s < D; ++s) {
    if (s < cnt) cp_async16_s(sb + 16u * s * THREADS, g + s * THREADS);
    cp_async_commit();
  }
  int j = 0;
  for (; j + D <= cnt; j += D) {
    const uint4* gn = g + static_cast<int64_t>(j + D) * THREADS;
#pragma unroll
    for (int s = 0; s < D; ++s) {
      cp_async_wait<D - 1>();  // item j + s has landed
      const uint4 v = mine[s * THREADS];
      f(v, tid + (j + s) * THREADS);
      if (j + s + D < cnt) cp_async16_s(sb + 16u * s * THREADS, gn + s * THREADS);
      cp_async_commit();
    }
  }
#pragma unroll
  for (int s = 0; s < D; ++s) {
    if (j + s < cnt) {
      cp_async_wait<D - 1>();
      const uint4 v = mine[s * THREADS];
      f(v, tid + (j + s) * THREADS);
      cp_async_commit();
    }
  }
  cp_async_wait<0>();
}

// Pairs of fp32 lanes (the packed fp32 instructions of sm_100 and later:
// each lane rounds exactly as the scalar operation).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 splat(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 exp2_2(float2 a) { return make_float2(fast_exp2(a.x), fast_exp2(a.y)); }

// s + (sum over even j of 2^(x_j c - mc), sum over odd j of the same): the
// two running sums of an online softmax, one per lane (N even).
template <int N>
__device__ __forceinline__ float2 exp2_sum_pairs(float2 s, const float* x, float c, float mc) {
  const float2 c2 = splat(c), nmc2 = splat(-mc);
#pragma unroll
  for (int j = 0; j < N; j += 2) s = add2(s, exp2_2(fma2(make_float2(x[j], x[j + 1]), c2, nmc2)));
  return s;
}

// s + (sum over j of 2^(x_j c.x - mc.x), sum over j of 2^(x_j c.y - mc.y)):
// one element's terms at two temperatures side by side in a register pair.
// (A polynomial 2^x on the FMA pipe for half of the second terms, to relieve
// the MUFU pipe, measured slower: the row stream is issue-bound.)
template <int N>
__device__ __forceinline__ float2 exp2_sum_two(float2 s, const float* x, float2 c, float2 mc) {
  const float2 nmc = make_float2(-mc.x, -mc.y);
#pragma unroll
  for (int j = 0; j < N; ++j) s = add2(s, exp2_2(fma2(splat(x[j]), c, nmc)));
  return s;
}

// Programmatic dependent launch.  Every kernel of the library is launched
// (launch_k) so that it may be scheduled before the previous kernel on the
// stream has finished; pdl_enter, its first statement, waits until that
// kernel has completed and its writes are visible, then lets the next kernel
// be scheduled.  A kernel must touch no global memory before pdl_enter.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The last launch_k failure of this thread since launch_status last ran.
inline cudaError_t& launch_error() {
  static thread_local cudaError_t e = cudaSuccess;
  return e;
}

// Launch configuration with programmatic stream serialization and, for
// cluster > 1, a thread-block cluster of that many CTAs along x.
struct LaunchCfg {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster = 1) {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (cluster > 1) {
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
  }
  LaunchCfg(const LaunchCfg&) = delete;
};

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             int cluster, Args&&... args) {
  LaunchCfg lc(grid, block, smem, s, cluster);
  const cudaError_t e = cudaLaunchKernelEx(&lc.cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) launch_error() = e;
  return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  return launch_kc(kernel, grid, block, smem, s, 1, std::forward<Args>(args)...);
}

// Thread-block clusters: this CTA's rank, a barrier over every thread of
// every CTA of the cluster (release / acquire: shared-memory writes before
// it, local or remote, are visible after it), and a store into the shared
// memory of another CTA of the cluster at the address that corresponds to
// a local one.
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_f32(float* local, unsigned rank, float v) {
  const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(local));
  unsigned ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_i32(int* local, unsigned rank, int v) {
  const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(local));
  unsigned ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// Flags between CTAs of one launch: a release store (the writer's earlier
// global stores are visible to whoever acquires the flag) and an acquire
// load, both at GPU scope.
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Asynchronous copy of the E elements [v0, v0 + E) of a row (element size
// ESZ, 16-byte aligned base, v0 * ESZ a multiple of 16) into E * ESZ / 16
// chunks slot[0], slot[stride], ...; elements at or past V are zero-filled.
template <int E, int ESZ>
__device__ __forceinline__ void issue_row(uint4* slot, int stride, const void* row, int64_t V, int64_t v0) {
  constexpr int per = 16 / ESZ, nch = E / per;
  const char* src = static_cast<const char*>(row) + v0 * ESZ;
  if (v0 + E <= V) {
#pragma unroll
    for (int c = 0; c < nch; ++c) cp_async16(slot + c * stride, src + 16 * c, 16);
    return;
  }
#pragma unroll
  for (int c = 0; c < nch; ++c) {
    const int64_t left = V - (v0 + c * per);
    const int n = left <= 0 ? 0 : (left >= per ? per : static_cast<int>(left));
    cp_async16(slot + c * stride, n > 0 ? src + 16 * c : row, n * ESZ);
  }
}

// Unpack one 16-byte vector into kVec floats.
template <int DT>
__device__ __forceinline__ void unpack(const uint4& v, float* x);

template <>
__device__ __forceinline__ void unpack<SPEC_F32>(const uint4& v, float* x) {
  x[0] = __uint_as_float(v.x);
  x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z);
  x[3] = __uint_as_float(v.w);
}

template <>
__device__ __forceinline__ void unpack<SPEC_BF16>(const uint4& v, float* x) {
  x[0] = bf16_lo(v.x);
  x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y);
  x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z);
  x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w);
  x[7] = bf16_hi(v.w);
}

// A 16-byte vector of -inf logits.
template <int DT>
__device__ __forceinline__ uint4 neg_inf_vec() {
  const uint32_t w = DT == SPEC_BF16 ? 0xff80ff80u : 0xff800000u;
  return make_uint4(w, w, w, w);
}

// Maximum of the 8 bf16 logits of a 16-byte vector, as a float: three packed
// bf16x2 max operations and one scalar.  NaN elements are ignored (the max
// of a NaN and a number is the number); eight NaNs give NaN.
__device__ __forceinline__ float max8_bf16(const uint4& w) {
  uint32_t a, b;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(w.x), "r"(w.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(w.z), "r"(w.w));
  asm("max.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(b));
  return fmaxf(bf16_lo(a), bf16_hi(a));
}

// (value desc, index asc): true if (va, ia) comes before (vb, ib).
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Warp-wide best (value desc, index asc).
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (before(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Merge two online-softmax partials (m, s), s = sum 2^((x - m) * c).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
  if (m2 > m) {
    s = (m == neg_inf() ? 0.0f : s * fast_exp2((m - m2) * c)) + s2;
    m = m2;
  } else if (m2 != neg_inf()) {
    s += s2 * fast_exp2((m2 - m) * c);
  }
}

__device__ __forceinline__ void warp_merge_ms(float& m, float& s, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge_ms(m, s, m2, s2, c);
  }
}

// Inclusive scan of one float per thread across a block, in thread order;
// also returns the block total.  `sh` holds at least 32 floats.  All threads
// of the block must call it.
__device__ __forceinline__ float block_inclusive_scan(float v, float* sh, float& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    float w = lane < nw ? sh[lane] : 0.0f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) sh[lane] = w;
  }
  __syncthreads();
  total = sh[nw - 1];
  return x + (warp > 0 ? sh[warp - 1] : 0.0f);
}

__device__ __forceinline__ void bump(int32_t* stats, int slot, int n = 1) {
  if (stats != nullptr && n != 0) atomicAdd(stats + slot, n);
}

// Bounds checks of the debug build (compiled with -DSPEC_DEBUG, the library
// libspecdec_debug.so): spec_in(i, n, stats) is whether 0 <= i < n; an index
// outside its buffer is counted (in this module's device counter, which
// spec_debug_bounds sums over the library's modules, and in the caller's
// SPEC_STAT_BOUNDS slot when it passes stats) and the caller skips the
// access: no trap, no assert.  In the release build it is true and costs
// nothing.
#ifdef SPEC_DEBUG
// each .cu file is a device module of its own, with its own counter
static __device__ unsigned int g_spec_bounds;

__device__ __forceinline__ bool spec_in(int64_t i, int64_t n, int32_t* stats) {
  if (i >= 0 && i < n) return true;
  atomicAdd(&g_spec_bounds, 1u);
  bump(stats, SPEC_STAT_BOUNDS);
  return false;
}

// Host: adds this module's count to *total (and zeroes it when reset).
using BoundsReader = int (*)(int64_t* total, int reset);
void register_bounds_reader(BoundsReader r);  // defined once, in verify.cu

namespace {
int read_module_bounds(int64_t* total, int reset) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_spec_bounds, sizeof(v)) != cudaSuccess) return SPEC_ERR_CUDA;
  *total += v;
  if (reset) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_spec_bounds, &z, sizeof(z)) != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}
struct BoundsRegistration {
  BoundsRegistration() { register_bounds_reader(read_module_bounds); }
};
const BoundsRegistration bounds_registration;
}  // namespace

// Whether the first `bytes` of dynamic shared memory that a kernel carves
// up lie within what its launch gave it (the same answer in every CTA of a
// launch, so a kernel may return on false without stranding a barrier).
__device__ __forceinline__ bool spec_smem_ok(size_t bytes, int32_t* stats) {
  uint32_t have;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(have));
  return bytes == 0 || spec_in(static_cast<int64_t>(bytes) - 1, have, stats);
}
#else
__device__ __forceinline__ bool spec_in(int64_t, int64_t, int32_t*) { return true; }
__device__ __forceinline__ bool spec_smem_ok(size_t, int32_t*) { return true; }
#endif

// Aligned vector span of a row: elements [head, head + nvec*kVec) start on a
// 16-byte boundary; [0, head) and the rest are handled one by one.
struct RowSpan {
  int64_t head, nvec;
};

// Visit every element of a row once.  Each thread sees its elements in
// increasing index order: a few leading scalars up to the first 16-byte
// boundary, then 16-byte vectors (UNROLL loads in flight per thread), then
// the trailing scalars.  F provides
//   template <int N> void visit(const float* x, int64_t first_index).
template <int DT, int UNROLL, class F>
__device__ __forceinline__ void for_row(const void* row, int64_t V, F& f);
template <int DT, int UNROLL, class F>
__device__ __forceinline__ void for_row(const void* row, int64_t V, F& f, int tid, int nthreads);

template <int DT>
__device__ __forceinline__ RowSpan row_span(const void* row, int64_t V) {
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kv = Logit<DT>::kVec;
  uintptr_t a = reinterpret_cast<uintptr_t>(row);
  int64_t head = static_cast<int64_t>(((16 - (a & 15)) & 15) / esz);
  if (head > V) head = V;
  int64_t nvec = (V - head) / kv;
  return {head, nvec};
}

inline int launch_status() {
  const cudaError_t e = cudaGetLastError();
  const cudaError_t k = launch_error();
  launch_error() = cudaSuccess;
  return (e == cudaSuccess && k == cudaSuccess) ? SPEC_OK : SPEC_ERR_CUDA;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace specdec

namespace specdec {

template <int DT, int UNROLL, class F>
__device__ __forceinline__ void for_row(const void* row, int64_t V, F& f, int tid, int nthreads) {
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const RowSpan sp = row_span<DT>(row, V);
  const int64_t nt = nthreads;
  for (int64_t i = tid; i < sp.head; i += nt) {
    float x = Logit<DT>::load1(row, i);
    f.template visit<1>(&x, i);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  int64_t i = tid;
  for (; i + (UNROLL - 1) * nt < sp.nvec; i += UNROLL * nt) {
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = ld_stream(vp + i + u * nt);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float x[kv];
      unpack<DT>(v[u], x);
      f.template visit<kv>(x, sp.head + (i + u * nt) * kv);
    }
  }
  for (; i < sp.nvec; i += nt) {
    float x[kv];
    unpack<DT>(ld_stream(vp + i), x);
    f.template visit<kv>(x, sp.head + i * kv);
  }
  for (int64_t t = sp.head + sp.nvec * kv + tid; t < V; t += nt) {
    float x = Logit<DT>::load1(row, t);
    f.template visit<1>(&x, t);
  }
}

template <int DT, int UNROLL, class F>
__device__ __forceinline__ void for_row(const void* row, int64_t V, F& f) {
  for_row<DT, UNROLL>(row, V, f, static_cast<int>(threadIdx.x), static_cast<int>(blockDim.x));
}

}  // namespace specdec

namespace specdec {

// Visit every element of a row once with 16-byte loads (UNROLL in flight per
// thread), handing the visitor raw vectors.  Every thread runs the same
// number of visits, so visitors may use warp votes and shuffles.  F provides
//   void visit_vec(const uint4& raw, int64_t first_index, bool ok)
//   void visit1(float x, int64_t index, bool ok)
// and an invalid slot passes -inf values with ok = false.  Thread t sees the
// vectors t, t + nthreads, ... (and the same for the scalar ends).
template <int DT, int UNROLL, class F>
__device__ __forceinline__ void for_row_raw(const void* row, int64_t V, F& f, int tid, int nthreads) {
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const RowSpan sp = row_span<DT>(row, V);
  const int64_t nt = nthreads;
  for (int64_t i0 = 0; i0 < sp.head; i0 += nt) {
    const int64_t i = i0 + tid;
    const bool ok = i < sp.head;
    f.visit1(ok ? Logit<DT>::load1(row, i) : neg_inf(), i, ok);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  for (int64_t i0 = 0; i0 < sp.nvec; i0 += UNROLL * nt) {
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + tid + u * nt;
      v[u] = i < sp.nvec ? ld_stream(vp + i) : neg_inf_vec<DT>();
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + tid + u * nt;
      f.visit_vec(v[u], sp.head + i * kv, i < sp.nvec);
    }
  }
  for (int64_t t0 = sp.head + sp.nvec * kv; t0 < V; t0 += nt) {
    const int64_t t = t0 + tid;
    const bool ok = t < V;
    f.visit1(ok ? Logit<DT>::load1(row, t) : neg_inf(), t, ok);
  }
}

// for_row_raw for rows of fewer than 2^31 elements, without per-vector
// bounds tests in the full rounds of UNROLL 16-byte vectors; the thread's
// remaining vectors (fewer than UNROLL) are loaded together in one last
// round.  Each thread still sees its elements (the same ones as in
// for_row_raw) in increasing index order; ok is always true.  Not
// warp-uniform (visitors must not use warp collectives).
template <int DT, int UNROLL, class F>
__device__ __forceinline__ void for_row_fast(const void* row, int64_t V64, F& f, int tid, int nthreads) {
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const RowSpan sp = row_span<DT>(row, V64);
  const int V = static_cast<int>(V64), head = static_cast<int>(sp.head), nvec = static_cast<int>(sp.nvec);
  if (tid < head) f.visit1(Logit<DT>::load1(row, tid), tid, true);  // head < kv <= nthreads
  const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + sp.head * esz);
  int i = tid;
  for (; i + (UNROLL - 1) * nthreads < nvec; i += UNROLL * nthreads) {
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = ld_stream(vp + i + u * nthreads);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) f.visit_vec(v[u], head + (i + u * nthreads) * kv, true);
  }
  if (i < nvec) {
    uint4 v[UNROLL - 1 > 0 ? UNROLL - 1 : 1];
#pragma unroll
    for (int u = 0; u < UNROLL - 1; ++u)
      if (i + u * nthreads < nvec) v[u] = ld_stream(vp + i + u * nthreads);
#pragma unroll
    for (int u = 0; u < UNROLL - 1; ++u)
      if (i + u * nthreads < nvec) f.visit_vec(v[u], head + (i + u * nthreads) * kv, true);
  }
  const int t = head + nvec * kv + tid;
  if (t < V) f.visit1(Logit<DT>::load1(row, t), t, true);  // tail < kv <= nthreads
}

}  // namespace specdec
