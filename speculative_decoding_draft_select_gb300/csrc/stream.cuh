// Row streaming through shared memory with bulk asynchronous copies.
//
// A persistent CTA owns rows r = blockIdx.x, blockIdx.x + gridDim.x, ...
// Each row's 16-byte-aligned body is cut into chunks of at most CHUNK bytes
// that thread 0 copies into a ring of NSTAGE shared-memory stages with
// cp.async.bulk (completion counted on one mbarrier per stage).  Up to NSTAGE
// chunks are in flight while the block works on the current one, across row
// boundaries, so HBM stays busy during each row's reductions.  The few
// elements before the first 16-byte boundary and after the last are read
// directly from global memory.
//
// Every wait on an mbarrier is bounded.  If a wait ever runs out, the block
// counts SPEC_STAT_WAIT_TIMEOUT, stops issuing, waits (again bounded) for the
// copies it has in flight and leaves the row loop.
#pragma once

#include "common.cuh"

namespace specdec {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bulk global -> shared copy; bytes and both addresses are multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait: each try_wait may itself suspend for a while; 1 << 22
// attempts is far beyond any copy's latency.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < (1 << 22); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Byte layout of one row for the streamer.
struct RowBody {
  int64_t head;   // leading elements read directly
  int64_t bytes;  // bulk-copied bytes (multiple of 16), starting after head
  int64_t tail0;  // first trailing element read directly
};

template <int ESZ>
__device__ __forceinline__ RowBody row_body(const char* row, int64_t V) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(row);
  int64_t head = static_cast<int64_t>(((16 - (a & 15)) & 15) / ESZ);
  if (head > V) head = V;
  const int64_t nvec = (V - head) * ESZ / 16;
  return {head, nvec * 16, head + nvec * 16 / ESZ};
}

// The shared-memory part a streamer needs: NSTAGE stages of CHUNK bytes
// (16-byte aligned) plus NSTAGE mbarriers.
template <int CHUNK, int NSTAGE>
struct StreamSmem {
  alignas(128) unsigned char stage[NSTAGE][CHUNK];
  uint64_t full[NSTAGE];
  int abort;
};

// Producer/consumer bookkeeping.  The producer (thread 0) walks the same
// (row, chunk) sequence as the consumers, NSTAGE chunks ahead.
template <int ESZ, int CHUNK, int NSTAGE>
struct RowStreamer {
  StreamSmem<CHUNK, NSTAGE>* sm;
  const char* base;  // row 0
  int64_t V, R, row_bytes;
  // producer cursor (thread 0 only)
  int64_t p_row, p_off;
  uint64_t issued;
  // consumer cursor (all threads)
  uint64_t consumed;

  __device__ void init(StreamSmem<CHUNK, NSTAGE>* s, const void* logits, int64_t V_, int64_t R_) {
    sm = s;
    base = static_cast<const char*>(logits);
    V = V_;
    R = R_;
    row_bytes = V_ * ESZ;
    issued = consumed = 0;
    p_row = blockIdx.x;
    p_off = 0;
    if (threadIdx.x == 0) {
      for (int i = 0; i < NSTAGE; ++i) mbar_init(&sm->full[i], 1);
      sm->abort = 0;
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int i = 0; i < NSTAGE; ++i) issue_next();
    __syncthreads();
  }

  // Thread 0: copy the next chunk of the sequence, if any, into its stage.
  __device__ void issue_next() {
    while (p_row < R) {
      const char* row = base + p_row * row_bytes;
      const RowBody rb = row_body<ESZ>(row, V);
      if (p_off < rb.bytes) {
        const int64_t left = rb.bytes - p_off;
        const uint32_t n = static_cast<uint32_t>(left < CHUNK ? left : CHUNK);
        const int st = static_cast<int>(issued % NSTAGE);
        mbar_expect_tx(&sm->full[st], n);
        bulk_g2s(sm->stage[st], row + rb.head * ESZ + p_off, n, &sm->full[st]);
        p_off += n;
        ++issued;
        return;
      }
      p_row += gridDim.x;
      p_off = 0;
    }
  }

  // All threads: wait for the next chunk; returns its stage pointer, or
  // nullptr when the wait ran out (the block then aborts).
  __device__ const unsigned char* acquire(int32_t* stats) {
    const int st = static_cast<int>(consumed % NSTAGE);
    const uint32_t parity = static_cast<uint32_t>((consumed / NSTAGE) & 1);
    if (!mbar_wait(&sm->full[st], parity)) atomicExch(&sm->abort, 1);
    __syncthreads();
    if (sm->abort) {
      if (threadIdx.x == 0) bump(stats, SPEC_STAT_WAIT_TIMEOUT);
      return nullptr;
    }
    return sm->stage[st];
  }

  // All threads: the current chunk has been consumed; thread 0 refills it.
  __device__ void release() {
    __syncthreads();
    ++consumed;
    if (threadIdx.x == 0) issue_next();
  }

  // After an abort: wait (bounded) for every copy still in flight.
  __device__ void drain() {
    if (threadIdx.x == 0) {
      for (uint64_t g = consumed; g < issued; ++g)
        mbar_wait(&sm->full[g % NSTAGE], static_cast<uint32_t>((g / NSTAGE) & 1));
    }
    __syncthreads();
  }
};

// Visit every element of row `r` once, through the streamer for the body and
// with direct loads for the ends.  All threads run the same number of
// visits (warp-uniform, like for_row_uniform): thread t sees the 16-byte
// vectors t, t + blockDim, ... of each chunk.  Returns false if the block
// aborted.
template <int DT, int CHUNK, int NSTAGE, class F>
__device__ __forceinline__ bool stream_row(RowStreamer<DT == SPEC_BF16 ? 2 : 4, CHUNK, NSTAGE>& s, int64_t r,
                                           F& f, int32_t* stats) {
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  const char* row = s.base + r * s.row_bytes;
  const RowBody rb = row_body<esz>(row, s.V);
  const int64_t nt = blockDim.x;
  for (int64_t i0 = 0; i0 < rb.head; i0 += nt) {
    const int64_t i = i0 + threadIdx.x;
    const bool ok = i < rb.head;
    float x = ok ? Logit<DT>::load1(row, i) : neg_inf();
    f.template visit<1>(&x, i, ok);
  }
  for (int64_t off = 0; off < rb.bytes; off += CHUNK) {
    const unsigned char* st = s.acquire(stats);
    if (st == nullptr) return false;
    const int64_t left = rb.bytes - off;
    const int64_t nvec = (left < CHUNK ? left : CHUNK) / 16;
    const int64_t first = rb.head + off / esz;
    for (int64_t v0 = 0; v0 < nvec; v0 += nt) {
      const int64_t v = v0 + threadIdx.x;
      const bool ok = v < nvec;
      float x[kv];
      if (ok) {
        unpack<DT>(*reinterpret_cast<const uint4*>(st + v * 16), x);
      } else {
#pragma unroll
        for (int j = 0; j < kv; ++j) x[j] = neg_inf();
      }
      f.template visit<kv>(x, first + v * kv, ok);
    }
    s.release();
  }
  for (int64_t t0 = rb.tail0; t0 < s.V; t0 += nt) {
    const int64_t t = t0 + threadIdx.x;
    const bool ok = t < s.V;
    float x = ok ? Logit<DT>::load1(row, t) : neg_inf();
    f.template visit<1>(&x, t, ok);
  }
  return true;
}

}  // namespace specdec
