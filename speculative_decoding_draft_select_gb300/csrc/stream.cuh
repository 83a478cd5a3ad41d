// Row streaming through shared memory: a warp-specialised bulk-copy pipeline.
//
// A persistent CTA owns rows r = blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp kConsumerWarps (the producer) walks that row sequence and copies each
// row's 16-byte-aligned body, CHUNK bytes at a time, into a ring of NSTAGE
// shared-memory stages with cp.async.bulk; completion is counted on the
// stage's "full" mbarrier.  The consumer warps wait on "full", each take a
// slice of the chunk, and release the stage by arriving on its "empty"
// mbarrier (one arrival per consumer warp); the producer waits on "empty"
// before refilling.  No block-wide barrier sits on the streaming path, so up
// to NSTAGE chunks stay in flight across row boundaries while the consumers
// reduce a row (they synchronise among themselves with a named barrier).
// The few elements before the first 16-byte boundary of a row and after the
// last are read directly from global memory.
//
// Every wait is bounded (a suspend-time hint per try_wait and an iteration
// cap).  If one ever runs out, the CTA counts SPEC_STAT_WAIT_TIMEOUT, the
// producer stops issuing, and before leaving the consumers wait (bounded)
// for every copy still in flight.
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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bulk global -> shared copy; bytes and both addresses are multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One bounded wait on an mbarrier phase: each try_wait suspends for at most
// about a microsecond; 1 << 16 of them bound the wait to well under a second.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (int i = 0; i < (1 << 16); ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(1000)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Named barrier over the consumer warps only (barrier 1; 0 is __syncthreads).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
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

template <int CHUNK, int NSTAGE>
struct PipeSmem {
  alignas(128) unsigned char stage[NSTAGE][CHUNK];
  uint64_t full[NSTAGE];
  uint64_t empty[NSTAGE];
  unsigned long long issued;  // chunks the producer issued (valid once done)
  int done;                   // producer finished
  int abort;
};

template <int ESZ, int CHUNK, int NSTAGE, int NCW>
struct RowPipe {
  static constexpr int kConsumers = NCW * 32;
  PipeSmem<CHUNK, NSTAGE>* sm;
  const char* base;
  int64_t V, R, row_bytes;
  uint64_t consumed;  // consumer side, identical in every consumer thread

  // All threads of the CTA.
  __device__ void init(PipeSmem<CHUNK, NSTAGE>* s, const void* rows, int64_t V_, int64_t R_) {
    sm = s;
    base = static_cast<const char*>(rows);
    V = V_;
    R = R_;
    row_bytes = V_ * ESZ;
    consumed = 0;
    if (threadIdx.x == 0) {
      for (int i = 0; i < NSTAGE; ++i) {
        mbar_init(&sm->full[i], 1);
        mbar_init(&sm->empty[i], NCW);
      }
      sm->issued = 0;
      sm->done = 0;
      sm->abort = 0;
      fence_mbar_init();
    }
    __syncthreads();
  }

  // Lane 0 of the producer warp: the whole chunk sequence of this CTA.
  __device__ void produce(int32_t* stats) {
    uint64_t g = 0;
    for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
      const char* row = base + r * row_bytes;
      const RowBody rb = row_body<ESZ>(row, V);
      for (int64_t off = 0; off < rb.bytes; off += CHUNK) {
        const int st = static_cast<int>(g % NSTAGE);
        if (g >= NSTAGE && !mbar_wait(&sm->empty[st], static_cast<uint32_t>((g / NSTAGE - 1) & 1))) {
          atomicExch(&sm->abort, 1);
          bump(stats, SPEC_STAT_WAIT_TIMEOUT);
        }
        if (*reinterpret_cast<volatile int*>(&sm->abort)) {
          r = R;
          break;
        }
        const int64_t left = rb.bytes - off;
        const uint32_t n = static_cast<uint32_t>(left < CHUNK ? left : CHUNK);
        mbar_expect_tx(&sm->full[st], n);
        bulk_g2s(sm->stage[st], row + rb.head * ESZ + off, n, &sm->full[st]);
        ++g;
      }
    }
    sm->issued = g;
    __threadfence_block();
    *reinterpret_cast<volatile int*>(&sm->done) = 1;
  }

  // Consumer threads: wait for the next chunk; nullptr when the CTA has
  // aborted or this wait ran out.
  __device__ const unsigned char* acquire(int32_t* stats) {
    const int lane = threadIdx.x & 31;
    int ab = lane == 0 ? *reinterpret_cast<volatile int*>(&sm->abort) : 0;
    if (__shfl_sync(0xffffffffu, ab, 0)) return nullptr;
    const int st = static_cast<int>(consumed % NSTAGE);
    const bool ok = mbar_wait(&sm->full[st], static_cast<uint32_t>((consumed / NSTAGE) & 1));
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0 && atomicExch(&sm->abort, 1) == 0) bump(stats, SPEC_STAT_WAIT_TIMEOUT);
      return nullptr;
    }
    return sm->stage[st];
  }

  // Consumer threads: this warp is done with the current chunk.
  __device__ void release() {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sm->empty[consumed % NSTAGE]);
    ++consumed;
  }

  // Consumer threads, at the end: after an abort, wait (bounded) for the
  // producer to stop and for every copy it issued to land, so that no copy
  // outlives the CTA.
  __device__ void finish() {
    if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&sm->abort)) {
      for (int i = 0; i < (1 << 20) && !*reinterpret_cast<volatile int*>(&sm->done); ++i) __nanosleep(1000);
      const uint64_t issued = *reinterpret_cast<volatile unsigned long long*>(&sm->issued);
      for (uint64_t g = consumed; g < issued; ++g)
        mbar_wait(&sm->full[g % NSTAGE], static_cast<uint32_t>((g / NSTAGE) & 1));
    }
  }
};

// Consumer threads: visit every element of row r once (the body through the
// pipe, the ends with direct loads).  Within a warp every lane runs the same
// number of visits (warp-uniform): consumer thread t sees the 16-byte vectors
// t, t + NCW*32, ... of each chunk.  F provides
//   void visit_vec(const uint4& raw, int64_t first_index, bool ok)
//   void visit1(float x, int64_t index, bool ok)
// (an invalid slot passes -inf values with ok = false).  After an abort (`aborted` set, here or
// earlier) the row is skipped, but the caller still runs its per-row
// barriers, so every consumer warp reaches the same barriers.
template <int DT, int CHUNK, int NSTAGE, int NCW, class F>
__device__ __forceinline__ void pipe_row(RowPipe<DT == SPEC_BF16 ? 2 : 4, CHUNK, NSTAGE, NCW>& p, int64_t r, F& f,
                                         int32_t* stats, bool& aborted) {
  if (aborted) return;
  constexpr int kv = Logit<DT>::kVec;
  constexpr int esz = DT == SPEC_BF16 ? 2 : 4;
  constexpr int nt = NCW * 32;
  const char* row = p.base + r * p.row_bytes;
  const RowBody rb = row_body<esz>(row, p.V);
  for (int64_t i0 = 0; i0 < rb.head; i0 += nt) {
    const int64_t i = i0 + threadIdx.x;
    const bool ok = i < rb.head;
    f.visit1(ok ? Logit<DT>::load1(row, i) : neg_inf(), i, ok);
  }
  for (int64_t off = 0; off < rb.bytes; off += CHUNK) {
    const unsigned char* st = p.acquire(stats);
    if (st == nullptr) {
      aborted = true;
      return;
    }
    const int64_t left = rb.bytes - off;
    const int nvec = static_cast<int>((left < CHUNK ? left : CHUNK) / 16);
    const int64_t first = rb.head + off / esz;
    for (int v0 = 0; v0 < nvec; v0 += nt) {
      const int v = v0 + static_cast<int>(threadIdx.x);
      const bool ok = v < nvec;
      const uint4 raw = ok ? *reinterpret_cast<const uint4*>(st + v * 16) : neg_inf_vec<DT>();
      f.visit_vec(raw, first + static_cast<int64_t>(v) * kv, ok);
    }
    p.release();
  }
  for (int64_t t0 = rb.tail0; t0 < p.V; t0 += nt) {
    const int64_t t = t0 + threadIdx.x;
    const bool ok = t < p.V;
    f.visit1(ok ? Logit<DT>::load1(row, t) : neg_inf(), t, ok);
  }
}

}  // namespace specdec
