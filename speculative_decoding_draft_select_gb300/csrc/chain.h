// Stochastic verify of chains (every node has at most one child): the launch
// that verify.cu's entry points call when the caller sets
// SPEC_VERIFY_CHAIN.  Defined in chain.cu.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace specdec {

// Where the draft distribution q comes from: fp32 rows, or draft logit rows
// (bf16 or fp32) with each row's (max, normaliser) at the temperature of cq.
struct ChainQ {
  int kind;  // 0: fp32 probabilities, 1: bf16 logits, 2: fp32 logits
  const void* q;
  const float* q_stats;
  float cq;
};

struct ChainIO {
  const int32_t *q_row, *dtok, *ntok, *nsib;
  const float *coins, *u_final;
  const int32_t* budget;
  int32_t eos;
  int32_t *committed, *num_committed, *accept_length, *accept_path, *next_root, *walk_info, *stats;
  // optional: committed ids mapped through a table (target -> draft ids),
  // table[id] when in range and >= 0, else the fallback; -1 padded
  const int32_t* map_table;
  int64_t map_len;
  int32_t map_fallback;
  int32_t* committed_mapped;
};

// Bytes of per-request workspace the chain verify needs beyond the per-row
// flags, maxima and normalisers.
size_t chain_ws_bytes(int B, int N);

// Enqueues the chain verify on s.  ready: B*N ints (zeroed here), m_row /
// z_row: B*N floats, req_ws: chain_ws_bytes(B) bytes, 256-byte aligned.
int chain_verify(int dtype, int B, int N, int64_t V, const void* target, float c, const ChainQ& q,
                 const ChainIO& io, int32_t* ready, float* m_row, float* z_row, void* req_ws, cudaStream_t s);

}  // namespace specdec
