// Internal launch interface between the C ABI (kda_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Arguments of the token-by-token kernel (verify).
struct RecurrentArgs {
  const uint16_t *q, *k, *v, *g, *beta;
  int64_t qkv_stride, g_stride, beta_stride, out_stride;
  const float *A_log, *dt_bias;
  float lower_bound, scale;
  int H;
  // token ranges: cu_seqlens (device) if non-null, else items of T tokens
  const int32_t *cu_seqlens;
  int T;
  // states
  const int32_t *slot_ids;   // non-null when a pool is read or written
  int num_slots;
  const float *state_in;     // pool to seed from (indexed by slot), or null = zero
  float *state_out_pool;     // pool to write the final state to (by slot), or null
  float *state_out_dense;    // [items, H, D, D] final states, or null
  float *inter;              // [items, T, H, D, D] per-step states, or null
  uint16_t *out;
  uint32_t *status;
};

cudaError_t launch_recurrent(const RecurrentArgs &args, int num_items, cudaStream_t stream);

// Arguments of the chunked prefill kernel.
struct ChunkArgs {
  const uint16_t *q, *k, *v, *g, *beta;
  int64_t qkv_stride, g_stride, beta_stride, out_stride;
  const float *A_log, *dt_bias;
  float lower_bound, scale;
  int H, num_seqs, total_tokens;
  const int32_t *cu_seqlens;
  const int32_t *slot_ids;
  int num_slots;
  const float *state_in;
  float *state_out_pool;
  float *state_out_dense;
  uint16_t *out;
  uint32_t *status;
};

// Arguments of the accept/commit copy.
struct CommitArgs {
  float *pool;
  int num_slots;
  const int32_t *slot_ids;
  const int32_t *num_accepted;
  const float *inter;   // [B, T, H, D, D]
  int B, T, H;
  uint32_t *status;
};

cudaError_t launch_commit(const CommitArgs &args, cudaStream_t stream);

// Host-side plan: sequences in the order their CTAs should start (longest
// first), computed from the host copy of cu_seqlens.
constexpr int kMaxPlannedSeqs = 2048;

cudaError_t launch_chunk_prefill(const ChunkArgs &args, const int32_t *cu_seqlens_host,
                                 cudaStream_t stream);

}  // namespace kda
