// Internal launch interface between the C ABI (kda_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kda.h"

namespace kda {

// Runs set() the first time a launcher runs on the current device (kernel attributes such as the dynamic
// shared-memory limit belong to the device's context) and returns its status; later calls on that device return
// cudaSuccess.  Thread-safe: concurrent first calls set the attributes once.
template <typename Set>
cudaError_t set_attributes_once(std::mutex &mu, uint64_t &done, Set set) {
  int dev = 0;
  if (const cudaError_t e = cudaGetDevice(&dev)) return e;
  if (dev < 0 || dev >= 64) return set();
  std::lock_guard<std::mutex> lock(mu);
  if ((done >> dev) & 1u) return cudaSuccess;
  const cudaError_t e = set();
  if (e == cudaSuccess) done |= uint64_t(1) << dev;
  return e;
}

// Sigmoid-gated RMSNorm of the output rows (gate == nullptr: none).
struct OutNorm {
  const uint16_t *gate;   // [rows, H, 128] bf16, indexed by the output row
  int64_t gate_stride;
  const float *weight;    // [128]
  float eps;
  float *rstd;            // [rows, H], or null
};

// Short causal convolutions of q, k, v (weight == nullptr: none).  Width 4.
constexpr int kConvW = 4;
struct ShortConv {
  const float *weight;        // [3, H, 128, 4]
  int silu;
  uint16_t *window_pool;      // [slots, 3, 3, H, 128] bf16
  uint16_t *window_dense;     // prefill: [num_seqs, 3, 3, H, 128], or null
  uint16_t *step_windows;     // verify: [B, T, 3, 3, H, 128]
};

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
  const int32_t *out_index;  // output row of each token, or null (row = token)
  int64_t num_out_rows;      // rows of out (bounds out_index)
  OutNorm norm;
  ShortConv conv;
  uint32_t *status;
  // non-null: the grid is launched as a programmatic dependent of the preceding grid; a zeroed counter in the
  // workspace (kDoneCounterOffset) through which the CTA that finishes last waits for that grid
  uint32_t *done_counter;
};

// Byte offset in the workspace of the counter a programmatic-dependent verify grid counts its CTAs with
// (inside the part kda_workspace_reset clears).
constexpr size_t kDoneCounterOffset = 128;
// Counters of the launches of a split prefill schedule (one per launch that waits for its predecessor, at most
// kMaxSplitCounters), from this byte offset of the workspace (also inside the cleared part).
constexpr size_t kSplitCounterOffset = 256;
constexpr int kMaxSplitCounters = 160;

cudaError_t launch_recurrent(const RecurrentArgs &args, int num_items, cudaStream_t stream);

// Host-side checks of one kda_recurrent_verify call without launching anything (the checks the call itself makes
// first); returns KDA_OK or the status the call would return.
int check_verify_call(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_token_stride,
                      const uint16_t *g, int64_t g_token_stride, const uint16_t *beta_logits,
                      int64_t beta_token_stride, const float *A_log, const float *dt_bias, float lower_bound,
                      float scale, int B, int T, int H, const float *state_pool, int num_slots,
                      const int32_t *slot_ids, uint16_t *out, int64_t out_token_stride, float *intermediate_states,
                      void *workspace, size_t workspace_bytes);

enum class PrefillPath { kAuto, kTwoPass, kFused, kOverlap };

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
  const int32_t *out_index;  // output row of each token, or null (row = token)
  int64_t num_out_rows;      // rows of out (bounds out_index)
  OutNorm norm;
  ShortConv conv;            // with conv.weight, q, k, v are the convolutions' raw inputs
  uint32_t *status;
  PrefillPath path;          // forced by the caller, or picked by launch_chunk_prefill
};

// Whether the fused prefill kernel serves a call (else the intra-chunk kernel + state pass do).
bool fused_prefill_applies(const ChunkArgs &args);

// Arguments of the accept/commit copy.
struct CommitArgs {
  float *pool;
  int num_slots;
  const int32_t *slot_ids;
  const int32_t *num_accepted;
  const float *inter;   // [B, T, H, D, D]
  const uint16_t *step_windows;   // [B, T, 3, 3, H, 128] conv windows, or null
  uint16_t *window_pool;          // [slots, 3, 3, H, 128]
  int B, T, H;
  uint32_t *status;
};

cudaError_t launch_commit(const CommitArgs &args, cudaStream_t stream);

// Sequences planned per launch pair of the chunked prefill (longer batches
// are split on the host into consecutive groups).
constexpr int kMaxSeqsPerLaunch = 1024;

// Chunk slots per intra-chunk launch (a group's slots are split on the host into consecutive launches).
constexpr int kMaxSlotsPerLaunch = 4096;

// Intra-chunk kernel: one CTA per (chunk slot, head) of a run of consecutive chunk slots.
struct IntraParams {
  CUtensorMap tq, tk, tv, tg;   // [tokens, H, 128] bf16, box 64 channels x 1 head x 64 tokens; q, k, g
                                // unswizzled, v with the 128-byte swizzle
  const uint16_t *beta;
  int64_t beta_stride;
  const float *A_log, *dt_bias;
  float lower_bound, scale;
  int H;
  int prefetch_ahead;           // a CTA prefetches into L2 the inputs of the CTA this many indices later
  uint8_t *blocks;              // block (local chunk slot g, head h) at blocks + (g H + h) kBlkBytes
  uint32_t *status;
  // short convolutions (conv.weight set): raw q, k, v, and the windows that a sequence's first chunk starts from
  ShortConv conv;
  const uint16_t *xq, *xk, *xv;
  int64_t qkv_stride;
  const int32_t *slot_ids;      // pool slot of each sequence (indexed by seq0 + local sequence)
  int num_slots;                // a slot outside [0, num_slots) reads a zero window (the state pass reports it)
  int seq0;
  int conv_load_initial;        // first chunks start from the slot's window (else from zeros)
  // non-null: the grid is launched as a programmatic dependent of a state pass (split state passes), and the CTA
  // that finishes last waits for that grid's completion through this zeroed counter in the workspace header
  uint32_t *done_counter;
  int32_t slot_tok0[kMaxSlotsPerLaunch];   // first token of each local chunk slot
  uint8_t slot_valid[kMaxSlotsPerLaunch];  // its tokens (1..64) | kSlotFirst for a sequence's first chunk
  int16_t slot_seq[kMaxSlotsPerLaunch];    // its sequence, local to the group
};
constexpr uint8_t kSlotFirst = 128;
static_assert(sizeof(IntraParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// State pass: one CTA per (item, head).  An item is a run of whole chunks of one sequence: the whole sequence,
// or one segment of it when a long sequence's state pass is split (its state then passes from one segment to the
// next through `state_mid`, in fp32 and in the caller's layout).
constexpr uint8_t kItemFromMid = 1;   // the item's initial state is state_mid[mid] (else the pool slot / zero)
constexpr uint8_t kItemToMid = 2;     // its final state goes to state_mid[mid] (else the pool slot / dense)
struct ChainParams {
  CUtensorMap tout;             // output [tokens, H, 128] bf16, box 64 channels x 1 head x 64 tokens
  const uint8_t *blocks;
  const int32_t *slot_ids;      // indexed by the item's sequence
  int num_slots;
  const float *state_in;
  float *state_out_pool;
  float *state_out_dense;       // indexed by the item's sequence
  float *state_mid;             // [segmented sequences, H, 128, 128] fp32, or null
  uint16_t *out;
  int64_t out_stride;
  const int32_t *out_index;     // output row of each token (global token index), or null (row = token)
  int64_t num_out_rows;
                                // (with out_index the rows are stored one by one, else by TMA)
  // short convolutions (conv.weight set): each sequence's final window goes to the pool with the final state,
  // else to conv.window_dense
  ShortConv conv;
  const uint16_t *xq, *xk, *xv;
  int64_t qkv_stride;
  int conv_load_initial;
  uint32_t *status;
  // Programmatic dependent launch.  wait_blocks: one thread waits for the preceding grid (the intra-chunk
  // launch that wrote this launch's blocks) before the first block is read; else the blocks are complete when
  // the grid is launched.  trigger_after_wait: the grid lets its own dependent launch only once that wait has
  // returned (else at its start).  done_counter (non-null): a zeroed counter in the workspace header through
  // which the CTA that finishes last waits for the preceding grid's completion.
  int wait_blocks, trigger_after_wait;
  uint32_t *done_counter;
  int H, num_seqs;              // num_seqs: items of the launch
  int32_t chunk_off[kMaxSeqsPerLaunch];       // first block of each item (its ceil(len / 64) blocks follow)
  int32_t tok0[kMaxSeqsPerLaunch];            // first token of each item
  int32_t len[kMaxSeqsPerLaunch];             // its tokens
  int32_t seq[kMaxSeqsPerLaunch];             // its sequence (index into slot_ids, state_out_dense, windows)
  uint8_t flags[kMaxSeqsPerLaunch];           // kItemFromMid | kItemToMid
  uint8_t mid[kMaxSeqsPerLaunch];             // its state's index in state_mid
  uint16_t order[kMaxSeqsPerLaunch];          // items, longest first
};
static_assert(sizeof(ChainParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// (sequence, head) pairs whose state passes may be split into segments at once, and the fp32 scratch their
// states pass through between segments (placed after the blocks in the prefill workspace)
constexpr int kMaxOverlapPairs = 96;
size_t overlap_scratch_bytes(int num_seqs, int H);

// Fused prefill: one CTA per (sequence, head) of a group builds each chunk's WY operands and runs the state
// recurrence over them without leaving the SM (kda_prefill_fused.cu).
struct FusedParams {
  CUtensorMap tq, tk, tg;       // [tokens, H, 128] bf16, box 64 channels x 1 head x 64 tokens, unswizzled
  CUtensorMap tv;               // the same for v, 128-byte swizzle (an MMA operand)
  CUtensorMap tout;             // output, 128-byte swizzle
  const uint16_t *beta;
  int64_t beta_stride;
  const float *A_log, *dt_bias;
  float lower_bound, scale;
  const int32_t *slot_ids;      // indexed by seq0 + local sequence
  int num_slots;
  const float *state_in;
  float *state_out_pool;
  float *state_out_dense;       // indexed by seq0 + local sequence
  uint16_t *out;
  int64_t out_stride;
  uint32_t *status;
  int H, num_seqs, seq0;
  int32_t tok_off[kMaxSeqsPerLaunch + 1];
  uint16_t order[kMaxSeqsPerLaunch];          // local sequences, longest first
};
static_assert(sizeof(FusedParams) <= 32764, "kernel parameters are limited to 32764 bytes");

cudaError_t launch_prefill_fused(const FusedParams &p, cudaStream_t stream);

// Gated RMSNorm of stored output rows, in place (the prefill's rows, after its state pass).
struct GatedNormArgs {
  uint16_t *out;
  int64_t out_stride;
  const int32_t *row_index;   // output row of token t, or null (row = t)
  int64_t num_rows;           // rows of out (bounds row_index)
  int num_tokens, H;
  OutNorm norm;
};

cudaError_t launch_gated_norm(const GatedNormArgs &args, cudaStream_t stream);

// programmatic: launched as a programmatic dependent of the preceding grid in the stream (a state pass)
cudaError_t launch_chunk_intra(const IntraParams &p, int num_chunks, cudaStream_t stream, bool programmatic);
// programmatic: launched as a programmatic dependent of the preceding grid in the stream (the intra-chunk grid);
// value_split: two CTAs per (item, head), each owning 64 of the value channels (shorter serial path per chunk)
cudaError_t launch_chunk_chain(const ChainParams &p, cudaStream_t stream, bool programmatic, bool value_split);

// Bytes of workspace kda_chunk_prefill needs (status header + one block per chunk and head); the split state
// passes also need overlap_scratch_bytes after the blocks.
size_t prefill_workspace_bytes(int64_t total_tokens, int num_seqs, int H);

// blocks: the workspace after its header, blocks_bytes long
cudaError_t launch_chunk_prefill(const ChunkArgs &args, const int32_t *cu_seqlens_host, uint8_t *blocks,
                                 size_t blocks_bytes, cudaStream_t stream);
// The schedule launch_chunk_prefill takes for `args` (host only, nothing launched): info[0] the kind (1 fused
// kernel, 2 plain schedule, 3 split schedule), info[1] whether the state passes take the value-split kernel,
// info[2] the split's segments, info[3] the sequences whose state passes are split.  sms <= 0: the current
// device's SM count (152 without one).
void describe_prefill_schedule(const ChunkArgs &args, const int32_t *cu_seqlens_host, size_t blocks_bytes, int sms,
                               int info[4]);

}  // namespace kda
