/*
 * kda.h -- C ABI of libkda: the Kimi Delta Attention (KDA) bounded-gate
 * recurrence on one GB300 (sm_103a) GPU.
 *
 * What the calls compute, per sequence n, head h and token t (token order):
 *
 *   q^ = q / sqrt(sum_c q_c^2 + 1e-6),  k^ likewise      ("in-kernel q/k l2norm")
 *   beta    = sigmoid(beta_logit)                           ("raw beta logits")
 *   lambda_c = lower_bound * sigmoid(exp(A_log[h]) * (g_c + dt_bias[h][c]))
 *   S_t = (I - beta k^ k^T) Diag(exp(lambda)) S_{t-1} + beta k^ v^T
 *   o_t = scale * S_t^T q^
 *
 * The gate, the in-kernel l2norm and the raw beta logits are the bounded-gate
 * KDA recurrence of vLLM PR #55737 "Use FlashKDA for KDA chunked prefill"
 * (PR summary and Purpose); the verify semantics (pool read-only, one state
 * record per draft step) are those of TensorRT-LLM PR #21179 "GLM-5.3-Flash
 * FP8 performance fixes on Hopper" (commit adding the one-launch KDA verify).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - head_dim is fixed at 128 for keys and values (dk = dv = 128).
 *  - Token tensors are [tokens, H, 128] with the 128 channels of a head
 *    contiguous and heads packed contiguously (head stride 128 elements); the
 *    token stride is given in ELEMENTS and may exceed H*128 (tensors read in
 *    place from a fused projection).  bf16 tensors are passed as uint16_t*
 *    holding bf16 bit patterns.
 *  - beta_logits is [tokens, H] bf16 with its own token stride (elements).
 *  - A_log is fp32 [H]; dt_bias is fp32 [H, 128].
 *  - States are fp32 [.., H, 128 (key channel), 128 (value channel)],
 *    row-major, 64 KiB per (slot or sequence, head).
 *  - Every pointer except cu_seqlens_host is a DEVICE pointer on the current
 *    device; all must be 16-byte aligned and the token strides multiples of 8
 *    elements (16 bytes).
 *  - Ownership: the caller allocates every buffer, including the workspace.
 *    The library never allocates device memory, never synchronises the
 *    stream or the device, and launches only on `stream` (a cudaStream_t;
 *    NULL = legacy default stream).
 *  - Errors: argument errors are detected on the host before any launch and
 *    returned as a KDA_ERR_* code with nothing launched.  Bad values that only
 *    the device can see (a slot id outside [0, num_slots)) make the kernel skip
 *    that sequence/request and OR a KDA_DEVICE_* bit into the status word at
 *    the start of the workspace; the word is sticky until kda_workspace_reset.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define KDA_OK 0
#define KDA_ERR_INVALID_ARG 1 /* NULL / misaligned pointer, bad size or stride, bad cu_seqlens */
#define KDA_ERR_UNSUPPORTED 2 /* lower_bound outside [-10, 0], non-finite scale, too many sequences */
#define KDA_ERR_WORKSPACE 3   /* workspace NULL, misaligned or smaller than kda_workspace_size() */
#define KDA_ERR_CUDA 4        /* a CUDA runtime call or kernel launch failed */

/* ---- bits of the device status word (first 4 bytes of the workspace) ---- */
#define KDA_DEVICE_BAD_SLOT 1u /* a slot id was outside [0, num_slots); that work item was skipped */
#define KDA_DEVICE_TIMEOUT 2u  /* a bounded wait inside a kernel gave up (a lost async completion); results are incomplete */
#define KDA_DEVICE_BAD_COUNT 4u /* an accepted-token count was outside [0, T]; that request was skipped */
#define KDA_DEVICE_BAD_INDEX 8u /* an output row index was outside [0, num_out_tokens); that row was not written */

/*
 * Slot id of a padding row.  A batch captured in a CUDA graph for a bucket of
 * B requests and replayed with fewer live requests fills the unused rows of
 * slot_ids with this value; kda_recurrent_verify and kda_commit_accepted skip
 * such rows without touching their outputs or setting a status bit (a padded
 * batch runs only its live rows, TensorRT-LLM PR #21179, breakable prefill
 * CUDA graphs commit).  Any other id outside [0, num_slots) is an error.
 */
#define KDA_PAD_SLOT_ID (-1)

/* ---- flags of kda_chunk_prefill ------------------------------------------ */
#define KDA_LOAD_INITIAL 1  /* S0 of sequence n = state_pool[slot_ids[n]]; else S0 = 0          */
#define KDA_FINAL_TO_POOL 2 /* final state of sequence n -> state_pool[slot_ids[n]]; else dense */
/* Execution path of kda_chunk_prefill (at most one of the three; none: the library picks).  All paths
 * compute the same result within rounding; KDA_TWO_PASS and KDA_OVERLAP the same bits.
 *  KDA_TWO_PASS  the intra-chunk kernel over every chunk and head, then the state pass over every
 *                (sequence, head), the chunks' operands handed over through the workspace;
 *  KDA_FUSED     one kernel, one CTA per (sequence, head), every chunk's operands kept on chip; it
 *                applies without short convolutions and with lower_bound >= -5 (else the call returns
 *                KDA_ERR_UNSUPPORTED);
 *  KDA_OVERLAP   the kernels of KDA_TWO_PASS, with the state passes of the longest sequences (as many
 *                (sequence, head) pairs as fit in half of the SMs, at most 96) split into segments of whole
 *                chunks.  The call is then one chain of programmatic dependent launches on `stream`:
 *                intra-chunk work of segment k, the state pass of segment k, intra-chunk work of segment
 *                k + 1 (beside it, on the SMs it leaves free), ..., and the state pass of the other
 *                sequences beside the last segment's.  A segment's final state reaches the next through
 *                the workspace (fp32), so the results are those of KDA_TWO_PASS bit for bit.  The
 *                workspace must hold kda_prefill_workspace_size() bytes (else KDA_ERR_WORKSPACE).
 * With no path flag the library takes KDA_FUSED for sequences of one chunk that fit one wave of SMs,
 * KDA_OVERLAP where the longest sequence has 64 chunks or more and every sequence of at least half its
 * length fits the split's budget (and the workspace holds the scratch), else KDA_TWO_PASS. */
#define KDA_TWO_PASS 4
#define KDA_FUSED 8
#define KDA_OVERLAP 16

/*
 * q, k, v, g and beta_logits of one set of tokens, laid out as in the
 * conventions above (used by kda_spec_step, which takes two such sets).
 */
typedef struct kda_token_tensors {
  const uint16_t *q, *k, *v;     /* [tokens, H, 128] bf16 */
  int64_t qkv_token_stride;      /* elements, shared by q, k, v */
  const uint16_t *g;             /* [tokens, H, 128] bf16 raw gate input */
  int64_t g_token_stride;
  const uint16_t *beta_logits;   /* [tokens, H] bf16 */
  int64_t beta_token_stride;
} kda_token_tensors;

/*
 * Optional sigmoid-gated RMSNorm applied to every output row before it is
 * stored ("sigmoid RMSNorm" / "gated norm" on BF16 D = 128 rows with output
 * and rstd compared: sglang PR #42489 "Improve GLM-5.3-Flash DFlash decoding
 * on B300", Modifications and review thread).  Per output row r and head h,
 * with o the attention output of that row and head:
 *   rstd = 1 / sqrt(mean_c o_c^2 + eps),  y_c = o_c * rstd * weight_c * sigmoid(gate_c)
 * and y (bf16) is stored instead of o.  The pages print no formula; this
 * normalise-then-gate form is the reading taken.  The verify kernel applies
 * it to its fp32 output in its epilogue; the prefill's rows are normalised
 * from their stored bf16 values by one more row-parallel kernel after the
 * state pass (on every SM, at HBM speed), which the call launches last.
 * Caller-owned device memory; gate and weight 16-byte aligned, rstd 4-byte;
 * a NULL gate or weight, a bad alignment or stride, or eps < 0 / NaN returns
 * KDA_ERR_INVALID_ARG before anything is launched.
 */
typedef struct kda_output_norm {
  const uint16_t *gate;          /* [rows, H, 128] bf16, row = the output row; token stride below */
  int64_t gate_token_stride;     /* elements, a multiple of 8 and >= H*128 */
  const float *weight;           /* [128] fp32, shared by the heads */
  float eps;                     /* >= 0 */
  float *rstd;                   /* [rows, H] fp32 (row-major), or NULL */
} kda_output_norm;

/*
 * Optional short causal convolutions of q, k and v ("three short
 * convolutions" per step with per-step windows: TensorRT-LLM PR #21179
 * "GLM-5.3-Flash FP8 performance fixes on Hopper", KDA verify commit).  With
 * one, the q, k, v tensors a call receives are the RAW inputs of the
 * convolutions; per channel c of each of the three and per token,
 *   y_c = act( w_c[0] x_{t-3} + w_c[1] x_{t-2} + w_c[2] x_{t-1} + w_c[3] x_t )
 * with act = SiLU or none, and y replaces q, k, v in the recurrence.  Inputs
 * before a sequence's first token come from its window: the 3 previous raw
 * inputs, oldest first, kept per pool slot beside the recurrent state.  The
 * pages print neither the width nor the activation: width 4 and SiLU are the
 * readings taken (the activation is selectable).
 * Caller-owned device memory, every pointer 16-byte aligned.  A NULL or
 * misaligned weight, an unknown activation, or a buffer the call needs that is
 * NULL or misaligned (the pool when the call reads or writes windows there,
 * window_dense for dense final states, step_windows for verify and commit)
 * returns KDA_ERR_INVALID_ARG before anything is launched.  Pool slots outside
 * [0, num_slots) behave as for the recurrent state (skipped, status bit).
 */
#define KDA_CONV_NONE 0
#define KDA_CONV_SILU 1
typedef struct kda_short_conv {
  const float *weight;           /* [3 (q, k, v), H, 128, 4] fp32; tap 3 on the current input */
  int activation;                /* KDA_CONV_SILU or KDA_CONV_NONE */
  uint16_t *window_pool;         /* [num_slots, 3, 3, H, 128] bf16 raw inputs: tensor, row (oldest first), head, channel */
  uint16_t *window_dense;        /* kda_chunk_prefill: [num_seqs, 3, 3, H, 128] final windows when the final
                                    states are dense (else NULL); ignored elsewhere */
  uint16_t *step_windows;        /* kda_recurrent_verify: [B, T, 3, 3, H, 128] window after each draft token;
                                    kda_commit_accepted: the same records, read */
} kda_short_conv;

/* Static, human-readable text for a status code. */
KDA_API const char *kda_status_string(int status);

/* Bytes of workspace every call needs (a multiple of 256). */
KDA_API size_t kda_workspace_size(void);

/*
 * Bytes of workspace kda_chunk_prefill needs for total_tokens tokens in
 * num_seqs sequences and H heads: kda_workspace_size() plus, for every chunk of
 * 64 tokens and head, the 74240-byte block the intra-chunk kernel hands to the
 * state pass (an upper bound: floor(total_tokens / 64) + num_seqs chunks), plus
 * 64 KiB for each of min(num_seqs * H, 96) (sequence, head) states that split
 * state passes (KDA_OVERLAP) hand from one segment to the next.  A call given
 * the blocks but not that scratch runs without the split.
 * Returns 0 for negative sizes or H <= 0.
 */
KDA_API size_t kda_prefill_workspace_size(int64_t total_tokens, int num_seqs, int H);

/*
 * The schedule kda_chunk_prefill takes for a call with these sequence lengths
 * (cu_seqlens_host [num_seqs + 1], host memory), H heads, flags, lower_bound,
 * short convolutions present (with_conv != 0) and workspace_bytes of workspace,
 * on a GPU with `sms` SMs (sms <= 0: the current device's, or 152 without one).
 * Host only: no device memory is read and nothing is launched, so it also runs
 * without a GPU.  The arguments are checked as kda_chunk_prefill checks them
 * (num_seqs >= 1).  On KDA_OK, info[4] holds:
 *   info[0]  KDA_SCHEDULE_FUSED (one fused kernel), KDA_SCHEDULE_PLAIN (the
 *            intra-chunk kernel, then the state pass over every chunk) or
 *            KDA_SCHEDULE_SPLIT (the longest sequences' state passes split into
 *            segments chained as programmatic dependent launches)
 *   info[1]  1 if the state passes (plain) or the split sequences' state passes
 *            run on two CTAs of 64 value channels per (sequence, head)
 *   info[2]  segments of the split schedule (0 otherwise)
 *   info[3]  sequences whose state passes are split (0 otherwise)
 * A spec step's prefill segment (rows stored by index) never takes the fused
 * kernel or the value split; this call describes kda_chunk_prefill.
 */
#define KDA_SCHEDULE_FUSED 1
#define KDA_SCHEDULE_PLAIN 2
#define KDA_SCHEDULE_SPLIT 3
KDA_API int kda_prefill_schedule(const int32_t *cu_seqlens_host, int num_seqs, int H, int flags,
                                 float lower_bound, int with_conv, size_t workspace_bytes, int sms,
                                 int *info);

/* Clear the device status word and the rest of the first kda_workspace_size()
 * bytes (an async memset on `stream`). */
KDA_API int kda_workspace_reset(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Debug helper: wait for `stream`, then copy the device status word into
 * *device_status.  This is the only call that synchronises.
 */
KDA_API int kda_read_device_status(const void *workspace, size_t workspace_bytes,
                           uint32_t *device_status, void *stream);

/*
 * Chunked varlen prefill.  Source: vLLM PR #55737 "Use FlashKDA for KDA
 * chunked prefill" (PR summary: bounded gate, in-kernel q/k l2norm, raw beta
 * logits, output plus final state, output written straight into the caller's
 * buffer); host cu_seqlens so that planning never reads device memory:
 * TensorRT-LLM PR #21179, commit passing cu_seqlens_cpu to chunked prefill.
 *
 *  q, k, v          [T_total, H, 128] bf16, token stride qkv_token_stride
 *  g                [T_total, H, 128] bf16 raw gate input, token stride g_token_stride
 *  beta_logits      [T_total, H] bf16, token stride beta_token_stride
 *  A_log [H], dt_bias [H,128] fp32; lower_bound in [-10, 0]; scale finite
 *  cu_seqlens_dev   [num_seqs + 1] int32 on the device, cu_seqlens_host the
 *                   same values in host memory (must be equal; starts at 0,
 *                   non-decreasing).  Zero-length sequences are allowed: their
 *                   final state is their initial state.
 *  state_pool       [num_slots, H, 128, 128] fp32; required when flags has
 *                   KDA_LOAD_INITIAL or KDA_FINAL_TO_POOL, with slot_ids
 *                   [num_seqs] int32 (distinct when KDA_FINAL_TO_POOL).
 *  out              [T_total, H, 128] bf16, token stride out_token_stride
 *  norm             NULL, or the gated RMSNorm applied to each output row
 *                   (gate and rstd rows are token rows)
 *  conv             NULL, or the short convolutions of q, k, v (q, k, v are then
 *                   their raw inputs): a sequence starts from its slot's window
 *                   with KDA_LOAD_INITIAL (else from zeros) and its final window
 *                   goes to the pool with KDA_FINAL_TO_POOL (else to window_dense)
 *  final_state      [num_seqs, H, 128, 128] fp32 dense final states; required
 *                   unless KDA_FINAL_TO_POOL (then ignored, may be NULL).
 *  Inputs and outputs must not overlap, except state_pool which may be both
 *  read and written (each sequence reads its slot before writing it).
 *  workspace        kda_prefill_workspace_size(cu_seqlens_host[num_seqs],
 *                   num_seqs, H) bytes (fewer than its header and blocks:
 *                   KDA_ERR_WORKSPACE; without its scratch states the call
 *                   takes no split schedule); its first word is the device
 *                   status word, the rest is scratch that the call overwrites
 *                   (the fused path uses only the header).
 *                   Concurrent calls need separate workspaces.
 *  flags            KDA_LOAD_INITIAL | KDA_FINAL_TO_POOL, and at most one of
 *                   KDA_TWO_PASS, KDA_FUSED, KDA_OVERLAP; other bits:
 *                   KDA_ERR_INVALID_ARG.
 */
KDA_API int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int64_t qkv_token_stride, const uint16_t *g, int64_t g_token_stride,
                      const uint16_t *beta_logits, int64_t beta_token_stride,
                      const float *A_log, const float *dt_bias, float lower_bound, float scale,
                      const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
                      int num_seqs, int H, float *state_pool, int num_slots,
                      const int32_t *slot_ids, int flags, uint16_t *out,
                      int64_t out_token_stride, const kda_output_norm *norm,
                      const kda_short_conv *conv, float *final_state, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * Speculative-decode verify over a pooled fp32 state.  Source: TensorRT-LLM
 * PR #21179 "GLM-5.3-Flash FP8 performance fixes on Hopper", commit fusing
 * the verify loop into one recurrent call that seeds from the pool state and
 * writes step t's state to row (b, t), the live pool staying read-only.
 *
 *  q, k, v, g       [B*T, H, 128] bf16 (request b's draft tokens are rows b*T .. b*T+T-1)
 *  beta_logits      [B*T, H] bf16
 *  state_pool       [num_slots, H, 128, 128] fp32, READ ONLY
 *  slot_ids         [B] int32, any values in [0, num_slots) (repeats allowed),
 *                   or KDA_PAD_SLOT_ID for a padding row (its out rows and
 *                   intermediate_states rows are left as they were)
 *  out              [B*T, H, 128] bf16
 *  norm             NULL, or the gated RMSNorm applied to each output row
 *                   (gate and rstd rows are token rows b*T + t)
 *  conv             NULL, or the short convolutions of q, k, v (q, k, v are then
 *                   their raw inputs): request b starts from window_pool[slot_ids[b]]
 *                   (read only) and the window after each draft token t goes to
 *                   step_windows[b, t]
 *  intermediate_states [B, T, H, 128, 128] fp32: row (b, t) = state after draft token t
 *  1 <= T <= 64.
 *
 * The call reads no device memory on the host and derives its launch from
 * (B, T, H) alone, so it can be captured in a CUDA graph once per (B, T)
 * bucket and replayed with new token data and slot ids in the same buffers.
 */
KDA_API int kda_recurrent_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t qkv_token_stride, const uint16_t *g, int64_t g_token_stride,
                         const uint16_t *beta_logits, int64_t beta_token_stride,
                         const float *A_log, const float *dt_bias, float lower_bound,
                         float scale, int B, int T, int H, const float *state_pool,
                         int num_slots, const int32_t *slot_ids, uint16_t *out,
                         int64_t out_token_stride, const kda_output_norm *norm,
                         const kda_short_conv *conv, float *intermediate_states, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Accept/commit after kda_recurrent_verify.  Source: vLLM PR #55737 "Use
 * FlashKDA for KDA chunked prefill" (follow-up commit: speculative tokens keep
 * the recurrent kernel "with num_accepted_tokens rollback"), over the per-step
 * states of TensorRT-LLM PR #21179's one-launch verify.
 *
 * For each request b with n = num_accepted[b] accepted draft tokens, copies
 * intermediate_states[b, n-1] (all heads) into state_pool[slot_ids[b]]; n = 0
 * leaves the slot untouched.  Counts outside [0, T] or slots outside
 * [0, num_slots) skip that request and set a device status bit, except
 * KDA_PAD_SLOT_ID rows, which are skipped without one.  With conv, the window
 * after token n-1 (conv->step_windows[b, n-1]) goes to conv->window_pool[slot]
 * in the same way.
 *
 *  state_pool          [num_slots, H, 128, 128] fp32, written
 *  slot_ids            [B] int32 device, distinct (padding rows excepted)
 *  num_accepted        [B] int32 device
 *  intermediate_states [B, T, H, 128, 128] fp32 (as written by kda_recurrent_verify)
 */
KDA_API int kda_commit_accepted(float *state_pool, int num_slots, const int32_t *slot_ids,
                                const int32_t *num_accepted, const float *intermediate_states,
                                const kda_short_conv *conv, int B, int T, int H, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * One speculative-decoding step of a KDA layer: the prefill segment (the
 * non-speculative tokens, chunked, as kda_chunk_prefill) and the verify
 * segment (B requests x T draft tokens, as kda_recurrent_verify) in one call,
 * both writing their outputs straight into the layer's output rows through
 * the step's index arrays.  Source: vLLM PR #55737 "Use FlashKDA for KDA
 * chunked prefill", follow-up commit: in a step that carries spec-decode
 * tokens the prefill segment runs on the chunked kernel, its outputs are
 * scattered by non_spec_token_indx, the spec tokens' by spec_token_indx
 * (recurrent kernel, num_accepted_tokens rollback), and the merge writes
 * directly into core_attn_out.  Here no intermediate output buffer and no
 * merge pass exist: each kernel stores its rows at their final place.
 *
 *  prefill          tokens of the prefill segment ([T_p, H, 128], T_p =
 *                   cu_seqlens_host[num_seqs]); may be NULL when num_seqs == 0
 *  cu_seqlens_dev / cu_seqlens_host / num_seqs / prefill_slot_ids / flags /
 *  final_state      as in kda_chunk_prefill (num_seqs == 0: no prefill segment)
 *  spec             tokens of the verify segment ([B*T, H, 128]); may be NULL when B == 0
 *  B, T, spec_slot_ids, intermediate_states
 *                   as in kda_recurrent_verify (B == 0: no verify segment;
 *                   KDA_PAD_SLOT_ID rows are skipped)
 *  A_log, dt_bias, lower_bound, scale, H, state_pool, num_slots
 *                   shared by both segments (one layer)
 *  core_attn_out    [num_out_tokens, H, 128] bf16, token stride out_token_stride
 *  non_spec_token_indx [T_p] int32 device: output row of prefill token i
 *  spec_token_indx  [B*T] int32 device: output row of verify token j (= b*T + t)
 *  norm             NULL, or the gated RMSNorm applied to each output row
 *                   (gate and rstd rows are output rows of core_attn_out)
 *  conv             NULL, or the short convolutions of q, k, v for both segments,
 *                   as in kda_chunk_prefill and kda_recurrent_verify
 *
 * Preconditions: the output rows named by the two index arrays are distinct
 * (rows named by neither are left as they were).  An index outside
 * [0, num_out_tokens) leaves that row unwritten and sets KDA_DEVICE_BAD_INDEX.
 * The pool slots the prefill segment writes back (KDA_FINAL_TO_POOL) are not
 * among spec_slot_ids.  Launch order on `stream`: the prefill's two kernels,
 * then the verify kernel as a programmatic dependent of the state pass, so
 * that verify CTAs run on the SMs the state pass leaves free; the call's work
 * is complete, for whatever the stream runs next, when its last kernel is.
 * workspace: at least kda_prefill_workspace_size(T_p, num_seqs, H) bytes,
 * cleared once by kda_workspace_reset before its first use (the step keeps a
 * counter beside the status word and leaves it at zero).  Arguments of both
 * segments are checked before anything is launched.
 */
KDA_API int kda_spec_step(const kda_token_tensors *prefill, const int32_t *cu_seqlens_dev,
                          const int32_t *cu_seqlens_host, int num_seqs, const int32_t *prefill_slot_ids,
                          int flags, float *final_state, const kda_token_tensors *spec, int B, int T,
                          const int32_t *spec_slot_ids, float *intermediate_states, const float *A_log,
                          const float *dt_bias, float lower_bound, float scale, int H, float *state_pool,
                          int num_slots, uint16_t *core_attn_out, int64_t out_token_stride,
                          int64_t num_out_tokens, const kda_output_norm *norm,
                          const kda_short_conv *conv, const int32_t *non_spec_token_indx,
                          const int32_t *spec_token_indx, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * kda_recurrent_verify without a workspace.  The pages have no counterpart:
 * this is a convenience for callers that cannot allocate device memory where
 * they run the layer (an engine plugin whose device memory is planned ahead
 * and may not grow while executing, or code that must avoid cudaMalloc because
 * it can synchronise the device).  Arguments and results are those of
 * kda_recurrent_verify minus the workspace; nothing is allocated.
 *
 *  - The scratch (the status word) lives in a fixed 4 KiB device array inside
 *    libkda, held by every GPU that loads the library until the process exits.
 *    A call needs kda_workspace_size() bytes of it; if that ever exceeded the
 *    array the call would return KDA_ERR_WORKSPACE without launching.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - The arguments are checked on the host first, exactly as
 *    kda_recurrent_verify checks them; a rejected call returns its status and
 *    queues nothing on the stream.
 *  - Every call shares the one array: an accepted call clears the status word
 *    (one memset on the stream) before its kernel, and calls whose work
 *    overlaps on the GPU (different streams, no ordering) race on it.  Slot ids outside [0, num_slots) are skipped as in
 *    kda_recurrent_verify, but this entry point does not report them.
 */
KDA_API int kda_recurrent_verify_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 int64_t qkv_token_stride, const uint16_t *g, int64_t g_token_stride,
                                 const uint16_t *beta_logits, int64_t beta_token_stride,
                                 const float *A_log, const float *dt_bias, float lower_bound,
                                 float scale, int B, int T, int H, const float *state_pool,
                                 int num_slots, const int32_t *slot_ids, uint16_t *out,
                                 int64_t out_token_stride, float *intermediate_states, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
