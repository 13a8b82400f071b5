// C ABI of libkda (declared in include/kda.h): host-side validation and
// launch planning.  Every check that can be made on the host is made here,
// before anything is launched; nothing here allocates device memory or
// synchronises (except kda_read_device_status, a debug helper).
#include <cmath>
#include <cstdint>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_block.h"

namespace {

constexpr size_t kWorkspaceBytes = 1024;
static_assert(kda::kDoneCounterOffset + sizeof(uint32_t) <= kWorkspaceBytes,
              "the spec step's CTA counter must sit in the cleared header");
static_assert(kda::kSplitCounterOffset >= kda::kDoneCounterOffset + sizeof(uint32_t) &&
                  kda::kSplitCounterOffset + kda::kMaxSplitCounters * sizeof(uint32_t) <= kWorkspaceBytes,
              "the split schedule's counters lie in the part kda_workspace_reset clears");

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool good_stride(int64_t stride, int64_t min_elems) { return stride >= min_elems && stride % 8 == 0; }

int check_workspace(const void *ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || bytes < kWorkspaceBytes) return KDA_ERR_WORKSPACE;
  return KDA_OK;
}

int check_gate(float lower_bound, float scale) {
  if (!std::isfinite(lower_bound) || !std::isfinite(scale)) return KDA_ERR_UNSUPPORTED;
  // The chunked kernel represents exp of up to 8 consecutive log-decays in
  // fp32; |lower_bound| <= 10 keeps that below e^80.  Positive bounds would
  // make the state grow and are outside the method's convention.
  if (lower_bound < -10.0f || lower_bound > 0.0f) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

int check_token_tensors(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_stride,
                        const uint16_t *g, int64_t g_stride, const uint16_t *beta,
                        int64_t beta_stride, const float *A_log, const float *dt_bias,
                        const uint16_t *out, int64_t out_stride, int H) {
  if (H <= 0 || H > 4096) return KDA_ERR_INVALID_ARG;
  const int64_t row = (int64_t)H * kda::kD;
  if (!q || !k || !v || !g || !beta || !A_log || !dt_bias || !out) return KDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(out) ||
      !aligned16(dt_bias))
    return KDA_ERR_INVALID_ARG;
  if (!good_stride(qkv_stride, row) || !good_stride(g_stride, row) || !good_stride(out_stride, row))
    return KDA_ERR_INVALID_ARG;
  if (beta_stride < H) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

// Host-side checks of the optional output norm; fills `n` (gate == nullptr when absent).
int check_norm(const kda_output_norm *norm, int H, kda::OutNorm *n) {
  *n = kda::OutNorm{};
  if (!norm) return KDA_OK;
  if (!norm->gate || !aligned16(norm->gate) || !good_stride(norm->gate_token_stride, (int64_t)H * kda::kD))
    return KDA_ERR_INVALID_ARG;
  if (!norm->weight || !aligned16(norm->weight)) return KDA_ERR_INVALID_ARG;
  if (!std::isfinite(norm->eps) || norm->eps < 0.0f) return KDA_ERR_INVALID_ARG;
  if (norm->rstd && (reinterpret_cast<uintptr_t>(norm->rstd) & 3u) != 0) return KDA_ERR_INVALID_ARG;
  n->gate = norm->gate;
  n->gate_stride = norm->gate_token_stride;
  n->weight = norm->weight;
  n->eps = norm->eps;
  n->rstd = norm->rstd;
  return KDA_OK;
}

// Host-side checks of the optional short convolutions; fills `c` (weight == nullptr when absent).
int check_conv(const kda_short_conv *conv, kda::ShortConv *c) {
  *c = kda::ShortConv{};
  if (!conv) return KDA_OK;
  if (!conv->weight || !aligned16(conv->weight)) return KDA_ERR_INVALID_ARG;
  if (conv->activation != KDA_CONV_NONE && conv->activation != KDA_CONV_SILU) return KDA_ERR_INVALID_ARG;
  c->weight = conv->weight;
  c->silu = conv->activation == KDA_CONV_SILU;
  c->window_pool = conv->window_pool;
  c->window_dense = conv->window_dense;
  c->step_windows = conv->step_windows;
  return KDA_OK;
}

// Host-side checks of one prefill call; on success fills `a` (no launch).
int prepare_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_token_stride,
                    const uint16_t *g, int64_t g_token_stride, const uint16_t *beta_logits,
                    int64_t beta_token_stride, const float *A_log, const float *dt_bias, float lower_bound,
                    float scale, const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host, int num_seqs,
                    int H, float *state_pool, int num_slots, const int32_t *slot_ids, int flags, uint16_t *out,
                    int64_t out_token_stride, const kda_output_norm *norm, const kda_short_conv *conv,
                    float *final_state, void *workspace, size_t workspace_bytes, kda::ChunkArgs *a) {
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  if (num_seqs < 0) return KDA_ERR_INVALID_ARG;
  if (!cu_seqlens_dev || !cu_seqlens_host) return KDA_ERR_INVALID_ARG;
  if (flags & ~(KDA_LOAD_INITIAL | KDA_FINAL_TO_POOL | KDA_TWO_PASS | KDA_FUSED | KDA_OVERLAP))
    return KDA_ERR_INVALID_ARG;
  const int path_flags = flags & (KDA_TWO_PASS | KDA_FUSED | KDA_OVERLAP);
  if (path_flags & (path_flags - 1)) return KDA_ERR_INVALID_ARG;   // at most one path
  if (cu_seqlens_host[0] != 0) return KDA_ERR_INVALID_ARG;
  for (int n = 0; n < num_seqs; ++n)
    if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
  *a = kda::ChunkArgs{};
  if (num_seqs == 0) return KDA_OK;   // a->num_seqs = 0: nothing to launch
  if (int rc = check_token_tensors(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits,
                                   beta_token_stride, A_log, dt_bias, out, out_token_stride, H))
    return rc;
  if (int rc = check_gate(lower_bound, scale)) return rc;
  const bool use_pool = flags & (KDA_LOAD_INITIAL | KDA_FINAL_TO_POOL);
  if (use_pool && (!state_pool || !slot_ids || num_slots <= 0 || !aligned16(state_pool)))
    return KDA_ERR_INVALID_ARG;
  if (!(flags & KDA_FINAL_TO_POOL) && (!final_state || !aligned16(final_state))) return KDA_ERR_INVALID_ARG;
  if (workspace_bytes < kda::prefill_workspace_bytes(cu_seqlens_host[num_seqs], num_seqs, H)) return KDA_ERR_WORKSPACE;
  if (int rc = check_norm(norm, H, &a->norm)) return rc;
  if (int rc = check_conv(conv, &a->conv)) return rc;
  if (conv && ((use_pool && (!conv->window_pool || !aligned16(conv->window_pool))) ||
               (!(flags & KDA_FINAL_TO_POOL) && (!conv->window_dense || !aligned16(conv->window_dense)))))
    return KDA_ERR_INVALID_ARG;

  a->q = q; a->k = k; a->v = v; a->g = g; a->beta = beta_logits;
  a->qkv_stride = qkv_token_stride; a->g_stride = g_token_stride;
  a->beta_stride = beta_token_stride; a->out_stride = out_token_stride;
  a->A_log = A_log; a->dt_bias = dt_bias;
  a->lower_bound = lower_bound; a->scale = scale;
  a->H = H; a->num_seqs = num_seqs; a->total_tokens = cu_seqlens_host[num_seqs];
  a->cu_seqlens = cu_seqlens_dev;
  a->slot_ids = use_pool ? slot_ids : nullptr;
  a->num_slots = num_slots;
  a->state_in = (flags & KDA_LOAD_INITIAL) ? state_pool : nullptr;
  a->state_out_pool = (flags & KDA_FINAL_TO_POOL) ? state_pool : nullptr;
  a->state_out_dense = (flags & KDA_FINAL_TO_POOL) ? nullptr : final_state;
  a->out = out;
  a->status = static_cast<uint32_t *>(workspace);
  a->path = (flags & KDA_TWO_PASS) ? kda::PrefillPath::kTwoPass
            : (flags & KDA_FUSED)  ? kda::PrefillPath::kFused
            : (flags & KDA_OVERLAP) ? kda::PrefillPath::kOverlap
                                   : kda::PrefillPath::kAuto;
  if (a->path == kda::PrefillPath::kFused && !kda::fused_prefill_applies(*a)) return KDA_ERR_UNSUPPORTED;
  if (a->path == kda::PrefillPath::kOverlap &&
      workspace_bytes < kda::prefill_workspace_bytes(cu_seqlens_host[num_seqs], num_seqs, H) +
                            kda::overlap_scratch_bytes(num_seqs, H))
    return KDA_ERR_WORKSPACE;
  return KDA_OK;
}

// Host-side checks of one verify call; on success fills `a` (no launch).
int prepare_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_token_stride,
                   const uint16_t *g, int64_t g_token_stride, const uint16_t *beta_logits, int64_t beta_token_stride,
                   const float *A_log, const float *dt_bias, float lower_bound, float scale, int B, int T, int H,
                   const float *state_pool, int num_slots, const int32_t *slot_ids, uint16_t *out,
                   int64_t out_token_stride, const kda_output_norm *norm, const kda_short_conv *conv,
                   float *intermediate_states, void *workspace, size_t workspace_bytes,
                   kda::RecurrentArgs *a) {
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  if (B < 0 || T < 1 || T > 64) return KDA_ERR_INVALID_ARG;
  *a = kda::RecurrentArgs{};
  if (B == 0) return KDA_OK;
  if (int rc = check_token_tensors(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits,
                                   beta_token_stride, A_log, dt_bias, out, out_token_stride, H))
    return rc;
  if (int rc = check_gate(lower_bound, scale)) return rc;
  if (!state_pool || !aligned16(state_pool) || num_slots <= 0 || !slot_ids) return KDA_ERR_INVALID_ARG;
  if (!intermediate_states || !aligned16(intermediate_states)) return KDA_ERR_INVALID_ARG;
  if (int rc = check_norm(norm, H, &a->norm)) return rc;
  if (int rc = check_conv(conv, &a->conv)) return rc;
  if (conv && (!conv->window_pool || !aligned16(conv->window_pool) || !conv->step_windows ||
               !aligned16(conv->step_windows)))
    return KDA_ERR_INVALID_ARG;

  a->q = q; a->k = k; a->v = v; a->g = g; a->beta = beta_logits;
  a->qkv_stride = qkv_token_stride; a->g_stride = g_token_stride;
  a->beta_stride = beta_token_stride; a->out_stride = out_token_stride;
  a->A_log = A_log; a->dt_bias = dt_bias;
  a->lower_bound = lower_bound; a->scale = scale;
  a->H = H;
  a->cu_seqlens = nullptr;
  a->T = T;
  a->slot_ids = slot_ids;
  a->num_slots = num_slots;
  a->state_in = state_pool;
  a->inter = intermediate_states;
  a->out = out;
  a->status = static_cast<uint32_t *>(workspace);
  return KDA_OK;
}

// The gated RMSNorm pass over a prefill's stored rows (nothing when the call has no norm).
cudaError_t launch_prefill_norm(const kda::ChunkArgs &a, cudaStream_t stream) {
  if (!a.norm.gate || a.num_seqs <= 0) return cudaSuccess;
  kda::GatedNormArgs n{};
  n.out = a.out;
  n.out_stride = a.out_stride;
  n.row_index = a.out_index;
  n.num_rows = a.out_index ? a.num_out_rows : a.total_tokens;
  n.num_tokens = a.total_tokens;
  n.H = a.H;
  n.norm = a.norm;
  return kda::launch_gated_norm(n, stream);
}

}  // namespace

int kda::check_verify_call(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_token_stride,
                           const uint16_t *g, int64_t g_token_stride, const uint16_t *beta_logits,
                           int64_t beta_token_stride, const float *A_log, const float *dt_bias, float lower_bound,
                           float scale, int B, int T, int H, const float *state_pool, int num_slots,
                           const int32_t *slot_ids, uint16_t *out, int64_t out_token_stride,
                           float *intermediate_states, void *workspace, size_t workspace_bytes) {
  kda::RecurrentArgs a;
  return prepare_verify(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits, beta_token_stride, A_log, dt_bias,
                        lower_bound, scale, B, T, H, state_pool, num_slots, slot_ids, out, out_token_stride, nullptr,
                        nullptr, intermediate_states, workspace, workspace_bytes, &a);
}

extern "C" {

const char *kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid pointer, size, stride or cu_seqlens";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: lower_bound outside [-10, 0], non-finite scale, or too many sequences";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call or kernel launch failed";
    default: return "KDA: unknown status";
  }
}

size_t kda_workspace_size(void) { return kWorkspaceBytes; }

size_t kda_prefill_workspace_size(int64_t total_tokens, int num_seqs, int H) {
  if (total_tokens < 0 || num_seqs < 0 || H <= 0) return 0;
  return kda::prefill_workspace_bytes(total_tokens, num_seqs, H) + kda::overlap_scratch_bytes(num_seqs, H);
}

int kda_prefill_schedule(const int32_t *cu_seqlens_host, int num_seqs, int H, int flags, float lower_bound,
                         int with_conv, size_t workspace_bytes, int sms, int *info) {
  if (!cu_seqlens_host || !info || num_seqs < 1 || H <= 0 || H > 4096) return KDA_ERR_INVALID_ARG;
  if (flags & ~(KDA_LOAD_INITIAL | KDA_FINAL_TO_POOL | KDA_TWO_PASS | KDA_FUSED | KDA_OVERLAP))
    return KDA_ERR_INVALID_ARG;
  const int path_flags = flags & (KDA_TWO_PASS | KDA_FUSED | KDA_OVERLAP);
  if (path_flags & (path_flags - 1)) return KDA_ERR_INVALID_ARG;
  if (cu_seqlens_host[0] != 0) return KDA_ERR_INVALID_ARG;
  for (int n = 0; n < num_seqs; ++n)
    if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
  if (int rc = check_gate(lower_bound, 1.0f)) return rc;
  const size_t need = kda::prefill_workspace_bytes(cu_seqlens_host[num_seqs], num_seqs, H);
  if (workspace_bytes < need) return KDA_ERR_WORKSPACE;
  kda::ChunkArgs a{};
  static const float kPresent = 0.f;   // the planner only asks whether the convolutions are there
  a.H = H;
  a.num_seqs = num_seqs;
  a.total_tokens = cu_seqlens_host[num_seqs];
  a.lower_bound = lower_bound;
  a.conv.weight = with_conv ? &kPresent : nullptr;
  a.path = (flags & KDA_TWO_PASS) ? kda::PrefillPath::kTwoPass
           : (flags & KDA_FUSED)  ? kda::PrefillPath::kFused
           : (flags & KDA_OVERLAP) ? kda::PrefillPath::kOverlap
                                  : kda::PrefillPath::kAuto;
  if (a.path == kda::PrefillPath::kFused && !kda::fused_prefill_applies(a)) return KDA_ERR_UNSUPPORTED;
  if (a.path == kda::PrefillPath::kOverlap && workspace_bytes < need + kda::overlap_scratch_bytes(num_seqs, H))
    return KDA_ERR_WORKSPACE;
  kda::describe_prefill_schedule(a, cu_seqlens_host, workspace_bytes - kda::kWorkspaceHeader, sms, info);
  return KDA_OK;
}

int kda_workspace_reset(void *workspace, size_t workspace_bytes, void *stream) {
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  return cudaMemsetAsync(workspace, 0, kWorkspaceBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

int kda_read_device_status(const void *workspace, size_t workspace_bytes, uint32_t *device_status,
                           void *stream) {
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  if (!device_status) return KDA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(device_status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_token_stride,
                      const uint16_t *g, int64_t g_token_stride, const uint16_t *beta_logits,
                      int64_t beta_token_stride, const float *A_log, const float *dt_bias,
                      float lower_bound, float scale, const int32_t *cu_seqlens_dev,
                      const int32_t *cu_seqlens_host, int num_seqs, int H, float *state_pool,
                      int num_slots, const int32_t *slot_ids, int flags, uint16_t *out,
                      int64_t out_token_stride, const kda_output_norm *norm, const kda_short_conv *conv,
                      float *final_state, void *workspace, size_t workspace_bytes, void *stream) {
  kda::ChunkArgs a;
  if (int rc = prepare_prefill(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits, beta_token_stride, A_log,
                               dt_bias, lower_bound, scale, cu_seqlens_dev, cu_seqlens_host, num_seqs, H, state_pool,
                               num_slots, slot_ids, flags, out, out_token_stride, norm, conv, final_state, workspace,
                               workspace_bytes, &a))
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = kda::launch_chunk_prefill(a, cu_seqlens_host,
                                              static_cast<uint8_t *>(workspace) + kda::kWorkspaceHeader,
                                              workspace_bytes - kda::kWorkspaceHeader, st);
  if (err == cudaSuccess) err = launch_prefill_norm(a, st);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_recurrent_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t qkv_token_stride,
                         const uint16_t *g, int64_t g_token_stride, const uint16_t *beta_logits,
                         int64_t beta_token_stride, const float *A_log, const float *dt_bias,
                         float lower_bound, float scale, int B, int T, int H, const float *state_pool,
                         int num_slots, const int32_t *slot_ids, uint16_t *out, int64_t out_token_stride,
                         const kda_output_norm *norm, const kda_short_conv *conv, float *intermediate_states,
                         void *workspace, size_t workspace_bytes, void *stream) {
  kda::RecurrentArgs a;
  if (int rc = prepare_verify(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits, beta_token_stride, A_log,
                              dt_bias, lower_bound, scale, B, T, H, state_pool, num_slots, slot_ids, out,
                              out_token_stride, norm, conv, intermediate_states, workspace, workspace_bytes, &a))
    return rc;
  cudaError_t err = kda::launch_recurrent(a, B, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_spec_step(const kda_token_tensors *prefill, const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
                  int num_seqs, const int32_t *prefill_slot_ids, int flags, float *final_state,
                  const kda_token_tensors *spec, int B, int T, const int32_t *spec_slot_ids,
                  float *intermediate_states, const float *A_log, const float *dt_bias, float lower_bound,
                  float scale, int H, float *state_pool, int num_slots, uint16_t *core_attn_out,
                  int64_t out_token_stride, int64_t num_out_tokens, const kda_output_norm *norm,
                  const kda_short_conv *conv, const int32_t *non_spec_token_indx, const int32_t *spec_token_indx,
                  void *workspace, size_t workspace_bytes, void *stream) {
  if (num_seqs < 0 || B < 0 || num_out_tokens < 0 || (num_seqs > 0 && !prefill) || (B > 0 && !spec))
    return KDA_ERR_INVALID_ARG;
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  kda::ChunkArgs pa{};       // an absent segment keeps num_seqs = 0 / B = 0 and is not checked further
  kda::RecurrentArgs va{};
  if (num_seqs > 0) {
    const kda_token_tensors &p = *prefill;
    if (int rc = prepare_prefill(p.q, p.k, p.v, p.qkv_token_stride, p.g, p.g_token_stride, p.beta_logits,
                                 p.beta_token_stride, A_log, dt_bias, lower_bound, scale, cu_seqlens_dev,
                                 cu_seqlens_host, num_seqs, H, state_pool, num_slots, prefill_slot_ids, flags,
                                 core_attn_out, out_token_stride, norm, conv, final_state, workspace, workspace_bytes,
                                 &pa))
      return rc;
  }
  if (B > 0) {
    const kda_token_tensors &s = *spec;
    if (int rc = prepare_verify(s.q, s.k, s.v, s.qkv_token_stride, s.g, s.g_token_stride, s.beta_logits,
                                s.beta_token_stride, A_log, dt_bias, lower_bound, scale, B, T, H, state_pool,
                                num_slots, spec_slot_ids, core_attn_out, out_token_stride, norm, conv,
                                intermediate_states, workspace, workspace_bytes, &va))
      return rc;
  }
  const bool has_prefill = pa.num_seqs > 0 && pa.total_tokens > 0, has_spec = B > 0;
  if ((has_prefill && !non_spec_token_indx) || (has_spec && !spec_token_indx)) return KDA_ERR_INVALID_ARG;
  if (num_out_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
  pa.out_index = non_spec_token_indx;
  pa.num_out_rows = num_out_tokens;
  va.out_index = spec_token_indx;
  va.num_out_rows = num_out_tokens;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the prefill's two kernels, then the verify grid as a programmatic dependent of the state pass: the state
  // pass occupies one SM per (sequence, head) and the verify CTAs fill the others while it runs
  if (pa.num_seqs > 0) {
    if (kda::launch_chunk_prefill(pa, cu_seqlens_host, static_cast<uint8_t *>(workspace) + kda::kWorkspaceHeader,
                                  workspace_bytes - kda::kWorkspaceHeader, st) != cudaSuccess)
      return KDA_ERR_CUDA;
    va.done_counter = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + kda::kDoneCounterOffset);
  }
  if (has_spec && kda::launch_recurrent(va, B, st) != cudaSuccess) return KDA_ERR_CUDA;
  if (launch_prefill_norm(pa, st) != cudaSuccess) return KDA_ERR_CUDA;   // the prefill rows' norm, last
  return KDA_OK;
}

int kda_commit_accepted(float *state_pool, int num_slots, const int32_t *slot_ids, const int32_t *num_accepted,
                        const float *intermediate_states, const kda_short_conv *conv, int B, int T, int H,
                        void *workspace, size_t workspace_bytes, void *stream) {
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  if (B < 0 || T < 1 || T > 64 || H <= 0 || H > 4096) return KDA_ERR_INVALID_ARG;
  if (B == 0) return KDA_OK;
  if (!state_pool || !aligned16(state_pool) || num_slots <= 0 || !slot_ids || !num_accepted) return KDA_ERR_INVALID_ARG;
  if (!intermediate_states || !aligned16(intermediate_states)) return KDA_ERR_INVALID_ARG;
  kda::CommitArgs a{};
  a.pool = state_pool;
  a.num_slots = num_slots;
  a.slot_ids = slot_ids;
  a.num_accepted = num_accepted;
  a.inter = intermediate_states;
  if (conv) {
    if (!conv->window_pool || !aligned16(conv->window_pool) || !conv->step_windows || !aligned16(conv->step_windows))
      return KDA_ERR_INVALID_ARG;
    a.step_windows = conv->step_windows;
    a.window_pool = conv->window_pool;
  }
  a.B = B;
  a.T = T;
  a.H = H;
  a.status = static_cast<uint32_t *>(workspace);
  return kda::launch_commit(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
