// kda_recurrent_verify_noalloc: the verify call for callers that cannot
// provide a workspace.
//
// The verify kernel needs a little global memory besides its inputs and
// outputs: the status word in which it records slot ids it had to skip.  The
// regular entry point takes that memory from the caller (the workspace).
// Some callers cannot allocate device memory at the point where they run the
// layer -- for example a plugin inside an inference engine that plans all
// device memory ahead of time and forbids allocation while executing, or code
// that must not call cudaMalloc because it can synchronise the device.  For
// them this file keeps the scratch in a fixed, file-scope device array that
// every GPU loading the library holds until the process exits.
#include <mutex>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace {

// Capacity of the built-in scratch.  A call needs kda_workspace_size() bytes.
constexpr size_t kNoAllocScratchBytes = 4096;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in; the kernel needs this address.
// Looked up once per device (the first call on a device), with that device
// current.
int noalloc_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" int kda_recurrent_verify_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                            int64_t qkv_token_stride, const uint16_t *g, int64_t g_token_stride,
                                            const uint16_t *beta_logits, int64_t beta_token_stride,
                                            const float *A_log, const float *dt_bias, float lower_bound,
                                            float scale, int B, int T, int H, const float *state_pool,
                                            int num_slots, const int32_t *slot_ids, uint16_t *out,
                                            int64_t out_token_stride, float *intermediate_states, void *stream) {
  const size_t need = kda_workspace_size();
  if (need > kNoAllocScratchBytes) return KDA_ERR_WORKSPACE;  // built-in scratch too small for this build
  void *scratch = nullptr;
  if (int rc = noalloc_scratch(&scratch)) return rc;
  // Every argument is checked before anything is queued on the stream: a rejected call adds no device work.
  if (int rc = kda::check_verify_call(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits, beta_token_stride,
                                      A_log, dt_bias, lower_bound, scale, B, T, H, state_pool, num_slots, slot_ids,
                                      out, out_token_stride, intermediate_states, scratch, kNoAllocScratchBytes))
    return rc;
  if (B == 0) return KDA_OK;
  // The array keeps whatever the previous call left; the status word must start at zero.
  if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_CUDA;
  return kda_recurrent_verify(q, k, v, qkv_token_stride, g, g_token_stride, beta_logits, beta_token_stride, A_log,
                              dt_bias, lower_bound, scale, B, T, H, state_pool, num_slots, slot_ids, out,
                              out_token_stride, nullptr, nullptr, intermediate_states, scratch, kNoAllocScratchBytes,
                              stream);
}
