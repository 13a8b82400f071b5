// Accept/commit after speculative verify: for request b with n accepted draft
// tokens, the pooled state becomes the state recorded after token n-1
// (vLLM PR #55737 "Use FlashKDA for KDA chunked prefill", follow-up commit:
// spec tokens keep the recurrent kernel "with num_accepted_tokens rollback";
// the per-step states are the rows written by the one-launch verify of
// TensorRT-LLM PR #21179).  n = 0 and padding rows leave the pool untouched.
//
// A pure HBM copy: one CTA per (request, head) moves 64 KiB with 16-byte
// loads and stores.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs p) {
  const int h = blockIdx.x % p.H;
  const int b = blockIdx.x / p.H;
  const int n = p.num_accepted[b];
  if (n == 0) return;
  const int slot = p.slot_ids[b];
  if (slot == KDA_PAD_SLOT_ID) return;   // padding row of a bucketed batch
  if (n < 0 || n > p.T || slot < 0 || slot >= p.num_slots) {
    if (threadIdx.x == 0) atomicOr(p.status, (n < 0 || n > p.T) ? KDA_DEVICE_BAD_COUNT : KDA_DEVICE_BAD_SLOT);
    return;
  }
  if (p.step_windows) {   // the conv window after token n-1: 3 tensors x 3 rows x 128 channels of this head
    constexpr int kRows = 3 * (kConvW - 1), kVec = kRows * kD / 8;   // 16-byte pieces
    for (int i = threadIdx.x; i < kVec; i += kThreads) {
      const int row = i / (kD / 8), piece = i % (kD / 8);   // row = tensor * 3 + window row
      const uint4 *wsrc = reinterpret_cast<const uint4 *>(
          p.step_windows + ((((size_t)b * p.T + (n - 1)) * kRows + row) * p.H + h) * kD) + piece;
      uint4 *wdst = reinterpret_cast<uint4 *>(p.window_pool + (((size_t)slot * kRows + row) * p.H + h) * kD) + piece;
      *wdst = *wsrc;
    }
  }
  const float4 *src = reinterpret_cast<const float4 *>(p.inter + (((size_t)b * p.T + (n - 1)) * p.H + h) * kD * kD);
  float4 *dst = reinterpret_cast<float4 *>(p.pool + ((size_t)slot * p.H + h) * kD * kD);
  constexpr int kVec = kD * kD / 4;   // 4096 float4
#pragma unroll 4
  for (int i = threadIdx.x; i < kVec; i += kThreads) dst[i] = __ldcs(src + i);
}

}  // namespace

cudaError_t launch_commit(const CommitArgs &args, cudaStream_t stream) {
  if (args.B <= 0) return cudaSuccess;
  commit_kernel<<<args.B * args.H, kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace kda
