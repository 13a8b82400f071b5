// Chunked prefill launcher.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

cudaError_t launch_chunk_prefill(const ChunkArgs &a, const int32_t *cu_seqlens_host, cudaStream_t stream) {
  (void)cu_seqlens_host;
  RecurrentArgs r{};
  r.q = a.q; r.k = a.k; r.v = a.v; r.g = a.g; r.beta = a.beta;
  r.qkv_stride = a.qkv_stride; r.g_stride = a.g_stride; r.beta_stride = a.beta_stride;
  r.out_stride = a.out_stride;
  r.A_log = a.A_log; r.dt_bias = a.dt_bias; r.lower_bound = a.lower_bound; r.scale = a.scale;
  r.H = a.H; r.cu_seqlens = a.cu_seqlens; r.T = 0;
  r.slot_ids = a.slot_ids; r.num_slots = a.num_slots;
  r.state_in = a.state_in; r.state_out_pool = a.state_out_pool; r.state_out_dense = a.state_out_dense;
  r.inter = nullptr; r.out = a.out; r.status = a.status;
  return launch_recurrent(r, a.num_seqs, stream);
}

}  // namespace kda
