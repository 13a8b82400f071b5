// Host planning of the chunked prefill: chunk slots per sequence, TMA tensor
// maps, and the two launches (intra-chunk kernel over every chunk and head,
// then the state pass over every sequence and head, longest sequences first).
// Everything is computed from the host copy of cu_seqlens; nothing here reads
// device memory or synchronises.
#include <cuda.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_block.h"

namespace kda {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [tokens, H, 128] bf16 with the given token stride; box = 64 channels x 1 head x 64 tokens, with the
// 128-byte swizzle (the row-swizzled tile layout of the MMA operands and the output staging) or
// unswizzled (tiles read only by CUDA cores); rows past the tensor's end read as zero
bool make_token_map(CUtensorMap *map, const void *base, int H, int total_tokens, int64_t token_stride,
                    bool swizzled = true) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(std::max(total_tokens, 1))};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD * 2), static_cast<cuuint64_t>(token_stride * 2)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kChunk)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_workspace_bytes(int64_t total_tokens, int num_seqs, int H) {
  // sum_n ceil(len_n / 64) <= floor(total / 64) + num_seqs
  const size_t chunks = static_cast<size_t>(std::max<int64_t>(total_tokens, 0) / kChunk) +
                        static_cast<size_t>(std::max(num_seqs, 0));
  return kWorkspaceHeader + chunks * static_cast<size_t>(std::max(H, 0)) * kBlkBytes;
}

bool fused_prefill_applies(const ChunkArgs &a) {
  // the fused kernel takes the 32-row anchored sub-blocks only, writes rows in token order and has no short
  // convolutions
  return a.conv.weight == nullptr && a.out_index == nullptr && a.lower_bound >= -5.0f;
}

namespace {

int sm_count() {
  static int sms = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 0;
  });
  return sms;
}

// The path the library takes when the caller does not force one.  The fused kernel walks a sequence's chunks
// one at a time at ~7 us per chunk (its producer's serial phases); the two-kernel path runs every chunk's
// producer work at once and then ~2 us per chunk of state pass.  Measured on GB300 as CUDA-graph replays
// (device time, H = 16): one-chunk sequences with up to 152 (sequence, head) pairs 12.9 us fused against
// 15.0 us; from two chunks per sequence on the two-kernel path is faster (1 x 128: 17.0 against 20.7 us,
// 1 x 256: 20.5 against 34.8 us, 2048 x 8: 207 against 245 us).  So the fused kernel is picked for one-chunk
// sequences that fit one wave of SMs.
bool fused_prefill_preferred(const ChunkArgs &a, const int32_t *cu_host) {
  if (!fused_prefill_applies(a)) return false;
  for (int i = 0; i < a.num_seqs; ++i)
    if (cu_host[i + 1] - cu_host[i] > kChunk) return false;
  const long pairs = static_cast<long>(a.num_seqs) * a.H;
  const long sms = sm_count() > 0 ? sm_count() : 152;
  return pairs <= sms;
}

cudaError_t launch_fused(const ChunkArgs &a, const int32_t *cu_host, cudaStream_t stream) {
  static FusedParams *fp = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!fp) fp = new FusedParams();
  if (!make_token_map(&fp->tq, a.q, a.H, a.total_tokens, a.qkv_stride, false) ||
      !make_token_map(&fp->tk, a.k, a.H, a.total_tokens, a.qkv_stride, false) ||
      !make_token_map(&fp->tg, a.g, a.H, a.total_tokens, a.g_stride, false) ||
      !make_token_map(&fp->tv, a.v, a.H, a.total_tokens, a.qkv_stride) ||
      !make_token_map(&fp->tout, a.out, a.H, a.total_tokens, a.out_stride))
    return cudaErrorInvalidValue;
  fp->beta = a.beta;
  fp->beta_stride = a.beta_stride;
  fp->A_log = a.A_log;
  fp->dt_bias = a.dt_bias;
  fp->lower_bound = a.lower_bound;
  fp->scale = a.scale;
  fp->slot_ids = a.slot_ids;
  fp->num_slots = a.num_slots;
  fp->state_in = a.state_in;
  fp->state_out_pool = a.state_out_pool;
  fp->state_out_dense = a.state_out_dense;
  fp->out = a.out;
  fp->out_stride = a.out_stride;
  fp->status = a.status;
  fp->H = a.H;
  std::vector<int> idx;
  for (int s0 = 0; s0 < a.num_seqs; s0 += kMaxSeqsPerLaunch) {
    const int ns = std::min(kMaxSeqsPerLaunch, a.num_seqs - s0);
    for (int i = 0; i <= ns; ++i) fp->tok_off[i] = cu_host[s0 + i];
    fp->num_seqs = ns;
    fp->seq0 = s0;
    idx.resize(ns);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
      return fp->tok_off[x + 1] - fp->tok_off[x] > fp->tok_off[y + 1] - fp->tok_off[y];
    });
    for (int i = 0; i < ns; ++i) fp->order[i] = static_cast<uint16_t>(idx[i]);
    const cudaError_t e = launch_prefill_fused(*fp, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_chunk_prefill(const ChunkArgs &a, const int32_t *cu_host, uint8_t *blocks, cudaStream_t stream) {
  if (a.num_seqs <= 0) return cudaSuccess;
  if (a.path == PrefillPath::kFused || (a.path == PrefillPath::kAuto && fused_prefill_preferred(a, cu_host)))
    return launch_fused(a, cu_host, stream);
  // host-side staging of the (large) kernel parameter structs; copied at launch
  static IntraParams *ip = nullptr;
  static ChainParams *cp = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!ip) {
    ip = new IntraParams();
    cp = new ChainParams();
  }
  if (!make_token_map(&ip->tq, a.q, a.H, a.total_tokens, a.qkv_stride, false) ||
      !make_token_map(&ip->tk, a.k, a.H, a.total_tokens, a.qkv_stride, false) ||
      !make_token_map(&ip->tv, a.v, a.H, a.total_tokens, a.qkv_stride) ||
      !make_token_map(&ip->tg, a.g, a.H, a.total_tokens, a.g_stride, false) ||
      (!a.out_index && !make_token_map(&cp->tout, a.out, a.H, a.total_tokens, a.out_stride)))
    return cudaErrorInvalidValue;
  ip->beta = a.beta;
  ip->beta_stride = a.beta_stride;
  ip->A_log = a.A_log;
  ip->dt_bias = a.dt_bias;
  ip->lower_bound = a.lower_bound;
  ip->scale = a.scale;
  ip->H = a.H;
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      ip->prefetch_ahead = 2 * sms;   // two intra-chunk CTAs per SM
    else
      ip->prefetch_ahead = 0;
  }
  ip->status = a.status;
  ip->conv = a.conv;
  ip->xq = a.q; ip->xk = a.k; ip->xv = a.v;
  ip->qkv_stride = a.qkv_stride;
  ip->slot_ids = a.slot_ids;
  ip->num_slots = a.num_slots;
  ip->conv_load_initial = a.state_in != nullptr;
  cp->conv = a.conv;
  cp->xq = a.q; cp->xk = a.k; cp->xv = a.v;
  cp->qkv_stride = a.qkv_stride;
  cp->conv_load_initial = a.state_in != nullptr;
  cp->blocks = blocks;
  cp->slot_ids = a.slot_ids;
  cp->num_slots = a.num_slots;
  cp->state_in = a.state_in;
  cp->state_out_pool = a.state_out_pool;
  cp->state_out_dense = a.state_out_dense;
  cp->out = a.out;
  cp->out_stride = a.out_stride;
  cp->out_index = a.out_index;   // with an index the output tensor map is not used
  cp->num_out_rows = a.num_out_rows;
  cp->status = a.status;
  cp->H = a.H;

  std::vector<int> idx;
  for (int s0 = 0; s0 < a.num_seqs; s0 += kMaxSeqsPerLaunch) {
    const int ns = std::min(kMaxSeqsPerLaunch, a.num_seqs - s0);
    int chunks = 0;
    for (int i = 0; i < ns; ++i) {
      const int len = cu_host[s0 + i + 1] - cu_host[s0 + i];
      cp->chunk_off[i] = chunks;
      cp->tok_off[i] = cu_host[s0 + i];
      chunks += (len + kChunk - 1) / kChunk;
    }
    cp->chunk_off[ns] = chunks;
    cp->tok_off[ns] = cu_host[s0 + ns];
    cp->num_seqs = ns;
    cp->seq0 = s0;
    ip->seq0 = s0;
    idx.resize(ns);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
      return cp->chunk_off[x + 1] - cp->chunk_off[x] > cp->chunk_off[y + 1] - cp->chunk_off[y];
    });
    for (int i = 0; i < ns; ++i) cp->order[i] = static_cast<uint16_t>(idx[i]);
    // intra-chunk launches over runs of at most kMaxSlotsPerLaunch chunk slots, each with its slot table
    cudaError_t e = cudaSuccess;
    for (int g0 = 0; g0 < chunks; g0 += kMaxSlotsPerLaunch) {
      const int ng = std::min(kMaxSlotsPerLaunch, chunks - g0);
      // the sequence holding slot g0, then its chunks in order
      int i = static_cast<int>(std::upper_bound(cp->chunk_off, cp->chunk_off + ns + 1, g0) - cp->chunk_off) - 1;
      for (int g = 0; g < ng; ++g) {
        while (cp->chunk_off[i + 1] <= g0 + g) ++i;
        const int j = g0 + g - cp->chunk_off[i];
        const int t = cp->tok_off[i] + j * kChunk;
        ip->slot_tok0[g] = t;
        ip->slot_valid[g] = static_cast<uint8_t>(std::min(kChunk, cp->tok_off[i + 1] - t) | (j == 0 ? kSlotFirst : 0));
        ip->slot_seq[g] = static_cast<int16_t>(i);
      }
      ip->blocks = blocks + static_cast<size_t>(g0) * a.H * kBlkBytes;
      e = launch_chunk_intra(*ip, ng, stream);
      if (e != cudaSuccess) return e;
    }
    e = launch_chunk_chain(*cp, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
