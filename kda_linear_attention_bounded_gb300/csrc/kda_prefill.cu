// Host planning of the chunked prefill: chunk slots per sequence, TMA tensor
// maps, and the launches.  The plain schedule is two launches per group of
// sequences (intra-chunk kernel over every chunk and head, then the state pass
// over every sequence and head, longest sequences first); the split schedule
// cuts the longest sequences' state passes into segments chained as
// programmatic dependent launches; one-chunk sequences may take the fused
// kernel.  Everything is computed from the host copy of cu_seqlens; nothing
// here reads device memory or synchronises.
#include <cuda.h>

#include <algorithm>
#include <functional>
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
bool fused_prefill_preferred(const ChunkArgs &a, const int32_t *cu_host, int sms) {
  if (!fused_prefill_applies(a)) return false;
  for (int i = 0; i < a.num_seqs; ++i)
    if (cu_host[i + 1] - cu_host[i] > kChunk) return false;
  const long pairs = static_cast<long>(a.num_seqs) * a.H;
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

// A run of whole chunks of one sequence that one state-pass CTA per head walks: the whole sequence, or one
// segment of it when the sequence's state pass is split.
struct Item {
  int seq, tok0, len;
  uint8_t flags, mid;
  int nchunks() const { return (len + kChunk - 1) / kChunk; }
};

// Programmatic chaining of the launches of a split schedule: each launch after the call's first one starts as a
// programmatic dependent of the launch before it, and the CTA of it that finishes last waits for that launch's
// completion through a counter of its own.
struct Chain {
  uint32_t *counters;
  int used;
  uint32_t *next() { return used < kMaxSplitCounters ? counters + used++ : nullptr; }
};

// Fills the state pass's tables for `items` whose blocks start at block index start[i] from cp->blocks.
void fill_chain(ChainParams *cp, const Item *items, const int *start, int n) {
  for (int i = 0; i < n; ++i) {
    cp->chunk_off[i] = start[i];
    cp->tok0[i] = items[i].tok0;
    cp->len[i] = items[i].len;
    cp->seq[i] = items[i].seq;
    cp->flags[i] = items[i].flags;
    cp->mid[i] = items[i].mid;
  }
  cp->num_seqs = n;
  std::vector<int> idx(n);
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) { return items[x].nchunks() > items[y].nchunks(); });
  for (int i = 0; i < n; ++i) cp->order[i] = static_cast<uint16_t>(idx[i]);
}

// Launches the intra-chunk kernel over the items' chunks, their blocks one after another from `blocks` (block
// (slot g, head h) at blocks + (g H + h) kBlkBytes), in runs of at most kMaxSlotsPerLaunch chunk slots.  seq0:
// the first sequence of a group of consecutive sequences (the short convolutions find a chunk's window slot as
// slot_ids[seq0 + slot_seq]); items that are not such a group run without convolutions.  chain: null for
// ordinary launches, else every run is a programmatic dependent of the launch before it.
cudaError_t launch_intra_runs(const Item *items, int n, int seq0, const int32_t *cu_host, uint8_t *blocks, int H,
                              IntraParams *ip, Chain *chain, cudaStream_t stream) {
  ip->seq0 = seq0;
  int g = 0, g0 = 0;
  auto run = [&]() -> cudaError_t {
    if (g == 0) return cudaSuccess;
    ip->blocks = blocks + static_cast<size_t>(g0) * H * kBlkBytes;
    ip->done_counter = chain ? chain->next() : nullptr;
    if (chain && !ip->done_counter) return cudaErrorInvalidValue;   // the planner sizes the chain; not reached
    const cudaError_t e = launch_chunk_intra(*ip, g, stream, chain != nullptr);
    g0 += g;
    g = 0;
    return e;
  };
  for (int i = 0; i < n; ++i) {
    const Item &it = items[i];
    for (int j = 0; j < it.nchunks(); ++j) {
      const int t = it.tok0 + j * kChunk;
      const bool first = j == 0 && it.tok0 == cu_host[it.seq];
      ip->slot_tok0[g] = t;
      ip->slot_valid[g] = static_cast<uint8_t>(std::min(kChunk, it.tok0 + it.len - t) | (first ? kSlotFirst : 0));
      ip->slot_seq[g] = static_cast<int16_t>(it.seq - seq0);
      if (++g == kMaxSlotsPerLaunch)
        if (cudaError_t e = run()) return e;
    }
  }
  return run();
}

// Split state passes.  The state pass of one (sequence, head) is a serial walk over its chunks (~1.85 us per
// chunk on GB300) that the plain schedule starts only once the intra-chunk kernel has covered every chunk of the
// call.  When a few long sequences dominate, their state passes are instead split into segments of whole chunks,
// and the call becomes one chain of programmatic dependent launches on the caller's stream:
//
//   I_0 -> C_0 -> I_1 -> C_1 -> ... -> I_{n-1} -> C_{n-1} [-> C_rest]
//
// I_k is the intra-chunk work of segment k (plus a share of the other sequences' chunks), C_k the state pass of
// segment k.  C_k is resident once I_k's last CTAs leave their SMs, and waits for I_k's completion before it
// reads a block; I_{k+1} may start only once every CTA of C_k has started, so it fills exactly the SMs C_k leaves
// free and cannot take those C_k needs.  The CTA of I_{k+1} that finishes last waits for C_k's completion, so
// C_{k+1} (which waits for I_{k+1}) finds the state C_k handed over through an fp32 scratch copy.  C_{n-1} lets
// its dependent start only once every block exists; C_rest, the plain state pass of the other sequences, then
// runs beside it.  The results are those of the plain schedule bit for bit (a segment's state pass rebuilds
// exactly the operands the unsplit one keeps on chip).
constexpr int kOverlapMinChunks = 64;     // the longest sequence's chunks below which the split does not pay
constexpr int kMaxSegments = 8;
constexpr double kIntraCtaUs = 8.5;       // one intra-chunk CTA, two resident per SM
constexpr double kChainChunkUs = 1.85;    // one chunk of state pass

// Segment bounds in chunks for state passes of up to max_chunks chunks with `pairs` (sequence, head) pairs.
// rest_chunks: the chunks of state pass that the other sequences' state pass (C_rest) needs, run beside the last
// segment's (0: no other sequences).  Measured on GB300 (CUDA-graph device time):
// - when the intra-chunk work of a segment, on the SMs the state passes leave free, is faster than the segment's
//   state pass (ratio < 1: few pairs), the state passes are the critical path: a short first segment so they
//   start early, then segments growing threefold (16384 x 1: 511-516 us over several such plans, 588 unsplit);
// - when it is slower (8192 x 4), the state pass and the intra-chunk work beside it share the HBM and every
//   segment boundary leaves SMs idle while the state pass's CTAs gather: three segments of about 3/8 of the
//   sequence measured best (48, 48, 32 chunks: 435 us; 4-8-16-32-32-32-4: 477, 32 x 4: 450, 64 x 2: 457;
//   488 unsplit);
// - with other sequences beside (16384 + 16 x [1, 4096]), their intra-chunk work must fit beside the lane's
//   long middle segment and their state pass beside its last one: growing head segments up to a quarter of
//   the sequence, a last segment of about the others' state pass (at most a quarter), the middle between
//   (4-12-36-140-64: 684 us; 4-16-64: 701, 4-12-36-124-80: 713; 890 unsplit).
std::vector<int> segment_bounds(int max_chunks, int pairs, int sms, int rest_chunks) {
  const double free_slots = 2.0 * std::max(sms - pairs, 1);
  const double ratio = pairs * kIntraCtaUs / free_slots / kChainChunkUs;   // intra-chunk / state-pass time per chunk
  std::vector<int> len;
  if (rest_chunks > 0) {
    const int quarter = std::max(1, max_chunks / 4);
    const int last = std::min(std::max(rest_chunks, 8), quarter);
    int head = 0;
    for (int s = 4; head + s <= quarter && head + s + last < max_chunks; s *= 3) {
      len.push_back(s);
      head += s;
    }
    if (max_chunks - head - last > 0) len.push_back(max_chunks - head - last);
    len.push_back(std::min(last, max_chunks - head));
  } else if (ratio < 1.0) {
    for (int s = 4, done = 0; done < max_chunks; done += s, s *= 3) len.push_back(std::min(s, max_chunks - done));
  } else {
    const int s = std::max(4, (3 * max_chunks + 7) / 8);
    for (int done = 0; done < max_chunks; done += s) len.push_back(std::min(s, max_chunks - done));
  }
  std::vector<int> b{0};
  for (int l : len)
    if (l > 0 && b.back() < max_chunks) b.push_back(std::min(max_chunks, b.back() + l));
  if (static_cast<int>(b.size()) > kMaxSegments + 1) {   // not reached by these rules; merge the tail
    b.resize(kMaxSegments);
    b.push_back(max_chunks);
  }
  return b;
}

// Chunks of state pass that C_rest takes for these (sequence, head) chunk counts on `sms` SMs: longest first,
// each onto the SM that frees first.
int rest_chain_chunks(std::vector<int> chunks, int sms) {
  if (chunks.empty() || sms <= 0) return 0;
  std::sort(chunks.begin(), chunks.end(), std::greater<int>());
  std::vector<long> load(sms, 0);   // a min-heap of the SMs' busy times
  for (int c : chunks) {
    std::pop_heap(load.begin(), load.end(), std::greater<long>());
    load.back() += c;
    std::push_heap(load.begin(), load.end(), std::greater<long>());
  }
  return static_cast<int>(*std::max_element(load.begin(), load.end()));
}

// The sequences whose state passes are split (indices into the call's sequences, longest first), or none.
// Automatic: every sequence of at least half the longest one's chunks, provided the longest has at least
// kOverlapMinChunks and their pairs fit in half of the SMs.  Forced: the longest sequences within that budget.
std::vector<int> overlap_lane(const ChunkArgs &a, const int32_t *cu_host, bool forced, int sms) {
  std::vector<int> idx(a.num_seqs);
  std::iota(idx.begin(), idx.end(), 0);
  auto nch = [&](int s) { return (cu_host[s + 1] - cu_host[s] + kChunk - 1) / kChunk; };
  std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) { return nch(x) > nch(y); });
  const int budget = std::min(sms / 2, kMaxOverlapPairs) / a.H;   // sequences
  std::vector<int> lane;
  if (a.num_seqs == 0 || budget <= 0 || nch(idx[0]) == 0) return lane;
  if (forced) {
    for (int i = 0; i < a.num_seqs && i < budget && nch(idx[i]) > 0; ++i) lane.push_back(idx[i]);
    return lane;
  }
  const int top = nch(idx[0]);
  if (top < kOverlapMinChunks) return lane;
  for (int i = 0; i < a.num_seqs && 2 * nch(idx[i]) >= top; ++i) {
    if (i == budget) return {};
    lane.push_back(idx[i]);
  }
  return lane;
}

// Whether a state-pass launch over `pairs` (item, head) pairs takes the value-split kernel: two CTAs per pair,
// 64 value channels each, which shortens the serial path per chunk from ~3.8 k to ~2.5 k cycles with
// bit-identical results, at the price of twice the SMs and twice the key-side block reads.  It pays where those
// SMs would otherwise idle: when both CTAs of every pair fit in `budget` SMs.  Not with rows stored by index
// (the spec step), whose verify grid runs beside the state pass on the SMs it leaves free: measured there,
// 210 us against 174.
bool use_vsplit(const ChunkArgs &a, long pairs, long budget) { return a.out_index == nullptr && 2 * pairs <= budget; }

// The schedule of one call, decided on the host from the sequence lengths alone: the fused kernel, the plain
// schedule (both kernels over every chunk, per group of sequences), or the split schedule (the lane's sequences
// in segments of chunks, the rest beside them).
struct PrefillPlan {
  enum Kind { kFusedKernel = 1, kPlain = 2, kSplit = 3 } kind = kPlain;
  std::vector<int> lane;     // split: the sequences whose state passes are split
  std::vector<int> bounds;   // split: segment bounds in chunks
  std::vector<Item> rest;    // split: the other sequences (whole)
  size_t all_blocks = 0;     // bytes of the blocks of every chunk
};

PrefillPlan plan_prefill(const ChunkArgs &a, const int32_t *cu_host, size_t blocks_bytes, int sms) {
  auto nch = [&](int s) { return (cu_host[s + 1] - cu_host[s] + kChunk - 1) / kChunk; };
  const size_t blk_bytes = static_cast<size_t>(a.H) * kBlkBytes;   // the blocks of one chunk

  PrefillPlan plan;
  if (a.path == PrefillPath::kFused || (a.path == PrefillPath::kAuto && fused_prefill_preferred(a, cu_host, sms))) {
    plan.kind = PrefillPlan::kFusedKernel;
    return plan;
  }
  // the split schedule, where it applies and the workspace holds the scratch states
  std::vector<int> &lane = plan.lane;
  std::vector<int> &bounds = plan.bounds;
  std::vector<Item> &rest = plan.rest;   // the other sequences (whole)
  size_t &all_blocks = plan.all_blocks;
  for (int s = 0; s < a.num_seqs; ++s) all_blocks += static_cast<size_t>(nch(s)) * blk_bytes;
  // (with the short convolutions a chunk finds its sequence's window slot through a 16-bit index)
  if ((a.path == PrefillPath::kAuto || a.path == PrefillPath::kOverlap) &&
      (a.conv.weight == nullptr || a.num_seqs <= INT16_MAX)) {
    lane = overlap_lane(a, cu_host, a.path == PrefillPath::kOverlap, sms);
    std::vector<char> in_lane(a.num_seqs, 0);
    int top = 0;
    for (int s : lane) {
      in_lane[s] = 1;
      top = std::max(top, nch(s));
    }
    for (int s = 0; s < a.num_seqs; ++s)
      if (!in_lane[s]) rest.push_back({s, cu_host[s], cu_host[s + 1] - cu_host[s], 0, 0});
    if (!lane.empty()) {
      const int pairs = static_cast<int>(lane.size()) * a.H;
      std::vector<int> rest_pairs;
      for (const Item &it : rest)
        for (int h = 0; h < a.H && it.nchunks() > 0; ++h) rest_pairs.push_back(it.nchunks());
      bounds = segment_bounds(top, pairs, sms, rest_chain_chunks(rest_pairs, std::max(sms - pairs, 1)));
    }
    // launches that wait for their predecessor (a bound): the intra-chunk runs of segments 1.. (the lane's
    // slots and a share of the rest's, kMaxSlotsPerLaunch per run) and the rest's state pass
    size_t runs = 1, rest_slots = 0;
    for (size_t k = 1; k + 1 < bounds.size(); ++k) {
      size_t slots = 0;
      for (int s : lane) slots += std::max(0, std::min(bounds[k + 1], nch(s)) - bounds[k]);
      runs += 2 + slots / kMaxSlotsPerLaunch;
    }
    for (const Item &it : rest) rest_slots += it.nchunks();
    runs += rest_slots / kMaxSlotsPerLaunch;
    if (lane.empty() || rest.size() > static_cast<size_t>(kMaxSeqsPerLaunch) || runs > kMaxSplitCounters ||
        all_blocks + lane.size() * a.H * kD * kD * sizeof(float) > blocks_bytes)
      lane.clear();
    // where the whole call's state passes fit the value-split kernel on the plain schedule, but the lane's would
    // keep the full-value kernel on more than 3/8 of the SMs (too few left for the intra-chunk work beside them),
    // the plain schedule wins up to ~160 chunks (graph replays, H = 16: 8192 x 4 424.4 against 430.7 us split,
    // 6000 x 4 315.5 against 327.2; the split stays ahead with 48 pairs, 8192 x 3: 355.0 against 362.3, and
    // for longer sequences, 12000 x 4: 613.5 against 617.3)
    const long lane_pairs = static_cast<long>(lane.size()) * a.H;
    if (a.path == PrefillPath::kAuto && !lane.empty() && a.num_seqs <= kMaxSeqsPerLaunch && top <= 160 &&
        use_vsplit(a, static_cast<long>(a.num_seqs) * a.H, sms) && 8 * lane_pairs > 3L * sms &&
        !(rest.empty() && use_vsplit(a, lane_pairs, sms / 2)))
      lane.clear();
  }
  if (!lane.empty()) plan.kind = PrefillPlan::kSplit;
  return plan;
}

}  // namespace

size_t overlap_scratch_bytes(int num_seqs, int H) {
  const long pairs = std::min<long>(static_cast<long>(std::max(num_seqs, 0)) * std::max(H, 0), kMaxOverlapPairs);
  return static_cast<size_t>(pairs) * kD * kD * sizeof(float);
}

cudaError_t launch_chunk_prefill(const ChunkArgs &a, const int32_t *cu_host, uint8_t *blocks, size_t blocks_bytes,
                                 cudaStream_t stream) {
  if (a.num_seqs <= 0) return cudaSuccess;
  const int sms = sm_count() > 0 ? sm_count() : 152;
  PrefillPlan plan = plan_prefill(a, cu_host, blocks_bytes, sms);
  if (plan.kind == PrefillPlan::kFusedKernel) return launch_fused(a, cu_host, stream);
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
  ip->prefetch_ahead = 2 * sms;   // two intra-chunk CTAs per SM
  ip->status = a.status;
  ip->conv = a.conv;
  ip->xq = a.q; ip->xk = a.k; ip->xv = a.v;
  ip->qkv_stride = a.qkv_stride;
  ip->slot_ids = a.slot_ids;
  ip->num_slots = a.num_slots;
  ip->conv_load_initial = a.state_in != nullptr;
  ip->done_counter = nullptr;
  cp->conv = a.conv;
  cp->xq = a.q; cp->xk = a.k; cp->xv = a.v;
  cp->qkv_stride = a.qkv_stride;
  cp->conv_load_initial = a.state_in != nullptr;
  cp->slot_ids = a.slot_ids;
  cp->num_slots = a.num_slots;
  cp->state_in = a.state_in;
  cp->state_out_pool = a.state_out_pool;
  cp->state_out_dense = a.state_out_dense;
  cp->state_mid = nullptr;
  cp->out = a.out;
  cp->out_stride = a.out_stride;
  cp->out_index = a.out_index;   // with an index the output tensor map is not used
  cp->num_out_rows = a.num_out_rows;
  cp->status = a.status;
  cp->H = a.H;
  cp->wait_blocks = 1;
  cp->trigger_after_wait = 0;
  cp->done_counter = nullptr;
  auto nch = [&](int s) { return (cu_host[s + 1] - cu_host[s] + kChunk - 1) / kChunk; };
  const size_t blk_bytes = static_cast<size_t>(a.H) * kBlkBytes;   // the blocks of one chunk
  std::vector<int> &lane = plan.lane;
  const std::vector<int> &bounds = plan.bounds;
  std::vector<Item> &rest = plan.rest;
  const size_t all_blocks = plan.all_blocks;

  if (lane.empty()) {   // plain schedule: per group of consecutive sequences, both kernels over all its chunks
    std::vector<Item> items;
    std::vector<int> start;
    size_t blk = 0;
    for (int s0 = 0; s0 < a.num_seqs; s0 += kMaxSeqsPerLaunch) {
      const int ns = std::min(kMaxSeqsPerLaunch, a.num_seqs - s0);
      items.clear();
      start.clear();
      int chunks = 0;
      for (int i = s0; i < s0 + ns; ++i) {
        items.push_back({i, cu_host[i], cu_host[i + 1] - cu_host[i], 0, 0});
        start.push_back(chunks);
        chunks += nch(i);
      }
      if (cudaError_t e = launch_intra_runs(items.data(), ns, s0, cu_host, blocks + blk, a.H, ip, nullptr, stream))
        return e;
      fill_chain(cp, items.data(), start.data(), ns);
      cp->blocks = blocks + blk;
      if (cudaError_t e = launch_chunk_chain(*cp, stream, true, use_vsplit(a, static_cast<long>(ns) * a.H, sms)))
        return e;
      blk += static_cast<size_t>(chunks) * blk_bytes;
    }
    return cudaSuccess;
  }

  // ---- split schedule
  cp->state_mid = reinterpret_cast<float *>(blocks + all_blocks);
  Chain chain{reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(a.status) + kSplitCounterOffset), 0};
  const int nseg = static_cast<int>(bounds.size()) - 1;
  const int pairs = static_cast<int>(lane.size()) * a.H;
  const double free_slots = 2.0 * std::max(sms - pairs, 1);
  // the other sequences' chunks go to the intra-chunk launches of segments 1.. where they fit beside the
  // previous segment's state pass (longest sequences first, each into the first launch with room); what is left
  // goes to the last one
  std::stable_sort(rest.begin(), rest.end(), [](const Item &x, const Item &y) { return x.nchunks() > y.nchunks(); });
  std::vector<std::vector<Item>> rest_in(nseg);
  {
    std::vector<double> room(nseg, 0.0);   // chunk-heads
    for (int k = 1; k < nseg; ++k) {
      int lane_chunks = 0;
      for (int s : lane) lane_chunks += std::max(0, std::min(bounds[k + 1], nch(s)) - bounds[k]);
      room[k] = free_slots * (bounds[k] - bounds[k - 1]) * kChainChunkUs / kIntraCtaUs -
                static_cast<double>(lane_chunks) * a.H;
    }
    for (const Item &it : rest) {
      const double need = static_cast<double>(it.nchunks()) * a.H;
      int k = 1;
      while (k < nseg && need > room[k]) ++k;
      if (k == nseg) k = nseg - 1;
      room[k] -= need;
      rest_in[k].push_back(it);
    }
  }
  std::vector<int> rest_start(rest.size());   // block index of each rest sequence, in rest_all's order
  std::vector<Item> rest_all;
  size_t blk = 0;   // in chunks
  std::vector<Item> items;
  std::vector<int> start;
  for (int k = 0; k < nseg; ++k) {
    items.clear();
    start.clear();
    int chunks = 0;
    for (size_t m = 0; m < lane.size(); ++m) {
      const int s = lane[m], c0 = bounds[k], c1 = std::min(bounds[k + 1], nch(s));
      if (c0 >= c1) continue;
      const int t0 = cu_host[s] + c0 * kChunk, t1 = std::min(cu_host[s + 1], cu_host[s] + c1 * kChunk);
      const uint8_t f = static_cast<uint8_t>((c0 > 0 ? kItemFromMid : 0) | (c1 < nch(s) ? kItemToMid : 0));
      items.push_back({s, t0, t1 - t0, f, static_cast<uint8_t>(m)});
      start.push_back(static_cast<int>(blk) + chunks);
      chunks += c1 - c0;
    }
    const int lane_items = static_cast<int>(items.size());
    for (const Item &it : rest_in[k]) {
      items.push_back(it);
      rest_all.push_back(it);
      rest_start[rest_all.size() - 1] = static_cast<int>(blk) + chunks;
      chunks += it.nchunks();
    }
    // I_k (a programmatic dependent of C_{k-1}; the call's first launch is an ordinary one)
    if (cudaError_t e = launch_intra_runs(items.data(), static_cast<int>(items.size()), 0, cu_host,
                                          blocks + blk * blk_bytes, a.H, ip, k > 0 ? &chain : nullptr, stream))
      return e;
    // C_k over the lane's items of segment k
    fill_chain(cp, items.data(), start.data(), lane_items);
    cp->blocks = blocks;
    cp->wait_blocks = 1;
    cp->trigger_after_wait = (k == nseg - 1 && !rest_all.empty()) ? 1 : 0;
    cp->done_counter = nullptr;
    // (the lane's state passes take the value split only with no other sequences beside them, whose work
    // would want those SMs: on 16384 + 16 varlen it measured 703 us against 670)
    if (cudaError_t e = launch_chunk_chain(*cp, stream, true, rest.empty() && use_vsplit(a, pairs, sms / 2)))
      return e;
    blk += chunks;
  }
  if (!rest_all.empty()) {   // C_rest beside C_{n-1}: every block exists once it may start
    fill_chain(cp, rest_all.data(), rest_start.data(), static_cast<int>(rest_all.size()));
    cp->blocks = blocks;
    cp->wait_blocks = 0;
    cp->trigger_after_wait = 0;
    cp->done_counter = chain.next();
    if (!cp->done_counter) return cudaErrorInvalidValue;   // the planner sizes the chain; not reached
    if (cudaError_t e = launch_chunk_chain(*cp, stream, true, false)) return e;
  }
  return cudaSuccess;
}

void describe_prefill_schedule(const ChunkArgs &a, const int32_t *cu_host, size_t blocks_bytes, int sms, int info[4]) {
  if (sms <= 0) sms = sm_count() > 0 ? sm_count() : 152;
  const PrefillPlan plan = plan_prefill(a, cu_host, blocks_bytes, sms);
  info[0] = plan.kind;
  info[1] = plan.kind == PrefillPlan::kPlain
                ? (a.num_seqs <= kMaxSeqsPerLaunch && use_vsplit(a, static_cast<long>(a.num_seqs) * a.H, sms))
                : plan.kind == PrefillPlan::kSplit ? (plan.rest.empty() &&
                                                      use_vsplit(a, static_cast<long>(plan.lane.size()) * a.H, sms / 2))
                                                   : 0;
  info[2] = plan.kind == PrefillPlan::kSplit ? static_cast<int>(plan.bounds.size()) - 1 : 0;
  info[3] = static_cast<int>(plan.lane.size());
}

}  // namespace kda
