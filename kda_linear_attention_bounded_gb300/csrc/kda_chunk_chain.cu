// State pass of the chunked KDA prefill on sm_103a.
//
// One CTA per (item, head) walks the item's chunks in order -- a whole
// sequence, or one segment of it when a long sequence's state pass is split
// (the state then arrives from and leaves to an fp32 scratch copy) -- with the
// state S (128 key x 128 value channels, fp32) resident in TMEM, and applies
// the state-dependent half of the chunk algebra to each chunk's block from the
// intra-chunk kernel (kda_prefill_block.h):
//
//   U  = U^ - W S                       (the delta-rule corrections)
//   O  = Q+ S + P U                     (scale already inside Q+ and P)
//   S' = Diag(e^(b_63)) S + K'^T U
//
// All products run transposed so that TMEM lane = value channel and M = 128:
// [U^T | O^T] = S^T [W | Q+]^T (N = 128), S'^T += U^T K' (N = 128) and
// O^T += U^T P^T (N = 64).  Their A operands S^T and U^T are bf16 copies kept
// in TMEM (tcgen05.mma with A in tensor memory); only the chunk's block comes
// from shared memory.  The state's key channels stay in the blocks' paired
// order rho; the caller's layout is used only to read S0 and to write the
// final state.
//
// Warps 0..7 run the epilogues (warp w owns TMEM lanes 32 (w % 4) .. +31 and
// half w / 4 of the columns); warp 8 only issues the MMAs and the bulk copies,
// so that a blocking MMA issue never delays an epilogue.  Per chunk the
// critical path is: first product -> U^T epilogue -> state product -> bf16
// copy of S' (which also stores the decayed state for the next state product).
// The previous chunk's output runs under the first product; blocks are
// triple-buffered, two chunks ahead.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_block.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = kChunk;
constexpr int kThreads = 288;   // 8 epilogue warps + 1 issuing warp
constexpr int kIssuer = 256;    // lane 0 of warp 8
constexpr int kNumBuf = 3;
constexpr uint32_t kBufStride = 75776;   // kBlkBytes rounded up to 1024
constexpr uint32_t OFF_SMALL = kNumBuf * kBufStride;
constexpr uint32_t SM_BAR = 0 /* full[3], m1, m2s, m2o */, SM_TMEM = 48, SM_ABORT = 52, SM_END = 64;
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kBufStride >= kBlkBytes && kBufStride % 1024 == 0, "block buffer");
// TMEM columns: S^T fp32 | two [U^T | O^T] accumulator pairs | S^T bf16 (A operand) | U^T bf16 (A operand)
constexpr uint32_t TM_S = 0, TM_UO0 = 128, TM_UO1 = 256, TM_SA = 384, TM_UA = 448, kTmemCols = 512;

__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              uint32_t *status) {
  if (*abort_flag) return;
  if (!mbar_wait(bar, parity)) {
    *abort_flag = 1;
    atomicOr(status, KDA_DEVICE_TIMEOUT);
  }
}

// 32 fp32 values -> 16 packed bf16 pairs in 16 TMEM columns
__device__ __forceinline__ void st_bf16_pairs(uint32_t taddr, const float *v) {
  float w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) w[j] = __uint_as_float(pack_bf16x2(v[2 * j], v[2 * j + 1]));
  tmem_st16(taddr, w);
}

__global__ void __launch_bounds__(kThreads, 1) chunk_chain_kernel(const __grid_constant__ ChainParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *small = sm + OFF_SMALL;
  uint64_t *bar_full = reinterpret_cast<uint64_t *>(small + SM_BAR);   // [3]: block landed in buffer b
  uint64_t *bar_m1 = bar_full + 3;    // first product done
  uint64_t *bar_m2s = bar_full + 4;   // state product done
  uint64_t *bar_m2o = bar_full + 5;   // output product done
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(small + SM_TMEM);
  volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(small + SM_ABORT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = prm.H;
  const int h = blockIdx.x % H;
  const int nl = static_cast<int>(prm.order[blockIdx.x / H]);   // item, longest first
  const int n = prm.seq[nl];
  const int t0 = prm.tok0[nl];
  const int len = prm.len[nl];
  const int nchunks = (len + kC - 1) / kC;
  const uint8_t item_flags = prm.flags[nl];
  const uint8_t *blk0 = prm.blocks + (static_cast<size_t>(prm.chunk_off[nl]) * H + h) * kBlkBytes;
  const size_t blk_step = static_cast<size_t>(H) * kBlkBytes;

  // every CTA of this grid has started once all have passed here: a grid launched after it as a programmatic
  // dependent (the verify segment of a spec step, the next intra-chunk launch of a split schedule) may then use
  // the SMs this grid leaves free
  if (!prm.trigger_after_wait) grid_launch_dependents();
  // the CTA that finishes last waits for the preceding grid (done_counter set; every exit passes here)
  auto finish = [&] {
    if (prm.done_counter && tid == 0 && atomicAdd(prm.done_counter, 1u) == gridDim.x - 1) {
      grid_dependency_wait();
      *prm.done_counter = 0;
    }
  };

  int slot = 0;
  if (prm.slot_ids) {
    slot = prm.slot_ids[n];
    if (slot < 0 || slot >= prm.num_slots) {
      if (tid == 0) atomicOr(prm.status, KDA_DEVICE_BAD_SLOT);
      finish();
      return;
    }
  }
  float *mid = prm.state_mid ? prm.state_mid + (static_cast<size_t>(prm.mid[nl]) * H + h) * kD * kD : nullptr;
  float *dst = (item_flags & kItemToMid) ? mid
               : prm.state_out_pool     ? prm.state_out_pool + (static_cast<size_t>(slot) * H + h) * kD * kD
                                        : prm.state_out_dense + (static_cast<size_t>(n) * H + h) * kD * kD;
  // epilogue thread = (value channel d, half hv of the key channels / tokens)
  const bool worker = warp < 8;
  const int quad = warp & 3, hv = (warp >> 2) & 1;
  const int d = quad * 32 + lane;
  const float *src = (item_flags & kItemFromMid) ? mid
                     : prm.state_in ? prm.state_in + (static_cast<size_t>(slot) * H + h) * kD * kD : nullptr;

  // The sequence's final short-convolution window (with conv): the last 3 raw inputs of q, k and v, rows of the
  // initial window (the slot's, else zeros) where the sequence has fewer than 3 tokens.  Every piece is read
  // before any is written (`sync` between), since the initial and final windows may be the same pool slot; the
  // intra-chunk grid, which reads initial windows, has completed when this runs.
  auto write_window = [&](auto sync) {
    constexpr int kRows = 3 * (kConvW - 1), kPieces = kRows * kD / 8;   // 144 pieces of 16 bytes
    const int row = tid / 16, cc = tid % 16, m = row / (kConvW - 1), j = row % (kConvW - 1);
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (tid < kPieces) {
      // rows before the sequence's first token come from the initial window (a segment that continues a
      // sequence has 64 or more of its tokens before it)
      if (!(item_flags & kItemFromMid) && len + j < kConvW - 1) {
        if (prm.conv_load_initial)
          val = *reinterpret_cast<const uint4 *>(
              prm.conv.window_pool + ((static_cast<size_t>(slot) * kRows + m * (kConvW - 1) + len + j) * H + h) * kD + 8 * cc);
      } else {
        const uint16_t *x = m == 0 ? prm.xq : m == 1 ? prm.xk : prm.xv;
        val = *reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t0 + len + j - (kConvW - 1)) * prm.qkv_stride +
                                               h * kD + 8 * cc);
      }
    }
    sync();
    if (tid < kPieces) {
      uint16_t *w = prm.state_out_pool
                        ? prm.conv.window_pool + ((static_cast<size_t>(slot) * kRows + row) * H + h) * kD
                        : prm.conv.window_dense + ((static_cast<size_t>(n) * kRows + row) * H + h) * kD;
      *reinterpret_cast<uint4 *>(w + 8 * cc) = val;
    }
  };

  if (nchunks == 0) {   // empty sequence: the final state is the initial one
    if (!worker) return;
    if (prm.conv.weight) write_window([] { named_bar_sync<1>(256); });
#pragma unroll 8
    for (int i = 0; i < 64; ++i) {
      const int kd = kd_of_rho(64 * hv + i);
      dst[static_cast<size_t>(kd) * kD + d] = src ? src[static_cast<size_t>(kd) * kD + d] : 0.f;
    }
    finish();
    return;
  }

  if (tid == kIssuer) {
    for (int i = 0; i < 6; ++i) mbar_init(&bar_full[i], 1);
    *s_abort = 0;
    fence_mbar_init();
    // this grid may start while the intra-chunk grid is still finishing: the blocks are read only once it
    // has completed and its writes are visible (everything above and the initial state do not depend on it)
    if (prm.wait_blocks) grid_dependency_wait();
    for (int c = 0; c < kNumBuf && c < nchunks; ++c) {
      mbar_arrive_expect_tx(&bar_full[c], kBlkBytes);
      bulk_load(sm + c * kBufStride, blk0 + c * blk_step, kBlkBytes, &bar_full[c]);
    }
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (prm.trigger_after_wait) grid_launch_dependents();   // the blocks' grid has completed
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  // S0 (this thread's 64 key channels rho = 64 hv + i) -> the bf16 A operand; once the first block is in,
  // Diag(gamma_0) S0 -> TMEM
  if (worker) {
    const int col = 64 * hv;
    float s[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const int kd = kd_of_rho(col + i);
      s[i] = src ? src[static_cast<size_t>(kd) * kD + d] : 0.f;
    }
    st_bf16_pairs(tmem + lane_base + TM_SA + col / 2, s);
    st_bf16_pairs(tmem + lane_base + TM_SA + col / 2 + 16, s + 32);
    wait_or_abort(&bar_full[0], 0, s_abort, prm.status);
    const float *gam = reinterpret_cast<const float *>(sm + kBlkGamma) + col;
#pragma unroll
    for (int i = 0; i < 64; ++i) s[i] *= gam[i];
#pragma unroll
    for (int k = 0; k < 4; ++k) tmem_st16(tmem + lane_base + TM_S + col + 16 * k, s + 16 * k);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();

  // output of a chunk (accumulated in pair ob) -> `stage` as the 64-token x 128-channel row-swizzled
  // tile the output tensor map stores (workers)
  // Scattered output (out_index set): item k of a thread is piece i = tid + k kThreads of the chunk's rows x 16
  // sixteen-byte pieces.  The output rows of a chunk are fetched one chunk ahead into registers, so the store
  // under the next chunk's first product waits on no global load.
  const bool row_pass = prm.out_index != nullptr;
  constexpr int kRowItems = (kC * 16 + kThreads - 1) / kThreads;
  int32_t orow[kRowItems];
  auto load_rows = [&](int tok, int rows) {
#pragma unroll
    for (int k = 0; k < kRowItems; ++k) {
      const int i = tid + k * kThreads;
      orow[k] = i < rows * 16 ? prm.out_index[tok + (i >> 4)] : 0;
    }
  };
  // staged rows 0 .. rows-1 -> the rows in orow (an index outside [0, num_out_rows) skips its piece)
  auto store_rows = [&](const uint8_t *stage, int rows) {
#pragma unroll
    for (int k = 0; k < kRowItems; ++k) {
      const int i = tid + k * kThreads;
      if (i >= rows * 16) break;
      const int r = i >> 4, cc = i & 15;
      const int64_t row = orow[k];
      if (row < 0 || row >= prm.num_out_rows) {
        if (cc == 0) atomicOr(prm.status, KDA_DEVICE_BAD_INDEX);
        continue;
      }
      *reinterpret_cast<uint4 *>(prm.out + row * prm.out_stride + h * kD + 8 * cc) =
          *reinterpret_cast<const uint4 *>(stage + swz_offset(64, r, 8 * cc));
    }
  };
  if (row_pass && nchunks > 0) load_rows(t0, min(kC, len));

  auto out_to_stage = [&](int ob, uint8_t *stage) {
    uint32_t ov[32];
    const uint32_t tb = tmem + lane_base + (ob ? TM_UO1 : TM_UO0) + 64 + 32 * hv;
    tmem_ld16_async(tb, ov);
    tmem_ld16_async(tb + 16, ov + 16);
    tmem_wait_ld();
    tmem_tie<32>(ov);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      *reinterpret_cast<uint16_t *>(stage + swz_offset(64, 32 * hv + i, d)) = f32_to_bf16_bits(__uint_as_float(ov[i]));
  };

  for (int c = 0; c < nchunks; ++c) {
    const int b = c % kNumBuf;
    uint8_t *buf = sm + b * kBufStride;
    const uint32_t tm_uo = c & 1 ? TM_UO1 : TM_UO0;
    wait_or_abort(&bar_full[b], (c / kNumBuf) & 1, s_abort, prm.status);

    // ---- [U^T | O^T] = S_c^T [W | Q+]^T  (one N = 128 product, A = S^T bf16 in TMEM)
    if (tid == kIssuer) {
      tc_fence_after();
      const uint64_t wq = desc_mnmajor_base(smem_u32(buf + kBlkWQ), 128);
      const uint32_t id = idesc_bf16(128, 128, false, true);
#pragma unroll
      for (int k = 0; k < 8; ++k) mma_bf16_tmem_a(tmem + tm_uo, tmem + TM_SA + 8 * k, wq + mnmajor_step(k), id, k > 0);
      mma_commit(bar_m1);
    }

    // ---- under the product: output of chunk c - 1 (its product is done) -> staged in its block buffer -> global
    if (c > 0) {
      uint8_t *prev = sm + ((c - 1) % kNumBuf) * kBufStride;
      wait_or_abort(bar_m2o, (c - 1) & 1, s_abort, prm.status);
      tc_fence_after();
      if (worker) out_to_stage((c - 1) & 1, prev);
      fence_async_smem();
      __syncthreads();
      if (row_pass) {    // rows scattered to the layer's output rows; then fetch chunk c's rows
        store_rows(prev, kC);
        load_rows(t0 + c * kC, min(kC, len - c * kC));
      } else if (tid == kIssuer) {   // chunk c - 1 is not the last one: all 64 rows are valid
        const int tok = t0 + (c - 1) * kC;
        tma_store_3d(&prm.tout, 0, h, tok, prev);
        tma_store_3d(&prm.tout, 64, h, tok, prev + 8192);
        bulk_commit();
      }
    }
    // ---- wait for the first product
    wait_or_abort(bar_m1, c & 1, s_abort, prm.status);
    tc_fence_after();

    // ---- U^T = U^^T - (W S)^T -> bf16 A operand in TMEM
    if (worker) {
      uint32_t v[32];
      tmem_ld16_async(tmem + lane_base + tm_uo + 32 * hv, v);
      tmem_ld16_async(tmem + lane_base + tm_uo + 32 * hv + 16, v + 16);
      tmem_wait_ld();
      tmem_tie<32>(v);
      float u[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = *reinterpret_cast<const uint4 *>(buf + kBlkUH + swz_offset(128, d, 32 * hv + 8 * j));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 uh = unpack_bf16x2(ws[e]);
          u[8 * j + 2 * e] = uh.x - __uint_as_float(v[8 * j + 2 * e]);
          u[8 * j + 2 * e + 1] = uh.y - __uint_as_float(v[8 * j + 2 * e + 1]);
        }
      }
      st_bf16_pairs(tmem + lane_base + TM_UA + 16 * hv, u);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();

    // ---- S^T += U^T K' (N = 128), then O^T += U^T P^T (N = 64), committed separately
    if (tid == kIssuer) {
      tc_fence_after();
      const uint64_t pk = desc_kmajor_base(smem_u32(buf + kBlkPK));
      const uint32_t id_s = idesc_bf16(128, 128, false, false), id_o = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16_tmem_a(tmem + TM_S, tmem + TM_UA + 8 * k, pk + desc_bytes(64 * 128) + kmajor_step(kBlkPKRows, k),
                        id_s, 1);
      mma_commit(bar_m2s);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16_tmem_a(tmem + tm_uo + 64, tmem + TM_UA + 8 * k, pk + kmajor_step(kBlkPKRows, k), id_o, 1);
      mma_commit(bar_m2o);
      // once the output store has read chunk c - 1's buffer, fetch the block two chunks ahead into it
      if (c > 0 && c + 2 < nchunks) {
        bulk_wait_read();
        const int bn = (c + 2) % kNumBuf;
        mbar_arrive_expect_tx(&bar_full[bn], kBlkBytes);
        bulk_load(sm + bn * kBufStride, blk0 + (c + 2) * blk_step, kBlkBytes, &bar_full[bn]);
      }
    }
    wait_or_abort(bar_m2s, c & 1, s_abort, prm.status);
    tc_fence_after();

    // ---- S_{c+1} -> the bf16 A operand of the next chunk's first product; Diag(gamma_{c+1}) S_{c+1} -> TMEM
    // (the decayed copy is only needed by the next chunk's state product)
    if (worker && c + 1 < nchunks) {
      const int col = 64 * hv;
      uint32_t sv[64];
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_ld16_async(tmem + lane_base + TM_S + col + 16 * k, sv + 16 * k);
      tmem_wait_ld();
      tmem_tie<64>(sv);
      float s[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(sv[i]);
      st_bf16_pairs(tmem + lane_base + TM_SA + col / 2, s);
      st_bf16_pairs(tmem + lane_base + TM_SA + col / 2 + 16, s + 32);
      const int bn = (c + 1) % kNumBuf;
      wait_or_abort(&bar_full[bn], ((c + 1) / kNumBuf) & 1, s_abort, prm.status);
      // the block's e^(b_63) for the thread's 64 key channels: 16-byte broadcast loads, packed multiplies
      const float4 *gam = reinterpret_cast<const float4 *>(sm + bn * kBufStride + kBlkGamma + 4 * col);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 g = gam[i];
        const float2 lo = mul2(make_float2(s[4 * i], s[4 * i + 1]), make_float2(g.x, g.y));
        const float2 hi = mul2(make_float2(s[4 * i + 2], s[4 * i + 3]), make_float2(g.z, g.w));
        s[4 * i] = lo.x;
        s[4 * i + 1] = lo.y;
        s[4 * i + 2] = hi.x;
        s[4 * i + 3] = hi.y;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_st16(tmem + lane_base + TM_S + col + 16 * k, s + 16 * k);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    if (*s_abort) break;
  }

  // output of the last chunk, and the final state
  wait_or_abort(bar_m2o, (nchunks - 1) & 1, s_abort, prm.status);
  tc_fence_after();
  uint8_t *last = sm + ((nchunks - 1) % kNumBuf) * kBufStride;
  const int last_valid = len - (nchunks - 1) * kC;
  if (worker) out_to_stage((nchunks - 1) & 1, last);
  fence_async_smem();
  __syncthreads();
  if (row_pass) {
    store_rows(last, last_valid);
  } else if (last_valid == kC) {
    if (tid == kIssuer) {
      const int tok = t0 + (nchunks - 1) * kC;
      tma_store_3d(&prm.tout, 0, h, tok, last);
      tma_store_3d(&prm.tout, 64, h, tok, last + 8192);
      bulk_commit();
    }
  } else {   // a ragged last chunk: only its valid rows, 16 bytes per thread and step
    uint16_t *o = prm.out + static_cast<size_t>(t0 + (nchunks - 1) * kC) * prm.out_stride + h * kD;
    for (int idx = tid; idx < last_valid * 16; idx += kThreads) {
      const int r = idx >> 4, cc = idx & 15;
      *reinterpret_cast<uint4 *>(o + static_cast<size_t>(r) * prm.out_stride + 8 * cc) =
          *reinterpret_cast<const uint4 *>(last + swz_offset(64, r, 8 * cc));
    }
  }
  if (tid == kIssuer) bulk_wait_all();
  if (worker) {
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int col = 64 * hv + 32 * part;
      uint32_t sv[32];
      tmem_ld16_async(tmem + lane_base + TM_S + col, sv);
      tmem_ld16_async(tmem + lane_base + TM_S + col + 16, sv + 16);
      tmem_wait_ld();
      tmem_tie<32>(sv);
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(kd_of_rho(col + i)) * kD + d] = __uint_as_float(sv[i]);
    }
  }
  if (prm.conv.weight && !(item_flags & kItemToMid)) write_window([] { __syncthreads(); });
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  finish();
}

}  // namespace

cudaError_t launch_chunk_chain(const ChainParams &p, cudaStream_t stream, bool programmatic) {
  if (p.num_seqs <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // programmatic dependent launch: the grid may be scheduled while the preceding intra-chunk grid drains
  // (it waits for that grid's completion before reading any block)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_seqs * p.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, chunk_chain_kernel, p);
}

}  // namespace kda
