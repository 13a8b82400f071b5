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


// ---------------------------------------------------------------- value-split state pass
// Two CTAs per (item, head), each owning 64 of the 128 value channels (v0 = 64 * (blockIdx.x & 1)): the
// columns of S, U^ and O are independent, and every key-side operand (W, Q+, K', P, the decay) is shared, so
// each CTA fetches the key-side tiles of the block and its half of U^^T.  The products run untransposed, with
// the 128 MMA rows on tokens or keys and both operands in shared memory:
//   D   = [W ; Q+] S                M = 128 (rows 0..63 W S, rows 64..127 Q+ S), N = 64 values, K = 128 keys
//   X   = -[I ; 0] U^               the CTA's U^ columns transposed into TMEM (an identity tile, negated by the
//                                   instruction, against the block's U^^T rows as a K-major B), so that the U
//                                   epilogue reads U^ and W S from TMEM and forms U = -(W S + X) in fp32
//   S  += K'^T U                    M = 128 keys, N = 64, K = 64 tokens (S fp32 in TMEM, lane = key rho)
//   D  += [U^^T ; P] U              rows 64..127 of D become O = Q+ S + P U; the A tile starts at the CTA's
//                                   U^^T rows just before P, whose products land in the rows the U epilogue
//                                   has already consumed
// with U = U^ - W S.  Since no product reads TMEM as an operand, the decay of S and the previous chunk's output
// read-out run beside the first product without slowing it; the serial path per chunk is the first product,
// the U epilogue, the state product and the bf16 copy of S.
//   warps 0, 1, 4, 5 (TMEM lanes 0..63): the U epilogue (a token row, 32 value columns each)
//   warps 2, 3, 6, 7 (lanes 64..127): the output epilogue of the previous chunk, then the fetch of the block
//                                     three chunks ahead into that chunk's buffer
//   all 8: the decay of S by the chunk's gamma (before the state product) and the bf16 copy of S after it
//   warp 8: MMA issue
// A chunk's buffer holds [W^T | Q+^T], then the U tile (over W^T, once the first product is done), then the
// chunk's output staging tile (over Q+^T, once its output product is done).
namespace vs {
constexpr int kThreads = 288;
constexpr int kIssuer = 256;
constexpr int kNumBuf = 3;
constexpr uint32_t BUF_WQ = 0, BUF_UH = 32768, BUF_PK = 40960, BUF_U = 0, BUF_STAGE = 16384;
constexpr uint32_t kBufStride = 65536;                 // [W^T | Q+^T] 32 KB, U^^T half 8 KB, [P ; K'^T] 24 KB
constexpr uint32_t kFetchBytes = 32768 + 8192 + 24576 + 512;   // + gamma (into its own ring)
constexpr uint32_t OFF_STILE = kNumBuf * kBufStride;   // bf16 S [key rho][64 values], MN-major B of the first product
constexpr uint32_t OFF_IDENT = OFF_STILE + 16384;      // bf16 [I ; 0], 128 rows x 64, K-major A
constexpr uint32_t OFF_SMALL = OFF_IDENT + 16384;
constexpr uint32_t SM_GAMMA = 0 /* [3][128] fp32 */, SM_BAR = 1536 /* full[3], m1, m2, m3 */, SM_TMEM = 1584,
                   SM_ABORT = 1588, SM_END = 1600;
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(OFF_STILE % 1024 == 0 && OFF_IDENT % 1024 == 0 && BUF_UH % 1024 == 0, "operand tiles");
static_assert(BUF_PK == BUF_UH + 8192, "the output product's A tile is the U^^T half followed by P");
constexpr uint32_t TM_D0 = 0, TM_D1 = 64, TM_S = 128, TM_X = 192, kTmemCols = 256;
constexpr int kBarU = 2, kBarO = 3;   // named barriers: U tile ready (all 9 warps), output warps among themselves
}  // namespace vs

template <int kId>
__device__ __forceinline__ void named_bar_arrive(int count) {
  static_assert(kId >= 1 && kId < 16, "barrier 0 is __syncthreads");
  asm volatile("bar.arrive %0, %1;" ::"n"(kId), "r"(count) : "memory");
}

__global__ void __launch_bounds__(vs::kThreads, 1) chunk_chain_vsplit_kernel(const __grid_constant__ ChainParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *small = sm + vs::OFF_SMALL;
  float *s_gamma = reinterpret_cast<float *>(small + vs::SM_GAMMA);   // [3][128]: e^(b_63) of the buffered chunks
  uint64_t *bar_full = reinterpret_cast<uint64_t *>(small + vs::SM_BAR);   // [3]: block landed in buffer b
  uint64_t *bar_m1 = bar_full + 3;    // first product done
  uint64_t *bar_m2 = bar_full + 4;    // state product done
  uint64_t *bar_m3 = bar_full + 5;    // output product done
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(small + vs::SM_TMEM);
  volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(small + vs::SM_ABORT);
  uint8_t *s_tile = sm + vs::OFF_STILE, *i_tile = sm + vs::OFF_IDENT;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = prm.H;
  const int half = blockIdx.x & 1, v0 = 64 * half;
  const int pair = blockIdx.x >> 1;
  const int h = pair % H;
  const int nl = static_cast<int>(prm.order[pair / H]);   // item, longest first
  const int n = prm.seq[nl];
  const int t0 = prm.tok0[nl];
  const int len = prm.len[nl];
  const int nchunks = (len + kChunk - 1) / kChunk;
  const uint8_t item_flags = prm.flags[nl];
  const uint8_t *blk0 = prm.blocks + (static_cast<size_t>(prm.chunk_off[nl]) * H + h) * kBlkBytes;
  const size_t blk_step = static_cast<size_t>(H) * kBlkBytes;

  if (!prm.trigger_after_wait) grid_launch_dependents();
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
  const float *src = (item_flags & kItemFromMid) ? mid
                     : prm.state_in ? prm.state_in + (static_cast<size_t>(slot) * H + h) * kD * kD : nullptr;
  // thread = (TMEM lane quadrant, 32 of the CTA's 64 value columns); lane = key rho for S, token row for D
  const bool worker = warp < 8;
  const int quad = warp & 3, vl = 32 * ((warp >> 2) & 1);
  const int rho = quad * 32 + lane;
  const size_t srow = static_cast<size_t>(kd_of_rho(rho)) * kD + v0 + vl;   // this thread's 32 state entries

  // the sequence's final short-convolution window (with conv), written by the first CTA of the pair: as in the
  // state pass above
  auto write_window = [&](auto sync) {
    constexpr int kRows = 3 * (kConvW - 1), kPieces = kRows * kD / 8;
    const int row = tid / 16, cc = tid % 16, m = row / (kConvW - 1), j = row % (kConvW - 1);
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (tid < kPieces) {
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
    if (prm.conv.weight && half == 0) write_window([] { named_bar_sync<1>(256); });
#pragma unroll 8
    for (int i = 0; i < 32; ++i) dst[srow + i] = src ? src[srow + i] : 0.f;
    finish();
    return;
  }

  // chunk c's key-side tiles, this CTA's U^^T rows and gamma -> buffer c % 3 (one thread)
  auto fetch = [&](int c) {
    const int b = c % vs::kNumBuf;
    uint8_t *buf = sm + b * vs::kBufStride;
    const uint8_t *g = blk0 + c * blk_step;
    mbar_arrive_expect_tx(&bar_full[b], vs::kFetchBytes);
    bulk_load(buf + vs::BUF_WQ, g + kBlkWQ, 32768, &bar_full[b]);
    bulk_load(buf + vs::BUF_UH, g + kBlkUH + v0 * 128, 8192, &bar_full[b]);
    bulk_load(buf + vs::BUF_PK, g + kBlkPK, 24576, &bar_full[b]);
    bulk_load(s_gamma + 128 * b, g + kBlkGamma, 512, &bar_full[b]);
  };
  if (tid == vs::kIssuer) {
    for (int i = 0; i < 6; ++i) mbar_init(&bar_full[i], 1);
    *s_abort = 0;
    fence_mbar_init();
    if (prm.wait_blocks) grid_dependency_wait();
    for (int c = 0; c < vs::kNumBuf && c < nchunks; ++c) fetch(c);
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, vs::kTmemCols);
    tmem_relinquish();
  }
  // the [I ; 0] tile: row r < 64 is e_r, rows 64..127 are zero (each thread one 16-byte piece of 4 rows)
  if (worker) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = tid + 256 * k, r = i >> 3, pc = i & 7;   // row r, columns 8 pc .. 8 pc + 7
      const bool on = r < 64 && (r >> 3) == pc;              // the piece holding column r of row r
      const int wi = (r & 7) >> 1;                           // its word; bf16 1.0 in the half of column r
      const uint32_t e = (r & 1) ? 0x3F800000u : 0x00003F80u;
      *reinterpret_cast<uint4 *>(i_tile + swz_offset(128, r, 8 * pc)) =
          make_uint4(on && wi == 0 ? e : 0u, on && wi == 1 ? e : 0u, on && wi == 2 ? e : 0u, on && wi == 3 ? e : 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (prm.trigger_after_wait) grid_launch_dependents();   // the blocks' grid has completed
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  // 32 fp32 state values -> their bf16 row piece of the S tile (4 x 16 bytes)
  auto store_s = [&](const float *s) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4 *>(s_tile + swz_offset(128, rho, vl + 8 * q)) =
          make_uint4(pack_bf16x2(s[8 * q], s[8 * q + 1]), pack_bf16x2(s[8 * q + 2], s[8 * q + 3]),
                     pack_bf16x2(s[8 * q + 4], s[8 * q + 5]), pack_bf16x2(s[8 * q + 6], s[8 * q + 7]));
  };
  // S0 -> the S tile and (undecayed) TMEM; each chunk decays its state by its own gamma before its state product
  if (worker) {
    float s[32];
    if (src) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = *reinterpret_cast<const float4 *>(src + srow + 4 * q);
        s[4 * q] = x.x; s[4 * q + 1] = x.y; s[4 * q + 2] = x.z; s[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = 0.f;
    }
    store_s(s);
    tmem_st16(tmem + lane_base + vs::TM_S + vl, s);
    tmem_st16(tmem + lane_base + vs::TM_S + vl + 16, s + 16);
    tmem_wait_st();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  const bool u_warp = worker && quad < 2, o_warp = worker && quad >= 2;
  const int orow = (quad - 2) * 32 + lane;   // output warps: token row of the chunk
  const int oi = orow + 64 * (vl >> 5);      // output warps: 0..127
  constexpr int kStoreThread = 64;           // lane 0 of warp 2
  // the output epilogue of chunk cc, whose output product the caller has waited for: its rows (D buffer
  // cc & 1, rows 64..127) -> the staging tile in its buffer -> global; then the block three chunks ahead into
  // that buffer (output warps only).  Rows go out in token order (the planner takes this kernel only without an
  // output row index).
  auto output_epilogue = [&](int cc, int rows) {
    uint8_t *buf = sm + (cc % vs::kNumBuf) * vs::kBufStride;
    uint8_t *stage = buf + vs::BUF_STAGE;
    tc_fence_after();
    uint32_t ov[32];
    const uint32_t tb = tmem + lane_base + ((cc & 1) ? vs::TM_D1 : vs::TM_D0) + vl;
    tmem_ld16_async(tb, ov);
    tmem_ld16_async(tb + 16, ov + 16);
    tmem_wait_ld();
    tmem_tie<32>(ov);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4 *>(stage + swz_offset(64, orow, vl + 8 * q)) =
          make_uint4(pack_bf16x2(__uint_as_float(ov[8 * q]), __uint_as_float(ov[8 * q + 1])),
                     pack_bf16x2(__uint_as_float(ov[8 * q + 2]), __uint_as_float(ov[8 * q + 3])),
                     pack_bf16x2(__uint_as_float(ov[8 * q + 4]), __uint_as_float(ov[8 * q + 5])),
                     pack_bf16x2(__uint_as_float(ov[8 * q + 6]), __uint_as_float(ov[8 * q + 7])));
    fence_async_smem();
    named_bar_sync<vs::kBarO>(128);
    const int tok = t0 + cc * kChunk;
    if (rows < kChunk) {   // a ragged last chunk: its valid rows one by one, 8 pieces of 16 bytes per row
      for (int i = oi; i < rows * 8; i += 128) {
        const int r = i >> 3, pc = i & 7;
        *reinterpret_cast<uint4 *>(prm.out + static_cast<int64_t>(tok + r) * prm.out_stride + h * kD + v0 + 8 * pc) =
            *reinterpret_cast<const uint4 *>(stage + swz_offset(64, r, 8 * pc));
      }
      named_bar_sync<vs::kBarO>(128);   // the staging tile has been read
      if (tid == kStoreThread && cc + vs::kNumBuf < nchunks) fetch(cc + vs::kNumBuf);
    } else if (tid == kStoreThread) {
      tma_store_3d(&prm.tout, v0, h, tok, stage);
      bulk_commit();
      if (cc + vs::kNumBuf < nchunks) {
        bulk_wait_read();
        fetch(cc + vs::kNumBuf);
      }
    }
  };

  for (int c = 0; c < nchunks; ++c) {
    const int b = c % vs::kNumBuf;
    uint8_t *buf = sm + b * vs::kBufStride;
    const uint32_t tm_d = (c & 1) ? vs::TM_D1 : vs::TM_D0;
    wait_or_abort(&bar_full[b], (c / vs::kNumBuf) & 1, s_abort, prm.status);

    // ---- D = [W ; Q+] S  (A: the [W^T | Q+^T] tile read MN-major, B: the S tile); X = -[I ; 0] U^ (the
    // identity tile against the U^^T half as a K-major B, negated)
    if (tid == vs::kIssuer) {
      tc_fence_after();
      const uint64_t a = desc_mnmajor_base(smem_u32(buf + vs::BUF_WQ), 128);
      const uint64_t bs = desc_mnmajor_base(smem_u32(s_tile), 128);
      const uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
      for (int k = 0; k < 8; ++k) mma_bf16(tmem + tm_d, a + mnmajor_step(k), bs + mnmajor_step(k), id, k > 0);
      const uint64_t ai = desc_kmajor_base(smem_u32(i_tile));
      const uint64_t bu = desc_kmajor_base(smem_u32(buf + vs::BUF_UH));
      const uint32_t idn = idesc_bf16(128, 64, false, false, true);
#pragma unroll
      for (int k = 0; k < 4; ++k) mma_bf16(tmem + vs::TM_X, ai + kmajor_step(128, k), bu + kmajor_step(64, k), idn, k > 0);
      mma_commit(bar_m1);
    }

    // ---- beside the product: S_c <- Diag(gamma_c) S_c in TMEM (all epilogue warps)
    if (worker) {
      const float g = s_gamma[128 * b + rho];
      uint32_t sv[32];
      tmem_ld16_async(tmem + lane_base + vs::TM_S + vl, sv);
      tmem_ld16_async(tmem + lane_base + vs::TM_S + vl + 16, sv + 16);
      tmem_wait_ld();
      tmem_tie<32>(sv);
      float s[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 p = mul2(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), make_float2(g, g));
        s[2 * i] = p.x;
        s[2 * i + 1] = p.y;
      }
      tmem_st16(tmem + lane_base + vs::TM_S + vl, s);
      tmem_st16(tmem + lane_base + vs::TM_S + vl + 16, s + 16);
      tmem_wait_st();
    }

    if (u_warp) {
      // ---- U = U^ - W S = -(D + X) (token rows 0..63) -> the U tile, over the W^T tile the first product has
      // consumed
      wait_or_abort(bar_m1, c & 1, s_abort, prm.status);
      tc_fence_after();
      uint32_t dv[32], xv[32];
      tmem_ld16_async(tmem + lane_base + tm_d + vl, dv);
      tmem_ld16_async(tmem + lane_base + tm_d + vl + 16, dv + 16);
      tmem_ld16_async(tmem + lane_base + vs::TM_X + vl, xv);
      tmem_ld16_async(tmem + lane_base + vs::TM_X + vl + 16, xv + 16);
      tmem_wait_ld();
      tmem_tie<32>(dv);
      tmem_tie<32>(xv);
      float u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) u[i] = -(__uint_as_float(dv[i]) + __uint_as_float(xv[i]));
      uint8_t *u_tile = buf + vs::BUF_U;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(u_tile + swz_offset(64, rho, vl + 8 * q)) =
            make_uint4(pack_bf16x2(u[8 * q], u[8 * q + 1]), pack_bf16x2(u[8 * q + 2], u[8 * q + 3]),
                       pack_bf16x2(u[8 * q + 4], u[8 * q + 5]), pack_bf16x2(u[8 * q + 6], u[8 * q + 7]));
      fence_async_smem();
      tc_fence_before();
      named_bar_sync<vs::kBarU>(vs::kThreads);
    } else if (o_warp) {
      // chunk c - 1's output product is waited for before this arrival lets chunk c's be issued (the
      // barrier's phases then cannot run two ahead of the wait)
      if (c > 0) wait_or_abort(bar_m3, (c - 1) & 1, s_abort, prm.status);
      tc_fence_before();
      named_bar_arrive<vs::kBarU>(vs::kThreads);   // the decay's TMEM stores are done
      if (c > 0) output_epilogue(c - 1, kChunk);   // chunk c - 1 is not the last one: all its rows are valid
    } else {   // the issuing warp
      named_bar_sync<vs::kBarU>(vs::kThreads);
      if (tid == vs::kIssuer) {
        tc_fence_after();
        // ---- S += K'^T U  (A: the K'^T rows of [P ; K'^T], K-major; B: the U tile)
        const uint64_t pk = desc_kmajor_base(smem_u32(buf + vs::BUF_PK));
        const uint64_t bu = desc_mnmajor_base(smem_u32(buf + vs::BUF_U), 64);
        const uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + vs::TM_S, pk + desc_bytes(64 * 128) + kmajor_step(kBlkPKRows, k), bu + mnmajor_step(k), id, 1);
        mma_commit(bar_m2);
        // ---- D += [U^^T half ; P] U: rows 64..127 of D become O = Q+ S + P U
        const uint64_t pj = desc_kmajor_base(smem_u32(buf + vs::BUF_UH));
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(tmem + tm_d, pj + kmajor_step(128, k), bu + mnmajor_step(k), id, 1);
        mma_commit(bar_m3);
      }
      __syncwarp();
    }

    // ---- S_{c+1} -> the S tile (the next chunk's first product)
    if (worker && c + 1 < nchunks) {
      wait_or_abort(bar_m2, c & 1, s_abort, prm.status);
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld16_async(tmem + lane_base + vs::TM_S + vl, sv);
      tmem_ld16_async(tmem + lane_base + vs::TM_S + vl + 16, sv + 16);
      tmem_wait_ld();
      tmem_tie<32>(sv);
      float s[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(sv[i]);
      store_s(s);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*s_abort) break;
  }

  // the last chunk's output and the final state
  const int last_valid = len - (nchunks - 1) * kChunk;
  if (o_warp) {
    wait_or_abort(bar_m3, (nchunks - 1) & 1, s_abort, prm.status);
    output_epilogue(nchunks - 1, last_valid);
  }
  if (worker) {
    wait_or_abort(bar_m2, (nchunks - 1) & 1, s_abort, prm.status);
    tc_fence_after();
    float s[32];
    tmem_ld16(tmem + lane_base + vs::TM_S + vl, s);
    tmem_ld16(tmem + lane_base + vs::TM_S + vl + 16, s + 16);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4 *>(dst + srow + 4 * q) = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
  }
  if (tid == kStoreThread) bulk_wait_all();
  if (prm.conv.weight && half == 0 && !(item_flags & kItemToMid)) write_window([] { __syncthreads(); });
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, vs::kTmemCols);
  }
  finish();
}

}  // namespace

cudaError_t launch_chunk_chain(const ChainParams &p, cudaStream_t stream, bool programmatic, bool value_split) {
  if (p.num_seqs <= 0) return cudaSuccess;
  static std::mutex mu;
  static uint64_t done = 0;
  if (const cudaError_t e = set_attributes_once(mu, done, [] {
        cudaError_t r = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (r == cudaSuccess)
          r = cudaFuncSetAttribute(chunk_chain_vsplit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   vs::kSmemBytes);
        return r;
      }))
    return e;
  // programmatic dependent launch: the grid may be scheduled while the preceding intra-chunk grid drains
  // (it waits for that grid's completion before reading any block)
  // (value_split: two CTAs per (item, head), each with 64 of the value channels)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_seqs * p.H * (value_split ? 2 : 1));
  cfg.blockDim = dim3(value_split ? vs::kThreads : kThreads);
  cfg.dynamicSmemBytes = value_split ? vs::kSmemBytes : kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return value_split ? cudaLaunchKernelEx(&cfg, chunk_chain_vsplit_kernel, p)
                     : cudaLaunchKernelEx(&cfg, chunk_chain_kernel, p);
}

}  // namespace kda
