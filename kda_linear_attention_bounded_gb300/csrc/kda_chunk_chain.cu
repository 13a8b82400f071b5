// State pass of the chunked KDA prefill on sm_103a.
//
// One CTA per (sequence, head) walks the sequence's chunks in order with the
// state S (128 key x 128 value channels, fp32) resident in TMEM, and applies
// the state-dependent half of the chunk algebra to each chunk's block from the
// intra-chunk kernel (kda_prefill_block.h):
//
//   U  = U^ - W S                       (the delta-rule corrections)
//   O  = Q+ S + P U                     (scale already inside Q+ and P)
//   S' = Diag(e^(b_63)) S + K'^T U
//
// All three products run transposed so that TMEM lane = value channel and M =
// 128: [U^T | O^T] = S^T [W | Q+]^T (N = 64 + 64) and [O^T | S'^T] += U^T [P ;
// K'^T]^T (N = 64 + 128).  The state's key channels are kept in the blocks'
// paired order rho; the caller's layout is used only to read S0 and to write
// the final state.
//
// Per chunk the critical path is the two tcgen05.mma groups and two short
// epilogues: U^T to bf16 (the A operand of the second product), and S' to the
// bf16 operand of the next chunk's first product while its decayed copy goes
// back to TMEM.  The next block arrives by bulk copy a whole chunk ahead.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_block.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = kChunk;
constexpr int kThreads = 256;
constexpr uint32_t kBufStride = 75776;      // kBlkBytes rounded up to 1024
constexpr uint32_t OFF_ST = 0;              // S^T bf16 K-major [dv][rho] (A of the first product), 32 KB
constexpr uint32_t OFF_BUF = 32768;         // two blocks
constexpr uint32_t OFF_UT = OFF_BUF + 2 * kBufStride;   // U^T bf16 K-major [dv][t], 16 KB
constexpr uint32_t OFF_OST = OFF_UT + 16384;             // output staging bf16 [64][136]
constexpr int kOStride = 136;
constexpr uint32_t OFF_SMALL = OFF_OST + 64 * kOStride * 2;
constexpr uint32_t SM_BAR = 0, SM_TMEM = 32, SM_ABORT = 36, SM_END = 64;
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kBufStride >= kBlkBytes && kBufStride % 1024 == 0, "block buffer");
constexpr uint32_t TM_U = 0, TM_O = 64, TM_S = 128, kTmemCols = 256;

__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              uint32_t *status) {
  if (*abort_flag) return;
  if (!mbar_wait(bar, parity)) {
    *abort_flag = 1;
    atomicOr(status, KDA_DEVICE_TIMEOUT);
  }
}

// 64 fp32 values -> bf16, 128 bytes of row `row` of a row-swizzled tile of R rows from column col0
__device__ __forceinline__ void store_row64(uint8_t *tile, int R, int row, int col0, const float *v) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4 *>(tile + swz_offset(R, row, col0 + 8 * j)) =
        make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                   pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
}

__global__ void __launch_bounds__(kThreads, 1) chunk_chain_kernel(const __grid_constant__ ChainParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *small = sm + OFF_SMALL;
  uint64_t *bar_full = reinterpret_cast<uint64_t *>(small + SM_BAR);   // [2]
  uint64_t *bar_mma = bar_full + 2;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(small + SM_TMEM);
  volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(small + SM_ABORT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = prm.H;
  const int h = blockIdx.x % H;
  const int nl = static_cast<int>(prm.order[blockIdx.x / H]);   // local sequence, longest first
  const int n = prm.seq0 + nl;
  const int t0 = prm.tok_off[nl];
  const int len = prm.tok_off[nl + 1] - t0;
  const int nchunks = prm.chunk_off[nl + 1] - prm.chunk_off[nl];
  const uint8_t *blk0 = prm.blocks + (static_cast<size_t>(prm.chunk_off[nl]) * H + h) * kBlkBytes;
  const size_t blk_step = static_cast<size_t>(H) * kBlkBytes;

  int slot = 0;
  if (prm.slot_ids) {
    slot = prm.slot_ids[n];
    if (slot < 0 || slot >= prm.num_slots) {
      if (tid == 0) atomicOr(prm.status, KDA_DEVICE_BAD_SLOT);
      return;
    }
  }
  float *dst = prm.state_out_pool ? prm.state_out_pool + (static_cast<size_t>(slot) * H + h) * kD * kD
                                  : prm.state_out_dense + (static_cast<size_t>(n) * H + h) * kD * kD;
  // thread = (value channel d, half of the key channels / tokens)
  const int quad = warp & 3, hv = warp >> 2;
  const int d = quad * 32 + lane;
  const float *src = prm.state_in ? prm.state_in + (static_cast<size_t>(slot) * H + h) * kD * kD : nullptr;

  if (nchunks == 0) {   // empty sequence: the final state is the initial one
#pragma unroll 8
    for (int i = 0; i < 64; ++i) {
      const int kd = kd_of_rho(64 * hv + i);
      dst[static_cast<size_t>(kd) * kD + d] = src ? src[static_cast<size_t>(kd) * kD + d] : 0.f;
    }
    return;
  }

  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(bar_mma, 1);
    *s_abort = 0;
    fence_mbar_init();
    for (int c = 0; c < 2 && c < nchunks; ++c) {
      mbar_arrive_expect_tx(&bar_full[c], kBlkBytes);
      bulk_load(sm + OFF_BUF + c * kBufStride, blk0 + c * blk_step, kBlkBytes, &bar_full[c]);
    }
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  // S0 -> bf16 operand, and Diag(gamma_0) S0 -> TMEM
  {
    float s[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const int kd = kd_of_rho(64 * hv + i);
      s[i] = src ? src[static_cast<size_t>(kd) * kD + d] : 0.f;
    }
    store_row64(sm + OFF_ST, 128, d, 64 * hv, s);
    wait_or_abort(&bar_full[0], 0, s_abort, prm.status);
    const float *gam = reinterpret_cast<const float *>(sm + OFF_BUF + kBlkGamma) + 64 * hv;
#pragma unroll
    for (int i = 0; i < 64; ++i) s[i] *= gam[i];
#pragma unroll
    for (int k = 0; k < 4; ++k) tmem_st16(tmem + lane_base + TM_S + 64 * hv + 16 * k, s + 16 * k);
    tmem_wait_st();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  uint32_t mma_phase = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int b = c & 1;
    uint8_t *buf = sm + OFF_BUF + b * kBufStride;
    const int tok0 = t0 + c * kC;
    const int valid = min(kC, len - c * kC);

    // ---- [U^T | O^T] = S^T [W | Q+]^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t st = smem_u32(sm + OFF_ST), wq = smem_u32(buf + kBlkWQ);
      const uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_bf16(tmem + TM_U, desc_kmajor(st, 128, s), desc_mnmajor(wq, 128, s), id, s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_bf16(tmem + TM_O, desc_kmajor(st, 128, s), desc_mnmajor(wq + 16384, 128, s), id, s > 0);
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_or_abort(bar_mma, mma_phase & 1, s_abort, prm.status);
    ++mma_phase;
    tc_fence_after();

    // ---- U^T = U^^T - (W S)^T -> bf16 [dv][t]
    {
      uint32_t v[32];
      tmem_ld16_async(tmem + lane_base + TM_U + 32 * hv, v);
      tmem_ld16_async(tmem + lane_base + TM_U + 32 * hv + 16, v + 16);
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
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(sm + OFF_UT + swz_offset(128, d, 32 * hv + 8 * j)) =
            make_uint4(pack_bf16x2(u[8 * j], u[8 * j + 1]), pack_bf16x2(u[8 * j + 2], u[8 * j + 3]),
                       pack_bf16x2(u[8 * j + 4], u[8 * j + 5]), pack_bf16x2(u[8 * j + 6], u[8 * j + 7]));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- [O^T | S^T] += U^T [P ; K'^T]^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ut = smem_u32(sm + OFF_UT), pk = smem_u32(buf + kBlkPK);
      const uint32_t id = idesc_bf16(128, kBlkPKRows, false, false);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_O, desc_kmajor(ut, 128, s), desc_kmajor(pk, kBlkPKRows, s), id, 1);
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_or_abort(bar_mma, mma_phase & 1, s_abort, prm.status);
    ++mma_phase;
    tc_fence_after();
    // the block is consumed: fetch chunk c + 2 into its buffer
    if (tid == 0 && c + 2 < nchunks) {
      mbar_arrive_expect_tx(&bar_full[b], kBlkBytes);
      bulk_load(buf, blk0 + (c + 2) * blk_step, kBlkBytes, &bar_full[b]);
    }

    // ---- S' -> bf16 operand and Diag(gamma_next) S' -> TMEM (or the final state); O -> staging
    {
      uint32_t sv[64];
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_ld16_async(tmem + lane_base + TM_S + 64 * hv + 16 * k, sv + 16 * k);
      uint32_t ov[32];
      tmem_ld16_async(tmem + lane_base + TM_O + 32 * hv, ov);
      tmem_ld16_async(tmem + lane_base + TM_O + 32 * hv + 16, ov + 16);
      tmem_wait_ld();
      tmem_tie<64>(sv);
      tmem_tie<32>(ov);
      float *s = reinterpret_cast<float *>(sv);
      if (c + 1 < nchunks) {
        store_row64(sm + OFF_ST, 128, d, 64 * hv, s);
        wait_or_abort(&bar_full[b ^ 1], ((c + 1) >> 1) & 1, s_abort, prm.status);
        const float *gam = reinterpret_cast<const float *>(sm + OFF_BUF + (b ^ 1) * kBufStride + kBlkGamma) + 64 * hv;
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] *= gam[i];
#pragma unroll
        for (int k = 0; k < 4; ++k) tmem_st16(tmem + lane_base + TM_S + 64 * hv + 16 * k, s + 16 * k);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[static_cast<size_t>(kd_of_rho(64 * hv + i)) * kD + d] = s[i];
      }
      uint16_t *sO = reinterpret_cast<uint16_t *>(sm + OFF_OST);
#pragma unroll
      for (int i = 0; i < 32; ++i) sO[(32 * hv + i) * kOStride + d] = f32_to_bf16_bits(__uint_as_float(ov[i]));
      tmem_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    {
      const uint16_t *sO = reinterpret_cast<const uint16_t *>(sm + OFF_OST);
      for (int idx = tid; idx < valid * 16; idx += kThreads) {
        const int r = idx >> 4, cc = idx & 15;
        *reinterpret_cast<uint4 *>(prm.out + static_cast<size_t>(tok0 + r) * prm.out_stride + h * kD + 8 * cc) =
            *reinterpret_cast<const uint4 *>(sO + r * kOStride + 8 * cc);
      }
    }
    if (*s_abort) break;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_chunk_chain(const ChainParams &p, cudaStream_t stream) {
  if (p.num_seqs <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  chunk_chain_kernel<<<p.num_seqs * p.H, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
