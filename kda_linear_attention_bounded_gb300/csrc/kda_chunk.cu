// Chunked prefill of the KDA bounded-gate recurrence on sm_103a.
//
// One CTA per (sequence, head) walks the sequence in chunks of C = 64
// tokens.  Within a chunk of rows r = 0..63 that starts from state S
// (dk x dv, kept in fp32 registers), with per-channel log-decays lambda and
// b_r = sum_{j<=r} lambda_j (the bounded gate and the in-kernel q/k l2norm
// of vLLM PR #55737 "Use FlashKDA for KDA chunked prefill", PR summary):
//
//   A[r,i] = beta_r sum_c k^_rc k^_ic e^(b_rc - b_ic)   (i < r)
//   P[r,i] =        sum_c q^_rc k^_ic e^(b_rc - b_ic)   (i <= r)
//   T      = (I + A)^-1 Diag(beta)
//   W = T (K^ o e^b),  U = T V - W S
//   O = scale ((Q^ o e^b) S + P U)
//   S' = Diag(e^b_63) S + (K^ o e^(b_63 - b))^T U
//
// which is the token recurrence S_t = (I - beta k^ k^T) Diag(alpha) S_{t-1}
// + beta k^ v^T, o_t = scale S_t^T q^ unrolled over the chunk (the
// corrections u_r solve (I + A) U = Diag(beta)(V - (K^ o e^b) S)).
//
// Where the work goes:
//  * the six dense contractions (W^T, U^T, O^T, the state update) are
//    tcgen05.mma (bf16 in, fp32 accumulate) with operands in 128-byte
//    swizzled shared memory and accumulators in TMEM, all with M = 128 so
//    that TMEM lane = value channel (W^T: lane = key channel);
//  * q, k, v, g arrive by TMA (3-D tensor maps over [tokens, H, 128] with the
//    caller's token stride);
//  * A and P need exp(b_r - b_i) inside the contraction over c, and b spans
//    up to 64 * |lower_bound| within a chunk -- far outside fp32.  They are
//    built from 16-row sub-blocks: with m_R = b at row 7 of block R and
//    a_I = b at row 15 of block I,
//      same block:  e^(b_r - b_i) = e^(b_r - m_R) * e^(m_R - b_i)   (|exponents| <= 8 |lb|)
//      block I < R: e^(b_r - b_i) = [e^(b_r - m_R) e^(m_R - a_I)] * e^(a_I - b_i)
//    The per-channel factor e^(m_R - a_I) (<= 1) depends on both blocks, so
//    these 16x16x128 products use warp-level mma.sync with that factor
//    applied to the operand fragments in registers; materialising one scaled
//    copy per block pair for tcgen05 would multiply the operand preparation.
//  * T by blocked forward substitution in fp32 on CUDA cores.
#include <cuda.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;          // chunk length
constexpr int kThreads = 256;   // 8 warps
constexpr int kTileBytes = 16384;  // one 64 x 128 bf16 tile

// ---- shared memory map (offsets from a 1024-byte aligned base) ----
constexpr uint32_t OFF_Q = 0;        // q (TMA) -> Q+ = q^ o e^b, in place
constexpr uint32_t OFF_K = 16384;    // k (TMA) -> K+ = k^ o e^b, in place
constexpr uint32_t OFF_V = 32768;    // v (TMA)
constexpr uint32_t OFF_G = 49152;    // g (TMA) -> K' = k^ o e^(b_63 - b), in place
constexpr uint32_t OFF_X = 65536;    // phase-dependent scratch, 66560 bytes:
//   prologue .. A/P products:  F^K, F^Q (k^, q^ o e^(b - m)), G (k^ o e^(m - b)), G' (k^ o e^(a - b))
constexpr uint32_t X_FK = 0, X_FQ = 16384, X_G = 32768, X_GP = 49152;
//   after the products:  A fp32 [64][68] | P bf16 | T bf16 | W bf16 [dk][r] | U^T bf16 [dv][i]
constexpr uint32_t X_A = 0, X_P = 17408, X_T = 25600, X_W = 33792, X_UT = 50176;
//   during the solve: (I + A)^-1 fp32 [64][68] over W and U^T; T region holds block products
constexpr uint32_t X_INV = 33792, X_Y = 25600;
constexpr int kAStride = 68;  // floats per row of A / (I+A)^-1
constexpr uint32_t OFF_ST = OFF_X + 66560;   // S^T bf16 [dv][dk] (K-major operand), 32 KB
constexpr uint32_t OFF_SMALL = OFF_ST + 32768;
constexpr uint32_t SM_NQ = 0, SM_NK = 256, SM_BETA = 512, SM_BSUM = 768, SM_GL = 2816, SM_C = 3328,
                   SM_DTB = 4864, SM_BAR = 5376, SM_TMEM = 5408, SM_ABORT = 5412, SM_END = 5440;
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;  // + alignment slack

// ---- TMEM columns (fp32 accumulators, lane = row of the M = 128 tile) ----
constexpr uint32_t TM_W = 0, TM_U = 64, TM_O = 128, TM_S = 256, TM_COLS = 512;

struct Params {
  CUtensorMap tq, tk, tv, tg;
  ChunkArgs a;
  int use_order;
  uint16_t order[kMaxPlannedSeqs];
};

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ void st_u32(uint8_t *p, uint32_t v) { *reinterpret_cast<uint32_t *>(p) = v; }

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ float exp_f(float x) { return fast_exp2(x * kLog2e); }

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Wait on an mbarrier phase; a wait that gives up records the fault and
// raises the CTA-wide abort flag (checked at chunk boundaries).
__device__ __forceinline__ void wait_or_flag(uint64_t *bar, uint32_t parity, uint32_t *abort_flag,
                                             uint32_t *status) {
  if (!mbar_wait(bar, parity)) {
    *abort_flag = 1;
    atomicOr(status, KDA_DEVICE_TIMEOUT);
  }
}

// Convert 32 fp32 values of one TMEM lane to bf16 and store them as four
// 16-byte chunks of row `row` (columns col0 .. col0+31) of a row-swizzled tile.
__device__ __forceinline__ void store_row32_bf16(uint8_t *tile, int R, int row, int col0, const float *v) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
    w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
    w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
    w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
    *reinterpret_cast<uint4 *>(tile + swz_offset(R, row, col0 + 8 * j)) = w;
  }
}

__global__ void __launch_bounds__(kThreads, 1) chunk_prefill_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem + OFF_Q, *sK = smem + OFF_K, *sV = smem + OFF_V, *sG = smem + OFF_G;
  uint8_t *sX = smem + OFF_X, *sST = smem + OFF_ST;
  uint8_t *small = smem + OFF_SMALL;
  float *s_nq = reinterpret_cast<float *>(small + SM_NQ);
  float *s_nk = reinterpret_cast<float *>(small + SM_NK);
  float *s_beta = reinterpret_cast<float *>(small + SM_BETA);
  float *s_bsum = reinterpret_cast<float *>(small + SM_BSUM);   // [4][128]
  float *s_gl = reinterpret_cast<float *>(small + SM_GL);       // [128] e^(b_63)
  uint32_t *s_c = reinterpret_cast<uint32_t *>(small + SM_C);   // [6][64] bf16x2 e^(m_R - a_I)
  float *s_dtb = reinterpret_cast<float *>(small + SM_DTB);     // [128]
  uint64_t *bar_qkv = reinterpret_cast<uint64_t *>(small + SM_BAR);
  uint64_t *bar_g = bar_qkv + 1;
  uint64_t *bar_mma = bar_qkv + 2;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(small + SM_TMEM);
  uint32_t *s_abort = reinterpret_cast<uint32_t *>(small + SM_ABORT);

  const ChunkArgs &a = p.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x % a.H;
  const int j_seq = blockIdx.x / a.H;
  const int n = p.use_order ? static_cast<int>(p.order[j_seq]) : j_seq;
  const int t0 = a.cu_seqlens[n];
  const int len = a.cu_seqlens[n + 1] - t0;
  const int nchunks = (len + kC - 1) / kC;

  int slot = 0;
  if (a.slot_ids) {
    slot = a.slot_ids[n];
    if (slot < 0 || slot >= a.num_slots) {
      if (tid == 0) atomicOr(a.status, KDA_DEVICE_BAD_SLOT);
      return;
    }
  }

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    mbar_init(bar_qkv, 1);
    mbar_init(bar_g, 1);
    mbar_init(bar_mma, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TM_COLS);
    tmem_relinquish();
  }
  if (tid < kD) s_dtb[tid] = a.dt_bias[h * kD + tid];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (tid == 0 && nchunks > 0) {
    prefetch_tensormap(&p.tq);
    prefetch_tensormap(&p.tk);
    prefetch_tensormap(&p.tv);
    prefetch_tensormap(&p.tg);
    mbar_arrive_expect_tx(bar_qkv, 3 * kTileBytes);
    tma_load_3d(sQ, &p.tq, 0, h, t0, bar_qkv);
    tma_load_3d(sQ + 8192, &p.tq, 64, h, t0, bar_qkv);
    tma_load_3d(sK, &p.tk, 0, h, t0, bar_qkv);
    tma_load_3d(sK + 8192, &p.tk, 64, h, t0, bar_qkv);
    tma_load_3d(sV, &p.tv, 0, h, t0, bar_qkv);
    tma_load_3d(sV + 8192, &p.tv, 64, h, t0, bar_qkv);
    mbar_arrive_expect_tx(bar_g, kTileBytes);
    tma_load_3d(sG, &p.tg, 0, h, t0, bar_g);
    tma_load_3d(sG + 8192, &p.tg, 64, h, t0, bar_g);
  }

  // State S^T in registers: thread owns value channel d and key channels
  // [64*hh, 64*hh + 64) -- exactly its TMEM lane / column half.
  const int quad = warp & 3, hh = warp >> 2;
  const int d = quad * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  float S[64];
  if (a.state_in) {
    const float *src = a.state_in + ((size_t)slot * a.H + h) * kD * kD + d;
#pragma unroll
    for (int i = 0; i < 64; ++i) S[i] = src[(size_t)(64 * hh + i) * kD];
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) S[i] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) store_row32_bf16(sST, 128, d, 64 * hh + 32 * j, S + 32 * j);
  fence_async_smem();
  __syncthreads();

  const float ea = __expf(a.A_log[h]);
  const float lb = a.lower_bound;
  uint32_t mma_phase = 0;

  for (int chunk = 0; chunk < nchunks; ++chunk) {
    const int tok0 = t0 + chunk * kC;
    const int valid = min(kC, len - chunk * kC);
    const uint32_t tma_parity = chunk & 1;
    wait_or_flag(bar_qkv, tma_parity, s_abort, a.status);
    wait_or_flag(bar_g, tma_parity, s_abort, a.status);

    // ---------------------------------------------- A1: norms, beta, padding
    {
      const int task = tid >> 1, half = tid & 1;
      const int r = task & 63;
      const uint8_t *tile = task < 64 ? sQ : sK;
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = *reinterpret_cast<const uint4 *>(tile + swz_offset(64, r, 64 * half + 8 * j));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(ws[e]);
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (half == 0) {
        const float nrm = r < valid ? rsqrtf(ss + kL2Eps) : 0.f;
        (task < 64 ? s_nq : s_nk)[r] = nrm;
      }
      if (tid < kC) {
        s_beta[tid] = tid < valid ? sigmoid_f(bf16_bits_to_f32(a.beta[(size_t)(tok0 + tid) * a.beta_stride + h]))
                                  : 0.f;
      }
      if (valid < kC) {  // rows past the sequence end: zero v (the others are masked through beta, norms, lambda)
        for (int idx = tid; idx < (kC - valid) * 16; idx += kThreads) {
          const int r2 = valid + idx / 16, cc = idx % 16;
          *reinterpret_cast<uint4 *>(sV + swz_offset(64, r2, 8 * cc)) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    __syncthreads();

    // ---------------------------------------------- A2: gate, decay, operands
    {
      const int cp = tid & 63;        // channel pair
      const int R = tid >> 6;         // 16-row block
      const int c0 = 2 * cp;
      const float dtb0 = s_dtb[c0], dtb1 = s_dtb[c0 + 1];
      float b0[16], b1[16];
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = 16 * R + j;
        const float2 gg = unpack_bf16x2(ld_u32(sG + swz_offset(64, r, c0)));
        const bool ok = r < valid;
        const float l0 = ok ? lb * sigmoid_f(ea * (gg.x + dtb0)) : 0.f;
        const float l1 = ok ? lb * sigmoid_f(ea * (gg.y + dtb1)) : 0.f;
        acc0 += l0;
        acc1 += l1;
        b0[j] = acc0;
        b1[j] = acc1;
      }
      s_bsum[R * kD + c0] = acc0;
      s_bsum[R * kD + c0 + 1] = acc1;
      __syncthreads();
      float pre[5][2];  // pre[I] = b at the end of block I-1 (prefix), pre[4] = chunk total
      pre[0][0] = pre[0][1] = 0.f;
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        pre[I + 1][0] = pre[I][0] + s_bsum[I * kD + c0];
        pre[I + 1][1] = pre[I][1] + s_bsum[I * kD + c0 + 1];
      }
      const float m0 = pre[R][0] + b0[7], m1 = pre[R][1] + b1[7];  // b at row 7 of the block
      if (R == 0) {
        s_gl[c0] = exp_f(pre[4][0]);
        s_gl[c0 + 1] = exp_f(pre[4][1]);
      }
      // e^(m_R - a_I) for the blocks I < R  (a_I = pre[I + 1])
#pragma unroll
      for (int I = 0; I < 3; ++I) {
        if (I < R) {
          const int pidx = R * (R - 1) / 2 + I;
          s_c[pidx * 64 + cp] = pack_bf16x2(exp_f(m0 - pre[I + 1][0]), exp_f(m1 - pre[I + 1][1]));
        }
      }
      const float em0 = exp_f(m0), em1 = exp_f(m1);                      // e^(m_R)
      const float el0 = exp_f(pre[4][0] - m0), el1 = exp_f(pre[4][1] - m1);  // e^(b_63 - m_R)
      const float eg0 = exp_f(b0[15] - b0[7]), eg1 = exp_f(b1[15] - b1[7]);  // e^(a_R - m_R)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = 16 * R + j;
        const float e0 = exp_f(b0[j] - b0[7]), e1 = exp_f(b1[j] - b1[7]);
        const float i0 = exp_f(b0[7] - b0[j]), i1 = exp_f(b1[7] - b1[j]);
        const uint32_t off = swz_offset(64, r, c0);
        const float2 qq = unpack_bf16x2(ld_u32(sQ + off));
        const float2 kk = unpack_bf16x2(ld_u32(sK + off));
        const float nq = s_nq[r], nk = s_nk[r];
        const float qh0 = qq.x * nq, qh1 = qq.y * nq, kh0 = kk.x * nk, kh1 = kk.y * nk;
        const float fk0 = kh0 * e0, fk1 = kh1 * e1, fq0 = qh0 * e0, fq1 = qh1 * e1;
        const float g0 = kh0 * i0, g1 = kh1 * i1;
        st_u32(sX + X_FK + off, pack_bf16x2(fk0, fk1));
        st_u32(sX + X_FQ + off, pack_bf16x2(fq0, fq1));
        st_u32(sX + X_G + off, pack_bf16x2(g0, g1));
        st_u32(sX + X_GP + off, pack_bf16x2(g0 * eg0, g1 * eg1));
        st_u32(sQ + off, pack_bf16x2(fq0 * em0, fq1 * em1));  // Q+
        st_u32(sK + off, pack_bf16x2(fk0 * em0, fk1 * em1));  // K+
        st_u32(sG + off, pack_bf16x2(g0 * el0, g1 * el1));    // K'
      }
    }
    __syncthreads();

    // ---------------------------------------------- B: A and P (16x16 sub-blocks, mma.sync)
    {
      const int g = lane >> 2, t = lane & 3;
      float accA[2][2][4], accP[2][2][4];  // [item][ntile][4]
      int items[2] = {warp, warp + 8};
#pragma unroll
      for (int it = 0; it < 2; ++it) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) accA[it][nt][e] = accP[it][nt][e] = 0.f;
      }
      // item index -> (R, I): 0:(0,0) 1:(1,0) 2:(1,1) 3:(2,0) 4:(2,1) 5:(2,2) 6:(3,0) 7:(3,1) 8:(3,2) 9:(3,3)
      const uint32_t base_fk = smem_u32(sX + X_FK), base_fq = smem_u32(sX + X_FQ);
      const uint32_t base_g = smem_u32(sX + X_G), base_gp = smem_u32(sX + X_GP);
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int item = items[it];
        if (item < 10) {
          const int R = item < 1 ? 0 : item < 3 ? 1 : item < 6 ? 2 : 3;
          const int I = item - R * (R + 1) / 2;
          const uint32_t bbase = (I == R) ? base_g : base_gp;
          const int pidx = R * (R - 1) / 2 + I;
          const int arow = 16 * R + (lane & 15);
          const int brow = 16 * I + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            uint32_t ak[4], aq[4], bb[4];
            const uint32_t aoff = swz_offset(64, arow, 16 * s + 8 * (lane >> 4));
            ldmatrix_x4(base_fk + aoff, ak[0], ak[1], ak[2], ak[3]);
            ldmatrix_x4(base_fq + aoff, aq[0], aq[1], aq[2], aq[3]);
            ldmatrix_x4(bbase + swz_offset(64, brow, 16 * s + 8 * ((lane >> 3) & 1)), bb[0], bb[1], bb[2], bb[3]);
            if (I < R) {
              const uint32_t clo = s_c[pidx * 64 + 8 * s + t], chi = s_c[pidx * 64 + 8 * s + t + 4];
              ak[0] = bf16x2_mul(ak[0], clo);
              ak[1] = bf16x2_mul(ak[1], clo);
              ak[2] = bf16x2_mul(ak[2], chi);
              ak[3] = bf16x2_mul(ak[3], chi);
              aq[0] = bf16x2_mul(aq[0], clo);
              aq[1] = bf16x2_mul(aq[1], clo);
              aq[2] = bf16x2_mul(aq[2], chi);
              aq[3] = bf16x2_mul(aq[3], chi);
            }
            mma_16816(accA[it][0], ak, bb[0], bb[1]);
            mma_16816(accA[it][1], ak, bb[2], bb[3]);
            mma_16816(accP[it][0], aq, bb[0], bb[1]);
            mma_16816(accP[it][1], aq, bb[2], bb[3]);
          }
        }
      }
      __syncthreads();  // every F / G read is done: the X region is reused below
      // zero the strictly-upper 16x16 blocks of P
      for (int idx = tid; idx < 6 * 128; idx += kThreads) {
        const int blk = idx / 128, e = idx % 128;
        const int R = blk < 3 ? 0 : blk < 5 ? 1 : 2;
        const int I = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
        const int r = 16 * R + e / 8, i = 16 * I + 2 * (e % 8);
        st_u32(sX + X_P + swz_offset(64, r, i), 0u);
      }
      float *sA = reinterpret_cast<float *>(sX + X_A);
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int item = items[it];
        if (item < 10) {
          const int R = item < 1 ? 0 : item < 3 ? 1 : item < 6 ? 2 : 3;
          const int I = item - R * (R + 1) / 2;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int r = 16 * R + g + 8 * hr;
              const int i = 16 * I + 8 * nt + 2 * t;
              float a0 = accA[it][nt][2 * hr] * s_beta[r], a1 = accA[it][nt][2 * hr + 1] * s_beta[r];
              float p0 = accP[it][nt][2 * hr], p1 = accP[it][nt][2 * hr + 1];
              if (I == R) {
                a0 = (i < r) ? a0 : 0.f;
                a1 = (i + 1 < r) ? a1 : 0.f;
                p0 = (i <= r) ? p0 : 0.f;
                p1 = (i + 1 <= r) ? p1 : 0.f;
              }
              *reinterpret_cast<float2 *>(sA + r * kAStride + i) = make_float2(a0, a1);
              st_u32(sX + X_P + swz_offset(64, r, i), pack_bf16x2(p0, p1));
            }
          }
        }
      }
    }
    __syncthreads();

    // ---------------------------------------------- C: T = (I + A)^-1 Diag(beta)
    {
      const float *sA = reinterpret_cast<const float *>(sX + X_A);
      float *sInv = reinterpret_cast<float *>(sX + X_INV);
      float *sY = reinterpret_cast<float *>(sX + X_Y);
      // C1: inverses of the unit-lower 16x16 diagonal blocks (warp R, lane = column)
      if (warp < 4 && lane < 16) {
        const int R = warp, jc = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float v = (r == jc) ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m) v = fmaf(-sA[(16 * R + r) * kAStride + 16 * R + m], x[m], v);
          x[r] = v;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sInv[(16 * R + r) * kAStride + 16 * R + jc] = x[r];
      }
      __syncthreads();
      // C2: off-diagonal blocks by distance dd = R - I:
      //   Inv_RI = -Inv_RR * sum_{J=I}^{R-1} A_RJ Inv_JI
      const int er = tid >> 4, ej = tid & 15;
#pragma unroll 1
      for (int dd = 1; dd < 4; ++dd) {
        for (int I = 0; I + dd < 4; ++I) {
          const int R = I + dd;
          float y = 0.f;
          for (int J = I; J < R; ++J) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
              y = fmaf(sA[(16 * R + er) * kAStride + 16 * J + m], sInv[(16 * J + m) * kAStride + 16 * I + ej], y);
          }
          sY[I * 256 + er * 16 + ej] = y;
        }
        __syncthreads();
        for (int I = 0; I + dd < 4; ++I) {
          const int R = I + dd;
          float x = 0.f;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            x = fmaf(sInv[(16 * R + er) * kAStride + 16 * R + m], sY[I * 256 + m * 16 + ej], x);
          sInv[(16 * R + er) * kAStride + 16 * I + ej] = -x;
        }
        __syncthreads();
      }
      // C3: T = Inv Diag(beta), lower triangle, bf16 K-major [r][i]
      for (int idx = tid; idx < kC * kC / 2; idx += kThreads) {
        const int r = idx / 32, i = 2 * (idx % 32);
        const float v0 = (i <= r) ? sInv[r * kAStride + i] * s_beta[i] : 0.f;
        const float v1 = (i + 1 <= r) ? sInv[r * kAStride + i + 1] * s_beta[i + 1] : 0.f;
        st_u32(sX + X_T + swz_offset(64, r, i), pack_bf16x2(v0, v1));
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------- D: W^T = K+^T T^T, U^T = V^T T^T, O^T = S^T Q+^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_w = idesc_bf16(128, 64, true, false);
      const uint32_t id_o = idesc_bf16(128, 64, false, false);
      const uint32_t kp = smem_u32(sK), v_ = smem_u32(sV), tt = smem_u32(sX + X_T);
      const uint32_t st = smem_u32(sST), qp = smem_u32(sQ);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_W, desc_mnmajor(kp, 64, s), desc_kmajor(tt, 64, s), id_w, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_U, desc_mnmajor(v_, 64, s), desc_kmajor(tt, 64, s), id_w, s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_bf16(tmem + TM_O, desc_kmajor(st, 128, s), desc_kmajor(qp, 64, s), id_o, s > 0);
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();

    // ---------------------------------------------- E: W^T (TMEM) -> W bf16 [dk][r]; U^T -= S^T W^T
    {
      float v[32];
      tmem_ld16(tmem + lane_base + TM_W + 32 * hh, v);
      tmem_ld16(tmem + lane_base + TM_W + 32 * hh + 16, v + 16);
      store_row32_bf16(sX + X_W, 128, d, 32 * hh, v);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_u = idesc_bf16(128, 64, false, true, /*negate_a=*/true);
      const uint32_t st = smem_u32(sST), w_ = smem_u32(sX + X_W);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_bf16(tmem + TM_U, desc_kmajor(st, 128, s), desc_mnmajor(w_, 128, s), id_u, 1);
      mma_commit(bar_mma);
      // q, k, v of the next chunk may now land (their tiles are no longer read)
      if (chunk + 1 < nchunks) {
        const int nt0 = tok0 + kC;
        mbar_arrive_expect_tx(bar_qkv, 3 * kTileBytes);
        tma_load_3d(sQ, &p.tq, 0, h, nt0, bar_qkv);
        tma_load_3d(sQ + 8192, &p.tq, 64, h, nt0, bar_qkv);
        tma_load_3d(sK, &p.tk, 0, h, nt0, bar_qkv);
        tma_load_3d(sK + 8192, &p.tk, 64, h, nt0, bar_qkv);
        tma_load_3d(sV, &p.tv, 0, h, nt0, bar_qkv);
        tma_load_3d(sV + 8192, &p.tv, 64, h, nt0, bar_qkv);
      }
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();

    // ---------------------------------------------- G: U^T (TMEM) -> bf16 [dv][i]; O^T += U^T P^T; S_acc = U^T K'
    {
      float v[32];
      tmem_ld16(tmem + lane_base + TM_U + 32 * hh, v);
      tmem_ld16(tmem + lane_base + TM_U + 32 * hh + 16, v + 16);
      store_row32_bf16(sX + X_UT, 128, d, 32 * hh, v);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_o = idesc_bf16(128, 64, false, false);
      const uint32_t id_s = idesc_bf16(128, 128, false, true);
      const uint32_t ut = smem_u32(sX + X_UT), pp = smem_u32(sX + X_P), kq = smem_u32(sG);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_O, desc_kmajor(ut, 128, s), desc_kmajor(pp, 64, s), id_o, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_S, desc_kmajor(ut, 128, s), desc_mnmajor(kq, 64, s), id_s, s > 0);
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();
    if (tid == 0 && chunk + 1 < nchunks) {
      const int nt0 = tok0 + kC;
      mbar_arrive_expect_tx(bar_g, kTileBytes);
      tma_load_3d(sG, &p.tg, 0, h, nt0, bar_g);
      tma_load_3d(sG + 8192, &p.tg, 64, h, nt0, bar_g);
    }

    // ---------------------------------------------- I: state update, output
    {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float acc[16];
        tmem_ld16(tmem + lane_base + TM_S + 64 * hh + 16 * j, acc);
#pragma unroll
        for (int i = 0; i < 16; ++i) S[16 * j + i] = fmaf(s_gl[64 * hh + 16 * j + i], S[16 * j + i], acc[i]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) store_row32_bf16(sST, 128, d, 64 * hh + 32 * j, S + 32 * j);
      float o[32];
      tmem_ld16(tmem + lane_base + TM_O + 32 * hh, o);
      tmem_ld16(tmem + lane_base + TM_O + 32 * hh + 16, o + 16);
      uint16_t *dst = a.out + (size_t)tok0 * a.out_stride + h * kD + d;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * hh + i;
        if (r < valid) dst[(size_t)r * a.out_stride] = f32_to_bf16_bits(a.scale * o[i]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*s_abort) break;
  }

  // ---------------------------------------------------------------- final state
  float *dst = nullptr;
  if (a.state_out_pool) dst = a.state_out_pool + ((size_t)slot * a.H + h) * kD * kD;
  else if (a.state_out_dense) dst = a.state_out_dense + ((size_t)n * a.H + h) * kD * kD;
  if (dst) {
#pragma unroll
    for (int i = 0; i < 64; ++i) dst[(size_t)(64 * hh + i) * kD + d] = S[i];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ---------------------------------------------------------------- host side
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

// [tokens, H, 128] bf16 with the given token stride; box = 64 channels x 1 head x 64 tokens
bool make_token_map(CUtensorMap *map, const void *base, int H, int total_tokens, int64_t token_stride) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(std::max(total_tokens, 1))};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD * 2), static_cast<cuuint64_t>(token_stride * 2)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kC)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_prefill(const ChunkArgs &a, const int32_t *cu_seqlens_host, cudaStream_t stream) {
  if (a.num_seqs <= 0) return cudaSuccess;
  static Params *prm_storage = nullptr;  // host-side staging only (kernel params are copied at launch)
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!prm_storage) prm_storage = new Params();
  Params &p = *prm_storage;
  p.a = a;
  if (!make_token_map(&p.tq, a.q, a.H, a.total_tokens, a.qkv_stride) ||
      !make_token_map(&p.tk, a.k, a.H, a.total_tokens, a.qkv_stride) ||
      !make_token_map(&p.tv, a.v, a.H, a.total_tokens, a.qkv_stride) ||
      !make_token_map(&p.tg, a.g, a.H, a.total_tokens, a.g_stride))
    return cudaErrorInvalidValue;
  // longest sequences start first
  p.use_order = a.num_seqs <= kMaxPlannedSeqs ? 1 : 0;
  if (p.use_order) {
    std::vector<int> idx(a.num_seqs);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) {
      return cu_seqlens_host[x + 1] - cu_seqlens_host[x] > cu_seqlens_host[y + 1] - cu_seqlens_host[y];
    });
    for (int i = 0; i < a.num_seqs; ++i) p.order[i] = static_cast<uint16_t>(idx[i]);
  }
  cudaError_t e = cudaFuncSetAttribute(chunk_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  chunk_prefill_kernel<<<a.num_seqs * a.H, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
