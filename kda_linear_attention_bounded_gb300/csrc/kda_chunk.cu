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
//    built from 16-row sub-blocks R.  With m_R = b at row 7 of block R:
//      same block:   e^(b_r - b_i) = e^(b_r - m_R) * e^(m_R - b_i)      (|exponents| <= 8 |lb|)
//      block I < R:  e^(b_r - b_i) = e^(b_r - m_R) * e^(m_R - b_i)      (second factor <= 1)
//    so one M = 128 tcgen05.mma of [F^K; F^Q] (k^, q^ o e^(b - m_R(row)))
//    against G (k^ o e^(m_R(row) - b)) yields every diagonal 16x16 block of A
//    and P, and one more MMA per row block R against k^_i o e^(m_R - b_i)
//    (i < 16R) yields its off-diagonal blocks;
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

constexpr int kC = 64;             // chunk length
constexpr int kThreads = 512;      // 16 warps
constexpr int kTileBytes = 16384;  // one 64 x 128 bf16 tile

// ---- shared memory map (offsets from a 1024-byte aligned base) ----
// WQ: stacked K-major operand [-W (64 rows r); Q+ (64 rows r)] x 128 key channels;
//     the raw q tile is loaded by TMA into the Q+ rows and converted in place.
constexpr uint32_t OFF_WQ = 0;       // 32 KB
constexpr uint32_t OFF_K = 32768;    // k (TMA) -> K+ = k^ o e^b, in place (MN-major operand of W^T)
constexpr uint32_t OFF_V = 49152;    // v (TMA)
constexpr uint32_t OFF_G = 65536;    // g (TMA), read by the gate only
// PK: stacked K-major operand [P (64 rows r); K'^T (128 rows c)] x 64 tokens i, one 128-byte panel
constexpr uint32_t OFF_PK = 81920;   // 24 KB
constexpr int kPKRows = 192;
constexpr uint32_t OFF_X = 106496;   // phase-dependent scratch, 73728 bytes:
//   prologue .. A/P:  [F^K; F^Q] (128 rows) | [G; B_1; B_2; B_3] (64 + 16 + 32 + 48 = 160 rows)
constexpr uint32_t X_FKQ = 0, X_GB = 32768;
constexpr int kGBRows = 160;
__host__ __device__ constexpr int gb_row0(int R) { return R == 0 ? 0 : R == 1 ? 64 : R == 2 ? 80 : 112; }
//   after A/P:  A fp32 [64][68] (later Inv_RR A_RJ) | T bf16 [r][i] | U^T bf16 [dv][i] | (I+A)^-1 fp32 [64][68]
constexpr uint32_t X_A = 0, X_T = 17408, X_UT = 25600, X_INV = 41984;
//   output staging: O bf16 [64][136] over A
constexpr uint32_t X_O = 0;
constexpr int kAStride = 68;   // floats per row of A / (I+A)^-1
constexpr int kOStride = 136;  // bf16 per row of the staged output
constexpr uint32_t OFF_ST = OFF_X + 73728;   // S^T bf16 [dv][dk] (K-major operand), 32 KB
constexpr uint32_t OFF_SMALL = OFF_ST + 32768;
constexpr uint32_t SM_NQ = 0, SM_NK = 256, SM_BETA = 512, SM_H0 = 768, SM_H1 = 2816, SM_GL = 4864,
                   SM_DTB = 5376, SM_BAR = 5888, SM_TMEM = 5928, SM_ABORT = 5932, SM_END = 5952;
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// offset of raw q / Q+ element (r, c) inside WQ
__device__ __forceinline__ uint32_t q_off(int r, int c) { return sm100::swz_offset(128, 64 + r, c); }

// ---- TMEM columns (fp32, lane = row of the M = 128 tile) ----
// W^T | U^T | O^T | S^T; U^T and O^T adjacent (one N = 128 product), O^T and
// S^T adjacent (one N = 192 product).  S^T (lane = value channel, column =
// key channel) lives in TMEM for the whole sequence.
constexpr uint32_t TM_W = 0, TM_U = 64, TM_O = 128, TM_S = 192, TM_COLS = 512;
// A / P products (same columns as W / U / O, which are free at that point)
constexpr uint32_t TM_AP_DIAG = 0;
__host__ __device__ constexpr uint32_t tm_ap_off(int R) { return R == 1 ? 64u : R == 2 ? 80u : 112u; }
static_assert(tm_ap_off(1) == 64 && tm_ap_off(3) + 48 == 160 && 160 <= TM_S, "A/P product columns");

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

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// D (16x8 fp32) += A (16x8 tf32, row) * B (8x8 tf32, col); fragments as in the PTX ISA m16n8k8 layout
__device__ __forceinline__ void mma_1688_tf32(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// Convert 8*n fp32 values to bf16 and store them as n 16-byte chunks of row
// `row` (columns col0 .. col0+8n-1) of a row-swizzled tile of R rows.
template <int N16>
__device__ __forceinline__ void store_row_bf16(uint8_t *tile, int R, int row, int col0, const float *v) {
#pragma unroll
  for (int j = 0; j < N16; ++j) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
    w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
    w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
    w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
    *reinterpret_cast<uint4 *>(tile + swz_offset(R, row, col0 + 8 * j)) = w;
  }
}


// ---- packed fp32x2 arithmetic (sm_100 family): one instruction per channel pair ----
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 exp2_2(float2 x) { return make_float2(fast_exp2(x.x), fast_exp2(x.y)); }
__device__ __forceinline__ uint32_t pack2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Operand pass of the prologue for one thread's 8 rows (block RB known at
// compile time) and one channel pair c0, c0 + 1.  x holds (b_r - m_R) log2(e).
template <int RB>
__device__ __forceinline__ void operand_rows(const float2 (&x)[8], int half, int c0, uint8_t *sWQ, uint8_t *sK,
                                            uint8_t *sX, uint8_t *sPK, const float *s_nq, const float *s_nk,
                                            float2 em, float2 el, float2 eg, const float2 (&cr)[4]) {
  const int rb = 16 * RB + 8 * half;
  uint32_t kq0[4], kq1[4];   // K'^T rows c0, c0 + 1 over this thread's 8 tokens
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = rb + j;
    const float2 e = exp2_2(x[j]);
    const float2 iv = exp2_2(make_float2(-x[j].x, -x[j].y));
    const uint32_t off = swz_offset(64, r, c0);
    const uint32_t qoff = q_off(r, c0);
    const float nq = s_nq[r], nk = s_nk[r];
    const float2 qh = mul2(unpack_bf16x2(ld_u32(sWQ + qoff)), make_float2(nq, nq));
    const float2 kh = mul2(unpack_bf16x2(ld_u32(sK + off)), make_float2(nk, nk));
    const float2 fk = mul2(kh, e), fq = mul2(qh, e), g = mul2(kh, iv);
    st_u32(sX + X_FKQ + swz_offset(128, r, c0), pack2(fk));
    st_u32(sX + X_FKQ + swz_offset(128, 64 + r, c0), pack2(fq));
    st_u32(sX + X_GB + swz_offset(kGBRows, r, c0), pack2(g));
    if (RB < 3) {
      const float2 gp = mul2(g, eg);  // k^ e^(a_R - b)
#pragma unroll
      for (int R2 = RB + 1; R2 < 4; ++R2)
        st_u32(sX + X_GB + swz_offset(kGBRows, gb_row0(R2) + r, c0), pack2(mul2(gp, cr[R2])));
    }
    st_u32(sWQ + qoff, pack2(mul2(fq, em)));  // Q+
    st_u32(sK + off, pack2(mul2(fk, em)));    // K+
    // K' = k^ e^(b_63 - b), collected along tokens for the transposed tile
    const uint32_t kp = pack2(mul2(g, el));
    if (j & 1) {
      kq0[j >> 1] |= kp << 16;
      kq1[j >> 1] |= kp & 0xFFFF0000u;
    } else {
      kq0[j >> 1] = kp & 0xFFFFu;
      kq1[j >> 1] = kp >> 16;
    }
  }
  *reinterpret_cast<uint4 *>(sPK + swz_offset(kPKRows, 64 + c0, rb)) = make_uint4(kq0[0], kq0[1], kq0[2], kq0[3]);
  *reinterpret_cast<uint4 *>(sPK + swz_offset(kPKRows, 65 + c0, rb)) = make_uint4(kq1[0], kq1[1], kq1[2], kq1[3]);
}

__global__ void __launch_bounds__(kThreads, 1) chunk_prefill_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sWQ = smem + OFF_WQ, *sK = smem + OFF_K, *sV = smem + OFF_V, *sG = smem + OFF_G;
  uint8_t *sPK = smem + OFF_PK, *sX = smem + OFF_X, *sST = smem + OFF_ST;
  uint8_t *small = smem + OFF_SMALL;
  float *s_nq = reinterpret_cast<float *>(small + SM_NQ);
  float *s_nk = reinterpret_cast<float *>(small + SM_NK);
  float *s_beta = reinterpret_cast<float *>(small + SM_BETA);
  float *s_h0 = reinterpret_cast<float *>(small + SM_H0);      // [4][128] sum of lambda over rows 0..7 of a block
  float *s_h1 = reinterpret_cast<float *>(small + SM_H1);      // [4][128] sum of lambda over rows 8..15
  float *s_gl = reinterpret_cast<float *>(small + SM_GL);      // [128] e^(b_63)
  float *s_dtb = reinterpret_cast<float *>(small + SM_DTB);    // [128]
  uint64_t *bar_q = reinterpret_cast<uint64_t *>(small + SM_BAR);
  uint64_t *bar_kv = bar_q + 1;
  uint64_t *bar_g = bar_q + 2;
  uint64_t *bar_mma = bar_q + 3;
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

  auto load_q = [&](int tok) {
    mbar_arrive_expect_tx(bar_q, kTileBytes);
    tma_load_3d(sWQ + 8192, &p.tq, 0, h, tok, bar_q);    // channels 0..63  -> rows 64..127 of panel 0
    tma_load_3d(sWQ + 24576, &p.tq, 64, h, tok, bar_q);  // channels 64..127 -> rows 64..127 of panel 1
  };
  auto load_kv = [&](int tok) {
    mbar_arrive_expect_tx(bar_kv, 2 * kTileBytes);
    tma_load_3d(sK, &p.tk, 0, h, tok, bar_kv);
    tma_load_3d(sK + 8192, &p.tk, 64, h, tok, bar_kv);
    tma_load_3d(sV, &p.tv, 0, h, tok, bar_kv);
    tma_load_3d(sV + 8192, &p.tv, 64, h, tok, bar_kv);
  };
  auto load_g = [&](int tok) {
    mbar_arrive_expect_tx(bar_g, kTileBytes);
    tma_load_3d(sG, &p.tg, 0, h, tok, bar_g);
    tma_load_3d(sG + 8192, &p.tg, 64, h, tok, bar_g);
  };

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_kv, 1);
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
    load_q(t0);
    load_kv(t0);
    load_g(t0);
  }
  // raw beta logits, fetched one chunk ahead (the sigmoid is applied when they are used)
  uint16_t beta_raw = (tid < kC && tid < len) ? a.beta[(size_t)(t0 + tid) * a.beta_stride + h] : uint16_t(0);

  // TMEM tiles are read / written by warp w on lanes 32*(w%4) .. +31 and a
  // quarter (w/4) of the columns.  For S^T: lane = value channel d.
  const int quad = warp & 3, qc = warp >> 2;
  const int d = quad * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  {
    float s0[32];
    if (a.state_in) {
      const float *src = a.state_in + ((size_t)slot * a.H + h) * kD * kD + d;
#pragma unroll
      for (int i = 0; i < 32; ++i) s0[i] = src[(size_t)(32 * qc + i) * kD];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) s0[i] = 0.f;
    }
    tmem_st16(tmem + lane_base + TM_S + 32 * qc, s0);
    tmem_st16(tmem + lane_base + TM_S + 32 * qc + 16, s0 + 16);
    store_row_bf16<4>(sST, 128, d, 32 * qc, s0);
    tmem_wait_st();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const float nea = -__expf(a.A_log[h]) * kLog2e;  // gate slope, log2 units
  const float lb2 = a.lower_bound * kLog2e;        // lower bound, log2 units
  uint32_t mma_phase = 0;

  for (int chunk = 0; chunk < nchunks; ++chunk) {
    const int tok0 = t0 + chunk * kC;
    const int valid = min(kC, len - chunk * kC);
    const uint32_t tma_parity = chunk & 1;
    const bool has_next = chunk + 1 < nchunks;
    // -- wait for inputs
    wait_or_flag(bar_q, tma_parity, s_abort, a.status);
    wait_or_flag(bar_kv, tma_parity, s_abort, a.status);

    // ---------------------------------------------- A: norms, beta, padding, gate, decay, operands
    // (decays are kept in log2 units: b2 = b * log2(e), so every factor is one ex2)
    {
      const int task = tid >> 2, part = tid & 3;   // norms: 128 (row, q|k) tasks x 4 threads of 32 channels
      const int r = task & 63;
      float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 32 * part + 8 * j;
        const uint8_t *src = task < 64 ? sWQ + q_off(r, c) : sK + swz_offset(64, r, c);
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(ws[e]);
          ss2 = fma2(f, f, ss2);
        }
      }
      float ss = ss2.x + ss2.y;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      if (part == 0) {
        const float nrm = r < valid ? rsqrtf(ss + kL2Eps) : 0.f;
        (task < 64 ? s_nq : s_nk)[r] = nrm;
      }
      if (tid < kC) {
        s_beta[tid] = tid < valid ? sigmoid_f(bf16_bits_to_f32(beta_raw)) : 0.f;
        const int nt = (chunk + 1) * kC + tid;   // next chunk's logit: a whole chunk to arrive
        beta_raw = nt < len ? a.beta[(size_t)(t0 + nt) * a.beta_stride + h] : uint16_t(0);
      }
      if (valid < kC) {  // rows past the sequence end: zero v (the others are masked through beta, norms, lambda)
        for (int idx = tid; idx < (kC - valid) * 16; idx += kThreads) {
          const int r2 = valid + idx / 16, cc = idx % 16;
          *reinterpret_cast<uint4 *>(sV + swz_offset(64, r2, 8 * cc)) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    wait_or_flag(bar_g, tma_parity, s_abort, a.status);
    {
      // thread = (channel pair, 16-row block R, half of the block): 8 rows x 2 channels
      const int cp = tid & 63, R = (tid >> 6) & 3, half = tid >> 8;
      const int c0 = 2 * cp;
      const int rb = 16 * R + 8 * half;   // first row of this thread
      // sigmoid(ea (g + dtb)) = 1 / (1 + 2^(nea g + nea dtb)),  nea = -ea log2(e)
      const float nd0 = nea * s_dtb[c0], nd1 = nea * s_dtb[c0 + 1];
      float b0[8], b1[8];   // cumulative log2-decay from the start of this half-block
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = rb + j;
        const float2 gg = unpack_bf16x2(ld_u32(sG + swz_offset(64, r, c0)));
        const bool ok = r < valid;
        const float l0 = ok ? lb2 * fast_rcp(1.f + fast_exp2(fmaf(nea, gg.x, nd0))) : 0.f;
        const float l1 = ok ? lb2 * fast_rcp(1.f + fast_exp2(fmaf(nea, gg.y, nd1))) : 0.f;
        acc0 += l0;
        acc1 += l1;
        b0[j] = acc0;
        b1[j] = acc1;
      }
      *reinterpret_cast<float2 *>((half ? s_h1 : s_h0) + R * kD + c0) = make_float2(acc0, acc1);
      // -- gate done
      __syncthreads();
      // raw g is no longer read: the next chunk's g may land
      if (tid == 0 && has_next) load_g(tok0 + kC);
      // absolute anchors of every block: m_I = b at row 7, a_I = b at row 15
      float mm[4][2], tot0 = 0.f, tot1 = 0.f, ar0 = 0.f, ar1 = 0.f, m0 = 0.f, m1 = 0.f;
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        const float2 x0 = *reinterpret_cast<const float2 *>(s_h0 + I * kD + c0);
        const float2 x1 = *reinterpret_cast<const float2 *>(s_h1 + I * kD + c0);
        mm[I][0] = tot0 + x0.x;
        mm[I][1] = tot1 + x0.y;
        tot0 += x0.x + x1.x;
        tot1 += x0.y + x1.y;
        if (I == R) {
          m0 = mm[I][0]; m1 = mm[I][1];
          ar0 = tot0; ar1 = tot1;
        }
      }
      const float2 t1 = *reinterpret_cast<const float2 *>(s_h1 + R * kD + c0);  // b_15 - b_7 of this block
      if (R == 0 && half == 0)
        *reinterpret_cast<float2 *>(s_gl + c0) = make_float2(fast_exp2(tot0), fast_exp2(tot1));
      const float em0 = fast_exp2(m0), em1 = fast_exp2(m1);              // e^(m_R)
      const float el0 = fast_exp2(tot0 - m0), el1 = fast_exp2(tot1 - m1);  // e^(b_63 - m_R)
      const float eg0 = fast_exp2(t1.x), eg1 = fast_exp2(t1.y);            // e^(a_R - m_R)
      // rows of this block feed the off-diagonal B tiles of every later block R2:
      //   B_R2[i] = k^_i e^(m_R2 - b_i) = (k^_i e^(a_R - b_i)) * e^(m_R2 - a_R), both factors <= 1
      float cr[4][2];
      cr[0][0] = cr[0][1] = 0.f;
#pragma unroll
      for (int R2 = 1; R2 < 4; ++R2) {
        cr[R2][0] = fast_exp2(fminf(mm[R2][0] - ar0, 0.f));
        cr[R2][1] = fast_exp2(fminf(mm[R2][1] - ar1, 0.f));
      }
      // b_r - m_R from the thread's own partial sums: half 0 ends at row 7, half 1 starts after it
      const float base0 = half ? 0.f : b0[7], base1 = half ? 0.f : b1[7];
      float2 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = make_float2(b0[j] - base0, b1[j] - base1);
      const float2 em = make_float2(em0, em1), el = make_float2(el0, el1), eg = make_float2(eg0, eg1);
      float2 crp[4];
#pragma unroll
      for (int R2 = 0; R2 < 4; ++R2) crp[R2] = make_float2(cr[R2][0], cr[R2][1]);
      switch (R) {   // warp-uniform
        case 0: operand_rows<0>(x, half, c0, sWQ, sK, sX, sPK, s_nq, s_nk, em, el, eg, crp); break;
        case 1: operand_rows<1>(x, half, c0, sWQ, sK, sX, sPK, s_nq, s_nk, em, el, eg, crp); break;
        case 2: operand_rows<2>(x, half, c0, sWQ, sK, sX, sPK, s_nq, s_nk, em, el, eg, crp); break;
        default: operand_rows<3>(x, half, c0, sWQ, sK, sX, sPK, s_nq, s_nk, em, el, eg, crp); break;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------- B: A and P from 16x16 sub-blocks (tcgen05)
    if (tid == 0) {
      tc_fence_after();
      // one 128 x 160 product: columns 0..63 diagonal blocks, then B_1, B_2, B_3
      const uint32_t fkq = smem_u32(sX + X_FKQ);
      const uint32_t gb = smem_u32(sX + X_GB);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_bf16(tmem + TM_AP_DIAG, desc_kmajor(fkq, 128, s), desc_kmajor(gb, kGBRows, s),
                 idesc_bf16(128, kGBRows, false, false), s > 0);
      mma_commit(bar_mma);
    }
    // while the A/P product runs (columns 0..159): S^T <- S^T Diag(e^(b_63)) in TMEM (columns 192..319)
    {
      uint32_t sv[32];
      tmem_ld16_async(tmem + lane_base + TM_S + 32 * qc, sv);
      tmem_ld16_async(tmem + lane_base + TM_S + 32 * qc + 16, sv + 16);
      tmem_wait_ld();
      tmem_tie<32>(sv);
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 g4 = *reinterpret_cast<const float4 *>(s_gl + 32 * qc + i);
        f[i] = __uint_as_float(sv[i]) * g4.x;
        f[i + 1] = __uint_as_float(sv[i + 1]) * g4.y;
        f[i + 2] = __uint_as_float(sv[i + 2]) * g4.z;
        f[i + 3] = __uint_as_float(sv[i + 3]) * g4.w;
      }
      tmem_st16(tmem + lane_base + TM_S + 32 * qc, f);
      tmem_st16(tmem + lane_base + TM_S + 32 * qc + 16, f + 16);
      tmem_wait_st();
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();
    // -- A/P products done
    {
      // lanes 0..63 of the products hold A rows (k), lanes 64..127 P rows (q);
      // warp = (lane quadrant, column block I)
      const bool is_p = quad >= 2;
      const int r = (quad & 1) * 32 + lane;     // row of A / P
      const int Rr = r >> 4;                     // its 16-row block
      const int Ra = (quad & 1) * 2;             // first of the two row blocks of this warp
      const int I = qc;
      float *sA = reinterpret_cast<float *>(sX + X_A);
      const float bscale = is_p ? 1.f : s_beta[r];
      uint32_t va[16], vb[16];
      const int srcA = (I == Ra) ? int(TM_AP_DIAG) + 16 * I : (I < Ra) ? int(tm_ap_off(Ra)) + 16 * I : -1;
      const int srcB = (I == Ra + 1) ? int(TM_AP_DIAG) + 16 * I : (I < Ra + 1) ? int(tm_ap_off(Ra + 1)) + 16 * I : -1;
      if (srcA >= 0) tmem_ld16_async(tmem + lane_base + srcA, va);
      if (srcB >= 0) tmem_ld16_async(tmem + lane_base + srcB, vb);
      tmem_wait_ld();
      tmem_tie<16>(va);
      tmem_tie<16>(vb);
      const bool mine_a = (Rr == Ra);
      const int src = mine_a ? srcA : srcB;
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int i = 16 * I + e;
        const float raw = __uint_as_float(mine_a ? va[e] : vb[e]);
        const bool keep = (src >= 0) && (is_p ? (i <= r) : (i < r));
        v[e] = keep ? raw * bscale : 0.f;
      }
      if (is_p) {
        store_row_bf16<2>(sPK, kPKRows, r, 16 * I, v);
      } else {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4 *>(sA + r * kAStride + 16 * I + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------- C: T = (I + A)^-1 Diag(beta)
    {
      const float *sA = reinterpret_cast<const float *>(sX + X_A);
      float *sInv = reinterpret_cast<float *>(sX + X_INV);
      // C1: inverses of the unit-lower 16x16 diagonal blocks (warp R, lane = column); their part
      // of T = Inv Diag(beta) goes straight to the bf16 T tile.  Warps 4..15 clear the upper blocks of T.
      uint16_t *sT16 = reinterpret_cast<uint16_t *>(sX + X_T);
      if (warp < 4) {
        if (lane < 16) {
          const int R = warp, jc = lane;
          const float bj = s_beta[16 * R + jc];
          float x[16];
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            float lrow[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float4 l4 = *reinterpret_cast<const float4 *>(sA + (16 * R + r) * kAStride + 16 * R + 4 * q4);
              lrow[4 * q4] = l4.x; lrow[4 * q4 + 1] = l4.y; lrow[4 * q4 + 2] = l4.z; lrow[4 * q4 + 3] = l4.w;
            }
            float v0 = (r == jc) ? 1.f : 0.f, v1 = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) {
              if (m & 1) v1 = fmaf(-lrow[m], x[m], v1);
              else v0 = fmaf(-lrow[m], x[m], v0);
            }
            x[r] = v0 + v1;
          }
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            sInv[(16 * R + r) * kAStride + 16 * R + jc] = x[r];
            sT16[swz_offset(64, 16 * R + r, 16 * R + jc) >> 1] = f32_to_bf16_bits(r >= jc ? x[r] * bj : 0.f);
          }
        }
      } else {
        // strictly-upper 16x16 blocks (R, I > R): 6 blocks x 16 rows x 2 chunks of 8 columns
        for (int idx = tid - 128; idx < 6 * 32; idx += kThreads - 128) {
          const int blk = idx >> 5, e = idx & 31;
          const int R = blk < 3 ? 0 : blk < 5 ? 1 : 2;
          const int I = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
          *reinterpret_cast<uint4 *>(sX + X_T + swz_offset(64, 16 * R + (e >> 1), 16 * I + 8 * (e & 1))) =
              make_uint4(0, 0, 0, 0);
        }
      }
      __syncthreads();
      // -- diagonal inverses done
      // C2: off-diagonal blocks.  With L~_RJ = Inv_RR A_RJ (J < R, computed in place over A):
      //   Inv_RI = - sum_{J=I}^{R-1} L~_RJ Inv_JI.
      // Each warp owns an 8-column half of one column block I and walks down it, reading only
      // its own earlier results, so the steps need no CTA-wide barrier.  TF32 m16n8k8 tensor-core MMAs.
      {
        float *sAw = reinterpret_cast<float *>(sX + X_A);
        const int g = lane >> 2, t = lane & 3;
        // pre-multiply: 6 block pairs x 2 column halves = 12 warps, all independent
        if (warp < 12) {
          const int pr = warp >> 1;                       // (R, J): (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
          const int R = pr < 1 ? 1 : pr < 3 ? 2 : 3;
          const int J = pr - (R * (R - 1)) / 2;
          const int n0 = 16 * J + 8 * (warp & 1);
          float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const float *ar = sInv + (16 * R + g) * kAStride + 16 * R + 8 * ks + t;
            const float *br = sAw + (16 * R + 8 * ks + t) * kAStride + n0 + g;
            mma_1688_tf32(y, to_tf32(ar[0]), to_tf32(ar[8 * kAStride]), to_tf32(ar[4]),
                          to_tf32(ar[8 * kAStride + 4]), to_tf32(br[0]), to_tf32(br[4 * kAStride]));
          }
          *reinterpret_cast<float2 *>(sAw + (16 * R + g) * kAStride + n0 + 2 * t) = make_float2(y[0], y[1]);
          *reinterpret_cast<float2 *>(sAw + (16 * R + g + 8) * kAStride + n0 + 2 * t) = make_float2(y[2], y[3]);
        }
        __syncthreads();
        // column walks: warp = (column block I in 0..2, half); I = 0 takes 3 steps, I = 2 one
        if (warp < 6) {
          const int I = warp >> 1;
          const int n0 = 16 * I + 8 * (warp & 1);
          const float2 bcol = *reinterpret_cast<const float2 *>(s_beta + n0 + 2 * t);
          for (int R = I + 1; R < 4; ++R) {
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            for (int J = I; J < R; ++J) {
#pragma unroll
              for (int ks = 0; ks < 2; ++ks) {
                const int kc = 16 * J + 8 * ks;
                const float *ar = sAw + (16 * R + g) * kAStride + kc + t;
                const float *br = sInv + (kc + t) * kAStride + n0 + g;
                mma_1688_tf32(x, to_tf32(ar[0]), to_tf32(ar[8 * kAStride]), to_tf32(ar[4]),
                              to_tf32(ar[8 * kAStride + 4]), to_tf32(br[0]), to_tf32(br[4 * kAStride]));
              }
            }
            *reinterpret_cast<float2 *>(sInv + (16 * R + g) * kAStride + n0 + 2 * t) = make_float2(-x[0], -x[1]);
            *reinterpret_cast<float2 *>(sInv + (16 * R + g + 8) * kAStride + n0 + 2 * t) = make_float2(-x[2], -x[3]);
            st_u32(sX + X_T + swz_offset(64, 16 * R + g, n0 + 2 * t), pack_bf16x2(-x[0] * bcol.x, -x[1] * bcol.y));
            st_u32(sX + X_T + swz_offset(64, 16 * R + g + 8, n0 + 2 * t), pack_bf16x2(-x[2] * bcol.x, -x[3] * bcol.y));
            __syncwarp();
          }
        }
      }
      // -- T done
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------- D: W^T = K+^T T^T, U^T = V^T T^T; clear O^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_w = idesc_bf16(128, 64, true, false);
      const uint32_t kp = smem_u32(sK), v_ = smem_u32(sV), tt = smem_u32(sX + X_T);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_W, desc_mnmajor(kp, 64, s), desc_kmajor(tt, 64, s), id_w, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_U, desc_mnmajor(v_, 64, s), desc_kmajor(tt, 64, s), id_w, s > 0);
      mma_commit(bar_mma);
    }
    // while the MMAs run: O^T <- 0 (its columns were A/P products until now), next beta
    {
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.f;
      tmem_st16(tmem + lane_base + TM_O + 16 * qc, z);
      tmem_wait_st();
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();
    // k, v of the next chunk may now land (K+ and V are no longer read)
    if (tid == 0 && has_next) load_kv(tok0 + kC);

    // ---------------------------------------------- E: -W into WQ; [U^T | O^T] += S^T [-W; Q+]^T
    {
      uint32_t v[16];
      tmem_ld16_async(tmem + lane_base + TM_W + 16 * qc, v);
      tmem_wait_ld();
      tmem_tie<16>(v);
      // W^T lane = key channel c; W row r = 16*qc + i, column c
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<uint16_t *>(sWQ + swz_offset(128, 16 * qc + i, d)) = f32_to_bf16_bits(-__uint_as_float(v[i]));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_uo = idesc_bf16(128, 128, false, false);
      const uint32_t st = smem_u32(sST), wq = smem_u32(sWQ);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma_bf16(tmem + TM_U, desc_kmajor(st, 128, s), desc_kmajor(wq, 128, s), id_uo, 1);
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();
    // q of the next chunk may now land (Q+ and W are no longer read)
    if (tid == 0 && has_next) load_q(tok0 + kC);

    // ---------------------------------------------- G: U^T -> bf16 [dv][i]; [O^T | S^T] += U^T [P; K'^T]^T
    {
      uint32_t v[16];
      tmem_ld16_async(tmem + lane_base + TM_U + 16 * qc, v);
      tmem_wait_ld();
      tmem_tie<16>(v);
      store_row_bf16<2>(sX + X_UT, 128, d, 16 * qc, reinterpret_cast<const float *>(v));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_os = idesc_bf16(128, kPKRows, false, false);
      const uint32_t ut = smem_u32(sX + X_UT), pk = smem_u32(sPK);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_O, desc_kmajor(ut, 128, s), desc_kmajor(pk, kPKRows, s), id_os, 1);
      mma_commit(bar_mma);
    }
    __syncwarp();
    wait_or_flag(bar_mma, mma_phase & 1, s_abort, a.status);
    ++mma_phase;
    tc_fence_after();

    // ---------------------------------------------- I: S^T -> bf16 operand, output
    {
      uint32_t sv[32];
      tmem_ld16_async(tmem + lane_base + TM_S + 32 * qc, sv);
      tmem_ld16_async(tmem + lane_base + TM_S + 32 * qc + 16, sv + 16);
      uint32_t o[16];
      tmem_ld16_async(tmem + lane_base + TM_O + 16 * qc, o);
      tmem_wait_ld();
      tmem_tie<32>(sv);
      tmem_tie<16>(o);
      store_row_bf16<4>(sST, 128, d, 32 * qc, reinterpret_cast<const float *>(sv));
      uint16_t *sO = reinterpret_cast<uint16_t *>(sX + X_O);
#pragma unroll
      for (int i = 0; i < 16; ++i) sO[(16 * qc + i) * kOStride + d] = f32_to_bf16_bits(a.scale * __uint_as_float(o[i]));
    }
    __syncthreads();
    {
      const uint16_t *sO = reinterpret_cast<const uint16_t *>(sX + X_O);
      for (int idx = tid; idx < valid * 16; idx += kThreads) {
        const int r = idx >> 4, cc = idx & 15;
        *reinterpret_cast<uint4 *>(a.out + (size_t)(tok0 + r) * a.out_stride + h * kD + 8 * cc) =
            *reinterpret_cast<const uint4 *>(sO + r * kOStride + 8 * cc);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // -- chunk done
    if (*s_abort) break;
  }

  // ---------------------------------------------------------------- final state
  float *dst = nullptr;
  if (a.state_out_pool) dst = a.state_out_pool + ((size_t)slot * a.H + h) * kD * kD;
  else if (a.state_out_dense) dst = a.state_out_dense + ((size_t)n * a.H + h) * kD * kD;
  if (dst) {
    uint32_t sv[32];
    tmem_ld16_async(tmem + lane_base + TM_S + 32 * qc, sv);
    tmem_ld16_async(tmem + lane_base + TM_S + 32 * qc + 16, sv + 16);
    tmem_wait_ld();
    tmem_tie<32>(sv);
#pragma unroll
    for (int i = 0; i < 32; ++i) dst[(size_t)(32 * qc + i) * kD + d] = __uint_as_float(sv[i]);
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
