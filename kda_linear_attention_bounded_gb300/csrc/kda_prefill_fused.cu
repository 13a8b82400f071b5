// Fused chunked prefill of the KDA bounded-gate recurrence on sm_103a.
//
// One CTA per (sequence, head) walks the sequence's chunks of C = 64 tokens.
// Its warps are split in two groups that work one chunk apart:
//
//  * producer warps 0..7 build the state-independent half of chunk n's algebra
//    (the bounded gate of vLLM PR #55737 "Use FlashKDA for KDA chunked prefill",
//    PR summary, with in-kernel q/k l2norm and sigmoid beta):
//      A[r,i] = beta_r sum_c k^_rc k^_ic e^(b_rc - b_ic)  (i < r)
//      P[r,i] = scale  sum_c q^_rc k^_ic e^(b_rc - b_ic)  (i <= r)
//      T = (I + A)^-1 Diag(beta),  W = T (k^ o e^b),  U^ = T V,
//      Q+ = scale q^ o e^b,  K' = k^ o e^(b_63 - b),  gamma = e^(b_63)
//    into one on-chip buffer laid out as the block image of kda_prefill_block.h;
//  * chain warps 8..15 apply chunk n - 1's buffer to the state S (128 key x
//    128 value channels, fp32, resident in TMEM):
//      U = U^ - W S,  O = Q+ S + P U,  S' = Diag(gamma) S + K'^T U.
//
// This is the token recurrence S_t = (I - beta k^ k^T) Diag(alpha) S_{t-1} +
// beta k^ v^T, o_t = scale S_t^T q^, unrolled over a chunk.  Nothing of a
// chunk but its output rows (and the final state) leaves the SM: per token and
// head the call moves q, k, v, g, beta and the output through HBM once.
//
// The producer follows the two-kernel path's intra-chunk kernel
// (kda_chunk_intra.cu) with 32-row anchored sub-blocks (lower_bound >= -5),
// reorganised so that less of it sits on the per-chunk critical path:
//  * the l2 norms are folded into scalings: the operand tiles hold the raw k, q
//    (times their decay factors), A and P take their row / column norms when
//    they are read out of TMEM, T is stored twice (T_U = Diag(n_k) T and
//    T_W = Diag(n_k) T Diag(n_k)), so that the chain's U' = Diag(n_k) U meets the
//    raw K' and P, and the output rows take n_q when they are read out; the norms
//    themselves are computed while the A/P product runs;
//  * W comes from the F tile (k e^(b - m_R)) in two K = 32 products, one per
//    32-row block, combined with the per-channel factors e^(m_R) when W^T is read
//    out, so there is no separate k e^b tile;
//  * U^' = T_U V is accumulated straight into the TMEM columns where the chain's
//    first product then adds -W'S (the chain keeps -S as its bf16 operand and the
//    producer stores -Q+), so U' arrives in TMEM in fp32 without a staging pass;
// The chain follows the state pass (kda_chunk_chain.cu): [U^T | O^T] =
// (-S)^T [W | -Q+]^T with the bf16 copy of -S as a TMEM A operand, the U^T
// epilogue (fp32 -> bf16 in place), S^T += U^T K' and O^T += U^T P^T, and the
// decay of the state by the next chunk's gamma.
//
// Synchronisation (mbarriers, one phase per chunk):
//   in / v / pmma / pw / pu   producer-internal (TMA landings, producer MMAs)
//   gamma                     producer -> chain: gamma of chunk n is in s_gamma[n & 1]
//   ready                     producer -> chain: chunk n's buffer is complete
//   m1u / m2s                 chain-internal (the U half of the first product, the state product)
//   free                      chain -> producer and chain: chunk n's output product is done, so its
//                             buffer may be overwritten and its output read out
// The producer is at most one chunk ahead, so no barrier is ever waited on two phases behind.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_block.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = kChunk;
constexpr int kThreads = 512;
constexpr int kProdThreads = 256;   // warps 0..7
constexpr int kChainThreads = 256;  // warps 8..15
constexpr int kChainIssuer = 256;   // first chain thread: issues the chain's MMAs and output stores
constexpr int kBarProd = 7, kBarChain = 8;   // hardware barriers of the two groups (1..6: the inverse's warp pairs)

// ---- shared memory (offsets from a 1024-byte aligned base) ----
constexpr uint32_t OFF_BUF = 0;                    // one chunk's operands for the chain, in the block layout
constexpr uint32_t OFF_TW = OFF_BUF + kBlkUH;      // (its U^ tile is unused here) T_W bf16 K-major [t][t'] (8 KB)
constexpr uint32_t OFF_TU = OFF_TW + 8192;         //                             T_U bf16 K-major (8 KB)
constexpr uint32_t OFF_QIN = 75776;                // q, k, g tiles (TMA, unswizzled), 16 KB each
constexpr uint32_t OFF_KIN = OFF_QIN + 16384;
constexpr uint32_t OFF_GIN = OFF_QIN + 32768;
constexpr uint32_t OFF_OPS = OFF_QIN + 49152;      // producer operand region (64 KB)
constexpr uint32_t OFF_FQ = OFF_OPS;               // [F | Q]: 128 rows rho x (64 + 64) tokens; F stays for W
constexpr uint32_t OFF_GB = OFF_OPS + 32768;       // [G | B_1]: 128 rows rho x 96 tokens in two panels
// after the A/P product
constexpr uint32_t OFF_A = OFF_OPS + 16384;        // A fp32 [64][68], inverted in place (over Q and G)
constexpr uint32_t OFF_V = OFF_OPS + 33792;        // v tile (TMA, 128-byte swizzle)
constexpr uint32_t OFF_STAGE = OFF_OPS + 65536;    // output tile staging for the TMA store (16 KB)
constexpr uint32_t OFF_SMALL = OFF_STAGE + 16384;
constexpr uint32_t SM_NQ = 0 /* [3][64] */, SM_NK = 768, SM_BETA = 1024 /* [2][64] */, SM_H = 1536 /* [8][128] */,
                   SM_GAMMA = 5632 /* [2][128] */, SM_EM = 6656 /* [2 blocks][128] */, SM_BAR = 7680,
                   SM_TMEM = 7808, SM_ABORT = 7812, SM_END = 7824;
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(OFF_QIN >= kBlkBytes && OFF_QIN % 1024 == 0 && OFF_V % 1024 == 0 && OFF_TW % 1024 == 0 &&
              OFF_STAGE % 1024 == 0 && OFF_TU + 8192 <= OFF_BUF + kBlkPK, "layout");
static_assert(OFF_A + 64 * 68 * 4 <= OFF_V && OFF_V + 16384 <= OFF_OPS + 65536, "operand region");
constexpr int kAStride = 68;

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;      // S^T fp32 (lane = value channel, column = key channel rho)
constexpr uint32_t TM_XU = 128;   // U^'^T from the producer, then U'^T after the first product; bf16 pairs in place
constexpr uint32_t TM_O0 = 192;   // O^T, two buffers (chunk parity)
constexpr uint32_t TM_SA = 320;   // -S^T bf16 (A operand of the first product)
constexpr uint32_t TM_P = 384;    // producer: A/P product (96 columns), then W's two block products (64 + 64)
constexpr uint32_t kTmemCols = 512;

// barrier indices in the SM_BAR array
enum { B_IN = 0, B_V, B_PMMA, B_PW, B_PU, B_GAMMA, B_READY, B_M1U, B_M2S, B_FREE, kNumBars };

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
// the q, k, g tiles are unswizzled: two 64-channel boxes of 64 rows x 128 bytes
__device__ __forceinline__ uint32_t in_offset(int r, int c) {
  return static_cast<uint32_t>((c >> 6) * 8192 + r * 128 + (c & 63) * 2);
}

__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              uint32_t *status) {
  if (*abort_flag) return;
  if (!mbar_wait(bar, parity)) {
    *abort_flag = 1;
    atomicOr(status, KDA_DEVICE_TIMEOUT);
  }
}

// barrier of `count` threads on hardware barrier kId that also returns whether any of them passed `pred`
template <int kId>
__device__ __forceinline__ bool bar_any(int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kId), "r"(count)
      : "memory");
  return r != 0;
}

// 8 consecutive tokens of the thread's two key channels -> two 16-byte chunks (rows rho, 64 + rho)
__device__ __forceinline__ void pack8(const float2 (&v)[8], uint4 &lo, uint4 &hi) {
  lo = make_uint4(pack_bf16x2(v[0].x, v[1].x), pack_bf16x2(v[2].x, v[3].x), pack_bf16x2(v[4].x, v[5].x),
                  pack_bf16x2(v[6].x, v[7].x));
  hi = make_uint4(pack_bf16x2(v[0].y, v[1].y), pack_bf16x2(v[2].y, v[3].y), pack_bf16x2(v[4].y, v[5].y),
                  pack_bf16x2(v[6].y, v[7].y));
}
// 16 x 8 tile of X Y (TF32 tensor cores, fp32 accumulate), as in the intra-chunk kernel
__device__ __forceinline__ void mm_16x8(float (&d)[4], const float *X, const float *Y, int ks, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k >= ks) break;
    const float *xa = X + g * kAStride + 8 * k + t;
    const float *yb = Y + (8 * k + t) * kAStride + g;
    mma_1688_tf32(d, to_tf32(xa[0]), to_tf32(xa[8 * kAStride]), to_tf32(xa[4]), to_tf32(xa[8 * kAStride + 4]),
                  to_tf32(yb[0]), to_tf32(yb[4 * kAStride]));
  }
}
__device__ __forceinline__ void st_16x8(float *D, const float (&d)[4], float sgn, int lane) {
  const int g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2 *>(D + g * kAStride + 2 * t) = make_float2(sgn * d[0], sgn * d[1]);
  *reinterpret_cast<float2 *>(D + (g + 8) * kAStride + 2 * t) = make_float2(sgn * d[2], sgn * d[3]);
}
// the same 16 x 8 tile of L^-1 (times sgn) as bf16 pairs into T_U (rows x n_k, columns x beta) and T_W (also
// columns x n_k); K-major, 128-byte swizzle
__device__ __forceinline__ void st_16x8_t(uint8_t *tU, uint8_t *tW, int row0, int col0, const float (&d)[4], float sgn,
                                          const float *s_beta, const float *s_nk, int lane) {
  const int g = lane >> 2, c = col0 + 2 * (lane & 3);
  const float r0 = sgn * s_nk[row0 + g], r1 = sgn * s_nk[row0 + g + 8];
  const float b0 = s_beta[c], b1 = s_beta[c + 1], n0 = s_nk[c], n1 = s_nk[c + 1];
  const float u00 = d[0] * r0 * b0, u01 = d[1] * r0 * b1, u10 = d[2] * r1 * b0, u11 = d[3] * r1 * b1;
  *reinterpret_cast<uint32_t *>(tU + swz_offset(64, row0 + g, c)) = pack_bf16x2(u00, u01);
  *reinterpret_cast<uint32_t *>(tU + swz_offset(64, row0 + g + 8, c)) = pack_bf16x2(u10, u11);
  *reinterpret_cast<uint32_t *>(tW + swz_offset(64, row0 + g, c)) = pack_bf16x2(u00 * n0, u01 * n1);
  *reinterpret_cast<uint32_t *>(tW + swz_offset(64, row0 + g + 8, c)) = pack_bf16x2(u10 * n0, u11 * n1);
}

struct Factors {
  float2 nems;  // -scale e^(m_R)
  float2 el;    // e^(b_63 - m_R)
  float2 eg;    // e^(a_R - m_R), a_R = b at the last row of block R
  float2 cr;    // e^(m_1 - a_0) (block 0 only), applied after eg: k e^(a_0 - b) <= |k| stays representable
};

// Operand rows of 8 tokens (rows t0 .. t0+7 of 32-row block R) for key channels (2p, 2p+1); x[j] = (b - m_R)
// log2(e) of those rows; k and q are the raw inputs (their norms are applied later as scalings).  F, Q, G and B_1
// go to the operand tiles, -Q+ and K' to the chunk's buffer.
template <int R>
__device__ __forceinline__ void build_rows(uint8_t *sm, const float2 (&x)[8], int t0, int p, const Factors &f) {
  const int c0 = 2 * p;
  // every tile row of this thread starts at the same swizzled offset within its 128-row panel
  const uint32_t o = swz_offset(128, p, t0);
  float2 e[8], v[8], w[8];
  uint32_t kw[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    kw[j] = ld_u32(sm + OFF_KIN + in_offset(t0 + j, c0));
    e[j] = exp2_2(x[j]);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = mul2(unpack_bf16x2(kw[j]), e[j]);               // F = k e^(b - m_R)
  {
    uint4 lo, hi;
    pack8(v, lo, hi);
    *reinterpret_cast<uint4 *>(sm + OFF_FQ + o) = lo;
    *reinterpret_cast<uint4 *>(sm + OFF_FQ + o + 8192) = hi;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    v[j] = mul2(unpack_bf16x2(kw[j]), exp2_2(make_float2(-x[j].x, -x[j].y)));        // G = k e^(m_R - b)
  {
    uint4 lo, hi;
    pack8(v, lo, hi);
    *reinterpret_cast<uint4 *>(sm + OFF_GB + o) = lo;
    *reinterpret_cast<uint4 *>(sm + OFF_GB + o + 8192) = hi;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = mul2(v[j], f.el);                               // K' = G e^(b_63 - m_R)
  {
    uint4 lo, hi;
    pack8(w, lo, hi);
    // PK rows 64 + rho: 192-row K-major tile, token columns < 64 (panel 0)
    *reinterpret_cast<uint4 *>(sm + OFF_BUF + kBlkPK + o + 64 * 128) = lo;
    *reinterpret_cast<uint4 *>(sm + OFF_BUF + kBlkPK + o + 128 * 128) = hi;
  }
  if (R == 0) {   // B_1: rows of block 0 anchored at m_1, k e^(m_1 - b) = (k e^(a_0 - b)) e^(m_1 - a_0)
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = mul2(mul2(v[j], f.eg), f.cr);
    uint4 lo, hi;
    pack8(w, lo, hi);
    *reinterpret_cast<uint4 *>(sm + OFF_GB + 16384 + o) = lo;          // columns 64 + t0: panel 1
    *reinterpret_cast<uint4 *>(sm + OFF_GB + 16384 + o + 8192) = hi;
  }
  // queries
#pragma unroll
  for (int j = 0; j < 8; ++j)
    v[j] = mul2(unpack_bf16x2(ld_u32(sm + OFF_QIN + in_offset(t0 + j, c0))), e[j]);  // Q = q e^(b - m_R)
  {
    uint4 lo, hi;
    pack8(v, lo, hi);
    *reinterpret_cast<uint4 *>(sm + OFF_FQ + 16384 + o) = lo;          // columns 64 + t0: panel 1
    *reinterpret_cast<uint4 *>(sm + OFF_FQ + 16384 + o + 8192) = hi;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = mul2(v[j], f.nems);                             // -Q+ = -scale Q e^(m_R)
  {
    uint4 lo, hi;
    pack8(w, lo, hi);
    *reinterpret_cast<uint4 *>(sm + OFF_BUF + kBlkWQ + 16384 + o) = lo;
    *reinterpret_cast<uint4 *>(sm + OFF_BUF + kBlkWQ + 16384 + o + 8192) = hi;
  }
}

// 32 fp32 values -> 16 packed bf16 pairs in 16 TMEM columns
__device__ __forceinline__ void st_bf16_pairs(uint32_t taddr, const float *v) {
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
  tmem_st16(taddr, w);
}

__global__ void __launch_bounds__(kThreads, 1) prefill_fused_kernel(const __grid_constant__ FusedParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *small = sm + OFF_SMALL;
  float *s_nq3 = reinterpret_cast<float *>(small + SM_NQ);     // [chunk % 3][64]: read by the chain a chunk later
  float *s_nk = reinterpret_cast<float *>(small + SM_NK);
  float *s_beta2 = reinterpret_cast<float *>(small + SM_BETA);
  float *s_h = reinterpret_cast<float *>(small + SM_H);
  float *s_gamma2 = reinterpret_cast<float *>(small + SM_GAMMA);
  float *s_em = reinterpret_cast<float *>(small + SM_EM);      // e^(m_0), e^(m_1) per key channel rho
  uint64_t *bars = reinterpret_cast<uint64_t *>(small + SM_BAR);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(small + SM_TMEM);
  volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(small + SM_ABORT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = prm.H;
  const int h = blockIdx.x % H;
  const int nl = static_cast<int>(prm.order[blockIdx.x / H]);   // local sequence, longest first
  const int n_seq = prm.seq0 + nl;
  const int t0 = prm.tok_off[nl];
  const int len = prm.tok_off[nl + 1] - t0;
  const int nchunks = (len + kC - 1) / kC;
  const bool producer = warp < 8;

  int slot = 0;
  if (prm.slot_ids) {
    slot = prm.slot_ids[n_seq];
    if (slot < 0 || slot >= prm.num_slots) {
      if (tid == 0) atomicOr(prm.status, KDA_DEVICE_BAD_SLOT);
      return;
    }
  }
  float *dst = prm.state_out_pool ? prm.state_out_pool + (static_cast<size_t>(slot) * H + h) * kD * kD
                                  : prm.state_out_dense + (static_cast<size_t>(n_seq) * H + h) * kD * kD;
  const float *src = prm.state_in ? prm.state_in + (static_cast<size_t>(slot) * H + h) * kD * kD : nullptr;
  // chain thread = (value channel d, half hv of the key channels / tokens)
  const int ctid = tid - kProdThreads;
  const int cw = warp - 8, quad = warp & 3, hv = (cw >> 2) & 1;
  const int d = quad * 32 + lane;

  if (nchunks == 0) {   // empty sequence: the final state is the initial one
    if (producer) return;
#pragma unroll 8
    for (int i = 0; i < 64; ++i) {
      const int kd = kd_of_rho(64 * hv + i);
      dst[static_cast<size_t>(kd) * kD + d] = src ? src[static_cast<size_t>(kd) * kD + d] : 0.f;
    }
    return;
  }

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    mbar_init(&bars[B_IN], 1);
    mbar_init(&bars[B_V], 1);
    mbar_init(&bars[B_PMMA], 1);
    mbar_init(&bars[B_PW], 1);
    mbar_init(&bars[B_PU], 1);
    mbar_init(&bars[B_GAMMA], 64);
    mbar_init(&bars[B_READY], 1);
    mbar_init(&bars[B_M1U], 1);
    mbar_init(&bars[B_M2S], 1);
    mbar_init(&bars[B_FREE], 1);
    *s_abort = 0;
    fence_mbar_init();
    // chunk 0's q, k, g
    mbar_arrive_expect_tx(&bars[B_IN], 3 * 16384);
#pragma unroll
    for (int x = 0; x < 128; x += 64) {
      tma_load_3d(sm + OFF_QIN + x * 128, &prm.tq, x, h, t0, &bars[B_IN]);
      tma_load_3d(sm + OFF_KIN + x * 128, &prm.tk, x, h, t0, &bars[B_IN]);
      tma_load_3d(sm + OFF_GIN + x * 128, &prm.tg, x, h, t0, &bars[B_IN]);
    }
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (producer) {
    // ================================================================ producer: the chunks' WY operands
    const int ptid = tid;
    const int p = ptid & 63, sel = ptid >> 6, c0 = 2 * p;
    const float2 dtb = *reinterpret_cast<const float2 *>(prm.dt_bias + h * kD + c0);
    const float nea = -__expf(prm.A_log[h]) * kLog2e;   // lambda = lb sigmoid(ea (g + dtb)); log2 units below
    const float lb2 = prm.lower_bound * kLog2e;
    const float2 nd = make_float2(nea * dtb.x, nea * dtb.y);
    const float2 nea2 = make_float2(nea, nea), lb22 = make_float2(lb2, lb2), one2 = make_float2(1.f, 1.f);
    const float2 zero2 = make_float2(0.f, 0.f);
    uint16_t beta_raw = ptid < min(kC, len) ? prm.beta[static_cast<size_t>(t0 + ptid) * prm.beta_stride + h] : uint16_t(0);
    bool stop = false;

    for (int n = 0; n < nchunks && !stop; ++n) {
      const int tok0 = t0 + n * kC;
      const int valid = min(kC, len - n * kC);
      float *s_beta = s_beta2 + 64 * (n & 1);
      float *s_nq = s_nq3 + 64 * (n % 3);
      // this chunk's beta (loaded one chunk earlier) to shared memory; the next chunk's load is issued here
      if (ptid < kC) {
        s_beta[ptid] = ptid < valid ? sigmoid_f(bf16_bits_to_f32(beta_raw)) : 0.f;
        const int nvalid = min(kC, len - (n + 1) * kC);
        beta_raw = ptid < nvalid ? prm.beta[static_cast<size_t>(tok0 + kC + ptid) * prm.beta_stride + h] : uint16_t(0);
      }
      wait_or_abort(&bars[B_IN], n & 1, s_abort, prm.status);

      // ---------------------------------------------------- gate and in-quarter decay sums
      // thread = (channel pair p, quarter `sel` of both 32-row blocks); a quarter before its block's anchor
      // (row 15 of the block) takes suffix sums up to its own last row, one after it prefix sums from its own
      // first row; the outer quarters add a neighbour quarter's sum below
      const bool before = sel < 2;
      float2 x[2][8];
#pragma unroll
      for (int bi = 0; bi < 2; ++bi) {
        const int qd = 4 * bi + sel;
        const int r0 = 8 * qd;
        float2 lam[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = r0 + j;
          const float2 gg = unpack_bf16x2(ld_u32(sm + OFF_GIN + in_offset(r, c0)));
          const float2 ex = exp2_2(fma2(gg, nea2, nd));
          const float2 den = fma2(ex, one2, one2);
          const float2 l = mul2(make_float2(fast_rcp(den.x), fast_rcp(den.y)), lb22);
          lam[j] = r < valid ? l : zero2;
        }
        float2 hs;
        if (before) {
          x[bi][7] = zero2;
#pragma unroll
          for (int j = 6; j >= 0; --j) x[bi][j] = make_float2(x[bi][j + 1].x - lam[j + 1].x, x[bi][j + 1].y - lam[j + 1].y);
          hs = make_float2(lam[0].x - x[bi][0].x, lam[0].y - x[bi][0].y);
        } else {
          float2 acc = zero2;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc = make_float2(acc.x + lam[j].x, acc.y + lam[j].y);
            x[bi][j] = acc;
          }
          hs = acc;
        }
        *reinterpret_cast<float2 *>(s_h + qd * kD + c0) = hs;
      }
      named_bar_sync<kBarProd>(kProdThreads);   // quarter sums and beta visible

      // ---------------------------------------------------- anchors, gamma, operand tiles
      // the chunk's buffer (and the producer's T tiles in it) and gamma slot are free once the chain's output
      // product of chunk n - 1 is done
      if (n > 0) wait_or_abort(&bars[B_FREE], (n - 1) & 1, s_abort, prm.status);
      {
        float2 sq[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) sq[q] = *reinterpret_cast<const float2 *>(s_h + q * kD + c0);
        auto add = [](float2 u, float2 v) { return make_float2(u.x + v.x, u.y + v.y); };
        const float2 m0 = add(sq[0], sq[1]);
        const float2 a0 = add(add(m0, sq[2]), sq[3]);
        const float2 m1 = add(add(a0, sq[4]), sq[5]);
        const float2 tot = add(add(m1, sq[6]), sq[7]);
        const float2 em0 = exp2_2(m0), em1 = exp2_2(m1);
        if (sel == 0) {   // gamma = e^(b_63) and the block factors e^(m_R) for rho = p and 64 + p
          float *gam = s_gamma2 + 128 * (n & 1);
          gam[p] = fast_exp2(tot.x);
          gam[64 + p] = fast_exp2(tot.y);
          s_em[p] = em0.x;
          s_em[64 + p] = em0.y;
          s_em[128 + p] = em1.x;
          s_em[192 + p] = em1.y;
          mbar_arrive(&bars[B_GAMMA]);
        }
        const float nsc = -prm.scale;
        Factors f0, f1;
        f0.nems = make_float2(nsc * em0.x, nsc * em0.y);
        f0.el = exp2_2(make_float2(tot.x - m0.x, tot.y - m0.y));
        f0.eg = exp2_2(make_float2(a0.x - m0.x, a0.y - m0.y));
        f0.cr = exp2_2(make_float2(fminf(m1.x - a0.x, 0.f), fminf(m1.y - a0.y, 0.f)));
        f1.nems = make_float2(nsc * em1.x, nsc * em1.y);
        f1.el = exp2_2(make_float2(tot.x - m1.x, tot.y - m1.y));
        f1.eg = zero2;
        f1.cr = zero2;
        // the outer quarters measure from the neighbour quarter's far end
        auto shift = [&](int bi, float2 off) {
#pragma unroll
          for (int j = 0; j < 8; ++j) x[bi][j] = add(x[bi][j], off);
        };
        shift(0, sel == 0 ? make_float2(-sq[1].x, -sq[1].y) : sel == 3 ? sq[2] : zero2);
        shift(1, sel == 0 ? make_float2(-sq[5].x, -sq[5].y) : sel == 3 ? sq[6] : zero2);
        build_rows<0>(sm, x[0], 8 * sel, p, f0);
        build_rows<1>(sm, x[1], 32 + 8 * sel, p, f1);
      }
      fence_async_smem();
      tc_fence_before();
      named_bar_sync<kBarProd>(kProdThreads);

      // ---------------------------------------------------- A/P product (one 128 x 96 tcgen05.mma)
      if (ptid == 0) {
        tc_fence_after();
        const uint64_t fq = desc_mnmajor_base(smem_u32(sm + OFF_FQ), 128);
        const uint64_t gb = desc_mnmajor_base(smem_u32(sm + OFF_GB), 128);
        const uint32_t id = idesc_bf16(128, 96, true, true);
#pragma unroll
        for (int s = 0; s < 8; ++s) mma_bf16(tmem + TM_P, fq + mnmajor_step(s), gb + mnmajor_step(s), id, s > 0);
        mma_commit(&bars[B_PMMA]);
      }
      // ---------------------------------------------------- l2 norms (token-major), under the product
      {
        const int r = ptid >> 2, part = ptid & 3;
        const int rot = (r & 1) * 2 + (part >> 1);
        float2 sqq = zero2, skk = zero2;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 32 * part + 8 * ((j + rot) & 3);
          const uint32_t off = in_offset(r, c);
          const uint4 wq = *reinterpret_cast<const uint4 *>(sm + OFF_QIN + off);
          const uint4 wk = *reinterpret_cast<const uint4 *>(sm + OFF_KIN + off);
          const uint32_t aq[4] = {wq.x, wq.y, wq.z, wq.w}, ak[4] = {wk.x, wk.y, wk.z, wk.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fq2 = unpack_bf16x2(aq[e]), fk2 = unpack_bf16x2(ak[e]);
            sqq = fma2(fq2, fq2, sqq);
            skk = fma2(fk2, fk2, skk);
          }
        }
        float ssq = sqq.x + sqq.y, ssk = skk.x + skk.y;
        ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
        ssk += __shfl_xor_sync(0xffffffffu, ssk, 1);
        ssq += __shfl_xor_sync(0xffffffffu, ssq, 2);
        ssk += __shfl_xor_sync(0xffffffffu, ssk, 2);
        if (part == 0) {
          s_nq[r] = r < valid ? rsqrtf(ssq + kL2Eps) : 0.f;
          s_nk[r] = r < valid ? rsqrtf(ssk + kL2Eps) : 0.f;
        }
      }
      named_bar_sync<kBarProd>(kProdThreads);   // norms visible; the input tiles are read for the last time
      if (ptid == 0) {
        // q, k, g of the next chunk into the input tiles; L2 prefetch of its v and of the inputs one chunk further
        if (n + 1 < nchunks) {
          mbar_arrive_expect_tx(&bars[B_IN], 3 * 16384);
#pragma unroll
          for (int x2 = 0; x2 < 128; x2 += 64) {
            tma_load_3d(sm + OFF_QIN + x2 * 128, &prm.tq, x2, h, tok0 + kC, &bars[B_IN]);
            tma_load_3d(sm + OFF_KIN + x2 * 128, &prm.tk, x2, h, tok0 + kC, &bars[B_IN]);
            tma_load_3d(sm + OFF_GIN + x2 * 128, &prm.tg, x2, h, tok0 + kC, &bars[B_IN]);
            tma_prefetch_3d(&prm.tv, x2, h, tok0 + kC);
          }
          if (n + 2 < nchunks) {
#pragma unroll
            for (int x2 = 0; x2 < 128; x2 += 64) {
              tma_prefetch_3d(&prm.tq, x2, h, tok0 + 2 * kC);
              tma_prefetch_3d(&prm.tk, x2, h, tok0 + 2 * kC);
              tma_prefetch_3d(&prm.tg, x2, h, tok0 + 2 * kC);
            }
          }
        }
      }
      wait_or_abort(&bars[B_PMMA], n & 1, s_abort, prm.status);
      tc_fence_after();
      if (ptid == 0) {   // the Q and G tiles are free: v may land (F stays for W)
        mbar_arrive_expect_tx(&bars[B_V], 16384);
        tma_load_3d(sm + OFF_V, &prm.tv, 0, h, tok0, &bars[B_V]);
        tma_load_3d(sm + OFF_V + 8192, &prm.tv, 64, h, tok0, &bars[B_V]);
      }

      // ---------------------------------------------------- A (fp32) and P (bf16 rows of the buffer) from TMEM
      {
        // lanes 0..63 of the product hold rows of A (k side), lanes 64..127 rows of P (q side); the warp's lanes
        // are one 32-row block R, ib picks the 32-column block I.  A takes beta_r n_r n_i (the key norms it was
        // built without), P only the scale (its norms go to U' and the output rows).
        const int q4 = warp & 3, ib = warp >> 2;
        const bool is_p = q4 >= 2;
        const int r = (q4 & 1) * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const float rscale = is_p ? prm.scale : s_beta[r] * s_nk[r];
        float *sA = reinterpret_cast<float *>(sm + OFF_A);
        const int R = q4 & 1, I = ib;
        const int srcc = I == R ? 32 * I : I < R ? 64 + 32 * I : -1;
        uint32_t va[32];
        if (srcc >= 0) {
          tmem_ld16_async(tmem + TM_P + lane_base + srcc, va);
          tmem_ld16_async(tmem + TM_P + lane_base + srcc + 16, va + 16);
        }
        tmem_wait_ld();
        tmem_tie<32>(va);
        const int lim = r - 32 * I + (is_p ? 1 : 0);
        float v[32];
        if (is_p) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = (srcc >= 0 && e < lim) ? __uint_as_float(va[e]) * rscale : 0.f;
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8)
            *reinterpret_cast<uint4 *>(sm + OFF_BUF + kBlkPK + swz_offset(kBlkPKRows, r, 32 * I + 8 * k8)) =
                make_uint4(pack_bf16x2(v[8 * k8], v[8 * k8 + 1]), pack_bf16x2(v[8 * k8 + 2], v[8 * k8 + 3]),
                           pack_bf16x2(v[8 * k8 + 4], v[8 * k8 + 5]), pack_bf16x2(v[8 * k8 + 6], v[8 * k8 + 7]));
        } else {
          const float4 *nk4 = reinterpret_cast<const float4 *>(s_nk + 32 * I);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 nc = nk4[e4];
            const float ncs[4] = {nc.x, nc.y, nc.z, nc.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = 4 * e4 + q;
              v[e] = (srcc >= 0 && e < lim) ? __uint_as_float(va[e]) * rscale * ncs[q] : 0.f;
            }
          }
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(sA + r * kAStride + 32 * I + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_bar_sync<kBarProd>(kProdThreads);

      // ---------------------------------------------------- T = (I + A)^-1 Diag(beta), as T_U and T_W
      // Blocked inverse of the unit-lower L = I + A in fp32, 16x16 blocks D_R = L_RR^-1:
      //   L^-1_10 = -D_1 A_10 D_0,  L^-1_32 = -D_3 A_32 D_2,  L^-1 (rows 32..63, cols 0..31) = -I_2 A_(23,01) I_1
      // in place in the A tile; each block of L^-1 goes to T_U (rows x n_k, columns x beta) and T_W (columns also
      // x n_k) in bf16; the six blocks above the diagonal of both are zero.
      {
        float *sA = reinterpret_cast<float *>(sm + OFF_A);
        float *sInv = sA;
        uint8_t *tU = sm + OFF_TU, *tW = sm + OFF_TW;
        if (ptid < 192) {   // zero blocks (I, J), J > I: 6 blocks x 16 rows x two 16-byte chunks, in both tiles
          const int z = ptid;
          const int b6 = z >> 5, rr = (z >> 1) & 15, hc = z & 1;
          const int I = b6 < 3 ? 0 : b6 < 5 ? 1 : 2;
          const int J = b6 < 3 ? b6 + 1 : b6 < 5 ? b6 - 1 : 3;
          const uint32_t o = swz_offset(64, 16 * I + rr, 16 * J + 8 * hc);
          *reinterpret_cast<uint4 *>(tU + o) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(tW + o) = make_uint4(0, 0, 0, 0);
        }
        // D_R: task (block R, column jc) = 8 warp + lane / 4, so warps 2R and 2R + 1 share block R; lane
        // q = lane % 4 of a task carries rows q, q + 4, q + 8, q + 12 of its column.  Right-looking: at step m
        // the lane holding row m broadcasts x_m to its task's lanes, and every later row takes one FMA.
        {
          const int q = lane & 3, jc = 8 * (warp & 1) + (lane >> 2), R = warp >> 1;
          const float *a = sA + (16 * R) * kAStride + 16 * R;
          float xs[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) xs[i] = 4 * i + q == jc ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < 15; ++m) {
            const float xm = __shfl_sync(0xffffffffu, xs[m >> 2], (lane & ~3) | (m & 3));
#pragma unroll
            for (int i = (m + 1) >> 2; i < 4; ++i) {
              const int r = 4 * i + q;
              if (r > m) xs[i] = fmaf(-a[r * kAStride + m], xm, xs[i]);
            }
          }
          switch (R) {   // both warps of the block have read its A entries (constant barrier ids)
            case 0: named_bar_sync<1>(64); break;
            case 1: named_bar_sync<2>(64); break;
            case 2: named_bar_sync<3>(64); break;
            default: named_bar_sync<4>(64); break;
          }
          const int c = 16 * R + jc;
          const float bc = s_beta[c], nc = s_nk[c];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = 16 * R + 4 * i + q;
            sInv[row * kAStride + c] = xs[i];
            const float u = xs[i] * s_nk[row] * bc;
            const uint32_t o = swz_offset(64, row, c);
            *reinterpret_cast<uint16_t *>(tU + o) = f32_to_bf16_bits(u);
            *reinterpret_cast<uint16_t *>(tW + o) = f32_to_bf16_bits(u * nc);
          }
        }
        named_bar_sync<kBarProd>(kProdThreads);
        // Every block product below is a set of 16 x 8 output tiles, one per warp task, on TF32 tensor cores.
        if (warp < 4) {
          const int lo = warp < 2 ? 0 : 32, nj = warp & 1;
          float dd[4] = {0.f, 0.f, 0.f, 0.f};
          mm_16x8(dd, sA + (lo + 16) * kAStride + lo, sInv + lo * kAStride + lo + 8 * nj, 2, lane);
          st_16x8(sA + lo * kAStride + lo + 16 + 8 * nj, dd, 1.f, lane);
          if (warp < 2) named_bar_sync<5>(64); else named_bar_sync<6>(64);
          float e4[4] = {0.f, 0.f, 0.f, 0.f};
          mm_16x8(e4, sInv + (lo + 16) * kAStride + lo + 16, sA + lo * kAStride + lo + 16 + 8 * nj, 2, lane);
          st_16x8(sInv + (lo + 16) * kAStride + lo + 8 * nj, e4, -1.f, lane);
          st_16x8_t(tU, tW, lo + 16, lo + 8 * nj, e4, -1.f, s_beta, s_nk, lane);
        }
        named_bar_sync<kBarProd>(kProdThreads);
        {
          const int mi = warp >> 2, nj = warp & 3;
          const int k0 = nj < 2 ? 0 : 16;
          float dd[4] = {0.f, 0.f, 0.f, 0.f};
          mm_16x8(dd, sA + (32 + 16 * mi) * kAStride + k0, sInv + k0 * kAStride + 8 * nj, (32 - k0) / 8, lane);
          st_16x8(sA + (16 * mi) * kAStride + 32 + 8 * nj, dd, 1.f, lane);
        }
        named_bar_sync<kBarProd>(kProdThreads);
        {
          const int mi = warp >> 2, nj = warp & 3;
          float dd[4] = {0.f, 0.f, 0.f, 0.f};
          mm_16x8(dd, sInv + (32 + 16 * mi) * kAStride + 32, sA + 32 + 8 * nj, mi ? 4 : 2, lane);
          st_16x8_t(tU, tW, 32 + 16 * mi, 8 * nj, dd, -1.f, s_beta, s_nk, lane);
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_bar_sync<kBarProd>(kProdThreads);

      // ---------------------------------------------------- W^T from F per 32-row block; U^'^T = V^T T_U^T
      const bool ragged = valid < kC;
      if (ragged) {   // rows past the sequence end: T's columns there are 0, but v may hold anything
        wait_or_abort(&bars[B_V], n & 1, s_abort, prm.status);
        for (int idx = ptid; idx < (kC - valid) * 16; idx += kProdThreads) {
          const int r2 = valid + idx / 16, cc = idx % 16;
          *reinterpret_cast<uint4 *>(sm + OFF_V + swz_offset(64, r2, 8 * cc)) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
        named_bar_sync<kBarProd>(kProdThreads);
      }
      if (ptid == 0) {
        tc_fence_after();
        const uint32_t id_w = idesc_bf16(128, 64, false, false);
        const uint32_t id_u = idesc_bf16(128, 64, true, false);
        const uint64_t ff = desc_kmajor_base(smem_u32(sm + OFF_FQ));
        const uint64_t vv = desc_mnmajor_base(smem_u32(sm + OFF_V), 64);
        const uint64_t tw = desc_kmajor_base(smem_u32(sm + OFF_TW));
        const uint64_t tu = desc_kmajor_base(smem_u32(sm + OFF_TU));
        // X_R^T = F_R^T T_W,R^T over the tokens of block R (K steps 2R, 2R + 1) -> TM_P + 64 R
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_bf16(tmem + TM_P + 64 * (s >> 1), ff + kmajor_step(128, s), tw + kmajor_step(64, s), id_w, s & 1);
        mma_commit(&bars[B_PW]);
        if (!ragged) wait_or_abort(&bars[B_V], n & 1, s_abort, prm.status);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16(tmem + TM_XU, vv + mnmajor_step(s), tu + kmajor_step(64, s), id_u, s > 0);
        mma_commit(&bars[B_PU]);
      }
      __syncwarp();
      // ---------------------------------------------------- W^T = Diag(e^(m_0)) X_0^T + Diag(e^(m_1)) X_1^T -> buffer
      {
        const int q4 = warp & 3, half = warp >> 2;   // lane = key channel rho; half = tokens 32 half .. +31
        wait_or_abort(&bars[B_PW], n & 1, s_abort, prm.status);
        tc_fence_after();
        const int row = q4 * 32 + lane;
        const uint32_t taddr = tmem + TM_P + (static_cast<uint32_t>(q4 * 32) << 16) + 32 * half;
        uint32_t x0[32], x1[32];
        tmem_ld16_async(taddr, x0);
        tmem_ld16_async(taddr + 16, x0 + 16);
        tmem_ld16_async(taddr + 64, x1);
        tmem_ld16_async(taddr + 80, x1 + 16);
        const float e0 = s_em[row], e1 = s_em[128 + row];
        tmem_wait_ld();
        tmem_tie<32>(x0);
        tmem_tie<32>(x1);
        const float2 e02 = make_float2(e0, e0), e12 = make_float2(e1, e1);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t wv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = 8 * k + 2 * q;
            const float2 wpair = fma2(make_float2(__uint_as_float(x1[i]), __uint_as_float(x1[i + 1])), e12,
                                      mul2(make_float2(__uint_as_float(x0[i]), __uint_as_float(x0[i + 1])), e02));
            wv[q] = pack2(wpair);
          }
          *reinterpret_cast<uint4 *>(sm + OFF_BUF + kBlkWQ + swz_offset(128, row, 32 * half + 8 * k)) =
              make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
      if (ptid == 0) wait_or_abort(&bars[B_PU], n & 1, s_abort, prm.status);   // U^' is in TMEM
      fence_async_smem();
      tc_fence_before();
      stop = bar_any<kBarProd>(kProdThreads, *s_abort != 0);
      if (ptid == 0) mbar_arrive(&bars[B_READY]);   // chunk n's buffer and U^' are complete
    }
  } else {
    // ================================================================ chain: the state recurrence
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    // -S0 (this thread's 64 key channels rho = 64 hv + i) -> the bf16 A operand; Diag(gamma_0) S0 -> TMEM
    {
      const int col = 64 * hv;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float s[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int kd = kd_of_rho(col + 32 * part + i);
          s[i] = src ? -src[static_cast<size_t>(kd) * kD + d] : 0.f;
        }
        st_bf16_pairs(tmem + lane_base + TM_SA + col / 2 + 16 * part, s);
      }
      wait_or_abort(&bars[B_GAMMA], 0, s_abort, prm.status);
      const float *gam = s_gamma2 + col;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float s[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int kd = kd_of_rho(col + 32 * part + i);
          s[i] = src ? src[static_cast<size_t>(kd) * kD + d] * gam[32 * part + i] : 0.f;
        }
        tmem_st16(tmem + lane_base + TM_S + col + 32 * part, s);
        tmem_st16(tmem + lane_base + TM_S + col + 32 * part + 16, s + 16);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    named_bar_sync<kBarChain>(kChainThreads);

    uint8_t *stage = sm + OFF_STAGE;
    // output of chunk cc (accumulated in O buffer cc & 1) -> staging, each token row times its query norm
    auto out_to_stage = [&](int cc) {
      uint32_t ov[32];
      const uint32_t tb = tmem + lane_base + TM_O0 + 64 * (cc & 1) + 32 * hv;
      tmem_ld16_async(tb, ov);
      tmem_ld16_async(tb + 16, ov + 16);
      tmem_wait_ld();
      tmem_tie<32>(ov);
      const float4 *nq4 = reinterpret_cast<const float4 *>(s_nq3 + 64 * (cc % 3) + 32 * hv);
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const float4 nq = nq4[i4];
        const float nqs[4] = {nq.x, nq.y, nq.z, nq.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = 4 * i4 + q;
          *reinterpret_cast<uint16_t *>(stage + swz_offset(64, 32 * hv + i, d)) =
              f32_to_bf16_bits(__uint_as_float(ov[i]) * nqs[q]);
        }
      }
    };
    const uint8_t *buf = sm + OFF_BUF;
    bool stop = false;
    for (int c = 0; c < nchunks && !stop; ++c) {
      const uint32_t tm_o = TM_O0 + 64 * (c & 1);
      wait_or_abort(&bars[B_READY], c & 1, s_abort, prm.status);

      // ---- [U'^T | O^T] = (-S_c)^T [W' | -Q+]^T: the U half accumulates onto U^'^T (it is on the critical path),
      //      then the O half
      if (tid == kChainIssuer) {
        // the previous chunk's output product has read U^T where the producer has put U^'^T and this product adds
        if (c > 0) wait_or_abort(&bars[B_FREE], (c - 1) & 1, s_abort, prm.status);
        tc_fence_after();
        const uint64_t wq = desc_mnmajor_base(smem_u32(buf + kBlkWQ), 128);
        const uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int k = 0; k < 8; ++k) mma_bf16_tmem_a(tmem + TM_XU, tmem + TM_SA + 8 * k, wq + mnmajor_step(k), id, 1);
        mma_commit(&bars[B_M1U]);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_tmem_a(tmem + tm_o, tmem + TM_SA + 8 * k, wq + desc_bytes(16384) + mnmajor_step(k), id, k > 0);
      }
      wait_or_abort(&bars[B_M1U], c & 1, s_abort, prm.status);
      // the previous chunk's output product (done before this step's first product was issued) -- waited on here,
      // before this step commits its own output product onto the same barrier
      if (c > 0) wait_or_abort(&bars[B_FREE], (c - 1) & 1, s_abort, prm.status);
      tc_fence_after();

      // ---- U'^T (fp32) -> bf16 pairs in place (columns 32 hv .. 32 hv + 15 of TM_XU)
      {
        uint32_t v[32];
        tmem_ld16_async(tmem + lane_base + TM_XU + 32 * hv, v);
        tmem_ld16_async(tmem + lane_base + TM_XU + 32 * hv + 16, v + 16);
        tmem_wait_ld();
        tmem_tie<32>(v);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        tmem_st16(tmem + lane_base + TM_XU + 32 * hv, w);
      }
      tmem_wait_st();
      tc_fence_before();
      if (tid == kChainIssuer) bulk_wait_read();   // the staging tile's previous store has read it
      named_bar_sync<kBarChain>(kChainThreads);

      // ---- S^T += U'^T K' (N = 128), then O^T += U'^T P^T (N = 64); U'^T's K steps: tokens 0..31 at TM_XU + 0, 8,
      //      tokens 32..63 at TM_XU + 32, 40
      if (tid == kChainIssuer) {
        tc_fence_after();
        const uint64_t pk = desc_kmajor_base(smem_u32(buf + kBlkPK));
        const uint32_t id_s = idesc_bf16(128, 128, false, false), id_o = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_tmem_a(tmem + TM_S, tmem + TM_XU + (k < 2 ? 8 * k : 32 + 8 * (k - 2)),
                          pk + desc_bytes(64 * 128) + kmajor_step(kBlkPKRows, k), id_s, 1);
        mma_commit(&bars[B_M2S]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_tmem_a(tmem + tm_o, tmem + TM_XU + (k < 2 ? 8 * k : 32 + 8 * (k - 2)), pk + kmajor_step(kBlkPKRows, k),
                          id_o, 1);
        mma_commit(&bars[B_FREE]);
      }
      // ---- the previous chunk's output -> staging (stored at the end of this step)
      if (c > 0) {
        out_to_stage(c - 1);
        fence_async_smem();
      }
      wait_or_abort(&bars[B_M2S], c & 1, s_abort, prm.status);
      tc_fence_after();

      // ---- -S_{c+1} -> the bf16 A operand of the next first product; Diag(gamma_{c+1}) S_{c+1} -> TMEM
      if (c + 1 < nchunks) {
        wait_or_abort(&bars[B_GAMMA], (c + 1) & 1, s_abort, prm.status);
        const float *gam = s_gamma2 + 128 * ((c + 1) & 1);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int col = 64 * hv + 32 * part;
          uint32_t sv[32];
          tmem_ld16_async(tmem + lane_base + TM_S + col, sv);
          tmem_ld16_async(tmem + lane_base + TM_S + col + 16, sv + 16);
          tmem_wait_ld();
          tmem_tie<32>(sv);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(-__uint_as_float(sv[2 * j]), -__uint_as_float(sv[2 * j + 1]));
          tmem_st16(tmem + lane_base + TM_SA + col / 2, w);
          float s[32];
          const float4 *g4 = reinterpret_cast<const float4 *>(gam + col);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 g = g4[i];
            const float2 lo = mul2(make_float2(__uint_as_float(sv[4 * i]), __uint_as_float(sv[4 * i + 1])), make_float2(g.x, g.y));
            const float2 hi = mul2(make_float2(__uint_as_float(sv[4 * i + 2]), __uint_as_float(sv[4 * i + 3])), make_float2(g.z, g.w));
            s[4 * i] = lo.x;
            s[4 * i + 1] = lo.y;
            s[4 * i + 2] = hi.x;
            s[4 * i + 3] = hi.y;
          }
          tmem_st16(tmem + lane_base + TM_S + col, s);
          tmem_st16(tmem + lane_base + TM_S + col + 16, s + 16);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      stop = bar_any<kBarChain>(kChainThreads, *s_abort != 0);
      if (c > 0 && tid == kChainIssuer) {   // chunk c - 1 is not the last one: all 64 rows are valid
        const int tok = t0 + (c - 1) * kC;
        tma_store_3d(&prm.tout, 0, h, tok, stage);
        tma_store_3d(&prm.tout, 64, h, tok, stage + 8192);
        bulk_commit();
      }
    }

    // output of the last chunk, and the final state
    if (!stop) {
      if (tid == kChainIssuer) bulk_wait_read();
      wait_or_abort(&bars[B_FREE], (nchunks - 1) & 1, s_abort, prm.status);
      named_bar_sync<kBarChain>(kChainThreads);
      tc_fence_after();
      const int last_valid = len - (nchunks - 1) * kC;
      out_to_stage(nchunks - 1);
      fence_async_smem();
      named_bar_sync<kBarChain>(kChainThreads);
      if (last_valid == kC) {
        if (tid == kChainIssuer) {
          const int tok = t0 + (nchunks - 1) * kC;
          tma_store_3d(&prm.tout, 0, h, tok, stage);
          tma_store_3d(&prm.tout, 64, h, tok, stage + 8192);
          bulk_commit();
        }
      } else {   // a ragged last chunk: only its valid rows, 16 bytes per thread and step
        uint16_t *o = prm.out + static_cast<size_t>(t0 + (nchunks - 1) * kC) * prm.out_stride + h * kD;
        for (int idx = ctid; idx < last_valid * 16; idx += kChainThreads) {
          const int r = idx >> 4, cc = idx & 15;
          *reinterpret_cast<uint4 *>(o + static_cast<size_t>(r) * prm.out_stride + 8 * cc) =
              *reinterpret_cast<const uint4 *>(stage + swz_offset(64, r, 8 * cc));
        }
      }
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
      if (tid == kChainIssuer) bulk_wait_all();
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill_fused(const FusedParams &p, cudaStream_t stream) {
  if (p.num_seqs <= 0) return cudaSuccess;
  static std::mutex mu;
  static uint64_t done = 0;
  if (const cudaError_t e = set_attributes_once(mu, done, [] {
        return cudaFuncSetAttribute(prefill_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      }))
    return e;
  prefill_fused_kernel<<<p.num_seqs * p.H, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
