// Intra-chunk half of the chunked KDA prefill on sm_103a.
//
// One CTA per (chunk of C = 64 tokens, head); every chunk of every sequence is
// independent here, so the grid covers them all at once, two CTAs per SM.
// With per-channel log-decays lambda (the bounded gate of vLLM PR #55737 "Use
// FlashKDA for KDA chunked prefill", PR summary), b_t = sum_{j<=t} lambda_j
// inside the chunk and k^, q^ the l2-normalised keys / queries, a CTA computes
// the part of the chunk algebra that does not depend on the state entering the
// chunk:
//
//   A[r,i] = beta_r sum_c k^_rc k^_ic e^(b_rc - b_ic)   (i < r)
//   P[r,i] = scale  sum_c q^_rc k^_ic e^(b_rc - b_ic)   (i <= r)
//   T      = (I + A)^-1 Diag(beta)
//   W = T (k^ o e^b),  U^ = T V,  Q+ = scale q^ o e^b,  K' = k^ o e^(b_63 - b),  e^(b_63)
//
// and writes them to the chunk's block of the workspace (kda_prefill_block.h)
// for the state pass.  This is the token recurrence S_t = (I - beta k^ k^T)
// Diag(alpha) S_{t-1} + beta k^ v^T unrolled over a chunk: the corrections
// U = U^ - W S solve (I + A) U = Diag(beta)(V - (k^ o e^b) S).
//
// exp(b_r - b_i) spans up to 64 |lower_bound| inside a chunk, far outside
// fp32.  A and P are built from sub-blocks R of 16 rows (32 rows when
// lower_bound >= -5) with anchors m_R = b at the middle row of block R:
//   same block:   e^(b_r - b_i) = e^(b_r - m_R) e^(m_R - b_i)     (|exponents| <= 8 |lb| or 16 |lb|)
//   block I < R:  e^(b_r - b_i) = e^(b_r - m_R) e^(m_R - b_i)     (second factor <= 1)
// so ONE tcgen05.mma (128 x 160, or 128 x 96) of [F; Q] = [k^; q^] o e^(b - m_R(row))
// against [G; B_1; ...] (G = k^ o e^(m_R(row) - b); B_R = the rows of blocks < R
// times e^(m_R - b)) yields every block of A and P that is needed.  T comes
// from blocked forward substitution (16x16 diagonal inverses on CUDA cores,
// off-diagonal blocks with TF32 mma.sync), W^T and U^^T from two more
// tcgen05.mma with M = 128 (lane = key / value channel).
//
// Operand tiles are key-channel-major ([channel][token], 128-byte rows): a
// thread owns two key channels and eight consecutive tokens of each, so every
// store is one 16-byte chunk; the two channels 2p, 2p + 1 go to rows p and
// 64 + p ("paired" order, kd_of_rho) so that a warp's stores hit all eight
// swizzle phases.
#include <cuda.h>

#include <type_traits>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_prefill_block.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = kChunk;
constexpr int kThreads = 256;   // 8 warps; two CTAs per SM

// ---- shared memory map (offsets from a 1024-byte aligned base) ----
// prologue .. A/P product
constexpr uint32_t OFF_FQ = 0;        // [F | Q]: 128 rows rho x (64 + 64) tokens, MN-major A operand (32 KB)
constexpr uint32_t OFF_GB = 32768;    // [G | B_1 | B_2 | B_3]: 128 rows rho x 160 tokens in 3 panels (48 KB)
constexpr uint32_t OFF_KP = 82944;    // K+^T = (k^ o e^b)^T: 128 rows rho x 64 tokens, K-major A operand (16 KB)
constexpr uint32_t OFF_QIN = 0, OFF_KIN = 16384, OFF_GIN = 32768;   // TMA tiles, consumed before the operands are written
// the q, k, g tiles are unswizzled (only CUDA cores read them): two 64-channel boxes of 64 rows x 128 bytes
__device__ __forceinline__ uint32_t in_offset(int r, int c) {
  return static_cast<uint32_t>((c >> 6) * 8192 + r * 128 + (c & 63) * 2);
}
// after the A/P product
constexpr uint32_t OFF_QST = 0;       // Q+^T rows of the block (16 KB), stored by bulk copy
constexpr uint32_t OFF_PKST = 16384;  // [P ; K'^T] rows of the block (24 KB), stored by bulk copy
constexpr uint32_t OFF_A = 40960;     // A fp32 [64][68], turned into (I + A)^-1 in place
constexpr uint32_t OFF_VIN = 58368;   // v tile (TMA) [token][value channel]
constexpr uint32_t OFF_T = 74752;     // T bf16 K-major [t][t'] (8 KB), written by the inverse's steps
// after the W / U^ products
constexpr uint32_t OFF_WST = 40960, OFF_UST = 57344;   // W^T and U^^T rows of the block
constexpr uint32_t OFF_SMALL = 99328;
constexpr uint32_t SM_NQ = 0, SM_NK = 256, SM_BETA = 512, SM_H = 768 /* [8 quarters][128] f32 */,
                   SM_BAR = 4864, SM_TMEM = 4888, SM_ABORT = 4892, SM_BARU = 4896,
                   SM_HALO = 4928 /* short convolutions: [3 tensors][3 rows][64 channel pairs] u32 */,
                   SM_VW = 7232 /* v's taps [128 channels][4] f32 */, SM_END = 9280;
constexpr int kCopyThread = 128;      // issues the block's early bulk stores (Q+, [P ; K'])
constexpr uint32_t kSmemBytes = OFF_SMALL + SM_END + 1024;   // + alignment slack
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
constexpr int kAStride = 68;
constexpr uint32_t kTmemCols = 256;   // A/P product: 160 columns; then W^T 0..63, U^^T 64..127

// Sub-blocks of BLK rows: 16, or 32 when lower_bound >= -5.  The anchored factors reach 2^(+-|x|) with |x| up to
// (BLK / 2) |lb| log2(e); both the large and the small side must stay inside fp32 / bf16 with room for small
// key components (2^-115.4 at the limit: 8 rows at |lb| = 10, or 16 rows at |lb| = 5; at 2^-127 the small
// factor flushes to zero and entries of A are lost).  The stacked tile [G | B_1 | ...] holds B_R2 (the rows
// of the blocks before R2, anchored at m_R2) from column gb_col0(R2); its width is gb_col0(64 / BLK).
template <int BLK>
__host__ __device__ constexpr int gb_col0(int R2) {
  return BLK == 16 ? (R2 == 1 ? 64 : R2 == 2 ? 80 : R2 == 3 ? 112 : 160) : (R2 == 1 ? 64 : 96);
}
template <int BLK>
constexpr int kGBCols = gb_col0<BLK>(64 / BLK);
constexpr float kLowerBound32 = -5.0f;   // lower bounds >= this take the 32-row sub-blocks

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Give up a wait after the mbarrier's time limit: record it in the status
// word and in the CTA's abort flag; later waits of the CTA return at once.
__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              uint32_t *status) {
  if (*abort_flag) return;
  if (!mbar_wait(bar, parity)) {
    *abort_flag = 1;
    atomicOr(status, KDA_DEVICE_TIMEOUT);
  }
}

// 8 consecutive tokens of the thread's two key channels -> two 16-byte chunks (rows rho, 64 + rho)
__device__ __forceinline__ void pack8(const float2 (&v)[8], uint4 &lo, uint4 &hi) {
  lo = make_uint4(pack_bf16x2(v[0].x, v[1].x), pack_bf16x2(v[2].x, v[3].x), pack_bf16x2(v[4].x, v[5].x),
                  pack_bf16x2(v[6].x, v[7].x));
  hi = make_uint4(pack_bf16x2(v[0].y, v[1].y), pack_bf16x2(v[2].y, v[3].y), pack_bf16x2(v[4].y, v[5].y),
                  pack_bf16x2(v[6].y, v[7].y));
}
__device__ __forceinline__ void put8(uint8_t *tile, int R_rows, int rho, int col0, const float2 (&v)[8]) {
  uint4 lo, hi;
  pack8(v, lo, hi);
  *reinterpret_cast<uint4 *>(tile + swz_offset(R_rows, rho, col0)) = lo;
  *reinterpret_cast<uint4 *>(tile + swz_offset(R_rows, 64 + rho, col0)) = hi;
}

// 16 x 8 tile of X Y for X (16 x 8ks) and Y (8ks x 8), both fp32 with row stride kAStride, on TF32
// tensor cores; fragments in the PTX ISA m16n8k8 layout (g = lane / 4, t = lane % 4)
__device__ __forceinline__ void mm_16x8(float (&d)[4], const float *X, const float *Y, int ks, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {   // ks <= 4
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

// the same 16 x 8 tile, times sgn and the column's beta, as bf16 pairs into T (K-major, 128-byte swizzle)
__device__ __forceinline__ void st_16x8_t(uint8_t *tT, int row0, int col0, const float (&d)[4], float sgn,
                                          const float *s_beta, int lane) {
  const int g = lane >> 2, c = col0 + 2 * (lane & 3);
  const float b0 = sgn * s_beta[c], b1 = sgn * s_beta[c + 1];
  *reinterpret_cast<uint32_t *>(tT + swz_offset(64, row0 + g, c)) = pack_bf16x2(d[0] * b0, d[1] * b1);
  *reinterpret_cast<uint32_t *>(tT + swz_offset(64, row0 + g + 8, c)) = pack_bf16x2(d[2] * b0, d[3] * b1);
}

struct BlockFactors {
  float2 em;      // e^(m_R)
  float2 ems;     // scale e^(m_R)
  float2 el;      // e^(b_63 - m_R)
  float2 eg;      // e^(a_R - m_R), a_R = b at the last row of block R
  float2 cr[4];   // e^(m_R2 - a_R) for R2 > R; applied after eg, since k^ e^(a_R - b) <= |k^| keeps the
                  // product representable where eg cr alone (up to 2^-230 at lower_bound -10) is not
};

// Operand rows of 8 tokens (rows t0 .. t0+7 of block R) for key channels
// (2p, 2p+1); x[j] = (b - m_R) log2(e) of those rows.  The block's Q+ and K'
// rows come back packed (qp, kq: rows p and 64 + p) and are stored once the
// operand tiles are free.
template <int R, int BLK>
__device__ __forceinline__ void build_rows(const uint32_t (&kqw)[16], const float2 (&x)[8],
                                           int t0, int p, const float *s_nq, const float *s_nk,
                                           const BlockFactors &f, uint8_t *sm, uint4 (&qp)[2], uint4 (&kq)[2]) {
  float2 kh[8], qh[8], e[8], ie[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float nk = s_nk[t0 + j], nq = s_nq[t0 + j];
    kh[j] = mul2(unpack_bf16x2(kqw[j]), make_float2(nk, nk));
    qh[j] = mul2(unpack_bf16x2(kqw[8 + j]), make_float2(nq, nq));
    e[j] = exp2_2(x[j]);
    ie[j] = exp2_2(make_float2(-x[j].x, -x[j].y));
  }
  float2 v[8], w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = mul2(kh[j], e[j]);   // F
  put8(sm + OFF_FQ, 128, p, t0, v);
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = mul2(v[j], f.em);    // K+ = F e^(m_R)
  put8(sm + OFF_KP, 128, p, t0, w);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = mul2(qh[j], e[j]);   // Q
  put8(sm + OFF_FQ, 128, p, 64 + t0, v);
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = mul2(v[j], f.ems);   // Q+ = scale Q e^(m_R)
  pack8(w, qp[0], qp[1]);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = mul2(kh[j], ie[j]);  // G
  put8(sm + OFF_GB, 128, p, t0, v);
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = mul2(v[j], f.el);    // K' = G e^(b_63 - m_R)
  pack8(w, kq[0], kq[1]);
  if (R < 64 / BLK - 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = mul2(v[j], f.eg);  // k^ e^(a_R - b) <= |k^|
#pragma unroll
    for (int R2 = R + 1; R2 < 64 / BLK; ++R2) {           // k^ e^(m_R2 - b) for the later blocks R2
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = mul2(v[j], f.cr[R2]);
      put8(sm + OFF_GB, 128, p, gb_col0<BLK>(R2) + t0, w);
    }
  }
}

// Short causal convolution down one channel pair of a bf16 tile, in place: rows r0 .. r0+n-1 at byte offsets
// off(r) from `tile`, the raw inputs of rows r0-3 .. r0-1 in x0 .. x2 (oldest first), taps wa / wb of the two
// channels (tap 3 on the current row).  Rows at or past `valid` become 0.
template <int N, typename Off>
__device__ __forceinline__ void conv_pair(uint8_t *tile, Off off, int r0, int valid, float2 x0, float2 x1,
                                          float2 x2, float4 wa, float4 wb, bool silu) {
  // the two channels side by side in packed fp32x2 arithmetic; the N inputs first (independent loads)
  const float2 w0 = make_float2(wa.x, wb.x), w1 = make_float2(wa.y, wb.y), w2 = make_float2(wa.z, wb.z),
               w3 = make_float2(wa.w, wb.w), half2 = make_float2(0.5f, 0.5f);
  uint32_t raw[N];
#pragma unroll
  for (int i = 0; i < N; ++i) raw[i] = *reinterpret_cast<const uint32_t *>(tile + off(r0 + i));
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int r = r0 + i;
    const float2 x = unpack_bf16x2(raw[i]);
    float2 y = fma2(w3, x, fma2(w2, x2, fma2(w1, x1, mul2(w0, x0))));
    if (silu) {   // x sigmoid(x) = x/2 + x/2 tanh(x/2)
      const float2 hy = mul2(y, half2);
      float t0, t1;
      asm("tanh.approx.f32 %0, %1;" : "=f"(t0) : "f"(hy.x));
      asm("tanh.approx.f32 %0, %1;" : "=f"(t1) : "f"(hy.y));
      y = fma2(hy, make_float2(t0, t1), hy);
    }
    *reinterpret_cast<uint32_t *>(tile + off(r)) = r < valid ? pack_bf16x2(y.x, y.y) : 0u;
    x0 = x1;
    x1 = x2;
    x2 = x;
  }
}

template <int BLK, bool kConv>
__global__ void __launch_bounds__(kThreads, 2) chunk_intra_kernel(const __grid_constant__ IntraParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *small = sm + OFF_SMALL;
  float *s_nq = reinterpret_cast<float *>(small + SM_NQ);
  float *s_nk = reinterpret_cast<float *>(small + SM_NK);
  float *s_beta = reinterpret_cast<float *>(small + SM_BETA);
  float *s_h = reinterpret_cast<float *>(small + SM_H);     // [quarter][channel]: sum of lambda over 8 rows
  uint64_t *bar_in = reinterpret_cast<uint64_t *>(small + SM_BAR);
  uint64_t *bar_v = bar_in + 1;
  uint64_t *bar_mma = bar_in + 2;
  uint64_t *bar_u = reinterpret_cast<uint64_t *>(small + SM_BARU);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(small + SM_TMEM);
  volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(small + SM_ABORT);

  // every CTA of this grid has started once all have passed here: the state pass may then be scheduled onto
  // SMs this grid no longer fills (it waits for this grid's completion before reading the blocks)
  grid_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = prm.H;
  const int h = blockIdx.x % H;
  const int gslot = blockIdx.x / H;
  // the chunk slot's first token and its tokens (a broadcast load each)
  const int tok0 = prm.slot_tok0[gslot], valid = prm.slot_valid[gslot] & (kSlotFirst - 1);
  uint8_t *blk = prm.blocks + (static_cast<size_t>(gslot) * H + h) * kBlkBytes;

  // ------------------------------------------------------------ setup: barriers, TMA of q, k, g, TMEM, beta
  if (tid == 0) {
    mbar_init(bar_in, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_u, 1);
    *s_abort = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_in, 3 * 16384);
    tma_load_3d(sm + OFF_QIN, &prm.tq, 0, h, tok0, bar_in);
    tma_load_3d(sm + OFF_QIN + 8192, &prm.tq, 64, h, tok0, bar_in);
    tma_load_3d(sm + OFF_KIN, &prm.tk, 0, h, tok0, bar_in);
    tma_load_3d(sm + OFF_KIN + 8192, &prm.tk, 64, h, tok0, bar_in);
    tma_load_3d(sm + OFF_GIN, &prm.tg, 0, h, tok0, bar_in);
    tma_load_3d(sm + OFF_GIN + 8192, &prm.tg, 64, h, tok0, bar_in);
  }
  if (warp == 1) {   // TMEM by warp 1, beside thread 0's barrier set-up and TMA issue
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  // short convolutions: the 3 raw inputs before the chunk for q, k, v (the previous tokens of the sequence,
  // else the slot's window for its first chunk, else zeros) and v's taps go to shared memory; this thread's
  // q or k taps to registers (thread = tensor tid / 128, channel pair tid % 64, half of the rows)
  // (the loads are issued here and land in shared memory after the wait for q, k, g, which hides them)
  uint32_t *s_halo = reinterpret_cast<uint32_t *>(small + SM_HALO);
  float4 cwa = make_float4(0.f, 0.f, 0.f, 0.f), cwb = cwa, vw = cwa;
  constexpr int kHaloWords = 3 * 3 * 64, kHaloPerThread = (kHaloWords + kThreads - 1) / kThreads;
  uint32_t halo[kHaloPerThread];
  if (kConv) {
    const bool first = prm.slot_valid[gslot] & kSlotFirst;
    int slot = first && prm.conv_load_initial ? prm.slot_ids[prm.seq0 + prm.slot_seq[gslot]] : -1;
    if (slot >= prm.num_slots) slot = -1;   // out of range: no window is read (the state pass sets the status bit)
#pragma unroll
    for (int k = 0; k < kHaloPerThread; ++k) {
      const int i = tid + k * kThreads;
      const int m = i / 192, j = (i / 64) % 3, w = i % 64;
      uint32_t x = 0u;
      if (i < kHaloWords) {
        if (!first) {
          const uint16_t *src = m == 0 ? prm.xq : m == 1 ? prm.xk : prm.xv;
          x = *reinterpret_cast<const uint32_t *>(src + static_cast<int64_t>(tok0 - 3 + j) * prm.qkv_stride + h * kD + 2 * w);
        } else if (slot >= 0) {
          x = *reinterpret_cast<const uint32_t *>(prm.conv.window_pool +
                                                  ((static_cast<size_t>(slot) * 9 + m * 3 + j) * H + h) * kD + 2 * w);
        }
      }
      halo[k] = x;
    }
    if (tid < kD) vw = *reinterpret_cast<const float4 *>(prm.conv.weight + ((2 * static_cast<size_t>(H) + h) * kD + tid) * 4);
    const int cm = tid >> 7, c = 2 * (tid & 63);
    cwa = *reinterpret_cast<const float4 *>(prm.conv.weight + ((static_cast<size_t>(cm) * H + h) * kD + c) * 4);
    cwb = *reinterpret_cast<const float4 *>(prm.conv.weight + ((static_cast<size_t>(cm) * H + h) * kD + c + 1) * 4);
  }
  // per-thread parameters, consumed after the wait for q, k, g (their latency hides under it)
  const int p = tid & 63, sel = tid >> 6;
  const int c0 = 2 * p;
  const float2 dtb = *reinterpret_cast<const float2 *>(prm.dt_bias + h * kD + c0);
  const uint16_t beta_raw = tid < valid ? prm.beta[(size_t)(tok0 + tid) * prm.beta_stride + h] : uint16_t(0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ------------------------------------------------------------ wait for q, k, g
  wait_or_abort(bar_in, 0, s_abort, prm.status);
  if (tid < kC) s_beta[tid] = tid < valid ? sigmoid_f(bf16_bits_to_f32(beta_raw)) : 0.f;

  // ------------------------------------------------------------ short convolutions of q and k, in place
  if (kConv) {
#pragma unroll
    for (int k = 0; k < kHaloPerThread; ++k)
      if (tid + k * kThreads < kHaloWords) s_halo[tid + k * kThreads] = halo[k];
    if (tid < kD) reinterpret_cast<float4 *>(small + SM_VW)[tid] = vw;
    const int cm = tid >> 7, cp = tid & 63, half = (tid >> 6) & 1;
    uint8_t *tile = sm + (cm == 0 ? OFF_QIN : OFF_KIN);
    const int c = 2 * cp;
    auto off = [c](int r) { return in_offset(r, c); };
    uint32_t h0 = 0u, h1 = 0u, h2 = 0u;
    if (half == 1) {   // rows 29 .. 31, read before the first half overwrites them
      h0 = ld_u32(tile + off(29)); h1 = ld_u32(tile + off(30)); h2 = ld_u32(tile + off(31));
    }
    __syncthreads();
    if (half == 0) {
      h0 = s_halo[cm * 192 + cp]; h1 = s_halo[cm * 192 + 64 + cp]; h2 = s_halo[cm * 192 + 128 + cp];
    }
    conv_pair<32>(tile, off, 32 * half, valid, unpack_bf16x2(h0), unpack_bf16x2(h1), unpack_bf16x2(h2), cwa, cwb,
                  prm.conv.silu != 0);
    __syncthreads();
  }

  // ------------------------------------------------------------ l2 norms (token-major)
  {
    // thread = (row r, quarter `part` of the channels); the 16-byte chunks of a quarter are visited in a
    // rotated order so that the eight threads of each quarter-warp read eight different bank groups
    const int r = tid >> 2, part = tid & 3;
    const int rot = (r & 1) * 2 + (part >> 1);
    float2 sq = make_float2(0.f, 0.f), sk = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = 32 * part + 8 * ((j + rot) & 3);
      const uint4 wq = *reinterpret_cast<const uint4 *>(sm + OFF_QIN + in_offset(r, c));
      const uint4 wk = *reinterpret_cast<const uint4 *>(sm + OFF_KIN + in_offset(r, c));
      const uint32_t aq[4] = {wq.x, wq.y, wq.z, wq.w}, ak[4] = {wk.x, wk.y, wk.z, wk.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fq = unpack_bf16x2(aq[e]), fk = unpack_bf16x2(ak[e]);
        sq = fma2(fq, fq, sq);
        sk = fma2(fk, fk, sk);
      }
    }
    float ssq = sq.x + sq.y, ssk = sk.x + sk.y;
    ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
    ssk += __shfl_xor_sync(0xffffffffu, ssk, 1);
    ssq += __shfl_xor_sync(0xffffffffu, ssq, 2);
    ssk += __shfl_xor_sync(0xffffffffu, ssk, 2);
    if (part == 0) {
      s_nq[r] = r < valid ? rsqrtf(ssq + kL2Eps) : 0.f;
      s_nk[r] = r < valid ? rsqrtf(ssk + kL2Eps) : 0.f;
    }
  }

  // ------------------------------------------------------------ gate and in-block decays
  // thread = (channel pair p, two 8-row quarters of the chunk); warp-uniform quarters.  16-row blocks: the
  // half `hf` of blocks Ra and Rb = 3 - Ra; 32-row blocks: quarter `sel` of both blocks.  A quarter before
  // its block's anchor takes its exponents as suffix sums up to its own last row, one after it as prefix sums
  // from its own first row; with 32-row blocks the outer quarters then add a neighbour quarter's sum.
  const int hf = sel & 1, Ra = sel >> 1, Rb = 3 - Ra;
  const bool before = BLK == 16 ? hf == 0 : sel < 2;
  const float nea = -__expf(prm.A_log[h]) * kLog2e;   // lambda = lb sigmoid(ea (g + dtb)); log2 units below
  const float lb2 = prm.lower_bound * kLog2e;
  const float2 nd = make_float2(nea * dtb.x, nea * dtb.y);
  const float2 nea2 = make_float2(nea, nea), lb22 = make_float2(lb2, lb2), one2 = make_float2(1.f, 1.f);
  float2 x[2][8];   // (b_t - m_R) log2(e), rows t0 .. t0+7 of each of the two blocks
  // the thread's k and q words and its decay exponents of each block wait in TMEM (its lane; columns 0..127,
  // 16 per block and kind) until the operand tiles are built: the input tiles are overwritten there, and
  // registers are short
  const uint32_t stash = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 32 * (warp >> 2);
#pragma unroll
  for (int bi = 0; bi < 2; ++bi) {
    const int R = BLK == 16 ? (bi ? Rb : Ra) : bi;
    const int qd = BLK == 16 ? 2 * R + hf : 4 * bi + sel;   // the quarter: rows 8 qd .. 8 qd + 7
    const int t0 = 8 * qd;
    float2 lam[8];
    uint32_t kq[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = t0 + j;
      const uint32_t off = in_offset(r, c0);
      kq[j] = ld_u32(sm + OFF_KIN + off);
      kq[8 + j] = ld_u32(sm + OFF_QIN + off);
      const float2 gg = unpack_bf16x2(ld_u32(sm + OFF_GIN + off));
      // lambda = lb2 / (1 + 2^(nea g + nea dtb)), channel pairs in packed fp32x2
      const float2 ex = exp2_2(fma2(gg, nea2, nd));
      const float2 den = fma2(ex, one2, one2);
      const float2 l = mul2(make_float2(fast_rcp(den.x), fast_rcp(den.y)), lb22);
      lam[j] = r < valid ? l : make_float2(0.f, 0.f);
    }
    float2 hs;
    if (before) {    // rows 0..7 of the quarter: b_t - (b at its last row) = -(lambda_{t+1} + ... + lambda_7)
      x[bi][7] = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 6; j >= 0; --j) x[bi][j] = make_float2(x[bi][j + 1].x - lam[j + 1].x, x[bi][j + 1].y - lam[j + 1].y);
      hs = make_float2(lam[0].x - x[bi][0].x, lam[0].y - x[bi][0].y);
    } else {         // b_t - (b before its first row) = lambda_0 + ... + lambda_t
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc = make_float2(acc.x + lam[j].x, acc.y + lam[j].y);
        x[bi][j] = acc;
      }
      hs = acc;
    }
    *reinterpret_cast<float2 *>(s_h + qd * kD + c0) = hs;   // the quarter's sum
    tmem_st16(stash + 16 * bi, kq);
    tmem_st16(stash + 64 + 16 * bi, reinterpret_cast<const float *>(x[bi]));
  }
  tmem_wait_st();
  __syncthreads();   // norms, half sums visible; q, k, g tiles fully read

  // ------------------------------------------------------------ anchors and operand tiles
  uint4 qp[2][2], kq[2][2];   // packed Q+ / K' rows of the thread's two quarters
  {
    // the k and q words and the exponents of quarter bi back from TMEM (exponents shifted by xoff)
    auto words = [&](int bi, uint32_t (&kqw)[16], float2 xoff) {
      uint32_t xw[16];
      tmem_ld16_async(stash + 16 * bi, kqw);
      tmem_ld16_async(stash + 64 + 16 * bi, xw);
      tmem_wait_ld();
      tmem_tie<16>(kqw);
      tmem_tie<16>(xw);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        x[bi][j] = make_float2(__uint_as_float(xw[2 * j]) + xoff.x, __uint_as_float(xw[2 * j + 1]) + xoff.y);
    };
    auto gamma_out = [&](float2 tot) {   // gamma = e^(b_63) for rho = p and 64 + p
      if (sel == 0) {
        float *gam = reinterpret_cast<float *>(blk + kBlkGamma);
        gam[p] = fast_exp2(tot.x);
        gam[64 + p] = fast_exp2(tot.y);
      }
    };
    using R0 = std::integral_constant<int, 0>;
    using R1 = std::integral_constant<int, 1>;
    using R2c = std::integral_constant<int, 2>;
    using R3 = std::integral_constant<int, 3>;
    const float2 zero2 = make_float2(0.f, 0.f);
    uint32_t kqw[16];
    if constexpr (BLK == 16) {
      float2 hh[2][4];   // half sums of block I: rows 0..7 (hh[0]) and 8..15 (hh[1])
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        hh[0][I] = *reinterpret_cast<const float2 *>(s_h + (2 * I) * kD + c0);
        hh[1][I] = *reinterpret_cast<const float2 *>(s_h + (2 * I + 1) * kD + c0);
      }
      float2 m[4], a[4], tot = zero2;   // anchors (b at row 7 of each block) and block ends (row 15)
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        m[I] = make_float2(tot.x + hh[0][I].x, tot.y + hh[0][I].y);
        a[I] = make_float2(m[I].x + hh[1][I].x, m[I].y + hh[1][I].y);
        tot = a[I];
      }
      gamma_out(tot);
      // the factors of block R (a compile-time block index, so only the later blocks' factors exist)
      auto factors = [&](auto Rc) {
        constexpr int R = decltype(Rc)::value;
        BlockFactors f;
        f.em = exp2_2(m[R]);
        f.ems = make_float2(f.em.x * prm.scale, f.em.y * prm.scale);
        f.el = exp2_2(make_float2(tot.x - m[R].x, tot.y - m[R].y));
        f.eg = exp2_2(hh[1][R]);
#pragma unroll
        for (int R2 = R + 1; R2 < 4; ++R2)
          f.cr[R2] = exp2_2(make_float2(fminf(m[R2].x - a[R].x, 0.f), fminf(m[R2].y - a[R].y, 0.f)));
        return f;
      };
      if (Ra == 0) {
        words(0, kqw, zero2);
        build_rows<0, 16>(kqw, x[0], 8 * hf, p, s_nq, s_nk, factors(R0{}), sm, qp[0], kq[0]);
        words(1, kqw, zero2);
        build_rows<3, 16>(kqw, x[1], 48 + 8 * hf, p, s_nq, s_nk, factors(R3{}), sm, qp[1], kq[1]);
      } else {
        words(0, kqw, zero2);
        build_rows<1, 16>(kqw, x[0], 16 + 8 * hf, p, s_nq, s_nk, factors(R1{}), sm, qp[0], kq[0]);
        words(1, kqw, zero2);
        build_rows<2, 16>(kqw, x[1], 32 + 8 * hf, p, s_nq, s_nk, factors(R2c{}), sm, qp[1], kq[1]);
      }
    } else {
      float2 sq[8];   // quarter sums
#pragma unroll
      for (int q = 0; q < 8; ++q) sq[q] = *reinterpret_cast<const float2 *>(s_h + q * kD + c0);
      auto add = [](float2 u, float2 v) { return make_float2(u.x + v.x, u.y + v.y); };
      // anchors m_R = b at row 15 of block R, block ends a_R = b at its row 31
      const float2 m0 = add(sq[0], sq[1]);
      const float2 a0 = add(add(m0, sq[2]), sq[3]);
      const float2 m1 = add(add(a0, sq[4]), sq[5]);
      const float2 tot = add(add(m1, sq[6]), sq[7]);
      gamma_out(tot);
      auto factors = [&](auto Rc) {
        constexpr int R = decltype(Rc)::value;
        const float2 mR = R ? m1 : m0, aR = R ? tot : a0;
        BlockFactors f;
        f.em = exp2_2(mR);
        f.ems = make_float2(f.em.x * prm.scale, f.em.y * prm.scale);
        f.el = exp2_2(make_float2(tot.x - mR.x, tot.y - mR.y));
        f.eg = exp2_2(make_float2(aR.x - mR.x, aR.y - mR.y));
        if (R == 0) f.cr[1] = exp2_2(make_float2(fminf(m1.x - a0.x, 0.f), fminf(m1.y - a0.y, 0.f)));
        return f;
      };
      // quarter sel of each block: the outer quarters measure from the neighbour quarter's far end
      auto xoff = [&](int R) {
        return sel == 0 ? make_float2(-sq[4 * R + 1].x, -sq[4 * R + 1].y) : sel == 3 ? sq[4 * R + 2] : zero2;
      };
      words(0, kqw, xoff(0));
      build_rows<0, 32>(kqw, x[0], 8 * sel, p, s_nq, s_nk, factors(R0{}), sm, qp[0], kq[0]);
      words(1, kqw, xoff(1));
      build_rows<1, 32>(kqw, x[1], 32 + 8 * sel, p, s_nq, s_nk, factors(R1{}), sm, qp[1], kq[1]);
    }
    // the packed Q+ and K' rows wait in TMEM columns 160..223 (beside the product's 160) until the
    // operand tiles are free
    tmem_st16(stash + 160, reinterpret_cast<const uint32_t *>(qp));
    tmem_st16(stash + 176, reinterpret_cast<const uint32_t *>(kq));
    tmem_wait_st();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------------------ A/P product (one 128 x 160 or 128 x 96 tcgen05.mma)
  if (tid == 0) {
    tc_fence_after();
    const uint64_t fq = desc_mnmajor_base(smem_u32(sm + OFF_FQ), 128);
    const uint64_t gb = desc_mnmajor_base(smem_u32(sm + OFF_GB), 128);
    const uint32_t id = idesc_bf16(128, kGBCols<BLK>, true, true);
#pragma unroll
    for (int s = 0; s < 8; ++s) mma_bf16(tmem, fq + mnmajor_step(s), gb + mnmajor_step(s), id, s > 0);
    mma_commit(bar_mma);
    // under the product: the CTA that starts about one wave after this one will find its q, k, v, g in L2
    const int nb = static_cast<int>(blockIdx.x) + prm.prefetch_ahead;
    if (prm.prefetch_ahead > 0 && nb < static_cast<int>(gridDim.x)) {
      const int t2 = prm.slot_tok0[nb / H], h2 = nb % H;
#pragma unroll
      for (int x = 0; x < 128; x += 64) {
        tma_prefetch_3d(&prm.tq, x, h2, t2);
        tma_prefetch_3d(&prm.tk, x, h2, t2);
        tma_prefetch_3d(&prm.tg, x, h2, t2);
        tma_prefetch_3d(&prm.tv, x, h2, t2);
      }
    }
  }
  __syncwarp();
  wait_or_abort(bar_mma, 0, s_abort, prm.status);
  tc_fence_after();
  if (tid == 0) {   // the operand tiles are free: v may land
    mbar_arrive_expect_tx(bar_v, 16384);
    tma_load_3d(sm + OFF_VIN, &prm.tv, 0, h, tok0, bar_v);
    tma_load_3d(sm + OFF_VIN + 8192, &prm.tv, 64, h, tok0, bar_v);
  }
  // the block's Q+ and K' rows go to their staging tiles
  {
    uint32_t w[32];
    tmem_ld16_async(stash + 160, w);
    tmem_ld16_async(stash + 176, w + 16);
    tmem_wait_ld();
    tmem_tie<32>(w);
    const uint4 *wq = reinterpret_cast<const uint4 *>(w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      (&qp[0][0])[i] = wq[i];
      (&kq[0][0])[i] = wq[4 + i];
    }
  }
#pragma unroll
  for (int bi = 0; bi < 2; ++bi) {
    const int t0 = BLK == 16 ? 16 * (bi ? Rb : Ra) + 8 * hf : 32 * bi + 8 * sel;
    *reinterpret_cast<uint4 *>(sm + OFF_QST + swz_offset(128, p, t0)) = qp[bi][0];
    *reinterpret_cast<uint4 *>(sm + OFF_QST + swz_offset(128, 64 + p, t0)) = qp[bi][1];
    *reinterpret_cast<uint4 *>(sm + OFF_PKST + swz_offset(kBlkPKRows, 64 + p, t0)) = kq[bi][0];
    *reinterpret_cast<uint4 *>(sm + OFF_PKST + swz_offset(kBlkPKRows, 128 + p, t0)) = kq[bi][1];
  }

  // ------------------------------------------------------------ A (fp32) and P (bf16 block rows) from TMEM
  {
    // lanes 0..63 of the product hold rows of A (k side), lanes 64..127 rows of P (q side)
    const int q4 = warp & 3, ib = warp >> 2;
    const bool is_p = q4 >= 2;                 // warp-uniform
    const int r = (q4 & 1) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const float bscale = is_p ? prm.scale : s_beta[r];
    float *sA = reinterpret_cast<float *>(sm + OFF_A);
    // column i of a row is kept iff i < r (A) or i <= r (P); this also zeroes the blocks above the diagonal,
    // whose registers are never loaded
    if constexpr (BLK == 16) {
      const int Ra2 = (q4 & 1) * 2;              // row blocks of this warp: Ra2 (lanes 0..15), Ra2 + 1
      const bool upper = lane >= 16;
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int I = 2 * ib + ii;   // column block
        // source columns of the two row blocks (warp-uniform); -1: the block is above the diagonal
        const int srcA = (I == Ra2) ? 16 * I : (I < Ra2) ? gb_col0<16>(Ra2) + 16 * I : -1;
        const int srcB = (I == Ra2 + 1) ? 16 * I : (I < Ra2 + 1) ? gb_col0<16>(Ra2 + 1) + 16 * I : -1;
        uint32_t va[16], vb[16];
        if (srcA >= 0) tmem_ld16_async(tmem + lane_base + srcA, va);
        if (srcB >= 0) tmem_ld16_async(tmem + lane_base + srcB, vb);
        tmem_wait_ld();
        tmem_tie<16>(va);
        tmem_tie<16>(vb);
        const int lim = r - 16 * I + (is_p ? 1 : 0);
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float raw = __uint_as_float(upper ? vb[e] : va[e]);
          v[e] = e < lim ? raw * bscale : 0.f;
        }
        if (is_p) {
#pragma unroll
          for (int k8 = 0; k8 < 2; ++k8)
            *reinterpret_cast<uint4 *>(sm + OFF_PKST + swz_offset(kBlkPKRows, r, 16 * I + 8 * k8)) =
                make_uint4(pack_bf16x2(v[8 * k8], v[8 * k8 + 1]), pack_bf16x2(v[8 * k8 + 2], v[8 * k8 + 3]),
                           pack_bf16x2(v[8 * k8 + 4], v[8 * k8 + 5]), pack_bf16x2(v[8 * k8 + 6], v[8 * k8 + 7]));
        } else {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4 *>(sA + r * kAStride + 16 * I + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
    } else {
      // 32-row blocks: the warp's lanes are one row block R; ib picks the 32-column block I
      const int R = q4 & 1, I = ib;
      const int src = I == R ? 32 * I : I < R ? gb_col0<32>(R) + 32 * I : -1;
      uint32_t va[32];
      if (src >= 0) {
        tmem_ld16_async(tmem + lane_base + src, va);
        tmem_ld16_async(tmem + lane_base + src + 16, va + 16);
      }
      tmem_wait_ld();
      tmem_tie<32>(va);
      const int lim = r - 32 * I + (is_p ? 1 : 0);
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = e < lim ? __uint_as_float(va[e]) * bscale : 0.f;
      if (is_p) {
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8)
          *reinterpret_cast<uint4 *>(sm + OFF_PKST + swz_offset(kBlkPKRows, r, 32 * I + 8 * k8)) =
              make_uint4(pack_bf16x2(v[8 * k8], v[8 * k8 + 1]), pack_bf16x2(v[8 * k8 + 2], v[8 * k8 + 3]),
                         pack_bf16x2(v[8 * k8 + 4], v[8 * k8 + 5]), pack_bf16x2(v[8 * k8 + 6], v[8 * k8 + 7]));
      } else {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4 *>(sA + r * kAStride + 32 * I + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------------------ T = (I + A)^-1 Diag(beta)
  // Blocked inverse of the unit-lower L = I + A in fp32, 16x16 blocks D_R = L_RR^-1:
  //   L^-1_10 = -D_1 A_10 D_0,  L^-1_32 = -D_3 A_32 D_2,
  //   L^-1 (rows 32..63, cols 0..31) = -I_2 A_(23,01) I_1,  I_1, I_2 the inverses of the diagonal 32x32 halves.
  // Everything happens in place in the A tile: each block of the inverse overwrites the block of A
  // that is no longer needed, and the temporaries live in its unused strictly-upper part.  Each step also
  // writes its block of T = L^-1 Diag(beta) in bf16; the six blocks above the diagonal of T are zero.
  {
    float *sA = reinterpret_cast<float *>(sm + OFF_A);
    float *sInv = sA;
    uint8_t *tT = sm + OFF_T;
    if (tid < 192) {   // zero blocks (I, J), J > I: 6 blocks x 16 rows x two 16-byte chunks
      const int b6 = tid >> 5, rr = (tid >> 1) & 15, hc = tid & 1;
      const int I = b6 < 3 ? 0 : b6 < 5 ? 1 : 2;
      const int J = b6 < 3 ? b6 + 1 : b6 < 5 ? b6 - 1 : 3;
      *reinterpret_cast<uint4 *>(tT + swz_offset(64, 16 * I + rr, 16 * J + 8 * hc)) = make_uint4(0, 0, 0, 0);
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
      const float bc = s_beta[16 * R + jc];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sInv[(16 * R + 4 * i + q) * kAStride + 16 * R + jc] = xs[i];
        *reinterpret_cast<uint16_t *>(tT + swz_offset(64, 16 * R + 4 * i + q, 16 * R + jc)) =
            f32_to_bf16_bits(xs[i] * bc);
      }
    }
    __syncthreads();
    // Every block product below is a set of 16 x 8 output tiles, one per warp task, on TF32
    // tensor cores (mma.sync m16n8k8) with fp32 accumulation.
    // Y_1 = A_10 D_0 -> A tile rows 0..15, cols 16..31;  Y_3 = A_32 D_2 -> rows 32..47, cols 48..63;
    // then L^-1_10 = -D_1 Y_1 -> sInv rows 16..31, cols 0..15;  L^-1_32 = -D_3 Y_3 -> rows 48..63, cols 32..47.
    // A warp's output tile needs only its own Y tile; the pair barrier keeps A_10 (A_32) intact until both
    // warps of the pair have read it.
    if (warp < 4) {
      const int lo = warp < 2 ? 0 : 32, nj = warp & 1;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mm_16x8(d, sA + (lo + 16) * kAStride + lo, sInv + lo * kAStride + lo + 8 * nj, 2, lane);
      st_16x8(sA + lo * kAStride + lo + 16 + 8 * nj, d, 1.f, lane);
      if (warp < 2) named_bar_sync<5>(64); else named_bar_sync<6>(64);
      float e[4] = {0.f, 0.f, 0.f, 0.f};
      mm_16x8(e, sInv + (lo + 16) * kAStride + lo + 16, sA + lo * kAStride + lo + 16 + 8 * nj, 2, lane);
      st_16x8(sInv + (lo + 16) * kAStride + lo + 8 * nj, e, -1.f, lane);
      st_16x8_t(tT, lo + 16, lo + 8 * nj, e, -1.f, s_beta, lane);
    } else if (tid == kCopyThread) {   // idle in this step: the Q+ and [P ; K'] rows (complete) to the block
      bulk_store(blk + kBlkWQ + 16384, sm + OFF_QST, 16384);
      bulk_store(blk + kBlkPK, sm + OFF_PKST, kBlkPKRows * 128);
      bulk_commit();
    }
    __syncthreads();
    // Z = A_(23,01) I_1 (32 x 32) -> A tile rows 0..31, cols 32..63; warp = (16-row half mi, 8 columns nj).
    // I_1 is block-lower: columns 16..31 only see its rows 16..31.
    {
      const int mi = warp >> 2, nj = warp & 3;
      const int k0 = nj < 2 ? 0 : 16;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mm_16x8(d, sA + (32 + 16 * mi) * kAStride + k0, sInv + k0 * kAStride + 8 * nj, (32 - k0) / 8, lane);
      st_16x8(sA + (16 * mi) * kAStride + 32 + 8 * nj, d, 1.f, lane);
    }
    __syncthreads();
    // L^-1 (rows 32..63, cols 0..31) = -I_2 Z; I_2 is block-lower: its rows 0..15 only see Z rows 0..15.
    // Only T is written: nothing reads this block of the inverse afterwards.
    {
      const int mi = warp >> 2, nj = warp & 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mm_16x8(d, sInv + (32 + 16 * mi) * kAStride + 32, sA + 32 + 8 * nj, mi ? 4 : 2, lane);
      st_16x8_t(tT, 32 + 16 * mi, 8 * nj, d, -1.f, s_beta, lane);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------------------ W^T = K+^T T^T, U^^T = V^T T^T
  // W^T (which needs no v) commits onto bar_mma, U^^T onto bar_u; each half of the warps then stages and
  // stores its own rows, so W^T leaves while U^^T is still being formed
  const bool ragged = valid < kC;
  if (kConv) {   // v's short convolution, in place in its swizzled operand tile (rows past the end become 0)
    wait_or_abort(bar_v, 0, s_abort, prm.status);
    const int cp = tid & 63, quarter = tid >> 6, c = 2 * cp;
    auto off = [c](int r) { return swz_offset(64, r, c); };
    const float4 *s_vw = reinterpret_cast<const float4 *>(small + SM_VW);
    const float4 wa = s_vw[c], wb = s_vw[c + 1];
    uint8_t *tile = sm + OFF_VIN;
    uint32_t h0, h1, h2;
    if (quarter == 0) {
      h0 = s_halo[2 * 192 + cp]; h1 = s_halo[2 * 192 + 64 + cp]; h2 = s_halo[2 * 192 + 128 + cp];
    } else {
      const int r0 = 16 * quarter;
      h0 = ld_u32(tile + off(r0 - 3)); h1 = ld_u32(tile + off(r0 - 2)); h2 = ld_u32(tile + off(r0 - 1));
    }
    __syncthreads();
    conv_pair<16>(tile, off, 16 * quarter, valid, unpack_bf16x2(h0), unpack_bf16x2(h1), unpack_bf16x2(h2), wa, wb,
                  prm.conv.silu != 0);
    fence_async_smem();
    __syncthreads();
  } else if (ragged) {   // rows past the sequence end: T's columns there are 0, but v may hold anything
    wait_or_abort(bar_v, 0, s_abort, prm.status);
    for (int idx = tid; idx < (kC - valid) * 16; idx += kThreads) {
      const int r2 = valid + idx / 16, cc = idx % 16;
      *reinterpret_cast<uint4 *>(sm + OFF_VIN + swz_offset(64, r2, 8 * cc)) = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    __syncthreads();
  }
  if (tid == 0) {
    tc_fence_after();
    const uint32_t id_w = idesc_bf16(128, 64, false, false);
    const uint32_t id_u = idesc_bf16(128, 64, true, false);
    const uint64_t kp = desc_kmajor_base(smem_u32(sm + OFF_KP));
    const uint64_t vv = desc_mnmajor_base(smem_u32(sm + OFF_VIN), 64);
    const uint64_t tt = desc_kmajor_base(smem_u32(sm + OFF_T));
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_bf16(tmem, kp + kmajor_step(128, s), tt + kmajor_step(64, s), id_w, s > 0);
    mma_commit(bar_mma);
    if (!ragged && !kConv) wait_or_abort(bar_v, 0, s_abort, prm.status);
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_bf16(tmem + 64, vv + mnmajor_step(s), tt + kmajor_step(64, s), id_u, s > 0);
    mma_commit(bar_u);
  }
  __syncwarp();
  // ------------------------------------------------------------ W^T, U^^T rows to the staging tiles
  {
    // warp = (lane quadrant, W^T | U^^T); the thread's row is one 128-byte line of the block tile
    const int q4 = warp & 3, which = warp >> 2;
    if (which) wait_or_abort(bar_u, 0, s_abort, prm.status); else wait_or_abort(bar_mma, 1, s_abort, prm.status);
    tc_fence_after();
    const int row = q4 * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + (which ? 64u : 0u);
    uint32_t v[64];
#pragma unroll
    for (int k = 0; k < 4; ++k) tmem_ld16_async(taddr + 16 * k, v + 16 * k);
    tmem_wait_ld();
    tmem_tie<64>(v);
    uint8_t *dst = sm + (which ? OFF_UST : OFF_WST);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float *f = reinterpret_cast<const float *>(v + 8 * k);
      *reinterpret_cast<uint4 *>(dst + swz_offset(128, row, 8 * k)) =
          make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                     pack_bf16x2(f[6], f[7]));
    }
    // ------------------------------------------------------------ block write-out, TMEM release
    // the warp's 32 staged rows are one contiguous 4 KB piece of the tile and of the block: it leaves at once
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      bulk_store(blk + (which ? kBlkUH : kBlkWQ) + q4 * 4096, dst + q4 * 4096, 4096);
      bulk_commit();
    }
  }
  __syncthreads();   // every TMEM read is done
  if (warp == 1) {   // the allocating warp, before its wait for its bulk store
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (lane == 0) bulk_wait_read();   // (the copy thread's wait also covers its earlier Q+ and [P ; K'] stores)
  // launched behind a state pass (a split prefill schedule): the CTA that finishes last waits for that grid's
  // completion, so that this grid completes after it (the next state pass waits for this grid and reads the state
  // the previous one wrote); it then clears the counter for the next call
  if (prm.done_counter && tid == 0 && atomicAdd(prm.done_counter, 1u) == gridDim.x - 1) {
    grid_dependency_wait();
    *prm.done_counter = 0;
  }
  // ------------------------------------------------------------ end
}

}  // namespace

cudaError_t launch_chunk_intra(const IntraParams &p, int num_chunks, cudaStream_t stream, bool programmatic) {
  if (num_chunks <= 0) return cudaSuccess;
  static std::mutex mu;
  static uint64_t done = 0;
  if (const cudaError_t e = set_attributes_once(mu, done, [] {
        cudaError_t r = cudaSuccess;
        for (auto fn : {chunk_intra_kernel<16, false>, chunk_intra_kernel<32, false>, chunk_intra_kernel<16, true>,
                        chunk_intra_kernel<32, true>})
          if (r == cudaSuccess) r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        return r;
      }))
    return e;
  const bool blk32 = p.lower_bound >= kLowerBound32, conv = p.conv.weight != nullptr;
  auto fn = blk32 ? (conv ? chunk_intra_kernel<32, true> : chunk_intra_kernel<32, false>)
                  : (conv ? chunk_intra_kernel<16, true> : chunk_intra_kernel<16, false>);
  if (!programmatic) {
    fn<<<num_chunks * p.H, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  }
  // a programmatic dependent of the preceding state pass: CTAs are scheduled onto the SMs that grid leaves free
  // once each of its CTAs has started
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_chunks * p.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace kda
