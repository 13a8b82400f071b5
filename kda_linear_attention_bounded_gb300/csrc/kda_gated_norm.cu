// Sigmoid-gated RMSNorm of stored output rows, in place: the norm of the prefill's rows.
//
// ("sigmoid RMSNorm" / "gated norm" on BF16 D = 128 rows with output and rstd compared: sglang PR #42489
// "Improve GLM-5.3-Flash DFlash decoding on B300", Modifications and review thread.)  Per (row, head):
//   rstd = 1 / sqrt(mean_c o_c^2 + eps),  y_c = o_c * rstd * w_c * sigmoid(z_c)
//
// The state pass of the prefill is a latency-bound chain on one CTA per SM; per-element work in its output
// epilogue lengthens every chunk of the chain (measured: +109 us on 8 x 2048 tokens, H = 16).  This pass instead
// runs over the stored bf16 rows on every SM at HBM speed: 16 lanes per (row, head), 16 bytes of o and of the
// gate per lane, so a warp moves two 256-byte rows of each.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr int kItemsPerCta = kThreads / 16;   // (row, head) items

__global__ void __launch_bounds__(kThreads) gated_norm_kernel(GatedNormArgs p) {
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kItemsPerCta + (threadIdx.x >> 4);
  const int cc = threadIdx.x & 15;
  const bool live = item < static_cast<int64_t>(p.num_tokens) * p.H;
  const int64_t tok = live ? item / p.H : 0;
  const int h = live ? static_cast<int>(item % p.H) : 0;
  int64_t row = tok;
  if (live && p.row_index) row = p.row_index[tok];
  const bool ok = live && row >= 0 && row < p.num_rows;
  // a bad row index was reported by the kernel that stored the row (or skipped it): nothing to normalise here
  uint4 piece = make_uint4(0u, 0u, 0u, 0u), zp = make_uint4(0u, 0u, 0u, 0u);
  uint16_t *dst = nullptr;
  if (ok) {
    dst = p.out + row * p.out_stride + h * kD + 8 * cc;
    piece = *reinterpret_cast<const uint4 *>(dst);
    zp = *reinterpret_cast<const uint4 *>(p.norm.gate + row * p.norm.gate_stride + h * kD + 8 * cc);
  }
  const float4 wa = *reinterpret_cast<const float4 *>(p.norm.weight + 8 * cc);
  const float4 wb = *reinterpret_cast<const float4 *>(p.norm.weight + 8 * cc + 4);
  const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
  const uint32_t pw[4] = {piece.x, piece.y, piece.z, piece.w};
  const uint32_t zw[4] = {zp.x, zp.y, zp.z, zp.w};
  float o[8], ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = unpack_bf16x2(pw[e]);
    o[2 * e] = x.x;
    o[2 * e + 1] = x.y;
    ss = fmaf(x.x, x.x, fmaf(x.y, x.y, ss));
  }
  // the 16 lanes of a (row, head) are 16 consecutive lanes of one warp
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rstd = rsqrtf(ss * (1.0f / kD) + p.norm.eps);
  uint32_t yw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 z = unpack_bf16x2(zw[e]);
    yw[e] = pack_bf16x2(o[2 * e] * rstd * w[2 * e] * sigmoid_f(z.x),
                        o[2 * e + 1] * rstd * w[2 * e + 1] * sigmoid_f(z.y));
  }
  if (ok) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
    if (cc == 0 && p.norm.rstd) p.norm.rstd[row * p.H + h] = rstd;
  }
}

}  // namespace

cudaError_t launch_gated_norm(const GatedNormArgs &args, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(args.num_tokens) * args.H;
  if (items <= 0 || !args.norm.gate) return cudaSuccess;
  const int64_t grid = (items + kItemsPerCta - 1) / kItemsPerCta;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  gated_norm_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace kda
