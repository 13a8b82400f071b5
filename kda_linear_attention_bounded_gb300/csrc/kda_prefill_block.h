// The per-(chunk, head) block that the intra-chunk kernel hands to the state
// pass of the chunked prefill.  Every tile is stored as the exact byte image
// of a 128-byte row-swizzled shared-memory operand (see kda_sm100.cuh), so the
// state pass fetches a block with plain bulk copies and feeds it to tcgen05.mma
// as is.
//
// Key channels are stored in the "paired" order rho: row rho < 64 holds key
// channel 2*rho, row 64 + rho holds key channel 2*rho + 1 (kd_of_rho).  A
// contraction over key channels does not depend on their order, and the state
// pass keeps its state columns in the same order (it permutes only when it
// reads or writes a state in the caller's layout).
//
// With b_t the cumulative log-decay of token t inside the chunk, k^, q^ the
// l2-normalised keys / queries, T = (I + A)^-1 Diag(beta) the chunk's WY
// factor and `scale` the output scale:
//   WQ     [W^T | Q+^T]: 128 rows rho x (64 + 64) tokens, MN-major B operand
//          W = T (k^ o e^b), Q+ = scale * q^ o e^b
//   UH     U^^T = (T V)^T: 128 value-channel rows x 64 tokens
//   PK     [P ; K'^T] K-major: rows 0..63 P[t][i] = scale * q^_t . k^_i e^(b_t - b_i) (i <= t),
//          rows 64 + rho: K'[i][rho] = k^_i e^(b_63 - b_i)
//   GAMMA  e^(b_63) per key channel rho, fp32
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace kda {

constexpr int kChunk = 64;
constexpr uint32_t kBlkWQ = 0;
constexpr uint32_t kBlkUH = 32768;
constexpr uint32_t kBlkPK = 49152;
constexpr uint32_t kBlkPKRows = 192;
constexpr uint32_t kBlkGamma = 73728;
constexpr uint32_t kBlkBytes = 74240;
// Device status word and padding in front of the blocks.
constexpr size_t kWorkspaceHeader = 1024;

__host__ __device__ constexpr int kd_of_rho(int rho) { return rho < 64 ? 2 * rho : 2 * (rho - 64) + 1; }
__host__ __device__ constexpr int rho_of_kd(int c) { return (c & 1) ? 64 + (c >> 1) : (c >> 1); }

}  // namespace kda
