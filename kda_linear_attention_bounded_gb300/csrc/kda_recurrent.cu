// Token-by-token KDA recurrence on CUDA cores: the speculative-verify kernel.
//
// Verify (TensorRT-LLM PR #21179 "GLM-5.3-Flash FP8 performance fixes on
// Hopper", commit fusing the verify loop): one launch seeds every (request,
// head) from the pooled fp32 state, runs the T draft tokens and writes the
// state after each token to intermediate_states[b, t]; the pool is only read.
//
// The work is HBM-bound: per (request, head) it reads 64 KiB of state and
// writes T x 64 KiB of per-step states.  Layout per CTA (one (b, h) pair,
// 256 threads = 8 warps): warp w owns key channels c = 16w .. 16w+15, lane l
// owns value channels d = 4l .. 4l+3, so every row of S moves as one
// coalesced 512-byte warp access of 16-byte vectors (loads of the pool,
// streaming stores of the per-step states).
//
// Per token the state update is rewritten so that ONE cross-warp reduction
// serves both the correction and the output:
//   u   = beta (v - S^T (alpha o k^))
//   o   = scale (S^T (alpha o q^) + (k^ . q^) u)          [= scale S_t^T q^]
//   S_t = Diag(alpha) S + k^ u^T
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = kWarps;      // tokens prepared per prologue pass (one per warp)
constexpr int kRows = kD / kWarps;  // key channels per warp (16)

// kVC consecutive floats (4, 2 or 1) as one load / store
template <int kVC>
__device__ __forceinline__ void load_vc(float *d, const float *src) {
  if constexpr (kVC == 4) {
    const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
    d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
  } else if constexpr (kVC == 2) {
    const float2 x = __ldg(reinterpret_cast<const float2 *>(src));
    d[0] = x.x; d[1] = x.y;
  } else {
    d[0] = __ldg(src);
  }
}
template <int kVC, bool kStream>
__device__ __forceinline__ void store_vc(float *dst, const float *v) {
  if constexpr (kVC == 4) {
    const float4 x = make_float4(v[0], v[1], v[2], v[3]);
    if (kStream) __stcs(reinterpret_cast<float4 *>(dst), x); else *reinterpret_cast<float4 *>(dst) = x;
  } else if constexpr (kVC == 2) {
    const float2 x = make_float2(v[0], v[1]);
    if (kStream) __stcs(reinterpret_cast<float2 *>(dst), x); else *reinterpret_cast<float2 *>(dst) = x;
  } else {
    if (kStream) __stcs(dst, v[0]); else *dst = v[0];
  }
}

// One work item: (request, head) and, with kP > 1, one of kP slices of the value channels (the columns of S are
// independent in the recurrence; every slice recomputes the key side).  Every return is taken by the whole CTA.
// The optional short convolutions and output norm are compile-time switches, so the plain call carries none of
// their code; they need whole rows (kP == 1).
template <bool kConv, bool kNorm, int kP>
__device__ __forceinline__ void recurrent_item(const RecurrentArgs &p) {
  static_assert(kP == 1 || (!kConv && !kNorm), "the value-channel split is for the plain call");
  constexpr int kVC = 4 / kP;          // value channels per lane
  constexpr int kCols = kD / kP;       // value channels per CTA
  __shared__ __align__(16) float s_khat[kTile][kD];
  __shared__ __align__(16) float s_kalpha[kTile][kD];
  __shared__ __align__(16) float s_qalpha[kTile][kD];
  __shared__ __align__(16) float s_alpha[kTile][kD];
  __shared__ __align__(16) float s_v[kTile][kD];
  __shared__ float s_beta[kTile], s_kq[kTile];
  __shared__ int64_t s_row[kTile];   // output row of each token of the tile
  __shared__ __align__(16) float s_gz[kTile][kD];   // sigmoid of the output norm's gate (with a norm)
  __shared__ float s_sq[4];                           // per-warp sums of o^2 (with a norm)
  __shared__ __align__(16) float s_redk[kWarps][kD];
  __shared__ __align__(16) float s_redq[kWarps][kD];
  __shared__ __align__(16) float s_u[kD];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = blockIdx.x % kP;
  const int h = (blockIdx.x / kP) % p.H;
  const int n = blockIdx.x / (kP * p.H);
  const int t_begin = p.cu_seqlens ? p.cu_seqlens[n] : n * p.T;
  const int t_end = p.cu_seqlens ? p.cu_seqlens[n + 1] : (n + 1) * p.T;

  int slot = -1;
  if (p.slot_ids) {
    slot = p.slot_ids[n];
    if (slot == KDA_PAD_SLOT_ID) return;   // padding row of a bucketed batch
    if (slot < 0 || slot >= p.num_slots) {
      if (tid == 0) atomicOr(p.status, KDA_DEVICE_BAD_SLOT);
      return;
    }
  }

  const int row0 = warp * kRows;
  const int col0 = lane * 4;                      // this lane's 4 key channels (q, k, gate)
  const int vcol = part * kCols + lane * kVC;     // this lane's kVC value channels (columns of S)
  float S[kRows][kVC];
  if (p.state_in) {
    const float *src = p.state_in + ((size_t)slot * p.H + h) * kD * kD;
#pragma unroll
    for (int i = 0; i < kRows; ++i) load_vc<kVC>(S[i], src + (size_t)(row0 + i) * kD + vcol);
  } else {
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < kVC; ++j) S[i][j] = 0.f;
  }

  // per-head gate constants for this lane's 4 channels
  const float ea = __expf(p.A_log[h]);
  float dtb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) dtb[j] = p.dt_bias[h * kD + col0 + j];

  for (int tile = t_begin; tile < t_end; tile += kTile) {
    const int nt = min(kTile, t_end - tile);
    // ---- prologue: warp w prepares token tile + w ----
    if (warp < nt) {
      const int t = tile + warp;
      // the output row of this token in the layer's output (-1: none; every lane loads the same index)
      int64_t row = t;
      if (p.out_index) {
        row = p.out_index[t];
        if (row < 0 || row >= p.num_out_rows) row = -1;
      }
      if (kNorm) {
        uint2 zr = make_uint2(0u, 0u);
        if (row >= 0) zr = *reinterpret_cast<const uint2 *>(p.norm.gate + row * p.norm.gate_stride + h * kD + col0);
        const float2 z01 = unpack_bf16x2(zr.x), z23 = unpack_bf16x2(zr.y);
        *reinterpret_cast<float4 *>(&s_gz[warp][col0]) =
            make_float4(sigmoid_f(z01.x), sigmoid_f(z01.y), sigmoid_f(z23.x), sigmoid_f(z23.y));
      }
      const uint2 gr = *reinterpret_cast<const uint2 *>(p.g + (size_t)t * p.g_stride + h * kD + col0);
      const uint16_t *gs = reinterpret_cast<const uint16_t *>(&gr);
      float qf[4], kf[4], vf[4], qq = 0.f, kk = 0.f;
      if (!kConv) {
        const uint2 qr = *reinterpret_cast<const uint2 *>(p.q + (size_t)t * p.qkv_stride + h * kD + col0);
        const uint2 kr = *reinterpret_cast<const uint2 *>(p.k + (size_t)t * p.qkv_stride + h * kD + col0);
        const float2 q01 = unpack_bf16x2(qr.x), q23 = unpack_bf16x2(qr.y);
        const float2 k01 = unpack_bf16x2(kr.x), k23 = unpack_bf16x2(kr.y);
        qf[0] = q01.x; qf[1] = q01.y; qf[2] = q23.x; qf[3] = q23.y;
        kf[0] = k01.x; kf[1] = k01.y; kf[2] = k23.x; kf[3] = k23.y;
        // this lane's kVC value channels of the CTA's slice
        const uint16_t *vp = p.v + (size_t)t * p.qkv_stride + h * kD + vcol;
        if constexpr (kVC == 4) {
          const uint2 vr = *reinterpret_cast<const uint2 *>(vp);
          const float2 v01 = unpack_bf16x2(vr.x), v23 = unpack_bf16x2(vr.y);
          vf[0] = v01.x; vf[1] = v01.y; vf[2] = v23.x; vf[3] = v23.y;
        } else if constexpr (kVC == 2) {
          const float2 v01 = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(vp));
          vf[0] = v01.x; vf[1] = v01.y;
        } else {
          vf[0] = bf16_bits_to_f32(*vp);
        }
      } else {
        // short causal convolutions of q, k, v over this lane's 4 channels: the raw inputs 3, 2, 1 and 0
        // tokens back (the request's own tokens, else its slot's window, oldest row first); the window
        // after this token (the inputs 2, 1, 0 back) is recorded for the commit
        const int r = t - t_begin;
        const uint16_t *base[3] = {p.q, p.k, p.v};
        float *dst[3] = {qf, kf, vf};
#pragma unroll
        for (int m = 0; m < 3; ++m) {
          uint2 xr[kConvW];
#pragma unroll
          for (int j = 0; j < kConvW; ++j) {
            const int back = kConvW - 1 - j;
            xr[j] = r - back >= 0
                        ? *reinterpret_cast<const uint2 *>(base[m] + (size_t)(t - back) * p.qkv_stride + h * kD + col0)
                        : *reinterpret_cast<const uint2 *>(
                              p.conv.window_pool +
                              ((((size_t)slot * 3 + m) * (kConvW - 1) + (kConvW - 1 + r - back)) * p.H + h) * kD + col0);
          }
          if (p.conv.step_windows) {
#pragma unroll
            for (int j = 0; j < kConvW - 1; ++j)
              *reinterpret_cast<uint2 *>(
                  p.conv.step_windows +
                  (((((size_t)n * p.T + r) * 3 + m) * (kConvW - 1) + j) * p.H + h) * kD + col0) = xr[j + 1];
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 w = *reinterpret_cast<const float4 *>(p.conv.weight + (((size_t)m * p.H + h) * kD + col0 + e) * kConvW);
            const float wt[kConvW] = {w.x, w.y, w.z, w.w};
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kConvW; ++j) {
              const float2 x2 = unpack_bf16x2(e < 2 ? xr[j].x : xr[j].y);
              acc = fmaf(wt[j], (e & 1) ? x2.y : x2.x, acc);
            }
            dst[m][e] = p.conv.silu ? acc * sigmoid_f(acc) : acc;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        qq += qf[j] * qf[j];
        kk += kf[j] * kf[j];
      }
      qq = warp_sum(qq);
      kk = warp_sum(kk);
      const float nq = rsqrtf(qq + kL2Eps), nk = rsqrtf(kk + kL2Eps);
      float kq = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float qh = qf[j] * nq, kh = kf[j] * nk;
        kq += qh * kh;
        const float lam = p.lower_bound * sigmoid_f(ea * (bf16_bits_to_f32(gs[j]) + dtb[j]));
        const float alpha = fast_exp2(lam * kLog2e);
        s_khat[warp][col0 + j] = kh;
        s_kalpha[warp][col0 + j] = alpha * kh;
        s_qalpha[warp][col0 + j] = alpha * qh;
        s_alpha[warp][col0 + j] = alpha;
      }
#pragma unroll
      for (int j = 0; j < kVC; ++j) s_v[warp][lane * kVC + j] = vf[j];
      kq = warp_sum(kq);
      if (lane == 0) {
        s_kq[warp] = kq;
        s_beta[warp] = sigmoid_f(bf16_bits_to_f32(p.beta[(size_t)t * p.beta_stride + h]));
        if (row < 0) atomicOr(p.status, KDA_DEVICE_BAD_INDEX);
        s_row[warp] = row;
      }
    }
    __syncthreads();

    for (int s = 0; s < nt; ++s) {
      const int t = tile + s;
      // partial S^T (alpha k^) and S^T (alpha q^) over this warp's 16 rows, for the lane's value channels
      float pk[kVC], pq[kVC];
#pragma unroll
      for (int j = 0; j < kVC; ++j) pk[j] = pq[j] = 0.f;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const float ka = s_kalpha[s][row0 + i], qa = s_qalpha[s][row0 + i];
#pragma unroll
        for (int j = 0; j < kVC; ++j) {
          pk[j] = fmaf(S[i][j], ka, pk[j]);
          pq[j] = fmaf(S[i][j], qa, pq[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < kVC; ++j) {
        s_redk[warp][lane * kVC + j] = pk[j];
        s_redq[warp][lane * kVC + j] = pq[j];
      }
      __syncthreads();
      if (tid < kCols) {   // thread = the slice's value channel tid
        float wk = 0.f, wq = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          wk += s_redk[w][tid];
          wq += s_redq[w][tid];
        }
        const float u = s_beta[s] * (s_v[s][tid] - wk);
        s_u[tid] = u;
        float o = p.scale * (wq + s_kq[s] * u);
        const int64_t row = s_row[s];
        if (kNorm) {   // gated RMSNorm over the 128 channels (warps 0..3)
          const float sq = warp_sum(o * o);
          if (lane == 0) s_sq[warp] = sq;
          named_bar_sync<1>(kD);
          const float rstd = rsqrtf((s_sq[0] + s_sq[1] + s_sq[2] + s_sq[3]) * (1.0f / kD) + p.norm.eps);
          o = o * rstd * p.norm.weight[tid] * s_gz[s][tid];
          if (tid == 0 && row >= 0 && p.norm.rstd) p.norm.rstd[row * p.H + h] = rstd;
        }
        if (row >= 0) p.out[row * p.out_stride + h * kD + part * kCols + tid] = f32_to_bf16_bits(o);
      }
      __syncthreads();
      float uu[kVC];
#pragma unroll
      for (int j = 0; j < kVC; ++j) uu[j] = s_u[lane * kVC + j];
      float *rec = p.inter ? p.inter + (((size_t)n * p.T + (t - t_begin)) * p.H + h) * kD * kD : nullptr;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const float a = s_alpha[s][row0 + i], kh = s_khat[s][row0 + i];
#pragma unroll
        for (int j = 0; j < kVC; ++j) S[i][j] = fmaf(a, S[i][j], kh * uu[j]);
        if (rec) store_vc<kVC, true>(rec + (size_t)(row0 + i) * kD + vcol, S[i]);
      }
    }
    __syncthreads();
  }

  float *dst = nullptr;
  if (p.state_out_pool) dst = p.state_out_pool + ((size_t)slot * p.H + h) * kD * kD;
  else if (p.state_out_dense) dst = p.state_out_dense + ((size_t)n * p.H + h) * kD * kD;
  if (dst) {
#pragma unroll
    for (int i = 0; i < kRows; ++i) store_vc<kVC, false>(dst + (size_t)(row0 + i) * kD + vcol, S[i]);
  }
}

// kMinB: CTAs per SM the registers are budgeted for (two, or three for the value-split form of large batches)
template <bool kConv, bool kNorm, int kP, int kMinB>
__global__ void __launch_bounds__(kThreads, kMinB) recurrent_kernel(RecurrentArgs p) {
  recurrent_item<kConv, kNorm, kP>(p);
  if (p.done_counter) {
    // launched as a programmatic dependent of the grid before it, which it does not read from: the CTA that
    // finishes last waits for that grid's completion, so this grid's completion implies it for whatever the
    // stream runs next; it then clears the counter for the next call on the same workspace
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(p.done_counter, 1u) == gridDim.x - 1) {
      sm100::grid_dependency_wait();
      *p.done_counter = 0;
    }
  }
}

}  // namespace

template <bool kConv, bool kNorm, int kP, int kMinB = 2>
cudaError_t launch_variant(const RecurrentArgs &args, int num_items, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(num_items) * args.H * kP;
  if (!args.done_counter) {
    recurrent_kernel<kConv, kNorm, kP, kMinB><<<grid, kThreads, 0, stream>>>(args);
    return cudaGetLastError();
  }
  // programmatic dependent launch: CTAs may be scheduled onto SMs the preceding grid leaves free once every
  // CTA of that grid has signalled launch_dependents
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, recurrent_kernel<kConv, kNorm, kP, kMinB>, args);
}

cudaError_t launch_recurrent(const RecurrentArgs &args, int num_items, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  const bool conv = args.conv.weight != nullptr, norm = args.norm.gate != nullptr;
  if (conv) return norm ? launch_variant<true, true, 1>(args, num_items, stream)
                        : launch_variant<true, false, 1>(args, num_items, stream);
  if (norm) return launch_variant<false, true, 1>(args, num_items, stream);
  // a small batch fills fewer SMs than one wave of (request, head) CTAs: split each item's value channels over
  // 2 or 4 CTAs while the grid still fits in one wave (two CTAs per SM)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  const long long items = static_cast<long long>(num_items) * args.H, wave = 2LL * sms;
  if (items * 4 <= wave) return launch_variant<false, false, 4>(args, num_items, stream);
  if (items * 2 <= wave) return launch_variant<false, false, 2>(args, num_items, stream);
  // more items than one wave, with four or more tokens each: half of an item's value channels per CTA in 80
  // registers, three CTAs per SM.  Measured as graph replays on H = 16: T = 8 at 32 / 48 / 64 requests 49.8 /
  // 74.6 / 97.9 us against 51.0 / 78.2 / 100.8 for whole items at two per SM, level at 256 requests; the spec
  // step 2048 x 4 + 64 x 4 171.6 against 173.4 us; T = 1 and 2 and batches below one wave are slower that way
  if (!args.cu_seqlens && args.T >= 4 && items > wave)
    return launch_variant<false, false, 2, 3>(args, num_items, stream);
  return launch_variant<false, false, 1>(args, num_items, stream);
}

}  // namespace kda
