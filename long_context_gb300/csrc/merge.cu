// Merge of stored per-step partials (the unfused path), HBM-bound.
//
// For every row (t, h) it folds S partials (O_s, m_s, l_s) with the
// online-softmax merge of "Megatron 架构与 6D 并行完整指南", section 六
// (m_new = max(m, m_s), alpha = exp(m - m_new), beta = exp(m_s - m_new),
// l = alpha l + beta l_s, O = alpha O + beta O_s), written in closed form:
//   m* = max_s m_s,  w_s = exp(m_s - m*),  l = sum_s w_s l_s,
//   O / l = sum_s (w_s / l) O_s,
// which is the same value as the step-by-step fold up to rounding (every
// alpha/beta product telescopes to one exp(m_s - m*)).  exp(-inf - x) = 0.
//
// Memory layout: O_s [S, rows, D], m_s and l_s [S, rows] (rows = T * H).
// Normalised partials (decode-time CP) come without l_s: l_s = 1 and m_s is
// the partial's LSE, which makes this the LSE-form merge.
// A warp owns a chunk of `chunk` consecutive rows (32, 16, 8 or 4, chosen by
// the host so that the last grid-stride round is nearly full): lane r reads
// m_s and l_s of row r (coalesced loads per step) and leaves that row's S
// coefficients w_s / l in shared memory; the warp then walks its rows while
// the lanes stream each row's S vectors of D floats as 16-byte loads, 8
// steps in flight.
#include <cuda_bf16.h>

#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kMergeThreads = 256;
constexpr float kNegInfM = -__builtin_huge_valf();

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  return __ldcs(p);
}

}  // namespace

template <int D, bool BF16_OUT>
__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const MergeParams p, int chunk) {
  constexpr int kLanesPerRow = D / 4;          // one float4 per lane
  constexpr int kRowsPerPass = 32 / kLanesPerRow;
  constexpr int kGroup = 8;                    // steps streamed together
  extern __shared__ float coef_smem[];         // per warp: [S][32]
  const int lane = threadIdx.x & 31;
  const int S = p.num_steps;
  float* coef = coef_smem + (threadIdx.x >> 5) * S * 32;
  const long long warp_global =
      (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kMergeThreads) >> 5;
  const long long rows = p.rows;
  const int sub = lane / kLanesPerRow;         // row within a pass
  const int col = (lane % kLanesPerRow) * 4;

  for (long long row0 = warp_global * chunk; row0 < rows; row0 += nwarps * chunk) {
    // Row statistics: lane r owns row row0 + r.
    const long long my_row = row0 + lane;
    const bool have = lane < chunk && my_row < rows;
    float mstar = kNegInfM;
    if (have)
      for (int s = 0; s < S; ++s)
        mstar = fmaxf(mstar, __ldg(p.m_steps + static_cast<long long>(s) * rows + my_row));
    float l = 0.f;
    for (int s = 0; s < S; ++s) {
      float w = 0.f;
      if (have) {
        const float m = __ldg(p.m_steps + static_cast<long long>(s) * rows + my_row);
        const float ls =
            p.l_steps ? __ldg(p.l_steps + static_cast<long long>(s) * rows + my_row) : 1.f;
        w = (m == kNegInfM) ? 0.f : expf(m - mstar);
        l += w * ls;
      }
      coef[s * 32 + lane] = w;
    }
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    for (int s = 0; s < S; ++s) coef[s * 32 + lane] *= inv_l;
    if (have) {
      if (p.out_lse) p.out_lse[my_row] = l > 0.f ? mstar + logf(l) : kNegInfM;
      if (!BF16_OUT) {
        if (p.out_m) p.out_m[my_row] = mstar;
        if (p.out_l) p.out_l[my_row] = l;
      }
    }
    __syncwarp();

    // Stream the O vectors of the warp's 32 rows, kGroup steps in flight.
#pragma unroll 2
    for (int q = 0; q < chunk / kRowsPerPass; ++q) {
      const int r = q * kRowsPerPass + sub;
      const long long row = row0 + r;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < rows) {
        for (int s0 = 0; s0 < S; s0 += kGroup) {
          float4 v[kGroup];
#pragma unroll
          for (int e = 0; e < kGroup; ++e) {
            if (s0 + e < S)
              v[e] = ld_stream(reinterpret_cast<const float4*>(
                  p.o_steps + (static_cast<long long>(s0 + e) * rows + row) * D + col));
            else
              v[e] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int e = 0; e < kGroup; ++e) {
            const float w = (s0 + e < S) ? coef[(s0 + e) * 32 + r] : 0.f;
            acc.x = fmaf(w, v[e].x, acc.x);
            acc.y = fmaf(w, v[e].y, acc.y);
            acc.z = fmaf(w, v[e].z, acc.z);
            acc.w = fmaf(w, v[e].w, acc.w);
          }
        }
        if (BF16_OUT) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(p.out_bf16 + row * D + col) = pk;
        } else {
          __stcs(reinterpret_cast<float4*>(p.out_o + row * D + col), acc);
        }
      }
    }
    __syncwarp();
  }
}

template <int D, bool BF16_OUT>
static cudaError_t launch_merge_d(const MergeParams& p, int num_sms,
                                  cudaStream_t stream) {
  // Grid-stride over at most 8 resident blocks per SM (the loads in flight
  // need them all).  Chunk size (a multiple of the rows one pass covers, 1 at
  // D = 128, 2 at D = 64): the largest of 32, 16, 8, 4 rows whose last
  // round keeps at least 99 % of the warps busy (U chunks over W warps: the
  // slowest warp does ceil(U / W) of them against U / W on average).
  const long long cap = static_cast<long long>(num_sms) * 8;
  const long long warps_per_block = kMergeThreads / 32;
  int chunk = 32;
  long long grid_ll = 0;
  double best = -1.0;
  for (int c = 32; c >= 4; c >>= 1) {
    const long long units = (p.rows + c - 1) / c;
    const long long b_needed = (units + warps_per_block - 1) / warps_per_block;
    const long long b = b_needed < cap ? b_needed : cap;
    const long long w = b * warps_per_block;
    const long long rounds = (units + w - 1) / w;
    const double eff = static_cast<double>(units) / static_cast<double>(rounds * w);
    if (eff > best + 1e-9) {
      best = eff;
      chunk = c;
      grid_ll = b;
    }
    if (eff >= 0.99) break;
  }
  const unsigned grid = static_cast<unsigned>(grid_ll);
  if (grid == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kMergeThreads / 32) * p.num_steps * 32 * sizeof(float);
  auto kern = merge_kernel<D, BF16_OUT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, kMergeThreads, smem, stream>>>(p, chunk);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, int D, bool bf16_out,
                         int num_sms, cudaStream_t stream) {
  if (D == 64)
    return bf16_out ? launch_merge_d<64, true>(p, num_sms, stream)
                    : launch_merge_d<64, false>(p, num_sms, stream);
  return bf16_out ? launch_merge_d<128, true>(p, num_sms, stream)
                  : launch_merge_d<128, false>(p, num_sms, stream);
}

}  // namespace cpattn
