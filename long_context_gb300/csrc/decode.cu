// Decode-time context parallelism ("VeRL Backend Parallelism": for the vLLM
// engines CP means decode context parallelism -- the KV cache of a sequence
// split over ranks).  One new query token per sequence attends to every
// cached key of that sequence; with decode CP size c the cache is cut into c
// contiguous shards, each shard gives a normalised partial (O_s, lse_s), and
// the partials merge in the LSE form (merge.cu with l_s = 1).
//
// One CTA (4 warps) per (sequence, head, shard): a key row of D bf16 values
// is read by D/8 lanes with 16-byte loads (two rows per warp instruction at
// D = 128), four K and four V loads in flight per lane; each group of lanes
// that shares a key keeps its own online-softmax state, and the CTA combines
// the groups at the end.  HBM bound (a single query per head is a
// matrix-vector product: no tensor-core contraction).
#include <cuda_bf16.h>

#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecUnroll = 4;  // loads of K (and of V) in flight per lane
constexpr float kDecNegInf = -__builtin_huge_valf();
constexpr float kDecLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void bf16x8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __bfloat1622float2(h[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kDecThreads) decode_partials_kernel(const DecodeParams p) {
  constexpr int kLanesPerKey = D / 8;             // 16-byte chunks of a row
  constexpr int kKeysPerLoad = 32 / kLanesPerKey;  // rows per warp instruction
  constexpr int kGroups = kDecWarps * kKeysPerLoad;
  constexpr int kKeysPerStep = kGroups * kDecUnroll;  // keys per CTA iteration
  __shared__ float g_m[kGroups], g_l[kGroups];
  __shared__ float g_o[kGroups][D];

  const int H = p.num_heads, c = p.cp;
  const int cta = static_cast<int>(blockIdx.x);
  const int s = cta % c;
  const int bh = cta / c;
  const int h = bh % H;
  const int b = bh / H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / kLanesPerKey;  // which row of a load
  const int dl = lane % kLanesPerKey;   // 8-feature chunk
  const int group = warp * kKeysPerLoad + sub;

  // Shard bounds (an inconsistent cu_seqlens gives an empty shard).
  const int s0 = p.cu_seqlens[b];
  const int s1 = p.cu_seqlens[b + 1];
  int L = s1 - s0;
  if (s0 < 0 || s1 > p.total_tokens || L < 0) L = 0;
  const int chunk = (L + c - 1) / c;
  const int a = min(s * chunk, L), z = min((s + 1) * chunk, L);

  float qf[8];
  {
    const uint4 qv = __ldg(reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * H + h) * D) + dl);
    bf16x8(qv, qf);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[e] *= p.scale_log2;
  }
  float m = kDecNegInf, l = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;

  for (int base = a + warp * kKeysPerLoad * kDecUnroll; base < z; base += kKeysPerStep) {
    uint4 kr[kDecUnroll], vr[kDecUnroll];
    bool valid[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int key = base + u * kKeysPerLoad + sub;
      valid[u] = key < z;
      if (valid[u]) {
        const size_t row = (static_cast<size_t>(s0 + key) * H + h) * D;
        kr[u] = __ldcs(reinterpret_cast<const uint4*>(p.k + row) + dl);
        vr[u] = __ldcs(reinterpret_cast<const uint4*>(p.v + row) + dl);
      }
    }
    float sc[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      float kf[8];
      bf16x8(valid[u] ? kr[u] : make_uint4(0, 0, 0, 0), kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(qf[e], kf[e], dot);
#pragma unroll
      for (int off = kLanesPerKey / 2; off > 0; off >>= 1)
        dot += __shfl_xor_sync(0xffffffffu, dot, off);
      sc[u] = valid[u] ? dot : kDecNegInf;
    }
    float mt = sc[0];
#pragma unroll
    for (int u = 1; u < kDecUnroll; ++u) mt = fmaxf(mt, sc[u]);
    const float mn = fmaxf(m, mt);
    if (mn == kDecNegInf) continue;  // no valid key yet in this group
    const float alpha = (m == kDecNegInf) ? 0.f : ex2f(m - mn);
    l *= alpha;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const float pu = valid[u] ? ex2f(sc[u] - mn) : 0.f;
      l += pu;
      float vf[8];
      bf16x8(valid[u] ? vr[u] : make_uint4(0, 0, 0, 0), vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = fmaf(pu, vf[e], o[e]);
    }
    m = mn;
  }

  // Combine the groups' states (log2 domain).
#pragma unroll
  for (int e = 0; e < 8; ++e) g_o[group][dl * 8 + e] = o[e];
  if (dl == 0) {
    g_m[group] = m;
    g_l[group] = l;
  }
  __syncthreads();
  float mstar = kDecNegInf;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) mstar = fmaxf(mstar, g_m[g]);
  const size_t out_row = (static_cast<size_t>(s) * p.num_seqs + b) * H + h;
  for (int t = threadIdx.x; t < D; t += kDecThreads) {
    float num = 0.f, den = 0.f;
    if (mstar != kDecNegInf) {
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        const float w = (g_m[g] == kDecNegInf) ? 0.f : ex2f(g_m[g] - mstar);
        num = fmaf(w, g_o[g][t], num);
        den = fmaf(w, g_l[g], den);
      }
    }
    p.o_steps[out_row * D + t] = den > 0.f ? num / den : 0.f;
    if (t == 0)
      p.lse_steps[out_row] = den > 0.f ? (mstar + __log2f(den)) * kDecLn2 : kDecNegInf;
  }
}

cudaError_t launch_decode_partials(const DecodeParams& p, int D, cudaStream_t stream) {
  const long long grid = static_cast<long long>(p.num_seqs) * p.num_heads * p.cp;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (D == 64)
    decode_partials_kernel<64><<<static_cast<unsigned>(grid), kDecThreads, 0, stream>>>(p);
  else
    decode_partials_kernel<128><<<static_cast<unsigned>(grid), kDecThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace cpattn
