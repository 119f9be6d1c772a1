// Work list for the attention kernel, built on the device from cu_seqlens and
// the per-sample CP sizes (so the host never has to read them back).
//
// A work item is one block of up to 256 query rows of one CP rank's chunk of
// one sample ("Dynamic Context Parallelism (DCP)": each sample gets its own CP
// size; "Megatron 架构与 6D 并行完整指南" section 六: rank i owns chunk i of the
// sequence).  Items are ordered by decreasing cost -- the number of KV tiles
// the block visits -- so that the long causal blocks start first and the
// short ones fill the tail.  The attention kernel maps CTA x to item x / H and
// head x % H, so all heads of one block run side by side and share K/V in L2.
#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kBuckets = 4096;  // cost histogram; costs above saturate

struct SampleGeom {
  int L, c, chunk, full, rem;  // full chunks of `chunk` tokens, then `rem`
};

__device__ __forceinline__ SampleGeom geom(const SchedParams& p, int b) {
  SampleGeom g;
  g.L = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
  g.c = p.cp_size ? p.cp_size[b] : 1;
  g.chunk = (g.L + g.c - 1) / g.c;
  g.full = g.chunk > 0 ? g.L / g.chunk : 0;
  g.rem = g.L - g.full * g.chunk;
  return g;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int items_of(const SampleGeom& g) {
  if (g.L == 0) return 0;
  return g.full * ceil_div(g.chunk, kRowsPerItem) +
         (g.rem > 0 ? ceil_div(g.rem, kRowsPerItem) : 0);
}

// Item `local` of a sample -> (rank, block) and its cost in KV tiles.
__device__ __forceinline__ void decode(const SampleGeom& g, int local,
                                       int causal, int& rank, int& blk,
                                       int& cost) {
  const int per = ceil_div(g.chunk, kRowsPerItem);
  rank = local / per;
  blk = local - rank * per;
  if (rank >= g.full) {  // the short last chunk
    rank = g.full;
    blk = local - g.full * per;
  }
  const int lo = rank * g.chunk;
  const int hi = min(lo + g.chunk, g.L);
  const int tiles_full_chunk = ceil_div(g.chunk, kBN);
  if (causal) {
    const int q_end = min(lo + (blk + 1) * kRowsPerItem, hi);
    cost = rank * tiles_full_chunk + ceil_div(q_end - lo, kBN);
  } else {
    cost = g.full * tiles_full_chunk + (g.rem > 0 ? ceil_div(g.rem, kBN) : 0);
  }
  (void)hi;
}

// Inclusive scan of one value per thread across the block.
__device__ __forceinline__ int block_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
  __syncthreads();
  return r;
}

}  // namespace

__global__ void __launch_bounds__(kSchedThreads)
    schedule_kernel(const SchedParams p) {
  __shared__ int s_bad;
  __shared__ int s_carry;
  __shared__ int warp_sums[32];
  __shared__ int hist[kBuckets];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = 0;
    s_carry = 0;
    p.hdr->error = 0;
    p.hdr->n_items = 0;
  }
  for (int k = tid; k < kBuckets; k += kSchedThreads) hist[k] = 0;
  __syncthreads();

  // Argument checks the host cannot make without reading device memory.
  if (tid == 0 && (p.cu_seqlens[0] != 0 ||
                   static_cast<long long>(p.cu_seqlens[p.num_seqs]) != p.total_tokens))
    s_bad = 1;
  for (int b = tid; b < p.num_seqs; b += kSchedThreads) {
    const int L = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
    const int c = p.cp_size ? p.cp_size[b] : 1;
    if (L < 0 || L > p.max_seqlen || c < 1 || c > p.max_cp) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) p.hdr->error = 1;  // CPATTN_ERR_INVALID_ARG
    return;
  }

  // Per-sample item counts -> exclusive prefix in p.prefix[0..B].
  for (int base = 0; base < p.num_seqs; base += kSchedThreads) {
    const int b = base + tid;
    const int cnt = b < p.num_seqs ? items_of(geom(p, b)) : 0;
    const int incl = block_scan(cnt, warp_sums);
    if (b < p.num_seqs) p.prefix[b] = s_carry + incl - cnt;
    __syncthreads();
    if (tid == kSchedThreads - 1) s_carry += incl;
    __syncthreads();
  }
  const int total = s_carry;
  if (tid == 0) p.prefix[p.num_seqs] = total;
  if (total > p.max_items) {
    if (tid == 0) p.hdr->error = 1;
    return;
  }
  __syncthreads();

  // Pass 1: cost histogram.
  for (int x = tid; x < total; x += kSchedThreads) {
    int lo = 0, hi = p.num_seqs - 1;  // last b with prefix[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.prefix[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const SampleGeom g = geom(p, lo);
    int rank, blk, cost;
    decode(g, x - p.prefix[lo], p.causal, rank, blk, cost);
    atomicAdd(&hist[min(cost, kBuckets - 1)], 1);
  }
  __syncthreads();

  // Bucket offsets, most expensive first.
  {
    constexpr int kPer = kBuckets / kSchedThreads;
    int loc[kPer];
    int sum = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      loc[e] = hist[kBuckets - 1 - (tid * kPer + e)];
      sum += loc[e];
    }
    const int incl = block_scan(sum, warp_sums);
    int run = incl - sum;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int bucket = kBuckets - 1 - (tid * kPer + e);
      hist[bucket] = run;
      run += loc[e];
    }
  }
  __syncthreads();

  // Pass 2: scatter.
  for (int x = tid; x < total; x += kSchedThreads) {
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.prefix[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const SampleGeom g = geom(p, lo);
    int rank, blk, cost;
    decode(g, x - p.prefix[lo], p.causal, rank, blk, cost);
    const int pos = atomicAdd(&hist[min(cost, kBuckets - 1)], 1);
    p.items[pos] = make_int2(lo, (rank << 20) | blk);
  }
  __syncthreads();
  if (tid == 0) p.hdr->n_items = total;
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream) {
  schedule_kernel<<<1, kSchedThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace cpattn
