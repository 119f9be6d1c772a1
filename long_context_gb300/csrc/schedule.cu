// CTA schedule for the attention kernel, built on the device from cu_seqlens
// and the per-sample CP sizes (so the host never reads them back).
//
// Work: one CTA per (block of up to 256 query rows of one CP rank's chunk,
// head) -- "Dynamic Context Parallelism (DCP)": each sample has its own CP
// size; "Megatron 架构与 6D 并行完整指南" section 六: rank i owns chunk i.
// Order (see work.cuh): samples by decreasing length, then head, then block
// by decreasing cost.  This kernel writes the sample order, for each position
// in it the first CTA index of that sample, and then the work of every CTA
// (sample start and length, CP size, head, rank, block) into a table that the
// attention kernel reads with one load per CTA.
#include "debug.cuh"
#include "kernels.h"
#include "work.cuh"

namespace cpattn {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kBuckets = 4096;  // length buckets of 128 tokens; longer saturate
// Batches of at most this many samples take a short path: one warp checks
// the arguments, orders the samples and forms the CTA prefix with shuffles
// (no block-wide barrier until the table fill), reading cu_seqlens and the
// CP sizes once.  The general path's time is a chain of block barriers and
// memory round trips (about 8 us), not arithmetic.
constexpr int kWarpSeqs = 32;

// Inclusive scan of one value per thread across the block.
__device__ __forceinline__ long long block_scan(long long v, long long* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const long long r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
  __syncthreads();
  return r;
}

// Work table: each thread fills a contiguous run of CTA indices, finding the
// sample position of the first one by binary search and walking on.  `cu`,
// `cps` (null: CP 1), `order` and `first_cta` may be in shared or global
// memory.
__device__ __forceinline__ void fill_table(const SchedParams& p, const int* cu, const int* cps,
                                           const int* order, const int* first_cta, int n_ctas,
                                           int tid) {
  const int per = (n_ctas + kSchedThreads - 1) / kSchedThreads;
  const int x_begin = min(tid * per, n_ctas);
  const int x_end = min(x_begin + per, n_ctas);
  if (x_begin >= x_end) return;
  int pos = 0;
  {
    int hi = p.num_seqs - 1;
    while (pos < hi) {
      const int mid = (pos + hi + 1) >> 1;
      if (first_cta[mid] <= x_begin) pos = mid; else hi = mid - 1;
    }
  }
  int next = first_cta[pos + 1];
  int b = order[pos];
  const int rows = p.rows_per_item;
  SampleGeom g = sample_geom(cu, cps, b);
  int n_b = sample_items(g, rows);
  int first = first_cta[pos];
  for (int x = x_begin; x < x_end; ++x) {
    while (x >= next) {  // samples without CTAs (L = 0) are passed over
      ++pos;
      first = next;
      next = first_cta[pos + 1];
      b = order[pos];
      g = sample_geom(cu, cps, b);
      n_b = sample_items(g, rows);
    }
    const int e = x - first;
    const int h = e / n_b;
    const int local = e - h * n_b;
    int rank, blk;
    item_coords(g, n_b - 1 - local, rank, blk, rows);
    const int tok0 = cu[b];
    if (!in_bounds(x, 0, p.max_ctas, p.hdr) || !in_bounds(b, 0, p.num_seqs, p.hdr) ||
        !in_bounds(h, 0, p.num_heads, p.hdr))
      continue;
    p.table[x] = make_int4(tok0, g.L, (h << 8) | g.c,
                           static_cast<int>((static_cast<unsigned>(blk) << 8) |
                                            static_cast<unsigned>(rank)));
    if (p.table_asc != nullptr) {
      item_coords(g, local, rank, blk, rows);
      p.table_asc[x] = make_int4(tok0, g.L, (h << 8) | g.c,
                                 static_cast<int>((static_cast<unsigned>(blk) << 8) |
                                                  static_cast<unsigned>(rank)));
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kSchedThreads)
    schedule_kernel(const SchedParams p) {
  __shared__ int s_bad;
  __shared__ long long s_carry;
  __shared__ long long warp_sums[32];
  __shared__ int hist[kBuckets];
  __shared__ int w_cu[kWarpSeqs + 1];
  __shared__ int w_cp[kWarpSeqs];
  __shared__ int w_order[kWarpSeqs];
  __shared__ int w_first[kWarpSeqs + 1];
  // The attention kernel (launched with programmatic stream serialization)
  // may start launching now; it waits for this grid's results before use.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;

  if (p.num_seqs <= kWarpSeqs) {
    // ---- short path: one warp, then the table fill by every thread.
    if (tid < 32) {
      const int lane = tid;
      const int B = p.num_seqs;
      int lo = 0, hi = 0, c = 1;
      if (lane < B) {
        lo = p.cu_seqlens[lane];
        hi = p.cu_seqlens[lane + 1];
        c = p.cp_size ? p.cp_size[lane] : 1;
      }
      const int L = hi - lo;
      bool bad = lane < B && (L < 0 || L > p.max_seqlen || c < 1 || c > p.max_cp);
      if (lane == 0) {
        const int cu_b = p.cu_seqlens[B];
        bad = bad || p.cu_seqlens[0] != 0 || static_cast<long long>(cu_b) != p.total_tokens;
        w_cu[B] = cu_b;
      }
      bad = __any_sync(0xffffffffu, bad);
      long long total = 0;
      if (!bad) {
        // Position of sample `lane`: longest bucket first, then by index (a
        // valid order of the general path's counting sort).
        const int bk = lane < B ? min(L >> 7, kBuckets - 1) : -1;
        int rank = 0;
        for (int j = 0; j < B; ++j) {
          const int bj = __shfl_sync(0xffffffffu, bk, j);
          rank += (bj > bk || (bj == bk && j < lane)) ? 1 : 0;
        }
        if (lane < B) {
          w_cu[lane] = lo;
          w_cp[lane] = c;
          w_order[rank] = lane;
        }
        __syncwarp();
        long long cnt = 0;
        if (lane < B)
          cnt = static_cast<long long>(
                    sample_items(sample_geom(w_cu, w_cp, w_order[lane]), p.rows_per_item)) *
                p.num_heads;
        long long incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        if (lane < B) w_first[lane] = static_cast<int>(incl - cnt);
        total = __shfl_sync(0xffffffffu, incl, 31);
        if (total > p.max_ctas) bad = true;
        if (lane == 0) w_first[B] = static_cast<int>(total);
      }
      if (lane == 0) {
        p.hdr->error = bad ? 1 : 0;  // CPATTN_ERR_INVALID_ARG
        p.hdr->n_items = 0;
        s_bad = bad ? 1 : 0;
        s_carry = total;
      }
    }
    __syncthreads();
    if (s_bad) return;
    fill_table(p, w_cu, w_cp, w_order, w_first, static_cast<int>(s_carry), tid);
    if (tid == 0) p.hdr->n_items = static_cast<int>(s_carry);
    return;
  }

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

  // Sample order: counting sort by length bucket, longest first.
  auto bucket = [&](int b) {
    return min((p.cu_seqlens[b + 1] - p.cu_seqlens[b]) >> 7, kBuckets - 1);
  };
  for (int b = tid; b < p.num_seqs; b += kSchedThreads) atomicAdd(&hist[bucket(b)], 1);
  __syncthreads();
  {
    constexpr int kPer = kBuckets / kSchedThreads;
    int loc[kPer];
    long long sum = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      loc[e] = hist[kBuckets - 1 - (tid * kPer + e)];
      sum += loc[e];
    }
    const long long incl = block_scan(sum, warp_sums);
    int run = static_cast<int>(incl - sum);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      hist[kBuckets - 1 - (tid * kPer + e)] = run;
      run += loc[e];
    }
  }
  __syncthreads();
  for (int b = tid; b < p.num_seqs; b += kSchedThreads) {
    const int slot = atomicAdd(&hist[bucket(b)], 1);
    if (in_bounds(slot, 0, p.num_seqs, p.hdr)) p.order[slot] = b;
  }
  __syncthreads();

  // First CTA of each sample position: prefix of items * heads.
  for (int base = 0; base < p.num_seqs; base += kSchedThreads) {
    const int k = base + tid;
    long long cnt = 0;
    if (k < p.num_seqs)
      cnt = static_cast<long long>(
                sample_items(sample_geom(p.cu_seqlens, p.cp_size, p.order[k]),
                             p.rows_per_item)) *
            p.num_heads;
    const long long incl = block_scan(cnt, warp_sums);
    if (k < p.num_seqs) p.first_cta[k] = static_cast<int>(s_carry + incl - cnt);
    __syncthreads();
    if (tid == kSchedThreads - 1) s_carry += incl;
    __syncthreads();
  }
  const long long total = s_carry;
  if (total > p.max_ctas) {
    if (tid == 0) p.hdr->error = 1;
    return;
  }
  if (tid == 0) p.first_cta[p.num_seqs] = static_cast<int>(total);
  __syncthreads();

  const int n_ctas = static_cast<int>(total);
  fill_table(p, p.cu_seqlens, p.cp_size, p.order, p.first_cta, n_ctas, tid);
  if (tid == 0) p.hdr->n_items = n_ctas;
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream) {
  schedule_kernel<<<1, kSchedThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace cpattn
