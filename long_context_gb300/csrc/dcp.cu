// Data movement around attention under dynamic CP ("Dynamic Context
// Parallelism (DCP)", verl documentation): every DPxCP rank selects its
// assigned samples from the shared mini-batch, the CP group's output is
// gathered, and the outputs are put back in the original sample order.  On one
// device both steps are permutations of whole samples between two packed THD
// arrays:
//   select  (gather):  sample ids[i] of the original array -> slot i of a
//                      packed array (cu_seqlens = prefix of the lengths)
//   restore (scatter): slot i of the packed array -> sample ids[i] of the
//                      original array
// HBM bound: one warp per token row, 16-byte vector copies.
#include <cuda_runtime.h>

#include <cstdint>

#include "cpattn.h"
#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kPermThreads = 256;
constexpr int kCuSmem = 4096;  // packed-side cu_seqlens staged in shared memory

// dst_cu[0] = 0, dst_cu[i + 1] = dst_cu[i] + length of sample ids[i]; also
// validates ids (an id out of range writes 0 lengths and sets *bad).
__global__ void __launch_bounds__(1024) select_cu_kernel(const int* __restrict__ src_cu,
                                                         int num_src, const int* __restrict__ ids,
                                                         int n, int* __restrict__ dst_cu,
                                                         int* __restrict__ bad) {
  __shared__ long long warp_sums[32];
  __shared__ long long carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    dst_cu[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int i = base + tid;
    long long len = 0;
    if (i < n) {
      const int b = ids[i];
      if (b < 0 || b >= num_src) {
        atomicExch(bad, 1);
      } else {
        len = src_cu[b + 1] - src_cu[b];
      }
    }
    long long v = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      long long w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const long long incl = v + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (i < n) dst_cu[i + 1] = static_cast<int>(incl);
    __syncthreads();
    if (tid == 1023) carry = incl;
    __syncthreads();
  }
}

// Copies whole samples between the original array (orig, orig_cu indexed by
// sample id) and a packed array (pack, pack_cu indexed by slot i).  gather:
// orig -> pack; otherwise pack -> orig.  Rows are row_bytes long (a multiple
// of 4; of 16 when vec16).
template <bool vec16>
__global__ void __launch_bounds__(kPermThreads) permute_kernel(
    const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, const int* __restrict__ orig_cu,
    const int* __restrict__ pack_cu, const int* __restrict__ ids, int n, long long row_bytes,
    bool gather, int num_orig, const int* __restrict__ bad) {
  __shared__ int s_cu[kCuSmem + 1];
  if (*bad) return;  // invalid ids: nothing is copied
  const bool staged = n <= kCuSmem;
  if (staged)
    for (int i = threadIdx.x; i <= n; i += kPermThreads) s_cu[i] = pack_cu[i];
  __syncthreads();
  const int* cu = staged ? s_cu : pack_cu;
  const long long rows = cu[n];
  const int lane = threadIdx.x & 31;
  const int n_vec = static_cast<int>(row_bytes / (vec16 ? 16 : 4));  // rows < 2^31 bytes
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kPermThreads + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * kPermThreads) >> 5;
  int slot = 0;
  for (long long t = warp0; t < rows; t += n_warps) {
    // Slot of packed row t: largest i with cu[i] <= t (starting from the
    // previous slot, rows only increase).
    if (t >= cu[slot + 1] || t < cu[slot]) {
      int lo = t >= cu[slot] ? slot : 0, hi = n - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
      }
      slot = lo;
    }
    const int b = ids[slot];
    if (b < 0 || b >= num_orig) continue;
    // A packed layout that does not match the original lengths copies nothing
    // beyond the original sample.
    if (t - cu[slot] >= static_cast<long long>(orig_cu[b + 1]) - orig_cu[b]) continue;
    const long long o_row = orig_cu[b] + (t - cu[slot]);
    const uint8_t* s = src + (gather ? o_row : t) * row_bytes;
    uint8_t* d = dst + (gather ? t : o_row) * row_bytes;
    if (vec16) {
      // Sixteen 16-byte loads in flight per lane before their stores (a whole
      // 8 KB row per warp), then four.
      const uint4* s4 = reinterpret_cast<const uint4*>(s);
      uint4* d4 = reinterpret_cast<uint4*>(d);
      int e = lane;
      for (; e + 15 * 32 < n_vec; e += 16 * 32) {
        uint4 a[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) a[j] = __ldcs(s4 + e + j * 32);
#pragma unroll
        for (int j = 0; j < 16; ++j) __stcs(d4 + e + j * 32, a[j]);
      }
      for (; e + 96 < n_vec; e += 128) {
        const uint4 a0 = __ldcs(s4 + e), a1 = __ldcs(s4 + e + 32);
        const uint4 a2 = __ldcs(s4 + e + 64), a3 = __ldcs(s4 + e + 96);
        __stcs(d4 + e, a0);
        __stcs(d4 + e + 32, a1);
        __stcs(d4 + e + 64, a2);
        __stcs(d4 + e + 96, a3);
      }
      for (; e < n_vec; e += 32) __stcs(d4 + e, __ldcs(s4 + e));
    } else {
      const uint32_t* s1 = reinterpret_cast<const uint32_t*>(s);
      uint32_t* d1 = reinterpret_cast<uint32_t*>(d);
      for (int e = lane; e < n_vec; e += 32) d1[e] = s1[e];
    }
  }
}

int dcp_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

}  // namespace

}  // namespace cpattn

using namespace cpattn;

extern "C" int cpattn_select_cu(const int32_t* src_cu, int32_t num_seqs, const int32_t* ids,
                                int32_t n, int32_t* dst_cu, int32_t* status, void* stream) {
  if (num_seqs < 0 || n < 0 || src_cu == nullptr || dst_cu == nullptr || status == nullptr)
    return CPATTN_ERR_INVALID_ARG;
  if (n > 0 && ids == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (!aligned(src_cu, 4) || !aligned(dst_cu, 4) || !aligned(status, 4) ||
      (ids && !aligned(ids, 4)))
    return CPATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return CPATTN_ERR_CUDA;
  select_cu_kernel<<<1, 1024, 0, s>>>(src_cu, num_seqs, ids, n, dst_cu, status);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

extern "C" int cpattn_permute_samples(const void* src, const int32_t* orig_cu,
                                      int32_t num_seqs, const int32_t* pack_cu,
                                      const int32_t* ids, int32_t n, int64_t row_bytes,
                                      int32_t gather, void* dst, const int32_t* status,
                                      void* stream) {
  if (num_seqs < 0 || n < 0 || row_bytes < 4 || row_bytes % 4 != 0 ||
      row_bytes >= (int64_t(1) << 31) || (gather != 0 && gather != 1))
    return CPATTN_ERR_INVALID_ARG;
  if (orig_cu == nullptr || pack_cu == nullptr || status == nullptr ||
      !aligned(orig_cu, 4) || !aligned(pack_cu, 4) || !aligned(status, 4))
    return CPATTN_ERR_INVALID_ARG;
  if (n == 0) return CPATTN_OK;
  if (src == nullptr || dst == nullptr || ids == nullptr || !aligned(ids, 4) ||
      !aligned(src, 4) || !aligned(dst, 4))
    return CPATTN_ERR_INVALID_ARG;
  const bool vec16 = row_bytes % 16 == 0 && aligned(src, 16) && aligned(dst, 16);
  const int sms = dcp_sms();
  if (sms <= 0) return CPATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(sms) * 8;
  if (vec16)
    permute_kernel<true><<<grid, kPermThreads, 0, s>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), orig_cu, pack_cu, ids, n,
        row_bytes, gather != 0, num_seqs, status);
  else
    permute_kernel<false><<<grid, kPermThreads, 0, s>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), orig_cu, pack_cu, ids, n,
        row_bytes, gather != 0, num_seqs, status);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}
