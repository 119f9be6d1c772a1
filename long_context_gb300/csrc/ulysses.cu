// Ulysses sequence parallelism ("VeRL Backend Parallelism", the USP section:
// ulysses_sequence_parallel_size splits the sequence over the SP group of a
// [dp, sp] mesh).  Before attention an all-to-all over the group trades
// sequence sharding for head sharding; after attention the inverse trades it
// back.  The concatenation of the sequence shards is the packed [T, H, E]
// array, so on one device both all-to-alls are a transpose of whole head
// groups between
//   sequence layout    [T, P, C]  (token t: its H heads, group by group)
//   head-group layout  [P, T, C]  (group p: heads [p H/P, (p+1) H/P) of all T)
// with C = (H / P) * E bytes (E = bytes of one head's row: D bf16 values for
// Q/K/V/O, one fp32 for the LSE).  A chunk of C bytes is contiguous on both
// sides, so the work is a [T, P] <-> [P, T] transpose of chunks: HBM bound,
// every byte read once and written once.
//
// Also here: the grouped cu_seqlens that lets one cpattn_fwd launch run the
// attention of all P head groups (group p's samples are the original samples
// shifted by p T rows).
#include <cuda_runtime.h>

#include <cstdint>

#include "cpattn.h"
#include "kernels.h"

namespace cpattn {

namespace {

constexpr int kUlyThreads = 256;

// One team of 2^log_team lanes copies one chunk of n_u units; up to sixteen
// loads in flight per lane before their stores (sixteen 16-byte loads per
// lane measured 3.5-4 % faster than four on 1 KB chunks: 0.96-0.97 of the
// copy bandwidth against 0.93).  Chunk r of dst comes from chunk
// src_row(r) of src:
//   to_groups:   dst [P, T] row r = p T + t   <-  src [T, P] row t P + p
//   from_groups: dst [T, P] row r = t P + p   <-  src [P, T] row p T + t
template <typename U>
__global__ void __launch_bounds__(kUlyThreads) ulysses_layout_kernel(
    const U* __restrict__ src, U* __restrict__ dst, uint32_t T, uint32_t P, int n_u,
    int log_team, bool to_groups) {
  const uint32_t n_rows = T * P;  // < 2^31, checked on the host
  const int team = 1 << log_team;
  const uint32_t gtid = blockIdx.x * kUlyThreads + threadIdx.x;
  const int tl = static_cast<int>(gtid & static_cast<uint32_t>(team - 1));
  const uint32_t n_teams = (gridDim.x * kUlyThreads) >> log_team;
  for (uint32_t r = gtid >> log_team; r < n_rows; r += n_teams) {
    uint32_t s_row;
    if (to_groups) {
      const uint32_t p = r / T, t = r - p * T;
      s_row = t * P + p;
    } else {
      const uint32_t t = r / P, p = r - t * P;
      s_row = p * T + t;
    }
    const U* s = src + static_cast<size_t>(s_row) * n_u;
    U* d = dst + static_cast<size_t>(r) * n_u;
    int e = tl;
    for (; e + 15 * team < n_u; e += 16 * team) {
      U a[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) a[j] = __ldcs(s + e + j * team);
#pragma unroll
      for (int j = 0; j < 16; ++j) __stcs(d + e + j * team, a[j]);
    }
    for (; e + 7 * team < n_u; e += 8 * team) {
      U a[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) a[j] = __ldcs(s + e + j * team);
#pragma unroll
      for (int j = 0; j < 8; ++j) __stcs(d + e + j * team, a[j]);
    }
    for (; e + 3 * team < n_u; e += 4 * team) {
      const U a0 = __ldcs(s + e), a1 = __ldcs(s + e + team);
      const U a2 = __ldcs(s + e + 2 * team), a3 = __ldcs(s + e + 3 * team);
      __stcs(d + e, a0);
      __stcs(d + e + team, a1);
      __stcs(d + e + 2 * team, a2);
      __stcs(d + e + 3 * team, a3);
    }
    for (; e < n_u; e += team) __stcs(d + e, __ldcs(s + e));
  }
}

__device__ __forceinline__ int sat_i32(long long x) {
  return x > 0x7fffffffLL ? 0x7fffffff : static_cast<int>(x);
}

// cu_out[p B + b] = cu[b] + p T (b < B), cu_out[P B] = cu[B] + (P - 1) T
// (cu[0] for an empty batch); cp_out[p B + b] = cp[b] (1 when cp is null).
// Out-of-range sums saturate, which the forward's cu_seqlens check rejects.
__global__ void ulysses_seqlens_kernel(const int* __restrict__ cu, const int* __restrict__ cp,
                                       int B, int P, int T, int* __restrict__ cu_out,
                                       int* __restrict__ cp_out) {
  const int n = P * B;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += gridDim.x * blockDim.x) {
    if (i == n) {
      cu_out[n] = B == 0 ? cu[0] : sat_i32(cu[B] + static_cast<long long>(P - 1) * T);
    } else {
      const int p = i / B, b = i - p * B;
      cu_out[i] = sat_i32(cu[b] + static_cast<long long>(p) * T);
      if (cp_out) cp_out[i] = cp ? cp[b] : 1;
    }
  }
}

int uly_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

template <typename U>
void launch_layout(const void* src, void* dst, uint32_t T, uint32_t P, long long chunk_bytes,
                   bool to_groups, int sms, cudaStream_t s) {
  const int n_u = static_cast<int>(chunk_bytes / static_cast<long long>(sizeof(U)));
  // Team: the largest power of two <= 32 that still gives each lane sixteen units.
  int log_team = 0;
  while (log_team < 5 && (16 << (log_team + 1)) <= n_u) ++log_team;
  const long long threads = static_cast<long long>(T) * P << log_team;
  long long blocks = (threads + kUlyThreads - 1) / kUlyThreads;
  const long long cap = 8LL * sms;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  ulysses_layout_kernel<U><<<static_cast<unsigned>(blocks), kUlyThreads, 0, s>>>(
      static_cast<const U*>(src), static_cast<U*>(dst), T, P, n_u, log_team, to_groups);
}

}  // namespace

}  // namespace cpattn

using namespace cpattn;

extern "C" int cpattn_ulysses_layout(const void* src, void* dst, int64_t num_tokens,
                                     int32_t num_heads, int64_t head_bytes, int32_t sp_size,
                                     int32_t to_head_groups, void* stream) {
  if (num_tokens < 0 || num_heads < 1 || sp_size < 1 || head_bytes < 1 ||
      num_heads % sp_size != 0 || (to_head_groups != 0 && to_head_groups != 1))
    return CPATTN_ERR_INVALID_ARG;
  const long long chunk = static_cast<long long>(num_heads / sp_size) * head_bytes;
  if (chunk % 4 != 0 || chunk >= (1LL << 31)) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens * static_cast<long long>(sp_size) >= (1LL << 31)) return CPATTN_ERR_INVALID_ARG;
  if (num_tokens == 0) return CPATTN_OK;
  if (src == nullptr || dst == nullptr || src == dst || !aligned(src, 4) || !aligned(dst, 4))
    return CPATTN_ERR_INVALID_ARG;
  const int sms = uly_sms();
  if (sms <= 0) return CPATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint32_t T = static_cast<uint32_t>(num_tokens), P = static_cast<uint32_t>(sp_size);
  const bool tg = to_head_groups != 0;
  if (chunk % 16 == 0 && aligned(src, 16) && aligned(dst, 16))
    launch_layout<uint4>(src, dst, T, P, chunk, tg, sms, s);
  else if (chunk % 8 == 0 && aligned(src, 8) && aligned(dst, 8))
    launch_layout<uint2>(src, dst, T, P, chunk, tg, sms, s);
  else
    launch_layout<unsigned int>(src, dst, T, P, chunk, tg, sms, s);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

extern "C" int cpattn_ulysses_seqlens(const int32_t* cu_seqlens, const int32_t* cp_size,
                                      int32_t num_seqs, int64_t num_tokens, int32_t sp_size,
                                      int32_t* cu_out, int32_t* cp_out, void* stream) {
  if (num_seqs < 0 || num_tokens < 0 || sp_size < 1 || cu_seqlens == nullptr ||
      cu_out == nullptr || !aligned(cu_seqlens, 4) || !aligned(cu_out, 4) ||
      (cp_size && !aligned(cp_size, 4)) || (cp_out && !aligned(cp_out, 4)))
    return CPATTN_ERR_INVALID_ARG;
  if (num_tokens * static_cast<long long>(sp_size) >= (1LL << 31) ||
      static_cast<long long>(num_seqs) * sp_size >= (1LL << 30))
    return CPATTN_ERR_INVALID_ARG;
  const int n = sp_size * num_seqs + 1;
  const int blocks = n / 256 + 1 < 1024 ? n / 256 + 1 : 1024;
  ulysses_seqlens_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      cu_seqlens, cp_size, num_seqs, sp_size, static_cast<int>(num_tokens), cu_out, cp_out);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}
