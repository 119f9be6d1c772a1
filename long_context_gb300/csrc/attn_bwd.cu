// Ring-attention backward for sm_103a: dQ, dK, dV of the forward in
// attn_fwd.cu, on the tensor cores (tcgen05, accumulators in TMEM, tiles
// staged by TMA).
//
// The gradient is the exact derivative of the forward's definition ("Megatron
// 架构与 6D 并行完整指南", section 六: every query attends to every visible
// key).  With P = exp(scale * Q K^T - LSE) over visible pairs and an upstream
// dO:
//   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
// LSE comes from the forward, so P needs no running max here.  The work is
// split by the ring's chunks as in the forward: the dQ kernel walks the KV
// chunks of its query block in the forward's ring order, and the dK/dV kernel
// walks the query chunks that see its key block in the order they visit it
// (chunk j, j + 1, ...).
//
// Both kernels: 384 threads, one CTA per SM (224 KB of shared memory: two
// stationary and five streamed 32 KB tiles; 512 TMEM columns):
//   warps 0-7  compute: warps w and w + 4 share the TMEM lanes of quarter w
//              (thread = one row of the stationary tile), for the first and
//              the second 64 columns of each streamed tile
//   warp  8    TMA producer
//   warp  9    MMA issuer (one thread) and TMEM owner
//   warp  10   waits for the streamed tiles' copies
//   warp  11   idle
// The MMA warp never waits on an mbarrier (a wait right after
// tcgen05.commit stalls the tensor queue).  It is released by hardware named
// barriers: barrier 3 for the first hand-off of each streamed tile and
// barrier 4 for the second, on which the compute warps arrive (bar.arrive)
// once their TMEM results are in place and warp 10 once the next tile's copy
// has landed; in the dK/dV kernel also barrier 5 (compute warps only), once
// the first half of P^T is in place.  A compute warp whose bounded wait failed switches to bar.sync
// for its remaining hand-offs, so it cannot arrive twice before a barrier
// completes, and every warp takes part in every hand-off: the MMA warp always
// runs to its end.
//
// dQ kernel, per 128-query tile, TMEM: S [0,128), dP [128,256), dQ [256,384).
//   S = Q K^T, dP = dO V^T; dS (bf16 pairs) of key columns [0,64) and
//   [64,128) overwrites dP columns [0,32) and [64,96); dQ += dS K (A from
//   TMEM, B = K MN-major).
// dK/dV kernel, per 128-key tile, TMEM: S^T [0,128), dP^T [128,256),
//   dV [256,384), dK [384,512).  S^T = K Q^T, dP^T = V dO^T; P^T and dS^T
//   (bf16 pairs) overwrite columns [0,32) and [64,96) of their regions;
//   dV += P^T dO, dK += dS^T Q.
#include <cuda_bf16.h>

#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "work.cuh"

namespace cpattn {

namespace {

constexpr int kBwdThreads = 384;
constexpr int kComputeThreads = 256;  // warps 0-7
// Named barriers 3 and 4: the compute warps, warp 10 and the MMA warp.
constexpr int kHandoffThreads = kComputeThreads + 64;
// Named barrier 5 (dK/dV kernel): the compute warps and the MMA warp.
constexpr int kHalfThreads = kComputeThreads + 32;
// Register split (setmaxnreg): launched at 168 per thread, the compute
// warpgroups rise to 224 and the control warpgroup drops to 56.
constexpr int kBwdLaunchRegs = 168;
constexpr int kBwdSoftmaxRegs = 224;
constexpr int kBwdCtrlRegs = 56;
static_assert(kBwdThreads * kBwdLaunchRegs == kComputeThreads * kBwdSoftmaxRegs + 128 * kBwdCtrlRegs,
              "the register split must add up to the launch total");
constexpr int kT = 128;  // rows of a tile (queries or keys)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInf = __builtin_huge_valf();
constexpr int kErrTimeout = 6;

// S0 / S1: stages of the rings of streamed tiles B0 / B1; kWithVec: room for
// the dK/dV kernel's per-tile column statistics.
template <int D, int S0, int S1, bool kWithVec>
struct BwdCfg {
  static constexpr int kTileBytes = kT * D * 2;
  static constexpr int kStages0 = S0;
  static constexpr int kStages1 = S1;
  // Stationary tiles A0, A1 (dQ kernel: Q, dO; dK/dV kernel: K, V) and the
  // stage rings B0, B1 of the streamed tiles (dQ: K, V; dK/dV: Q, dO).
  static constexpr int kA0Off = 0;
  static constexpr int kA1Off = kTileBytes;
  static constexpr int kB0Off = 2 * kTileBytes;
  static constexpr int kB1Off = kB0Off + S0 * kTileBytes;
  // dK/dV kernel: LSE * log2 e and D of the current streamed query tile's
  // 128 queries (float [2][128]).
  static constexpr int kVecOff = kB1Off + S1 * kTileBytes;
  static constexpr int kBarOff = kVecOff + (kWithVec ? 2 * kT * 4 : 0);
  // a_full, b0_full[S0], b0_empty[S0], b1_full[S1], b1_empty[S1], s_full,
  // o_done, drain, dp_full
  static constexpr int kNumBars = 1 + 2 * S0 + 2 * S1 + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + align slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
};

// dK/dV: Q is read twice per tile (S^T = K Q^T, then dK += dS^T Q), so its
// stage is freed late, after dK; a third Q stage lets the copy of tile x + 1
// start a whole tile earlier.  dO's stage is freed after dV.
template <int D>
using DkdvCfg = BwdCfg<D, 3, 2, true>;
// dQ: K is read twice per tile (S = Q K^T, then dQ += dS K), so its stage is
// freed late; a third K stage gives its copy a full tile period more.
template <int D>
using DqCfg = BwdCfg<D, 3, 2, false>;

// Query chunks visited by a stationary query block: the forward's ring (KV
// chunk (i - s) mod c at step s), restricted to keys below q_blk_end on the
// diagonal when causal.
struct QRing {
  int L, c, chunk, i, causal, q_blk_end;
  __device__ __forceinline__ void seg(int s, int& lo, int& n_tiles, int& end) const {
    n_tiles = 0;
    lo = 0;
    end = 0;
    if (s >= c) return;
    int j = i - s;
    if (j < 0) j += c;
    lo = min(j * chunk, L);
    end = min((j + 1) * chunk, L);
    int hi = end;
    if (causal) {
      if (j > i) return;
      if (j == i) hi = min(hi, q_blk_end);
    }
    if (hi > lo) n_tiles = (hi - lo + kT - 1) / kT;
  }
};

// Query chunks that see a stationary key block of chunk j, in the order they
// visit it around the ring: chunk (j + s) mod c at step s; causal keeps the
// chunks at or after j, and on chunk j the query tiles from the key block on.
struct KRing {
  int L, c, chunk, j, causal, kv0;
  __device__ __forceinline__ void seg(int s, int& lo, int& n_tiles, int& end) const {
    n_tiles = 0;
    lo = 0;
    end = 0;
    if (s >= c) return;
    int i = j + s;
    if (i >= c) i -= c;
    if (causal && i < j) return;
    lo = min(i * chunk, L);
    end = min((i + 1) * chunk, L);
    if (causal && i == j) lo = kv0;
    if (end > lo) n_tiles = (end - lo + kT - 1) / kT;
  }
};

template <class R>
struct Walk {  // flattened (step, tile) sequence of a ring
  int s, kt, nt, lo, end;
  __device__ __forceinline__ void skip_empty(const R& r) {
    while (s < r.c) {
      r.seg(s, lo, nt, end);
      if (nt > 0) return;
      ++s;
    }
  }
  __device__ __forceinline__ void start(const R& r) {
    s = 0;
    kt = 0;
    skip_empty(r);
  }
  __device__ __forceinline__ void advance(const R& r) {
    if (++kt < nt) return;
    kt = 0;
    ++s;
    skip_empty(r);
  }
  __device__ __forceinline__ bool done(const R& r) const { return s >= r.c; }
  __device__ __forceinline__ int tile_row() const { return lo + kt * kT; }
};

template <class R>
__device__ __forceinline__ int count_tiles(const R& r) {
  Walk<R> w;
  w.start(r);
  int n = 0;
  for (; !w.done(r); w.advance(r)) ++n;
  return n;
}

__device__ __forceinline__ void raise_error(WsHeader* hdr, int code) {
  atomicCAS(&hdr->error, 0, code);
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 200000000ull) return false;  // 0.2 s
  }
  return true;
}

// Shared-memory descriptor words (start address >> 4 in the low 14 bits plus
// the leading byte offset; the high word is constant).
template <int D>
struct Desc {
  uint32_t hi_k, hi_mn;
  __device__ __forceinline__ Desc() {
    hi_k = static_cast<uint32_t>(sdesc_sw128(0, 16, 1024) >> 32);
    hi_mn = static_cast<uint32_t>(sdesc_sw128(0, 16384, 1024) >> 32);
  }
  __device__ __forceinline__ uint32_t lo_k(uint32_t addr) const {
    return static_cast<uint32_t>(sdesc_sw128(addr, 16, 1024));
  }
  __device__ __forceinline__ uint32_t lo_mn(uint32_t addr) const {
    return static_cast<uint32_t>(sdesc_sw128(addr, 16384, 1024));
  }
};

// C[128 x 128] (TMEM col d) = A[128 x D] B[128 x D]^T, both K-major in
// shared memory (descriptor low words a, b).
template <int D>
__device__ __forceinline__ void mma_abt(uint32_t d, uint32_t a, uint32_t b, uint32_t hi) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, kT, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
    mma_ss(d, pack_u64(a + off, hi), pack_u64(b + off, hi), idesc, kk > 0 ? 1u : 0u);
  }
}

// C[128 x D] (TMEM col d) (+)= A[128 x 128] * B[128 x D], B MN-major in
// shared memory (descriptor low word b).  A is in TMEM as bf16 pairs: its
// first 64 K-columns packed in columns [a, a + 32), the last 64 in
// [a + 64, a + 96) (each half written by the warps that own those columns).
template <int D>
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a, uint32_t b, uint32_t hi,
                                           bool acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, D, true);
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    mma_ts(d, a + kk * 8 + (kk >= 4 ? 32 : 0), pack_u64(b + ((kk * 2048) >> 4), hi), idesc,
           (acc || kk > 0) ? 1u : 0u);
}

// The half of mma_tmem_a over the K-columns that the compute warps write
// first (half 0: [0, 32) and [64, 96); half 1: [32, 64) and [96, 128)), so
// that the product can start before all of A is in TMEM.
template <int D>
__device__ __forceinline__ void mma_tmem_a_half(uint32_t d, uint32_t a, uint32_t b, uint32_t hi,
                                                bool acc, int half) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, D, true);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int kk = (j & 1) + 2 * half + 4 * (j >> 1);
    mma_ts(d, a + kk * 8 + (kk >= 4 ? 32 : 0), pack_u64(b + ((kk * 2048) >> 4), hi), idesc,
           (acc || j > 0) ? 1u : 0u);
  }
}

// Loads a 128-row bf16 tile (rows row0.., head h) into shared memory.  (The
// debug build checks row0 against the T rows of the tensor.)
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int h, int row0, uint64_t pol, const BwdParams& p) {
  row0 = checked_coord(row0, 0, static_cast<int>(p.total_tokens), p.hdr);
#pragma unroll
  for (int hf = 0; hf < D / 64; ++hf)
    tma_load_3d(dst + hf * 16384, map, bar, hf * 64, h, row0, pol);
}

// The debug build's check of a work entry: rows of this batch, a valid head,
// CP size, rank and block start (false: the CTA does nothing).
__device__ __forceinline__ bool unit_in_bounds(int tok0, int L, int h, int c, int rank,
                                               int first, int chunk_end, const BwdParams& p) {
  if (!kDebugChecks) return true;
  return in_bounds(tok0, 0, p.total_tokens + 1, p.hdr) &&
         in_bounds(static_cast<long long>(tok0) + L, 0, p.total_tokens + 1, p.hdr) &&
         in_bounds(h, 0, p.num_heads, p.hdr) && in_bounds(c, 1, kMaxCp + 1, p.hdr) &&
         in_bounds(rank, 0, c, p.hdr) && in_bounds(first, 0, chunk_end, p.hdr);
}

// Byte offset of 16-byte chunk c of row r in a 128-row tile buffer laid out
// as 64-column halves of 128-byte rows with the 128-byte swizzle (the TMA
// load layout).
__device__ __forceinline__ int swizzle128(int r, int c) {
  return (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Columns [col0, col0 + NC) of this thread's row r of a [128 x D] fp32 TMEM
// accumulator (TMEM address `taddr` = that row at column col0), times `mul`,
// to bf16 in global memory, where tile row i starts at g0 + i * ld.  The
// rows go out through `stage`, a free 128-row tile buffer: each thread writes
// its row there in the swizzled layout (conflict-free), then the warp copies
// its own 32 rows (from row0) out with NC / 8 lanes per row, so each store
// instruction writes whole row segments instead of 16 bytes of 32 rows.
// Rows i >= n_rows are not written.
template <int NC>
__device__ __forceinline__ void store_rows_staged(uint32_t taddr, float mul, uint8_t* stage,
                                                  int r, int col0, int lane, int row0,
                                                  __nv_bfloat16* g0, size_t ld, int n_rows) {
  uint32_t v[NC];
#pragma unroll
  for (int q = 0; q < NC / 32; ++q) tmem_ld32(taddr + q * 32, v + q * 32);
  tmem_wait_ld();
#pragma unroll
  for (int q = 0; q < NC / 32; ++q) reg_fence32(v + q * 32);
  fence_proxy_async_smem();
#pragma unroll
  for (int q = 0; q < NC / 32; ++q) {
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = pack_bf16x2(__uint_as_float(v[q * 32 + 2 * e]) * mul,
                         __uint_as_float(v[q * 32 + 2 * e + 1]) * mul);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint4*>(stage + swizzle128(r, (col0 + q * 32) / 8 + e)) =
          make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
  }
  __syncwarp();
  constexpr int kLpr = NC / 8;      // lanes per row: one 16-byte chunk each
  constexpr int kRpi = 32 / kLpr;  // rows per store instruction
  const int c = col0 / 8 + lane % kLpr;
#pragma unroll 4
  for (int it = 0; it < 32 / kRpi; ++it) {
    const int rr = row0 + it * kRpi + lane / kLpr;
    const uint4 val = *reinterpret_cast<const uint4*>(stage + swizzle128(rr, c));
    if (rr < n_rows) *reinterpret_cast<uint4*>(g0 + rr * ld + c * 8) = val;
  }
}

// A compute warp's arrival on hand-off barrier `id`: non-blocking while its
// waits succeed; blocking once one has failed (it then skips its work, and
// must not run ahead of the barrier).
__device__ __forceinline__ void handoff(uint32_t id, bool ok, uint32_t n = kHandoffThreads) {
  if (ok)
    named_bar_arrive(id, n);
  else
    named_bar_sync(id, n);
}

struct UnitIds {
  int tok0, L, h, c, rank, blk, chunk;
};

__device__ __forceinline__ UnitIds decode(const CtaWork& w) {
  UnitIds u;
  u.tok0 = w.x;
  u.L = w.y;
  u.h = static_cast<int>(static_cast<unsigned>(w.z) >> 8);
  u.c = w.z & 0xff;
  u.rank = w.w & 0xff;
  u.blk = static_cast<int>(static_cast<unsigned>(w.w) >> 8);
  u.chunk = cdiv(u.L, u.c);
  return u;
}

}  // namespace

// ------------------------------------------------------------------ delta --
// Two rows per warp: 16 lanes x 8 features (16-byte loads) per row at D=128.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ out,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta,
                                                        long long rows) {
  constexpr int kLanesPerRow = D / 8;                // 16 at D=128, 8 at D=64
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r0 = warp_id * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
    const long long r = r0 + lane / kLanesPerRow;
    float acc = 0.f;
    if (r < rows) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(out + r * D) + lane % kLanesPerRow);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + r * D) + lane % kLanesPerRow);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(a2[e]);
        const float2 y = __bfloat1622float2(b2[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int o = kLanesPerRow / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (r < rows && lane % kLanesPerRow == 0) delta[r] = acc;
  }
}

// -------------------------------------------------------------- dK / dV --
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = DkdvCfg<D>;
  // Programmatic dependent of the schedule kernel: wait for its table, then
  // let the dQ kernel (independent of this one) start launching.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int x_cta = static_cast<int>(blockIdx.x);
  const int n_ctas = __ldcg(&p.hdr->n_items);
  const int err0 = __ldcg(&p.hdr->error);
  const CtaWork work = __ldg(&p.table[x_cta]);
  if (x_cta >= n_ctas) return;
  if (err0 == kErrTimeout) return;

  const UnitIds u = decode(work);
  const int kv0 = min(u.rank * u.chunk, u.L) + u.blk * kT;        // first key of the tile
  const int kv_blk_end = min(kv0 + kT, min((u.rank + 1) * u.chunk, u.L));
  KRing ring{u.L, u.c, u.chunk, u.rank, p.causal, kv0};
  if (!unit_in_bounds(u.tok0, u.L, u.h, u.c, u.rank, kv0, min((u.rank + 1) * u.chunk, u.L), p))
    return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* a_full = bars;
  uint64_t* b0_full = bars + 1;
  uint64_t* b0_empty = b0_full + C::kStages0;
  uint64_t* b1_full = b0_empty + C::kStages0;
  uint64_t* b1_empty = b1_full + C::kStages1;
  uint64_t* s_full = b1_empty + C::kStages1;
  uint64_t* o_done = s_full + 1;
  uint64_t* drain = o_done + 1;
  uint64_t* dp_full = drain + 1;  // dP^T ready (S^T ready is s_full)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  float* vec = reinterpret_cast<float*>(smem + C::kVecOff);  // [lse2 | delta][128]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 8 && lane == 0) {
    mbar_init(a_full, 1);
    for (int st = 0; st < C::kStages0; ++st) {
      mbar_init(&b0_full[st], 1);
      mbar_init(&b0_empty[st], 1);
    }
    for (int st = 0; st < C::kStages1; ++st) {
      mbar_init(&b1_full[st], 1);
      mbar_init(&b1_empty[st], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(dp_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    mbar_arrive_expect_tx(a_full, 2 * C::kTileBytes);
    load_tile<D>(smem + C::kA0Off, &tm_k, a_full, u.h, u.tok0 + kv0, pol_kv, p);
    load_tile<D>(smem + C::kA1Off, &tm_v, a_full, u.h, u.tok0 + kv0, pol_kv, p);
    Walk<KRing> w;
    w.start(ring);
    if (!w.done(ring)) {  // query tile 0 goes to stage 0, which is free
      const int row = u.tok0 + w.tile_row();
      mbar_arrive_expect_tx(&b0_full[0], C::kTileBytes);
      load_tile<D>(smem + C::kB0Off, &tm_q, &b0_full[0], u.h, row, pol_q, p);
      mbar_arrive_expect_tx(&b1_full[0], C::kTileBytes);
      load_tile<D>(smem + C::kB1Off, &tm_do, &b1_full[0], u.h, row, pol_q, p);
    }
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  static_assert(kBwdSoftmaxRegs == 224 && kBwdCtrlRegs == 56, "immediates below");
  if (warp >= 8) {
    regs_lower_56();
    // Work decoded again after the register split (values live across it
    // would be spilled there).
    const UnitIds u = decode(__ldg(&p.table[x_cta]));
    const int kv0 = min(u.rank * u.chunk, u.L) + u.blk * kT;
    const int kv_blk_end = min(kv0 + kT, min((u.rank + 1) * u.chunk, u.L));
    const KRing ring{u.L, u.c, u.chunk, u.rank, p.causal, kv0};
    if (warp == 8) {
      // -------------------------------------------------------- TMA producer --
      if (lane == 0) {
        const uint64_t pol_q = l2_policy_evict_last();
        Walk<KRing> w;
        w.start(ring);
        int nb0 = 0, nb1 = 0;
        if (!w.done(ring)) {
          nb0 = nb1 = 1;
          w.advance(ring);
        }
        bool ok = true;
        for (; !w.done(ring); w.advance(ring)) {
          const int x = nb0;
          const int st0 = x % C::kStages0;
          const uint32_t ph0 = (x / C::kStages0) & 1;
          const int st1 = x % C::kStages1;
          const uint32_t ph1 = (x / C::kStages1) & 1;
          const int row = u.tok0 + w.tile_row();
          ok = wait_bounded(&b0_empty[st0], ph0 ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&b0_full[st0], C::kTileBytes);
          load_tile<D>(smem + C::kB0Off + st0 * C::kTileBytes, &tm_q, &b0_full[st0], u.h, row, pol_q, p);
          ++nb0;
          ok = wait_bounded(&b1_empty[st1], ph1 ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&b1_full[st1], C::kTileBytes);
          load_tile<D>(smem + C::kB1Off + st1 * C::kTileBytes, &tm_do, &b1_full[st1], u.h, row, pol_q, p);
          ++nb1;
        }
        if (!ok) {
          raise_error(p.hdr, kErrTimeout);
          *abort_flag = 1;
        }
        wait_drain(a_full, 0);
        for (int st = 0; st < C::kStages0; ++st)
          if (st < nb0) wait_drain(&b0_full[st], (((nb0 - 1 - st) / C::kStages0)) & 1);
        for (int st = 0; st < C::kStages1; ++st)
          if (st < nb1) wait_drain(&b1_full[st], (((nb1 - 1 - st) / C::kStages1)) & 1);
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer --
      const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
      const Desc<D> dsc;
      const uint32_t k_lo = dsc.lo_k(smem_u32(smem + C::kA0Off));
      const uint32_t v_lo = dsc.lo_k(smem_u32(smem + C::kA1Off));
      const uint32_t q_lo_k = dsc.lo_k(smem_u32(smem + C::kB0Off));
      const uint32_t do_lo_k = dsc.lo_k(smem_u32(smem + C::kB1Off));
      const uint32_t q_lo_mn = dsc.lo_mn(smem_u32(smem + C::kB0Off));
      const uint32_t do_lo_mn = dsc.lo_mn(smem_u32(smem + C::kB1Off));
      constexpr uint32_t kStageLo = C::kTileBytes >> 4;
      const int n = count_tiles(ring);
      // Three hand-offs per query tile x: once the first half of P^T(x) (the
      // compute warps' first 32 columns each) is in TMEM, the half of dV(x)
      // over those queries; once all of P^T(x) is, the other half and then
      // S^T(x + 1) (which overwrites P^T(x) after dV(x) has read it); once
      // dS^T(x) is in TMEM, dK(x) and then dP^T(x + 1).  The exponentials of
      // tile x + 1 thus overlap dK(x) and dP^T(x + 1), and the second half of
      // P^T(x) overlaps the first half of dV(x).
      named_bar_sync(1, 64);  // K, V and query tile 0 landed
      if (lane == 0 && n > 0) {
        tc_fence_after();
        mma_abt<D>(tmem, k_lo, q_lo_k, dsc.hi_k);            // S^T = K Q^T
        mma_commit(s_full);
        mma_abt<D>(tmem + kT, v_lo, do_lo_k, dsc.hi_k);      // dP^T = V dO^T
        mma_commit(dp_full);
      }
      __syncwarp();
      for (int x = 0; x < n; ++x) {
        // Q (ring B0) and dO (ring B1) of tile x and x + 1.
        const uint32_t q_st = static_cast<uint32_t>(x) % C::kStages0;
        const uint32_t q_st1 = static_cast<uint32_t>(x + 1) % C::kStages0;
        const uint32_t do_st = static_cast<uint32_t>(x) % C::kStages1;
        const uint32_t do_st1 = static_cast<uint32_t>(x + 1) % C::kStages1;
        named_bar_sync(5, kHalfThreads);  // the first half of P^T(x) in TMEM
        if (lane == 0) {
          tc_fence_after();
          mma_tmem_a_half<D>(tmem + 2 * kT, tmem, do_lo_mn + do_st * kStageLo, dsc.hi_mn, x > 0, 0);
        }
        __syncwarp();
        named_bar_sync(3, kHandoffThreads);  // P^T(x) in TMEM; query tile x + 1 landed
        if (lane == 0) {
          tc_fence_after();
          mma_tmem_a_half<D>(tmem + 2 * kT, tmem, do_lo_mn + do_st * kStageLo, dsc.hi_mn, true, 1);
          mma_commit(&b1_empty[do_st]);  // dO(x): last read by dV(x)
          if (x + 1 < n) {
            mma_abt<D>(tmem, k_lo, q_lo_k + q_st1 * kStageLo, dsc.hi_k);
            mma_commit(s_full);
          }
        }
        __syncwarp();
        named_bar_sync(4, kHandoffThreads);  // dS^T(x) in TMEM; dO tile x + 1 landed
        if (lane == 0) {
          tc_fence_after();
          mma_tmem_a<D>(tmem + 3 * kT, tmem + kT, q_lo_mn + q_st * kStageLo, dsc.hi_mn, x > 0);  // dK
          mma_commit(&b0_empty[q_st]);
          if (x == n - 1) mma_commit(o_done);
          if (x + 1 < n) {
            mma_abt<D>(tmem + kT, v_lo, do_lo_k + do_st1 * kStageLo, dsc.hi_k);
            mma_commit(dp_full);
          }
        }
        __syncwarp();
      }
      if (lane == 0) {
        mma_commit(drain);
        wait_drain(drain, 0);
      }
      __syncwarp();
    } else if (warp == 10) {
      // --------------------------------------------- waits for the MMA warp --
      const int n = count_tiles(ring);
      bool ok = true;
      if (lane == 0) {
        ok = wait_bounded(a_full, 0, abort_flag);
        if (ok && n > 0) ok = wait_bounded(&b0_full[0], 0, abort_flag);
        if (ok && n > 0) ok = wait_bounded(&b1_full[0], 0, abort_flag);
      }
      __syncwarp();
      named_bar_sync(1, 64);
      for (int x = 0; x < n; ++x) {
        const int st0n = (x + 1) % C::kStages0;
        const uint32_t ph0n = ((x + 1) / C::kStages0) & 1;
        const int st1n = (x + 1) % C::kStages1;
        const uint32_t ph1n = ((x + 1) / C::kStages1) & 1;
        if (lane == 0 && ok && x + 1 < n) ok = wait_bounded(&b0_full[st0n], ph0n, abort_flag);
        __syncwarp();
        named_bar_sync(3, kHandoffThreads);
        if (lane == 0 && ok && x + 1 < n) ok = wait_bounded(&b1_full[st1n], ph1n, abort_flag);
        __syncwarp();
        named_bar_sync(4, kHandoffThreads);
      }
      if (lane == 0 && !ok) {
        raise_error(p.hdr, kErrTimeout);
        *abort_flag = 1;
      }
      __syncwarp();
    }
  } else {
    regs_raise_224();
    // Work decoded again after the register split (values live across it
    // would be spilled there).
    const UnitIds u = decode(__ldg(&p.table[x_cta]));
    const int kv0 = min(u.rank * u.chunk, u.L) + u.blk * kT;
    const int kv_blk_end = min(kv0 + kT, min((u.rank + 1) * u.chunk, u.L));
    const KRing ring{u.L, u.c, u.chunk, u.rank, p.causal, kv0};
    // -------------------------------------------------------------- compute --
    // Thread r of warps 0-3 and thread r of warps 4-7 own key kv0 + r (TMEM
    // lane r), the first for query columns [0, 64), the second for [64, 128).
    // For each streamed query tile: P^T[r, i] = 2^(S^T[r, i] scale log2 e -
    // LSE_i log2 e) over the queries i that see key r, and
    // dS^T[r, i] = P^T[r, i] (dP^T[r, i] - D_i).
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const int r = threadIdx.x & (kT - 1);
    const int ch = warp >> 2;  // column half
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t row_addr = tmem + lane_base;
    const int k_pos = kv0 + r;
    const float c2 = p.scale_log2;
    const float2 c22 = make_float2(c2, c2);
    const int n = count_tiles(ring);
    bool ok = true;
    Walk<KRing> w;
    w.start(ring);
    // Column statistics, one tile ahead: for column r of a tile (query
    // tile_row + r, if it belongs to the chunk) warps 0-3 load its LSE and
    // warps 4-7 its D.  The load for tile x + 1 is issued at the top of tile
    // x and consumed at the top of tile x + 1, so its round trip to L2 or
    // DRAM overlaps a whole tile's work instead of preceding its exponentials.
    // One shared-memory buffer: it is rewritten once every compute warp is
    // done with the previous tile.
    Walk<KRing> w_next = w;
    float col_raw = 0.f;
    bool col_ok = false;
    auto fetch_col = [&](const Walk<KRing>& wt) {
      const int qp = wt.tile_row() + r;
      col_ok = qp < wt.end && in_bounds(u.tok0 + qp, 0, p.total_tokens, p.hdr);
      if (col_ok) {
        const size_t ri = static_cast<size_t>(u.tok0 + qp) * p.num_heads + u.h;
        col_raw = __ldg(ch == 0 ? &p.lse[ri] : &p.delta[ri]);
      }
    };
    if (n > 0) fetch_col(w_next);
    for (int x = 0; x < n; ++x, w.advance(ring)) {
      const int qt0 = w.tile_row();  // first query of the tile (sample position)
      float* lse_s = vec;
      float* dlt_s = vec + kT;
      if (x > 0) named_bar_sync(2, kComputeThreads);  // tile x - 1's statistics are read
      // +inf LSE outside the chunk: P = 0 there.
      if (ch == 0)
        lse_s[r] = col_ok ? col_raw * kLog2e : kInf;
      else
        dlt_s[r] = col_ok ? col_raw : 0.f;
      if (x + 1 < n) {
        w_next.advance(ring);
        fetch_col(w_next);
      }
      named_bar_sync(2, kComputeThreads);  // the column statistics are in shared memory
#ifdef CPATTN_FAULT_INJECT_DROP_P
      // Test-only build: in CTA 0, compute warp 0 waits for its first S^T on
      // the drain barrier, which completes only after the last MMA, so its
      // bounded wait runs out; the warp then takes part in the remaining
      // hand-offs with bar.sync, and the kernels end with a timeout status.
      uint64_t* s_wait = (blockIdx.x == 0 && warp == 0 && x == 0) ? drain : s_full;
#else
      uint64_t* s_wait = s_full;
#endif
      if (ok) ok = __all_sync(0xffffffffu, wait_bounded(s_wait, x & 1, abort_flag));
      const float4* lse4 = reinterpret_cast<const float4*>(lse_s);
      const float4* dlt4 = reinterpret_cast<const float4*>(dlt_s);
      float pv[64];
      if (ok) {
        tc_fence_after();
        // Causal: query i sees key k_pos iff qt0 + i >= k_pos.
        const int col_lo = p.causal ? max(0, k_pos - qt0) : 0;
        const bool masked = __any_sync(0xffffffffu, col_lo > 64 * ch);
        // Phase 1: P^T of this half's columns [64 ch, 64 ch + 64), kept in
        // registers and stored packed to columns [64 ch, 64 ch + 32) of the
        // S^T region (columns this thread has already read).
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t sv[32];
          tmem_ld32(row_addr + ch * 64 + q * 32, sv);
          tmem_wait_ld();
          reg_fence32(sv);
          uint32_t pw[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int c0 = ch * 64 + q * 32 + 4 * e4;
            const float4 l4 = lse4[c0 / 4];
#pragma unroll
            for (int j2 = 0; j2 < 2; ++j2) {
              const int e = 4 * e4 + 2 * j2;
              const float2 nl = j2 ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
              const float2 xs = __ffma2_rn(
                  make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c22, nl);
              float2 pp = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
              if (masked) {
                if (c0 + 2 * j2 < col_lo) pp.x = 0.f;
                if (c0 + 2 * j2 + 1 < col_lo) pp.y = 0.f;
              }
              pv[q * 32 + e] = pp.x;
              pv[q * 32 + e + 1] = pp.y;
              pw[2 * e4 + j2] = pack_bf16x2(pp.x, pp.y);
            }
          }
          tmem_st16(row_addr + ch * 64 + q * 16, pw);
          if (q == 0) {  // the first half of P^T: dV can start on it
            tmem_wait_st();
            tc_fence_before();
            named_bar_arrive(5, kHalfThreads);
          }
        }
        tmem_wait_st();
        tc_fence_before();
      } else {
        named_bar_sync(5, kHalfThreads);
      }
      handoff(3, ok);
      // Phase 2: dS^T = P^T (dP^T - D), stored packed over the dP^T region
      // the same way.
      if (ok) ok = __all_sync(0xffffffffu, wait_bounded(dp_full, x & 1, abort_flag));
      {
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t dv[32];
            tmem_ld32(row_addr + kT + ch * 64 + q * 32, dv);
            tmem_wait_ld();
            reg_fence32(dv);
            uint32_t dw[16];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int c0 = ch * 64 + q * 32 + 4 * e4;
              const float4 d4 = dlt4[c0 / 4];
#pragma unroll
              for (int j2 = 0; j2 < 2; ++j2) {
                const int e = 4 * e4 + 2 * j2;
                const float2 nd = j2 ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
                const float2 ds = __fmul2_rn(
                    make_float2(pv[q * 32 + e], pv[q * 32 + e + 1]),
                    __fadd2_rn(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd));
                dw[2 * e4 + j2] = pack_bf16x2(ds.x, ds.y);
              }
            }
            tmem_st16(row_addr + kT + ch * 64 + q * 16, dw);
          }
          tmem_wait_st();
          tc_fence_before();
        }
      }
      handoff(4, ok);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, wait_bounded(o_done, 0, abort_flag));
      if (ok) {
        tc_fence_after();
        // dV goes out through the K buffer, dK through the V buffer (every
        // MMA reading them has completed).
        const size_t ri0 = static_cast<size_t>(u.tok0 + kv0) * p.num_heads + u.h;
        const size_t ld = static_cast<size_t>(p.num_heads) * D;
        const int n_rows =
            in_bounds(static_cast<long long>(u.tok0) + kv_blk_end, 1, p.total_tokens + 1, p.hdr)
                ? kv_blk_end - kv0
                : 0;
        if (ch == 0)
          store_rows_staged<D>(row_addr + 2 * kT, 1.f, smem + C::kA0Off, r, 0, lane,
                               (warp & 3) * 32, p.dv + ri0 * D, ld, n_rows);
        else
          store_rows_staged<D>(row_addr + 3 * kT, p.scale, smem + C::kA1Off, r, 0, lane,
                               (warp & 3) * 32, p.dk + ri0 * D, ld, n_rows);
        tc_fence_before();
      }
    }
    if (!ok) {
      raise_error(p.hdr, kErrTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), C::kTmemCols);
  }
}

// ------------------------------------------------------------------- dQ --
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = DqCfg<D>;
  const int x_cta = static_cast<int>(blockIdx.x);
  const int n_ctas = __ldcg(&p.hdr->n_items);
  const int err0 = __ldcg(&p.hdr->error);
  const CtaWork work = __ldg(&p.table[x_cta]);
  // Programmatic dependent of the dK/dV kernel, which it does not read: it
  // starts while dK/dV's last CTAs run, and every CTA waits for dK/dV before
  // it exits, so the backward completes only when both have.
  if (x_cta >= n_ctas || err0 == kErrTimeout) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }

  const UnitIds u = decode(work);
  const int q0 = min(u.rank * u.chunk, u.L) + u.blk * kT;
  const int q_blk_end = min(q0 + kT, min((u.rank + 1) * u.chunk, u.L));
  QRing ring{u.L, u.c, u.chunk, u.rank, p.causal, q_blk_end};
  if (!unit_in_bounds(u.tok0, u.L, u.h, u.c, u.rank, q0, min((u.rank + 1) * u.chunk, u.L), p)) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* a_full = bars;
  uint64_t* b0_full = bars + 1;
  uint64_t* b0_empty = b0_full + C::kStages0;
  uint64_t* b1_full = b0_empty + C::kStages0;
  uint64_t* b1_empty = b1_full + C::kStages1;
  uint64_t* s_full = b1_empty + C::kStages1;
  uint64_t* o_done = s_full + 1;
  uint64_t* drain = o_done + 1;
  uint64_t* dp_full = drain + 1;   // dP ready (S ready is s_full)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 8 && lane == 0) {
    mbar_init(a_full, 1);
    for (int st = 0; st < C::kStages0; ++st) {
      mbar_init(&b0_full[st], 1);
      mbar_init(&b0_empty[st], 1);
    }
    for (int st = 0; st < C::kStages1; ++st) {
      mbar_init(&b1_full[st], 1);
      mbar_init(&b1_empty[st], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(dp_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();
    mbar_arrive_expect_tx(a_full, 2 * C::kTileBytes);
    load_tile<D>(smem + C::kA0Off, &tm_q, a_full, u.h, u.tok0 + q0, pol_q, p);
    load_tile<D>(smem + C::kA1Off, &tm_do, a_full, u.h, u.tok0 + q0, pol_q, p);
    Walk<QRing> w;
    w.start(ring);
    if (!w.done(ring)) {
      const int row = u.tok0 + w.tile_row();
      mbar_arrive_expect_tx(&b0_full[0], C::kTileBytes);
      load_tile<D>(smem + C::kB0Off, &tm_k, &b0_full[0], u.h, row, pol_kv, p);
      mbar_arrive_expect_tx(&b1_full[0], C::kTileBytes);
      load_tile<D>(smem + C::kB1Off, &tm_v, &b1_full[0], u.h, row, pol_kv, p);
    }
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  static_assert(kBwdSoftmaxRegs == 224 && kBwdCtrlRegs == 56, "immediates below");
  if (warp >= 8) {
    regs_lower_56();
    // Work decoded again after the register split (values live across it
    // would be spilled there).
    const UnitIds u = decode(__ldg(&p.table[x_cta]));
    const int q0 = min(u.rank * u.chunk, u.L) + u.blk * kT;
    const int q_blk_end = min(q0 + kT, min((u.rank + 1) * u.chunk, u.L));
    const QRing ring{u.L, u.c, u.chunk, u.rank, p.causal, q_blk_end};
    if (warp == 8) {
      // -------------------------------------------------------- TMA producer --
      if (lane == 0) {
        const uint64_t pol_kv = l2_policy_evict_last();
        Walk<QRing> w;
        w.start(ring);
        int nb0 = 0, nb1 = 0;
        if (!w.done(ring)) {
          nb0 = nb1 = 1;
          w.advance(ring);
        }
        bool ok = true;
        for (; !w.done(ring); w.advance(ring)) {
          const int x = nb0;
          const int st0 = x % C::kStages0;
          const uint32_t ph0 = (x / C::kStages0) & 1;
          const int st1 = x % C::kStages1;
          const uint32_t ph1 = (x / C::kStages1) & 1;
          const int row = u.tok0 + w.tile_row();
          ok = wait_bounded(&b0_empty[st0], ph0 ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&b0_full[st0], C::kTileBytes);
          load_tile<D>(smem + C::kB0Off + st0 * C::kTileBytes, &tm_k, &b0_full[st0], u.h, row, pol_kv, p);
          ++nb0;
          ok = wait_bounded(&b1_empty[st1], ph1 ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&b1_full[st1], C::kTileBytes);
          load_tile<D>(smem + C::kB1Off + st1 * C::kTileBytes, &tm_v, &b1_full[st1], u.h, row, pol_kv, p);
          ++nb1;
        }
        if (!ok) {
          raise_error(p.hdr, kErrTimeout);
          *abort_flag = 1;
        }
        wait_drain(a_full, 0);
        for (int st = 0; st < C::kStages0; ++st)
          if (st < nb0) wait_drain(&b0_full[st], (((nb0 - 1 - st) / C::kStages0)) & 1);
        for (int st = 0; st < C::kStages1; ++st)
          if (st < nb1) wait_drain(&b1_full[st], (((nb1 - 1 - st) / C::kStages1)) & 1);
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer --
      const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
      const Desc<D> dsc;
      const uint32_t q_lo = dsc.lo_k(smem_u32(smem + C::kA0Off));
      const uint32_t do_lo = dsc.lo_k(smem_u32(smem + C::kA1Off));
      const uint32_t k_lo_k = dsc.lo_k(smem_u32(smem + C::kB0Off));
      const uint32_t v_lo_k = dsc.lo_k(smem_u32(smem + C::kB1Off));
      const uint32_t k_lo_mn = dsc.lo_mn(smem_u32(smem + C::kB0Off));
      constexpr uint32_t kStageLo = C::kTileBytes >> 4;
      const int n = count_tiles(ring);
      // Two hand-offs per KV tile x: once the compute warps have read S(x),
      // S(x + 1); once dS(x) is in TMEM (over the dP region), dQ(x) and then
      // dP(x + 1).  S(x + 1) thus overlaps the dS phase of tile x, and dQ(x),
      // dP(x + 1) the exponentials of tile x + 1.
      named_bar_sync(1, 64);  // Q, dO and KV tile 0 landed
      if (lane == 0 && n > 0) {
        tc_fence_after();
        mma_abt<D>(tmem, q_lo, k_lo_k, dsc.hi_k);          // S = Q K^T
        mma_commit(s_full);
        mma_abt<D>(tmem + kT, do_lo, v_lo_k, dsc.hi_k);    // dP = dO V^T
        mma_commit(dp_full);
        mma_commit(&b1_empty[0]);                          // V consumed
      }
      __syncwarp();
      for (int x = 0; x < n; ++x) {
        // K (ring B0) and V (ring B1) of tile x and x + 1.
        const uint32_t k_st = static_cast<uint32_t>(x) % C::kStages0;
        const uint32_t k_st1 = static_cast<uint32_t>(x + 1) % C::kStages0;
        const uint32_t v_st1 = static_cast<uint32_t>(x + 1) % C::kStages1;
        named_bar_sync(3, kHandoffThreads);  // S(x) read out; KV tile x + 1's K landed
        if (lane == 0 && x + 1 < n) {
          tc_fence_after();
          mma_abt<D>(tmem, q_lo, k_lo_k + k_st1 * kStageLo, dsc.hi_k);
          mma_commit(s_full);
        }
        __syncwarp();
        named_bar_sync(4, kHandoffThreads);  // dS(x) in TMEM; KV tile x + 1's V landed
        if (lane == 0) {
          tc_fence_after();
          mma_tmem_a<D>(tmem + 2 * kT, tmem + kT, k_lo_mn + k_st * kStageLo, dsc.hi_mn, x > 0);  // dQ
          mma_commit(&b0_empty[k_st]);                                                            // K done
          if (x == n - 1) mma_commit(o_done);
          if (x + 1 < n) {
            mma_abt<D>(tmem + kT, do_lo, v_lo_k + v_st1 * kStageLo, dsc.hi_k);
            mma_commit(dp_full);
            mma_commit(&b1_empty[v_st1]);
          }
        }
        __syncwarp();
      }
      if (lane == 0) {
        mma_commit(drain);
        wait_drain(drain, 0);
      }
      __syncwarp();
    } else if (warp == 10) {
      // --------------------------------------------- waits for the MMA warp --
      const int n = count_tiles(ring);
      bool ok = true;
      if (lane == 0) {
        ok = wait_bounded(a_full, 0, abort_flag);
        if (ok && n > 0) ok = wait_bounded(&b0_full[0], 0, abort_flag);
        if (ok && n > 0) ok = wait_bounded(&b1_full[0], 0, abort_flag);
      }
      __syncwarp();
      named_bar_sync(1, 64);
      for (int x = 0; x < n; ++x) {
        const int st0n = (x + 1) % C::kStages0;
        const uint32_t ph0n = ((x + 1) / C::kStages0) & 1;
        const int st1n = (x + 1) % C::kStages1;
        const uint32_t ph1n = ((x + 1) / C::kStages1) & 1;
        if (lane == 0 && ok && x + 1 < n) ok = wait_bounded(&b0_full[st0n], ph0n, abort_flag);
        __syncwarp();
        named_bar_sync(3, kHandoffThreads);
        if (lane == 0 && ok && x + 1 < n) ok = wait_bounded(&b1_full[st1n], ph1n, abort_flag);
        __syncwarp();
        named_bar_sync(4, kHandoffThreads);
      }
      if (lane == 0 && !ok) {
        raise_error(p.hdr, kErrTimeout);
        *abort_flag = 1;
      }
      __syncwarp();
    }
  } else {
    regs_raise_224();
    // Work decoded again after the register split (values live across it
    // would be spilled there).
    const UnitIds u = decode(__ldg(&p.table[x_cta]));
    const int q0 = min(u.rank * u.chunk, u.L) + u.blk * kT;
    const int q_blk_end = min(q0 + kT, min((u.rank + 1) * u.chunk, u.L));
    const QRing ring{u.L, u.c, u.chunk, u.rank, p.causal, q_blk_end};
    // -------------------------------------------------------------- compute --
    // Thread r of warps 0-3 and of warps 4-7 own query q0 + r (TMEM lane r),
    // for key columns [0, 64) and [64, 128) of each KV tile:
    // P = 2^(S scale log2 e - LSE log2 e) over the visible keys (a prefix of
    // the tile) and dS = P (dP - D).
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const int r = threadIdx.x & (kT - 1);
    const int ch = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t row_addr = tmem + lane_base;
    const int q_pos = q0 + r;
    const bool row_valid =
        q_pos < q_blk_end && in_bounds(u.tok0 + q_pos, 0, p.total_tokens, p.hdr);
    const size_t ri = static_cast<size_t>(u.tok0 + q_pos) * p.num_heads + u.h;
    const float lse2 = row_valid ? __ldg(&p.lse[ri]) * kLog2e : 0.f;
    const float dlt = row_valid ? __ldg(&p.delta[ri]) : 0.f;
    const float c2 = p.scale_log2;
    const float2 c22 = make_float2(c2, c2);
    const float2 nl = make_float2(-lse2, -lse2);
    const float2 nd = make_float2(-dlt, -dlt);
    const int n = count_tiles(ring);
    bool ok = true;
    Walk<QRing> w;
    w.start(ring);
    for (int x = 0; x < n; ++x, w.advance(ring)) {
      if (ok) ok = __all_sync(0xffffffffu, wait_bounded(s_full, x & 1, abort_flag));
      float pv[64];
      if (ok) {
        tc_fence_after();
        const int kv0 = w.tile_row();
        const int lim = p.causal ? min(w.end, q_pos + 1) : w.end;
        const int nvis = lim - kv0;  // visible keys: a prefix of the tile
        const bool masked = __any_sync(0xffffffffu, nvis < 64 * ch + 64);
        // Phase 1: P of this half's key columns [64 ch, 64 ch + 64), kept in
        // registers; then S's region is released for S(x + 1).
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t sv[32];
          tmem_ld32(row_addr + ch * 64 + q * 32, sv);
          tmem_wait_ld();
          reg_fence32(sv);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = ch * 64 + q * 32 + 2 * e;
            const float2 xs = __ffma2_rn(
                make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), c22, nl);
            float2 pp = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
            if (masked) {
              if (c0 >= nvis) pp.x = 0.f;
              if (c0 + 1 >= nvis) pp.y = 0.f;
            }
            pv[q * 32 + 2 * e] = pp.x;
            pv[q * 32 + 2 * e + 1] = pp.y;
          }
        }
        tc_fence_before();
      }
      handoff(3, ok);
      // Phase 2: dS = P (dP - D), stored packed to columns
      // [64 ch, 64 ch + 32) of the dP region (already read here).
      if (ok) ok = __all_sync(0xffffffffu, wait_bounded(dp_full, x & 1, abort_flag));
      {
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t dv[32];
            tmem_ld32(row_addr + kT + ch * 64 + q * 32, dv);
            tmem_wait_ld();
            reg_fence32(dv);
            uint32_t dw[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 ds = __fmul2_rn(
                  make_float2(pv[q * 32 + 2 * e], pv[q * 32 + 2 * e + 1]),
                  __fadd2_rn(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nd));
              dw[e] = pack_bf16x2(ds.x, ds.y);
            }
            tmem_st16(row_addr + kT + ch * 64 + q * 16, dw);
          }
          tmem_wait_st();
          tc_fence_before();
        }
      }
      handoff(4, ok);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, wait_bounded(o_done, 0, abort_flag));
      if (ok) {
        tc_fence_after();
        // Warps 0-3 write output columns [0, D/2), warps 4-7 [D/2, D), both
        // through the Q buffer (every MMA reading it has completed).
        const size_t ri0 = static_cast<size_t>(u.tok0 + q0) * p.num_heads + u.h;
        store_rows_staged<D / 2>(row_addr + 2 * kT + ch * (D / 2), p.scale, smem + C::kA0Off, r,
                                 ch * (D / 2), lane, (warp & 3) * 32, p.dq + ri0 * D,
                                 static_cast<size_t>(p.num_heads) * D,
                                 in_bounds(static_cast<long long>(u.tok0) + q_blk_end, 1,
                                           p.total_tokens + 1, p.hdr)
                                     ? q_blk_end - q0
                                     : 0);
        tc_fence_before();
      }
    }
    if (!ok) {
      raise_error(p.hdr, kErrTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), C::kTmemCols);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}


cudaError_t launch_bwd_delta(const __nv_bfloat16* out, const __nv_bfloat16* dout,
                             float* delta, long long rows, int D, int num_sms,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long warps_needed = (rows + 1) / 2;
  long long blocks = (warps_needed + 7) / 8;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (D == 64)
    bwd_delta_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, dout, delta, rows);
  else
    bwd_delta_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, dout, delta, rows);
  return cudaGetLastError();
}

template <int kSmem>
static cudaError_t launch_kernel(void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                                              BwdParams),
                                 const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo,
                                 const BwdParams& p, long long grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  // The register split inside the kernel assumes exactly kBwdLaunchRegs per
  // thread at launch; with any other count the raise could wait forever.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != kBwdLaunchRegs)
    return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, p);
}

cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const BwdParams& p, int D, long long grid, cudaStream_t stream) {
  if (D == 64) return launch_kernel<DkdvCfg<64>::kSmemBytes>(attn_bwd_dkdv_kernel<64>, tq, tk, tv, tdo, p, grid, stream);
  return launch_kernel<DkdvCfg<128>::kSmemBytes>(attn_bwd_dkdv_kernel<128>, tq, tk, tv, tdo, p, grid, stream);
}

cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo,
                          const BwdParams& p, int D, long long grid, cudaStream_t stream) {
  if (D == 64) return launch_kernel<DqCfg<64>::kSmemBytes>(attn_bwd_dq_kernel<64>, tq, tk, tv, tdo, p, grid, stream);
  return launch_kernel<DqCfg<128>::kSmemBytes>(attn_bwd_dq_kernel<128>, tq, tk, tv, tdo, p, grid, stream);
}

}  // namespace cpattn
