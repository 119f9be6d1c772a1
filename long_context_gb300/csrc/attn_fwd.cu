// Ring-attention forward for sm_103a: block attention on the tensor cores
// (tcgen05, accumulators in TMEM, Q/K/V tiles staged by TMA) with the
// online-softmax merge of the ring folded into the same kernel.
//
// What is computed follows the ring_attention listing of "Megatron 架构与 6D
// 并行完整指南", section 六: a sample split into c CP chunks; rank i holds Q chunk
// i and at ring step s the KV chunk (i - s) mod c; each step's block attention
// (O_step, m_step, l_step) is folded into (O, m, l) with
//   m_new = max(m, m_step), alpha = exp(m - m_new), beta = exp(m_step - m_new),
//   l = alpha l + beta l_step, O = alpha O + beta O_step,
// and the result is O / l.  The kernel walks the same chunks in the same ring
// order, 128 keys at a time, and applies that merge after every KV tile
// rather than only at chunk boundaries (a KV tile is a sub-block of a chunk,
// so the fold is the same operation at a finer grain).  In partials mode the
// running state restarts at every ring step and each step's (O_step, m_step,
// l_step) is written out for the standalone merge kernel.
//
// CTA organisation (384 threads, one CTA per SM):
//   warps 0-3   softmax for Q tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q tile 1
//   warp  8     TMA producer (Q once, then K/V tiles through a stage ring)
//   warp  9     MMA issuer (one thread) and TMEM owner
//   warp  10    waits on the hand-offs (mbarriers) for the MMA issuer and
//               releases it through a named barrier: an mbarrier wait in the
//               issuing thread right after tcgen05.commit stalls until the
//               queued MMAs drain (measured on GB300: about 300 cycles of
//               idle tensor pipe per wait)
//   warp  11    idle
// The softmax warpgroups take 224 registers per thread and the control
// warpgroup (warps 8-11) gives its share up, down to 56.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 and O1 at 256 + t*D.
// P_t (bf16, two per column) overwrites the first 64 columns of S_t; the
// next S_t is issued after PV_t, and tcgen05 MMAs of one thread run in order.
#include <cuda_bf16.h>

#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "work.cuh"

namespace cpattn {

namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLn2 = 0.69314718055994530942f;
// The running max is only moved when a tile's max exceeds it by more than
// this many powers of two; until then exp2 values stay below 2^8.  O and l
// share the stale reference, so O / l and m + ln l are unchanged.
constexpr float kRescaleThreshold = 8.0f;
// A tile whose exponentials, taken against the running max as it stands,
// sum above this bound is redone with its own row max (so every P value
// stays below 2^16).
constexpr float kMaxLazyTileSum = 65536.0f;

enum : int {
  kErrInvalid = 1,
  kErrTimeout = 6,
};

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;          // 128-byte swizzle atoms
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kNQ * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[NQ],
  // p_full[NQ], o_done[NQ], drain, staged[NQ]
  static constexpr int kNumBars = 1 + 4 * kStages + 3 * kNQ + 1 + kNQ;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + align slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 2 * kBN;
};

// The KV chunks one CTA visits, in ring order.
struct Ring {
  int L, c, chunk, i, causal, q_blk_end, num_steps;

  // Ring step s: keys [kv_lo, kv_lo + 128 * n_tiles) of chunk (i - s) mod c
  // are processed; kv_end is that chunk's end (keys at or beyond it are
  // masked).
  __device__ __forceinline__ void seg(int s, int& kv_lo, int& n_tiles,
                                      int& kv_end) const {
    n_tiles = 0;
    kv_lo = 0;
    kv_end = 0;
    if (s >= c) return;
    int j = i - s;
    if (j < 0) j += c;
    kv_lo = min(j * chunk, L);
    kv_end = min((j + 1) * chunk, L);
    int hi = kv_end;
    if (causal) {
      if (j > i) return;
      if (j == i) hi = min(hi, q_blk_end);
    }
    if (hi > kv_lo) n_tiles = (hi - kv_lo + kBN - 1) / kBN;
  }
};

// Cursor over the flattened (step, tile) sequence of a Ring.
struct Cursor {
  int s, kt, nt, kv_lo, kv_end;
  __device__ __forceinline__ void skip_empty(const Ring& r) {
    while (s < r.num_steps) {
      r.seg(s, kv_lo, nt, kv_end);
      if (nt > 0) return;
      ++s;
    }
  }
  __device__ __forceinline__ void start(const Ring& r) {
    s = 0;
    kt = 0;
    skip_empty(r);
  }
  __device__ __forceinline__ void advance(const Ring& r) {
    if (++kt < nt) return;
    kt = 0;
    ++s;
    skip_empty(r);
  }
  __device__ __forceinline__ bool first() const { return kt == 0; }
  __device__ __forceinline__ bool last() const { return kt == nt - 1; }
};

// Byte offset of 16-byte chunk c of row r in a tile stored as 64-column
// halves of 128-byte rows with the 128-byte swizzle (the TMA load layout).
__device__ __forceinline__ int swizzle128(int r, int c) {
  return (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void raise_error(WsHeader* hdr, int code) {
  atomicCAS(&hdr->error, 0, code);
}

// Wait that ignores the CTA abort flag (used to drain copies in flight).
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 200000000ull) return false;  // 0.2 s
  }
  return true;
}

}  // namespace

template <int D, bool PARTIALS>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
  using C = Cfg<D>;
  // Launched as a programmatic dependent of the schedule kernel: wait for
  // its table (a no-op when launched normally).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The three loads are independent, so they are in flight together.  The
  // table holds an entry for every CTA of the grid (used or not).
  const int x_cta = static_cast<int>(blockIdx.x);
  const int n_ctas = __ldcg(&p.hdr->n_items);
  const int err0 = __ldcg(&p.hdr->error);
  const CtaWork work = __ldg(&p.table[x_cta]);
  if (x_cta >= n_ctas) return;
  // After one CTA gave up on a wait, the rest of the grid does no work.
  if (err0 == kErrTimeout) return;

  // CTA -> (sample, head, rank, block): see work.cuh for the order.
  SampleGeom geo;
  geo.L = work.y;
  geo.c = work.z & 0xff;
  geo.chunk = cdiv(geo.L, geo.c);
  const int h = static_cast<int>(static_cast<unsigned>(work.z) >> 8);
  const int rank = work.w & 0xff;
  const int blk = static_cast<int>(static_cast<unsigned>(work.w) >> 8);
  const int tok0 = work.x;
  Ring ring;
  ring.L = geo.L;
  ring.c = geo.c;
  ring.chunk = geo.chunk;
  ring.i = rank;
  ring.causal = p.causal;
  ring.num_steps = p.num_steps;
  // The chunk's query blocks are aligned to its end: block blk covers rows
  // [q_lo, q_hi) with q_hi = chunk end - (blocks after it) * 256, so only
  // block 0 can be short, and a short block is the chunk's cheapest (its
  // rows see the fewest keys) rather than its costliest.  Its Q tiles start
  // before the chunk (q0 may even be negative: TMA fills those rows with
  // zeros); the rows before q_lo are computed but never stored.
  const int qc_lo = min(rank * ring.chunk, ring.L);
  const int qc_hi = min((rank + 1) * ring.chunk, ring.L);
  const int n_blk = cdiv(qc_hi - qc_lo, kRowsPerItem);
  const int q_hi = qc_hi - (n_blk - 1 - blk) * kRowsPerItem;
  const int q_lo = max(q_hi - kRowsPerItem, qc_lo);
  ring.q_blk_end = q_hi;
  // The first Q tile is skipped when the block has no rows for it.
  const int nq = (q_lo + kBM < q_hi) ? kNQ : 1;
  const int q0 = q_hi - nq * kBM;  // first row of Q tile 0
  if (kDebugChecks) {
    // The work entry must address rows of this batch and a valid head, CP
    // size, rank and block (every CTA thread reads the same entry, so the
    // whole CTA leaves together, before any barrier or TMEM allocation).
    const bool ok = in_bounds(tok0, 0, p.total_tokens + 1, p.hdr) &&
                    in_bounds(static_cast<long long>(tok0) + geo.L, 0, p.total_tokens + 1,
                              p.hdr) &&
                    in_bounds(h, 0, p.num_heads, p.hdr) &&
                    in_bounds(geo.c, 1, kMaxCp + 1, p.hdr) &&
                    in_bounds(rank, 0, geo.c, p.hdr) && in_bounds(blk, 0, n_blk, p.hdr) &&
                    in_bounds(q_lo, qc_lo, qc_hi, p.hdr);
    if (!ok) return;
  }
  const int T32 = static_cast<int>(p.total_tokens);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::kStages;
  uint64_t* v_full = k_empty + C::kStages;
  uint64_t* v_empty = v_full + C::kStages;
  uint64_t* s_full = v_empty + C::kStages;
  uint64_t* p_full = s_full + kNQ;
  uint64_t* o_done = p_full + kNQ;
  uint64_t* drain = o_done + kNQ;
  uint64_t* staged = drain + 1;  // O tile t staged in shared memory (128 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The producer thread sets up the barriers and starts the copies of Q and
  // of the first K/V tile before the CTA-wide barrier, so that their latency
  // overlaps the TMEM allocation and the barrier.
  if (warp == 8 && lane == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(&k_full[st], 1);
      mbar_init(&k_empty[st], 1);
      mbar_init(&v_full[st], 1);
      mbar_init(&v_empty[st], 1);
    }
    for (int t = 0; t < kNQ; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], kBM);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    for (int t = 0; t < kNQ; ++t) mbar_init(&staged[t], kBM);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();
    mbar_arrive_expect_tx(q_full, nq * C::kTileBytes);
    for (int t = 0; t < nq; ++t) {
      const int qrow = checked_coord(tok0 + q0 + t * kBM, -kBM, T32, p.hdr);
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(smem + C::kQOff + t * C::kTileBytes + hf * 16384, &tm_q, q_full,
                    hf * 64, h, qrow, pol_q);
    }
    Cursor cur;
    cur.start(ring);
    if (cur.s < ring.num_steps) {  // tile 0 goes to stage 0, which is free
      const int row = checked_coord(tok0 + cur.kv_lo, 0, T32, p.hdr);
      mbar_arrive_expect_tx(&k_full[0], C::kTileBytes);
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(smem + C::kKOff + hf * 16384, &tm_k, &k_full[0], hf * 64, h, row,
                    pol_kv);
      mbar_arrive_expect_tx(&v_full[0], C::kTileBytes);
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(smem + C::kVOff + hf * 16384, &tm_v, &v_full[0], hf * 64, h, row,
                    pol_kv);
    }
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  static_assert(kSoftmaxRegs == 224 && kCtrlRegs == 56, "immediates below");

  if (warp >= 8) {
    regs_lower_56();
    if (warp == 8) {
      // ------------------------------------------------------ TMA producer --
      if (lane == 0) {
        const uint64_t pol_kv = l2_policy_evict_last();
        uint8_t* sk = smem + C::kKOff;
        uint8_t* sv = smem + C::kVOff;
        // Warm L2 with the Q tiles of CTA x_cta + num_sms, which in table
        // order starts about when one of the running CTAs ends: its first
        // copy then reads L2 instead of DRAM.
        {
          const int nx = x_cta + p.num_sms;
          if (nx < n_ctas) {
            const CtaWork wn = __ldg(&p.table[nx]);
            const int Ln = wn.y, cn = wn.z & 0xff;
            const int hn = static_cast<int>(static_cast<unsigned>(wn.z) >> 8);
            const int rankn = wn.w & 0xff;
            const int blkn = static_cast<int>(static_cast<unsigned>(wn.w) >> 8);
            const int chunkn = cdiv(Ln, cn);
            const int qc_lon = min(rankn * chunkn, Ln);
            const int qc_hin = min((rankn + 1) * chunkn, Ln);
            const int q_hin = qc_hin - (cdiv(qc_hin - qc_lon, kRowsPerItem) - 1 - blkn) *
                                           kRowsPerItem;
            const int nqn = (max(q_hin - kRowsPerItem, qc_lon) + kBM < q_hin) ? kNQ : 1;
            const int q0n = q_hin - nqn * kBM;
            for (int t = 0; t < nqn; ++t)
              for (int hf = 0; hf < C::kHalves; ++hf)
                tma_prefetch_l2_3d(&tm_q, hf * 64, hn, wn.x + q0n + t * kBM);
          }
        }
        // Q and tile 0 were issued before the CTA barrier.
        Cursor cur;
        cur.start(ring);
        int nk = 0, nv = 0;  // K and V tiles whose copies were issued
        if (cur.s < ring.num_steps) {
          nk = nv = 1;
          cur.advance(ring);
        }
        bool ok = true;
        for (; cur.s < ring.num_steps; cur.advance(ring)) {
          const int x = nk;
          const int st = x % C::kStages;
          const uint32_t ph = (x / C::kStages) & 1;
          const int row = checked_coord(tok0 + cur.kv_lo + cur.kt * kBN, 0, T32, p.hdr);
          ok = wait_bounded(&k_empty[st], ph ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&k_full[st], C::kTileBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(sk + st * C::kTileBytes + hf * 16384, &tm_k, &k_full[st],
                        hf * 64, h, row, pol_kv);
          ++nk;
          ok = wait_bounded(&v_empty[st], ph ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full[st], C::kTileBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(sv + st * C::kTileBytes + hf * 16384, &tm_v, &v_full[st],
                        hf * 64, h, row, pol_kv);
          ++nv;
        }
        if (!ok) {
          raise_error(p.hdr, kErrTimeout);
          *abort_flag = 1;
        }
        // Drain: every copy issued into shared memory must land before exit.
        wait_drain(q_full, 0);
        for (int st = 0; st < C::kStages; ++st) {
          if (st < nk) {
            const int last = st + ((nk - 1 - st) / C::kStages) * C::kStages;
            wait_drain(&k_full[st], (last / C::kStages) & 1);
          }
          if (st < nv) {
            const int last = st + ((nv - 1 - st) / C::kStages) * C::kStages;
            wait_drain(&v_full[st], (last / C::kStages) & 1);
          }
        }
      }
    } else if (warp == 9) {
      // ------------------------------------------------------- MMA issuer --
      // Lane 0 issues every MMA and never touches an mbarrier in the loop: a
      // wait right after a commit stalls the tensor queue.  Warp 10 does the
      // waiting and releases this warp through named barrier 1 before each
      // block of MMAs (both warps run the same number of rendezvous).
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, true);
      const uint32_t sq = smem_u32(smem + C::kQOff);
      const uint32_t sk = smem_u32(smem + C::kKOff);
      const uint32_t sv = smem_u32(smem + C::kVOff);

      // Descriptor words: the high word is constant; the low word holds the
      // start address >> 4 (14 bits, shared memory is below 2^18 bytes) and
      // the leading byte offset, so tile and k-step offsets are 32-bit adds.
      const uint32_t hi_kq = static_cast<uint32_t>(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t hi_v = static_cast<uint32_t>(sdesc_sw128(0, 16384, 1024) >> 32);
      const uint32_t lo_q = static_cast<uint32_t>(sdesc_sw128(sq, 16, 1024));
      const uint32_t lo_k = static_cast<uint32_t>(sdesc_sw128(sk, 16, 1024));
      const uint32_t lo_v = static_cast<uint32_t>(sdesc_sw128(sv, 16384, 1024));
      auto issue_s = [&](int t, int st) {
        const uint32_t d = tmem + t * kBN;
        const uint32_t a0 = lo_q + t * (C::kTileBytes >> 4);
        const uint32_t b0 = lo_k + st * (C::kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(d, pack_u64(a0 + off, hi_kq), pack_u64(b0 + off, hi_kq), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[t]);
      };
      auto issue_pv = [&](int t, int st, bool acc) {
        const uint32_t d = tmem + C::kOCol + t * D;
        const uint32_t a = tmem + t * kBN;
        const uint32_t b0 = lo_v + st * (C::kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(d, a + kk * 8, pack_u64(b0 + ((kk * 2048) >> 4), hi_v), idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
      };

      Cursor cur;
      cur.start(ring);
      int n = 0;
      {
        Cursor c2 = cur;
        for (; c2.s < ring.num_steps; c2.advance(ring)) ++n;
      }
      named_bar_sync(1, 64);  // Q and K(0) landed
      if (lane == 0 && n > 0) {
        tc_fence_after();
        for (int t = 0; t < nq; ++t) issue_s(t, 0);
        mma_commit(&k_empty[0]);
      }
      __syncwarp();
      for (int x = 0; x < n; ++x, cur.advance(ring)) {
        const int st = x % C::kStages;
        // Fused: one accumulation over every ring step.  Partials: O restarts
        // at each ring step and is read out at its end.
        const bool zero_init = PARTIALS ? cur.first() : (x == 0);
        const bool seg_end = PARTIALS ? cur.last() : (x == n - 1);
        const bool has_next = x + 1 < n;
        const int st1 = (x + 1) % C::kStages;
        for (int t = 0; t < nq; ++t) {
          named_bar_sync(1, 64);  // P_t(x), V(x) and K(x+1) are ready
          if (lane == 0) {
            tc_fence_after();
            issue_pv(t, st, !zero_init);
            if (seg_end) mma_commit(&o_done[t]);
            if (t == nq - 1) mma_commit(&v_empty[st]);
            if (has_next) {
              issue_s(t, st1);
              if (t == nq - 1) mma_commit(&k_empty[st1]);
            }
          }
          __syncwarp();
        }
      }
      if (lane == 0) {
        mma_commit(drain);
        wait_drain(drain, 0);
      }
      __syncwarp();
    } else if (warp == 10) {
      // ------------------------------------------------ waits for the MMAs --
      // After a failed (bounded) wait the remaining rendezvous still happen,
      // without waiting, so the MMA warp always runs to its end.
      Cursor cur;
      cur.start(ring);
      int n = 0;
      for (; cur.s < ring.num_steps; cur.advance(ring)) ++n;
      bool ok = true;
      if (lane == 0) {
        ok = wait_bounded(q_full, 0, abort_flag);
        if (ok && n > 0) ok = wait_bounded(&k_full[0], 0, abort_flag);
      }
      __syncwarp();
      named_bar_sync(1, 64);
      for (int x = 0; x < n; ++x) {
        const int st = x % C::kStages;
        const uint32_t ph = (x / C::kStages) & 1;
        const int st1 = (x + 1) % C::kStages;
        const uint32_t ph1 = ((x + 1) / C::kStages) & 1;
        for (int t = 0; t < nq; ++t) {
          if (lane == 0 && ok) {
            if (t == 0) {
              ok = wait_bounded(&v_full[st], ph, abort_flag);
              if (ok && x + 1 < n) ok = wait_bounded(&k_full[st1], ph1, abort_flag);
            }
            if (ok) ok = wait_bounded(&p_full[t], x & 1, abort_flag);
          }
          __syncwarp();
          named_bar_sync(1, 64);
        }
      }
      if (lane == 0 && !ok) {
        raise_error(p.hdr, kErrTimeout);
        *abort_flag = 1;
      }
      __syncwarp();
    }
  } else {
    regs_raise_224();
    if (warp < 4 * nq) {
      // ---------------------------------------------------------- softmax --
      const int t = warp >> 2;
      const int r = threadIdx.x & 127;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t s_addr = tmem + lane_base + t * kBN;
      const uint32_t o_addr = tmem + lane_base + C::kOCol + t * D;
      const int q_pos = q0 + t * kBM + r;
      const bool row_valid = q_pos >= q_lo && q_pos < q_hi;
      const size_t row_idx = static_cast<size_t>(tok0 + q_pos) * p.num_heads + h;
      const float c_log2 = p.scale_log2;

      float m_run = kNegInf;  // running max, log2 domain (scaled score * log2 e)
      float l_run = 0.f;
      int x = 0;
      int seg_done = 0;
      bool ok = true;
      bool any_pv = false;  // a PV has accumulated into O_t (this segment)

      for (int s = 0; s < ring.num_steps && ok; ++s) {
        int kv_lo, nt, kv_end;
        ring.seg(s, kv_lo, nt, kv_end);
        if (PARTIALS) {
          if (nt == 0) {
            if (row_valid &&
                in_bounds(static_cast<long long>(row_idx), 0, p.total_tokens * p.num_heads,
                          p.hdr)) {
              const size_t so = static_cast<size_t>(s) * p.total_tokens * p.num_heads + row_idx;
              float4* dst = reinterpret_cast<float4*>(p.o_steps + so * D);
              for (int q = 0; q < D / 4; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
              p.m_steps[so] = kNegInf;
              p.l_steps[so] = 0.f;
            }
            continue;
          }
          m_run = kNegInf;
          l_run = 0.f;
          any_pv = false;
        }
        for (int kt = 0; kt < nt; ++kt, ++x) {
          ok = __all_sync(0xffffffffu, wait_bounded(&s_full[t], x & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          // The row max is taken only when the warp has a row without a
          // reference yet; otherwise the exponentials use the running max as
          // it is, and the tile is redone with its own max only if that
          // reference was too low (a tile sum above 2^16, or not finite).  S
          // is still in TMEM for the redo, since P has not been written yet.
          bool with_max = __any_sync(0xffffffffu, m_run == kNegInf);
          float2 acc0, acc1;
          uint32_t pk[kBN / 2];
#pragma unroll 1
          for (;;) {
          uint32_t sr[kBN];
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q) tmem_ld32(s_addr + q * 32, sr + q * 32);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q) reg_fence32(sr + q * 32);

          // Visible keys of this row form a prefix of the tile.
          const int kv0 = kv_lo + kt * kBN;
          const int lim = ring.causal ? min(kv_end, q_pos + 1) : kv_end;
          const int nvis = lim - kv0;
          if (nvis < kBN) {
#pragma unroll
            for (int cc = 0; cc < kBN; ++cc)
              if (cc >= nvis) sr[cc] = __float_as_uint(kNegInf);
          }
          if (with_max) {
          // Row max: four chains of 3-input max.
          float mx0 = fmaxf(__uint_as_float(sr[0]), __uint_as_float(sr[1]));
          float mx1 = fmaxf(__uint_as_float(sr[2]), __uint_as_float(sr[3]));
          float mx2 = fmaxf(__uint_as_float(sr[4]), __uint_as_float(sr[5]));
          float mx3 = fmaxf(__uint_as_float(sr[6]), __uint_as_float(sr[7]));
#pragma unroll
          for (int cc = 8; cc < kBN; cc += 8) {
            mx0 = fmax3(mx0, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
            mx1 = fmax3(mx1, __uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3]));
            mx2 = fmax3(mx2, __uint_as_float(sr[cc + 4]), __uint_as_float(sr[cc + 5]));
            mx3 = fmax3(mx3, __uint_as_float(sr[cc + 6]), __uint_as_float(sr[cc + 7]));
          }
          const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c_log2;
          const float m_new = fmaxf(m_run, m_tile);
          const bool need = m_new > m_run + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = (m_run == kNegInf) ? 0.f : ex2_approx(m_run - m_new);
            if (any_pv) {
              // PV of the previous tile completed before S of this tile (same
              // issuing thread, committed in order), so O_t is stable here.
#pragma unroll
              for (int q = 0; q < D / 32; ++q) {
                uint32_t orr[32];
                tmem_ld32(o_addr + q * 32, orr);
                tmem_wait_ld();
                reg_fence32(orr);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                tmem_st32(o_addr + q * 32, orr);
              }
            }
            l_run *= alpha;
            m_run = m_new;
          }
          }
          const float mref = (m_run == kNegInf) ? 0.f : m_run;
          // p = 2^(s * scale * log2 e - m): packed FMA on pairs, one ex2 each.
          const float2 c2 = make_float2(c_log2, c_log2);
          const float2 nm2 = make_float2(-mref, -mref);
          acc0 = make_float2(0.f, 0.f);
          acc1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k2 = 0; k2 < kBN / 2; ++k2) {
            const float2 xs = __ffma2_rn(
                make_float2(__uint_as_float(sr[2 * k2]), __uint_as_float(sr[2 * k2 + 1])), c2, nm2);
            const float2 pp = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
            if (k2 & 1) acc1 = __fadd2_rn(acc1, pp); else acc0 = __fadd2_rn(acc0, pp);
            pk[k2] = pack_bf16x2(pp.x, pp.y);
          }
          if (with_max) break;
          const float l_tile = (acc0.x + acc1.x) + (acc0.y + acc1.y);
          if (!__any_sync(0xffffffffu, !(l_tile <= kMaxLazyTileSum))) break;
          with_max = true;
          }
          l_run += (acc0.x + acc1.x) + (acc0.y + acc1.y);
          tmem_st32(s_addr, pk);
          tmem_st32(s_addr + 32, pk + 32);
          tmem_wait_st();
          tc_fence_before();
#ifdef CPATTN_FAULT_INJECT_DROP_P
          // Test-only build: CTA 0 never hands its first P tile of Q tile 0
          // to the MMA warp, whose bounded wait then runs out (no trap, no
          // fault).
          if (!(blockIdx.x == 0 && t == 0 && x == 0))
#endif
            mbar_arrive(&p_full[t]);
          any_pv = true;
        }
        if (PARTIALS && ok) {
          // End of ring step s: write (O_step, m_step, l_step) and restart.
          ok = __all_sync(0xffffffffu,
                          wait_bounded(&o_done[t], seg_done & 1, abort_flag));
          ++seg_done;
          if (!ok) break;
          tc_fence_after();
          const size_t so = static_cast<size_t>(s) * p.total_tokens * p.num_heads + row_idx;
          float4* dst = reinterpret_cast<float4*>(p.o_steps + so * D);
          const bool row_store =
              row_valid && in_bounds(static_cast<long long>(row_idx), 0,
                                     p.total_tokens * p.num_heads, p.hdr);
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t orr[32];
            tmem_ld32(o_addr + q * 32, orr);
            tmem_wait_ld();
            reg_fence32(orr);
            if (row_store) {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[q * 8 + e / 4] =
                    make_float4(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1]),
                                __uint_as_float(orr[e + 2]), __uint_as_float(orr[e + 3]));
            }
          }
          if (row_store) {
            p.m_steps[so] = (m_run == kNegInf) ? kNegInf : m_run * kLn2;
            p.l_steps[so] = l_run;
          }
          tc_fence_before();
        }
      }
      if (!PARTIALS && ok) {
        // Epilogue: O / l in bf16 and LSE = m + ln l.
        ok = __all_sync(0xffffffffu, wait_bounded(&o_done[t], 0, abort_flag));
        if (ok) {
          tc_fence_after();
          const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
          // The rows go out through Q tile t's buffer, free now (every MMA
          // reading it completed before o_done[t]): each thread writes its
          // row there in the 128-byte-swizzled layout (conflict-free), then
          // the warp copies its own 32 rows out with D / 8 lanes per row, so
          // every global store instruction writes whole rows.
          uint8_t* stage = smem + C::kQOff + t * C::kTileBytes;
          fence_proxy_async_smem();
          // All D columns of the row in flight before one wait.
          uint32_t orr[D];
#pragma unroll
          for (int q = 0; q < D / 32; ++q) tmem_ld32(o_addr + q * 32, orr + q * 32);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < D / 32; ++q) reg_fence32(orr + q * 32);
          const float2 il2 = make_float2(inv_l, inv_l);
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(orr[q * 32 + 2 * e]),
                                                       __uint_as_float(orr[q * 32 + 2 * e + 1])),
                                           il2);
              w[e] = pack_bf16x2(o2.x, o2.y);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4*>(stage + swizzle128(r, q * 4 + e)) =
                  make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
          if (q0 + t * kBM >= q_lo && q0 + t * kBM + kBM <= q_hi) {
            // A full tile: the staged layout is the TMA layout, so one thread
            // stores it with the bulk engine once every row is staged (each
            // thread makes its writes visible to the async proxy first).  The
            // issuing thread waits only until the engine has read shared
            // memory, before the CTA's final barrier.
            fence_proxy_async_smem();
            mbar_arrive(&staged[t]);
            if ((warp & 3) == 0 && lane == 0) {
              if (wait_bounded(&staged[t], 0, abort_flag)) {
                const int orow = tok0 + q0 + t * kBM;
                if (in_bounds(orow, 0, p.total_tokens - kBM + 1, p.hdr)) {
#pragma unroll
                  for (int hf = 0; hf < C::kHalves; ++hf)
                    tma_store_3d(&tm_o, stage + hf * 16384, hf * 64, h, orow);
                }
                bulk_commit_group();
                bulk_wait_group_read0();
              } else {
                ok = false;
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
          } else {
            // The tile that starts a short block: its rows before the block
            // belong to another block, rank or sample, so the warp copies its
            // own 32 rows out with D / 8 lanes per row (every store
            // instruction writes whole rows), skipping those.
            __syncwarp();
            constexpr int kLpr = D / 8;      // lanes per row: one 16-byte chunk each
            constexpr int kRpi = 32 / kLpr;  // rows per store instruction
            const int c = lane % kLpr;
            const int row_w = (warp & 3) * 32;
#pragma unroll 4
            for (int it = 0; it < 32 / kRpi; ++it) {
              const int rr = row_w + it * kRpi + lane / kLpr;
              const uint4 val = *reinterpret_cast<const uint4*>(stage + swizzle128(rr, c));
              const int qp = q0 + t * kBM + rr;
              if (qp >= q_lo && qp < q_hi && in_bounds(tok0 + qp, 0, p.total_tokens, p.hdr))
                *reinterpret_cast<uint4*>(
                    p.out + (static_cast<size_t>(tok0 + qp) * p.num_heads + h) * D + c * 8) = val;
            }
          }
          if (row_valid && p.lse != nullptr &&
              in_bounds(static_cast<long long>(row_idx), 0, p.total_tokens * p.num_heads,
                        p.hdr))
            p.lse[row_idx] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : kNegInf;
          tc_fence_before();
        }
      }
      if (!ok) {
        raise_error(p.hdr, kErrTimeout);
        *abort_flag = 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

int attn_smem_bytes(int D) {
  return D == 64 ? Cfg<64>::kSmemBytes : Cfg<128>::kSmemBytes;
}

template <int D, bool PARTIALS>
static cudaError_t launch_attn_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& to,
                                 const FwdParams& p,
                                 long long grid, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, PARTIALS>;
  // The register split inside the kernel assumes exactly kLaunchRegs per
  // thread at launch; with any other count the raise could wait forever.
  static const int regs = [&] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : -1;
  }();
  if (regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, p);
}

cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int D,
                        bool partials, long long grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (D == 64)
    return partials ? launch_attn_t<64, true>(tq, tk, tv, to, p, grid, stream)
                    : launch_attn_t<64, false>(tq, tk, tv, to, p, grid, stream);
  return partials ? launch_attn_t<128, true>(tq, tk, tv, to, p, grid, stream)
                  : launch_attn_t<128, false>(tq, tk, tv, to, p, grid, stream);
}

}  // namespace cpattn
