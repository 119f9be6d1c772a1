// Dynamic-CP planner (host).  See cpattn_plan in include/cpattn.h.
//
// Rules (a reading of "Dynamic Context Parallelism (DCP)", verl 0.9.0 docs,
// and section 4 of "20-Megatron-MCore-TP-PP-EP如何支撑MoE"; the pages name the
// scheduler but do not give its algorithm):
//   * CP size: smallest allowed c with ceil(L / c) <= limit, where the allowed
//     sizes are the powers of two below max_cp and max_cp itself;
//   * placement order: longest first, ties by ascending sample index;
//   * a micro-batch has W rank slots of `limit` tokens; a CP-c sample takes the
//     aligned rank group [g*c, (g+1)*c) and adds ceil(L / c) to each slot;
//   * first fit over micro-batches in creation order and groups in order,
//     opening a new micro-batch when nothing fits.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "cpattn.h"

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool is_pow2(int64_t x) { return x >= 1 && (x & (x - 1)) == 0; }

// Smallest allowed CP size for a sample, or 0 when none fits.
int32_t pick_cp(int64_t len, int64_t limit, int32_t max_cp) {
  for (int32_t c = 1; c < max_cp; c *= 2)
    if (ceil_div(len, c) <= limit) return c;
  return ceil_div(len, max_cp) <= limit ? max_cp : 0;
}

}  // namespace

extern "C" int cpattn_plan(const int32_t* seqlens, int32_t n, int32_t world,
                           int32_t limit, int32_t max_cp, int32_t* cp_size,
                           int32_t* micro_batch, int32_t* first_rank,
                           int32_t* order, int32_t* num_micro_batches,
                           int32_t* rank_load) {
  if (n < 0 || world < 2 || world % 2 != 0 || world > 4096 || limit < 1)
    return CPATTN_ERR_INVALID_ARG;
  if (max_cp < 1 || max_cp > world || !(is_pow2(max_cp) || max_cp == world))
    return CPATTN_ERR_INVALID_ARG;
  if (num_micro_batches == nullptr) return CPATTN_ERR_INVALID_ARG;
  if (n > 0 && (seqlens == nullptr || cp_size == nullptr ||
                micro_batch == nullptr || first_rank == nullptr ||
                order == nullptr))
    return CPATTN_ERR_INVALID_ARG;
  for (int32_t b = 0; b < n; ++b)
    if (seqlens[b] < 0) return CPATTN_ERR_INVALID_ARG;

  std::vector<int32_t> cp(n);
  for (int32_t b = 0; b < n; ++b) {
    cp[b] = pick_cp(seqlens[b], limit, max_cp);
    if (cp[b] == 0) return CPATTN_ERR_PLAN_INFEASIBLE;
  }

  std::vector<int32_t> ord(n);
  std::iota(ord.begin(), ord.end(), 0);
  std::stable_sort(ord.begin(), ord.end(), [&](int32_t a, int32_t b) {
    return seqlens[a] > seqlens[b];
  });

  // loads[mb * world + r]: tokens already placed on rank r of micro-batch mb.
  std::vector<int64_t> loads;
  std::vector<int32_t> mb_of(n), first_of(n);
  int32_t nmb = 0;
  for (int32_t b : ord) {
    const int32_t c = cp[b];
    const int64_t need = ceil_div(seqlens[b], c);
    bool placed = false;
    for (int32_t mb = 0; mb < nmb && !placed; ++mb) {
      int64_t* slot = loads.data() + static_cast<size_t>(mb) * world;
      for (int32_t g = 0; g < world / c; ++g) {
        bool fits = true;
        for (int32_t r = g * c; r < (g + 1) * c; ++r)
          if (slot[r] + need > limit) { fits = false; break; }
        if (!fits) continue;
        for (int32_t r = g * c; r < (g + 1) * c; ++r) slot[r] += need;
        mb_of[b] = mb;
        first_of[b] = g * c;
        placed = true;
        break;
      }
    }
    if (!placed) {
      loads.resize(static_cast<size_t>(nmb + 1) * world, 0);
      int64_t* slot = loads.data() + static_cast<size_t>(nmb) * world;
      for (int32_t r = 0; r < c; ++r) slot[r] += need;
      mb_of[b] = nmb;
      first_of[b] = 0;
      ++nmb;
    }
  }

  for (int32_t b = 0; b < n; ++b) {
    cp_size[b] = cp[b];
    micro_batch[b] = mb_of[b];
    first_rank[b] = first_of[b];
    order[b] = ord[b];
  }
  *num_micro_batches = nmb;
  if (rank_load != nullptr)
    for (size_t x = 0; x < loads.size(); ++x)
      rank_load[x] = static_cast<int32_t>(loads[x]);
  return CPATTN_OK;
}
