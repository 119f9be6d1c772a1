// Work decomposition shared by the schedule kernel and the attention kernel.
//
// A sample of length L at CP size c is split into c contiguous chunks of
// ceil(L / c) tokens (rank r owns chunk r); each non-empty chunk is cut into
// blocks of kRowsPerItem query rows.  A "work item" is one such block; the
// attention kernel runs one CTA per (item, head).
//
// CTA order: samples by decreasing length; within a sample, head by head;
// within a head, items by decreasing cost.  CTAs resident together therefore
// read the K/V of one (sample, head) -- a working set that stays in L2 -- and
// the heaviest causal blocks of the longest samples start first.
#pragma once

#include "kernels.h"

namespace cpattn {

struct SampleGeom {
  int L, c, chunk, full, rem;  // `full` chunks of `chunk` tokens, then `rem`
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ SampleGeom sample_geom(const int* cu, const int* cp,
                                                  int b) {
  SampleGeom g;
  g.L = cu[b + 1] - cu[b];
  g.c = cp ? cp[b] : 1;
  g.chunk = cdiv(g.L, g.c);
  g.full = g.chunk > 0 ? g.L / g.chunk : 0;
  g.rem = g.L - g.full * g.chunk;
  return g;
}

// Work items of one sample (its blocks of `rows` rows over all ranks).
__device__ __forceinline__ int sample_items(const SampleGeom& g, int rows = kRowsPerItem) {
  if (g.L == 0) return 0;
  return g.full * cdiv(g.chunk, rows) + (g.rem > 0 ? cdiv(g.rem, rows) : 0);
}

// Item `local` of a sample -> (rank, block).  For causal attention the cost
// of a query block (KV tiles visited) never decreases with `local`; the cost
// of a key block (query tiles that see it) never increases with it.
__device__ __forceinline__ void item_coords(const SampleGeom& g, int local,
                                            int& rank, int& blk, int rows = kRowsPerItem) {
  const int per = cdiv(g.chunk, rows);
  rank = local / per;
  blk = local - rank * per;
  if (rank >= g.full) {  // the short last chunk
    rank = g.full;
    blk = local - g.full * per;
  }
}

}  // namespace cpattn
