// Bounds checks of the debug build (compiled with -DCPATTN_DEBUG).
//
// In the debug build every global-memory index and every TMA coordinate the
// attention kernels derive from their work entry is checked against the
// tensor it addresses.  A check that fails records CPATTN_ERR_DEVICE_BOUNDS
// in the workspace error word (first error wins) and the access is skipped
// -- or, for a TMA load whose mbarrier must still complete, issued at a
// clamped in-range coordinate -- so a wrong index shows up as a status the
// host reads, never as a trap or a memory fault.  In the regular build the
// checks compile to nothing.
#pragma once

#include "kernels.h"

namespace cpattn {

constexpr int kErrBounds = 7;  // CPATTN_ERR_DEVICE_BOUNDS

#ifdef CPATTN_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// lo <= x < hi; otherwise (debug build only) the error word is set and the
// result is false.
__device__ __forceinline__ bool in_bounds(long long x, long long lo, long long hi,
                                          WsHeader* hdr) {
  if (!kDebugChecks) return true;
  if (x >= lo && x < hi) return true;
  if (hdr != nullptr) atomicCAS(&hdr->error, 0, kErrBounds);
  return false;
}

// A coordinate for a load that must be issued: x itself when lo <= x < hi,
// else (debug build only) the error is recorded and lo is used instead.
__device__ __forceinline__ int checked_coord(int x, int lo, int hi, WsHeader* hdr) {
  return in_bounds(x, lo, hi, hdr) ? x : lo;
}

}  // namespace cpattn
