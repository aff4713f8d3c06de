// sched.cuh -- the m-tile schedule of the CUDA-core and decode engines: the
// tiles of `bm` rows of every group, numbered group by group, as an exclusive
// prefix sched[G + 1] over the groups (sched[G] = the number of tiles).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

// Group g of linear m-tile j (sched non-decreasing, j < sched[G]).
__device__ __forceinline__ int find_group(const int32_t* sched, int G, int j) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (sched[mid] <= j) lo = mid; else hi = mid;
  }
  return lo;
}

// The schedule built by one warp of the block in shared memory (G <= a few
// thousand): a warp-wide scan of the groups' tile counts, 32 groups at a
// time.  Offsets that are not a valid partition (offsets[0] != 0, a negative
// count, offsets[G] above the stated bound) give no tiles and raise the
// rows flag.
__device__ __forceinline__ void block_schedule(const GemmArgs& a, int bm, int32_t* sched, int lane) {
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < a.G; base += 32) {
    const int g = base + lane;
    int v = 0;
    if (g < a.G) {
      int64_t cnt = a.offsets ? (int64_t)a.offsets[g + 1] - a.offsets[g] : a.single_rows;
      if (cnt < 0) { bad = true; cnt = 0; }
      v = (int)((cnt + bm - 1) / bm);
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (g < a.G) sched[g] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    if (a.offsets) bad |= a.offsets[0] != 0 || (int64_t)a.offsets[a.G] > a.rows_bound;
    else bad |= a.single_rows > a.rows_bound || a.single_rows < 0;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sched[a.G] = bad ? 0 : carry;
    if (bad && blockIdx.x == 0 && blockIdx.y == 0) set_flag(a.flags, kFlagRows);
  }
}

}  // namespace moe
