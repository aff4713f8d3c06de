// tc_pair.cuh -- inline-PTX wrappers for the tcgen05 kernels that run on
// pairs of SMs (2-CTA clusters, tcgen05 cta_group::2): cluster ranks and
// addresses, cluster-scope mbarrier arrivals and bounded waits, TMA loads
// that complete on the even CTA's barrier, pair TMEM allocation, the pair
// MMA and its commits.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace moe {
namespace tc {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Cluster-scope test of a barrier phase (test_wait: never suspends the
// thread).  Every wait of this kernel polls with it.
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (about 2 s of SM clocks, then the abort flag).
__device__ __forceinline__ bool wait2(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void wait2_quiet(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test_cluster(bar, parity))
    if (clock64() - t0 > kWaitCycles) return;
}
// TMA tile loads into this CTA's shared memory whose completion is counted
// on a barrier of the even CTA (cta_group::2 form: the barrier may sit in
// either CTA of the pair; `bar` is its cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma2(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive (once) on the barrier at this offset in both CTAs of the pair when
// every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void commit2_both(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void commit2_self(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Tile -> (group, row tile, n-tile) from the prefix of row tiles per group:
// n-tile major, row tile minor within a group, so the tiles that share a
// weight tile run side by side.
template <class A>
__device__ __forceinline__ void pair_decode_tile(const A& a, const int32_t* sched, int64_t tile,
                                            int& g, int& mp, int& nt) {
  int lo = 0, hi = a.G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)sched[mid] * a.NT <= tile) lo = mid; else hi = mid;
  }
  g = lo;
  const int mtg = sched[g + 1] - sched[g];
  const int64_t local = tile - (int64_t)sched[g] * a.NT;
  nt = (int)(local / mtg);
  mp = (int)(local % mtg);
}

// Prefix of ceil(rows_g / ROWS) over the groups (one warp, shared memory);
// sched[G] = 0 when the offsets are inconsistent or exceed the row bound.
template <int ROWS, class A>
__device__ void pair_schedule(const A& a, int32_t* sched, int lane) {
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < a.G; base += 32) {
    const int g = base + lane;
    int v = 0;
    if (g < a.G) {
      int64_t cnt = a.offsets ? (int64_t)a.offsets[g + 1] - a.offsets[g] : a.single_rows;
      if (cnt < 0) { bad = true; cnt = 0; }
      v = (int)((cnt + ROWS - 1) / ROWS);
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
    if (bad && blockIdx.x == 0) set_flag(a.flags, kFlagRows);
  }
}

}  // namespace tc
}  // namespace moe
