// gemm_tc2.cu -- grouped bf16 GEMM on pairs of SMs (tcgen05 cta_group::2).
//
// Same contract as the one-SM engine in gemm_tc.cu ("Fused MoE Kernel Notes",
// group_gemm_same_nk: groups of rows with shared N and K, the m-tile schedule
// built from the real group sizes).  The two CTAs of a cluster share one
// 256 x 256 output tile (a group's last tile, when at most 128 of its rows
// are left, is a half tile: M = 128, see IDESC_HALF): CTA r keeps rows 128r .. 128r+127 of the A tile and
// rows (N) 128r .. 128r+127 of the B tile in its own shared memory, and the
// even CTA's MMA thread issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
// K = 16), which reads both CTAs' operands and writes each CTA's 128 rows x
// 256 columns of the fp32 accumulator into that CTA's TMEM.  Per SM a 64-wide
// k-block then needs 32 KB of operands instead of the 48 KB of a one-SM
// 128 x 256 tile, so six stages fit where four did and the loads in flight per
// SM cover 50 % more latency.  For SwiGLU CTA 0 loads the 128 gate rows and
// CTA 1 the 128 up rows of the n-tile, so accumulator columns 0-127 are gate
// and 128-255 up in both CTAs, as in the one-SM engine.
//
// Roles, in each CTA of the pair:
//   warp 0     TMA A producer (its 128 rows), warp 6 TMA B producer (its half);
//              the loads of both CTAs complete on the even CTA's "full"
//              barrier of the stage (cta_group::2 TMA), on which the even
//              CTA's producers expect the pair's bytes;
//   warp 1     TMEM allocation, collective over the pair; in the even CTA
//              also the MMA issuer;
//   warps 2-5  epilogue over the CTA's own TMEM lanes; they tell the even CTA
//              that an accumulator is drained (remote arrive, 256 a phase).
// The MMA completion (tcgen05.commit ... multicast) frees the stage in both
// CTAs and marks the accumulator full in both.  Every wait is bounded as in
// the one-SM engine; a CTA that gives up raises its abort flag, its partner's
// waits run out in turn, and both meet at the closing cluster barrier before
// TMEM is released.
#include <atomic>
#include "common.cuh"
#include "internal.h"
#include "tc_pair.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace tc2 {

using namespace tc;

constexpr int BMP = 256, BMC = 128;     // rows of a pair tile, of one CTA's half
constexpr int BN = 256, BNC = 128, BK = 64;
constexpr int S = 6;                    // stages
constexpr int A_BYTES = BMC * BK * 2;   // 16 KB
constexpr int B_BYTES = BNC * BK * 2;   // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RING_BYTES = S * STAGE_BYTES;
constexpr int THREADS = 224;            // warps 0-6
constexpr uint32_t TMEM_COLS = 512;     // two 256-column accumulators
constexpr int BAR_BYTES = 512;
// Dynamic tile order: the even CTA's A producer takes tiles from a counter in
// global memory (atomicAdd) and hands each tile number to every role of both
// CTAs through a ring of NSLOT shared-memory slots, so the tiles in progress
// across the GPU always form one window of consecutive tile numbers (a static
// round-robin drifts apart, and then the CTAs that share a weight tile no
// longer read it while it is in L2).
constexpr int NSLOT = 4;
// A group of at least this many pair m-tiles is ordered m-tile major when
// its weights fit in half the L2 (they stay there while every m-tile passes
// over them); other groups n-tile major (the m-tiles sharing a weight tile
// run side by side, and a weight tile is read from DRAM once).
constexpr int MMAJOR_TILES = 8;
constexpr int64_t MMAJOR_WEIGHT_BYTES = 64ll << 20;
constexpr int MAX_SMEM_G = 1024;
constexpr int SCHED_BYTES = (MAX_SMEM_G + 1) * 4;
constexpr int OUT_ROW_BYTES = 80;
constexpr int OUT_WARP_BYTES = 32 * OUT_ROW_BYTES;
constexpr int OUT_BYTES = 4 * OUT_WARP_BYTES;
// half tiles with SwiGLU: the up values of a 32 x 32 chunk handed from the
// warps holding TMEM lanes 64-127 to those holding lanes 0-63 (fp32, [32][33]
// for each of the two warp pairs)
constexpr int XCH_STRIDE = 33;
constexpr int XCH_BYTES = 2 * 32 * XCH_STRIDE * 4;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES + OUT_BYTES + XCH_BYTES + SCHED_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
static_assert((2 * S + 5 + 3 * NSLOT + 1) * 8 + 12 <= BAR_BYTES, "barrier area");
// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major,
// N >> 3 at bits 17-22, M >> 4 at bits 24-28 (M = 256 across the pair).
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BMP >> 4) << 24);
// The last tile of a group with at most 128 rows left is a half tile: M = 128
// over the pair (64 rows a CTA), full MMA rate per row, so it costs half a
// tile instead of a whole one.  Its accumulator takes 128 TMEM columns: lane
// l < 64 holds row l of the CTA's half, columns 0-127 of the tile's N; lane
// 64 + l the same row, columns 128-255.
constexpr uint32_t IDESC_HALF = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((BMP / 2) >> 4) << 24);

struct Args {
  int mode, N, K, G, NT, KB;
  const int32_t* offsets;
  int64_t single_rows;
  int64_t rows_bound;
  const int32_t* sched;   // global pair-tile prefix, or NULL: built in shared memory
  int32_t* ctr;           // zeroed tile counter (dynamic order), or NULL: round-robin
  int mmajor;             // 1: large groups may be ordered m-tile major
  // K split (few-tile calls): up to ksmax splits, chosen in the kernel from
  // the real tile count; partial sums to part [split][row][NT * 256] (fp32),
  // the number of splits to *ks_out; part == NULL: no split
  int ksmax;
  int ks_clusters;   // clusters the split count is sized for: all the GPU
                     // holds, so a call held to fewer SMs sums in the same order
  float* part;
  int64_t part_ld, part_stride;
  int32_t* ks_out;
  void* out;
  int64_t ldo;
  uint32_t* flags;
  // grouped calls: group g's A maps at amaps[2 g] (BMC-row box) and
  // amaps[2 g + 1] (BMC / 2 rows), spanning only the group's rows, so the
  // padding rows of its last tile load as zeros (less power in the tensor
  // cores than the next group's rows; the results do not change); NULL: the
  // global maps
  const CUtensorMap* amaps;
};

// Pair tile -> (group, pair m-tile, n-tile), pair m-tiles of BMP rows; within
// a group n-tile major, or m-tile major for groups of MMAJOR_TILES m-tiles
// or more.
__device__ __forceinline__ void decode_tile(const Args& a, const int32_t* sched, int64_t tile,
                                            int& g, int& mp, int& nt) {
  pair_decode_tile(a, sched, tile, g, mp, nt);
  const int mtg = sched[g + 1] - sched[g];
  if (a.mmajor && mtg >= MMAJOR_TILES) {
    const int64_t local = tile - (int64_t)sched[g] * a.NT;
    mp = (int)(local / a.NT);
    nt = (int)(local % a.NT);
  }
}
__device__ void build_schedule(const Args& a, int32_t* sched, int lane) {
  pair_schedule<BMP>(a, sched, lane);
}

// Rows of the group left from pair m-tile mp on (> 0 for every scheduled tile).
__device__ __forceinline__ int64_t tile_rows_left(const Args& a, int g, int mp) {
  const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
  const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
  return gend - (gbeg + (int64_t)mp * BMP);
}

// Named barrier of the four epilogue warps (barrier 0 is __syncthreads).
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA64,
                    const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                    const Args a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  // bars: full[S] empty[S] tfull[2] tempty[2] final tfill[NSLOT] tdrain[NSLOT];
  // then the tile slots, the epilogue's copy of its tile, and the scalars
  volatile int64_t* s_tile = reinterpret_cast<volatile int64_t*>(bars + 2 * S + 5 + 2 * NSLOT);
  volatile int64_t* s_etile = s_tile + NSLOT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5 + 3 * NSLOT + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_slot + 2);
  unsigned char* s_out = smem + RING_BYTES + BAR_BYTES;
  float* s_xch = reinterpret_cast<float*>(s_out + OUT_BYTES);
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_out + OUT_BYTES + XCH_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const uint32_t ring = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[S + s]); };
  auto tfull = [&](int b) { return smem_u32(&bars[2 * S + b]); };
  auto tempty = [&](int b) { return smem_u32(&bars[2 * S + 2 + b]); };
  const uint32_t final_bar = smem_u32(&bars[2 * S + 4]);
  auto tfill = [&](int i) { return smem_u32(&bars[2 * S + 5 + i]); };
  auto tdrain = [&](int i) { return smem_u32(&bars[2 * S + 5 + NSLOT + i]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 2);      // the even CTA's A and B producers (pair's bytes)
      mbar_init(empty(s), 1);     // the pair's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 2 * 128);   // both CTAs' epilogue threads
    }
    mbar_init(final_bar, 1);
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(tfill(i), 1);   // the even CTA's tile taker
      mbar_init(tdrain(i), 6);  // three readers in each CTA (see next_tile)
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 2 && a.sched == nullptr) build_schedule(a, s_sched, lane);
  cluster_sync();   // barriers of both CTAs initialised before any remote arrive
  if (warp == 1) {
    tmem_alloc2(smem_u32(tmem_slot), TMEM_COLS);   // collective over the pair
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t* sched = a.sched ? a.sched : s_sched;
  const int64_t cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  // K splits: as many as keep every cluster busy (at most ksmax, at least 4
  // k-blocks a split); the same in every CTA, recorded for the reduction.
  const int64_t tiles1 = (int64_t)sched[a.G] * a.NT;
  int ks = 1;
  if (a.part != nullptr) {
    int64_t k = tiles1 > 0 ? (int64_t)a.ks_clusters / tiles1 : 1;
    if (k > a.ksmax) k = a.ksmax;
    if (k > a.KB / 4) k = a.KB / 4;
    ks = k < 1 ? 1 : (int)k;
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.ks_out = ks;
  }
  const int64_t total = tiles1 * ks;
  // k-blocks of split sp of a tile
  auto kb_range = [&](int sp, int& kb0, int& kb1) {
    kb0 = (int)((int64_t)sp * a.KB / ks);
    kb1 = (int)((int64_t)(sp + 1) * a.KB / ks);
  };

  // Tile n of this pair (n = 0, 1, ...), or -1 when there is none left (or a
  // wait ran out).  The even CTA's A producer takes it (take = true) and
  // writes it to slot n % NSLOT of both CTAs; every other reader -- the A
  // producer of the odd CTA, both B producers, the MMA issuer and one thread
  // of each CTA's epilogue -- reads it from its own CTA's slot and tells the
  // even CTA that it has (six readers a slot use).
  // The taker claims its tiles one ahead: the counter's reply for the next
  // tile arrives while the loads of this one go out.
  int64_t reserve = a.ctr && threadIdx.x == 0 && leader ? (int64_t)atomicAdd(a.ctr, 1) : -1;
  auto next_tile = [&](int64_t n, bool take) -> int64_t {
    const int slot = (int)(n % NSLOT);
    const uint32_t use = (uint32_t)(n / NSLOT);
    if (take) {
      if (!wait2(tdrain(slot), (use & 1u) ^ 1u, abort_flag)) return -1;
      int64_t t = cl + n * ncl;
      if (a.ctr) {
        t = reserve;
        reserve = (int64_t)atomicAdd(a.ctr, 1);
      }
      if (t >= total) t = -1;
      s_tile[slot] = t;
      const uint32_t remote = map_to_rank(smem_u32((const void*)&s_tile[slot]), 1);
      asm volatile("st.shared::cluster.b64 [%0], %1;" ::"r"(remote), "l"(t) : "memory");
      mbar_arrive(tfill(slot));
      mbar_arrive_cluster(map_to_rank(tfill(slot), 1));
      return t;
    }
    if (!wait2(tfill(slot), use & 1u, abort_flag)) return -1;
    const int64_t t = s_tile[slot];
    mbar_arrive_cluster(map_to_rank(tdrain(slot), 0));
    return t;
  };

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ---------------- TMA producers ----------------
    const bool is_a = warp == 0;
    const CUtensorMap* bmap = (a.mode == kSwiGLU && rank == 1) ? &tmB1 : &tmB0;
    auto b_row = [&](int nt) { return a.mode == kSwiGLU ? nt * BNC : nt * BN + (int)rank * BNC; };
    int s = 0;
    uint32_t ph = 0, issued = 0, par = 0;
    bool ok = true;
    const CUtensorMap* acquired = nullptr;   // per-group map last made visible
    for (int64_t n = 0; ok; ++n) {
      const int64_t tile = next_tile(n, is_a && leader);
      if (tile < 0) break;
      int g, mp, nt, kb0, kb1;
      decode_tile(a, sched, tile / ks, g, mp, nt);
      kb_range((int)(tile % ks), kb0, kb1);
      const int64_t gbase = a.offsets ? a.offsets[g] : 0;
      const bool half = tile_rows_left(a, g, mp) <= BMC;
      const int64_t local = (int64_t)mp * BMP + (int64_t)rank * (half ? BMC / 2 : BMC);
      const CUtensorMap* amap = half ? &tmA64 : &tmA;
      int arow = (int)(gbase + local);
      if (is_a && a.amaps) {
        amap = a.amaps + 2 * g + (half ? 1 : 0);
        arow = (int)local;
        if (amap != acquired) {   // written by the preceding kernel
          asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                           reinterpret_cast<uint64_t>(amap))
                       : "memory");
          acquired = amap;
        }
      }
      const int brow = b_row(nt);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait2(empty(s), ph ^ 1u, abort_flag)) { ok = false; break; }
        const uint32_t st = ring + s * STAGE_BYTES;
        // the even CTA's "full" barrier counts both CTAs' bytes; only the
        // even CTA's producers arrive on it (with the pair's byte count)
        const uint32_t fb = map_to_rank(full(s), 0);
        if (leader) mbar_expect_tx(full(s), 2 * (is_a ? (half ? A_BYTES / 2 : A_BYTES) : B_BYTES));
        if (is_a) tma_load_2d_pair(st, amap, kb * BK, arow, fb);
        else tma_load_3d_pair(st + A_BYTES, bmap, kb * BK, brow, g, fb);
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (*abort_flag && leader) {
      // loads still in flight land before the pair goes away (the odd CTA's
      // are counted on these barriers too; its own waits run out seconds
      // after any load of its could have landed)
      for (int i = 0; i < S; ++i)
        if (issued & (1u << i)) wait2_quiet(full(i), (par >> i) & 1u);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- even CTA: MMA issuer for the pair ----------------
    int s = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int64_t n = 0; ok; ++n) {
      const int64_t tile = next_tile(n, false);
      if (tile < 0) break;
      int g, mp, nt, kb0, kb1;
      decode_tile(a, sched, tile / ks, g, mp, nt);
      kb_range((int)(tile % ks), kb0, kb1);
      const uint32_t idesc = tile_rows_left(a, g, mp) <= BMC ? IDESC_HALF : IDESC;
      if (!wait2(tempty(acc), aph ^ 1u, abort_flag)) break;
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)acc * BN;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait2(full(s), ph, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = ring + s * STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma2(d, sw128_desc(st + kk * 32), sw128_desc(st + A_BYTES + kk * 32), idesc,
               (kb != kb0 || kk != 0) ? 1u : 0u);
        commit2_both(empty(s));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      commit2_both(tfull(acc));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (*abort_flag) {
      commit2_self(final_bar);
      wait2_quiet(final_bar, 0);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue (warps 2..5, both CTAs) ----------------
    const int q = warp & 3;   // TMEM lanes 32q .. 32q+31 of this CTA
    const int et = threadIdx.x - 64;   // 0 .. 127
    unsigned char* stage = s_out + (warp - 2) * OUT_WARP_BYTES;
    unsigned char* my_row = stage + lane * OUT_ROW_BYTES;
    const bool swiglu = a.mode == kSwiGLU;
    bf16* out = reinterpret_cast<bf16*>(a.out);
    int acc = 0;
    uint32_t aph = 0;
    // a 32 x 32 chunk of finished rows (my_row of each lane) to global rows
    // row0 .. row0+31 (nvalid of them), columns n .. n+31
    auto store_chunk = [&](const uint4 (&packed)[4], int64_t row0, int nvalid, int n) {
#pragma unroll
      for (int v = 0; v < 4; ++v) reinterpret_cast<uint4*>(my_row)[v] = packed[v];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int p = lane + 32 * i;   // 128 pieces: 32 rows x 4 x 16 B
        const int rr = p >> 2, pc = p & 3;
        const int col = n + pc * 8;
        if (rr < nvalid && col < a.N)
          *reinterpret_cast<uint4*>(out + (row0 + rr) * a.ldo + col) =
              *reinterpret_cast<const uint4*>(stage + rr * OUT_ROW_BYTES + pc * 16);
      }
      __syncwarp();
    };
    for (int64_t n = 0;; ++n) {
      // one thread takes the tile and waits for its accumulator; the four
      // warps follow its result together (the half tiles' hand-over meets
      // at named barriers)
      if (et == 0) {
        const int64_t t = next_tile(n, false);
        *s_etile = t;
        *s_ok = t >= 0 && wait2(tfull(acc), aph, abort_flag) ? 1 : 0;
      }
      epi_bar();
      const int okv = *s_ok;
      const int64_t tile = *s_etile;
      epi_bar();
      if (!okv) break;
      int g, mp, nt;
      decode_tile(a, sched, tile / ks, g, mp, nt);
      const int sp = (int)(tile % ks);
      const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
      const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
      const bool half = tile_rows_left(a, g, mp) <= BMC;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * BN;
      if (ks > 1) {
        // K split: this lane's row of the fp32 accumulator (256 columns of a
        // full tile; 128 of a half tile) to the split's partial sums,
        // columns nt * 256 + c; the reduction applies the epilogue
        const int64_t row = half
            ? gbeg + (int64_t)mp * BMP + (int64_t)rank * (BMC / 2) + (q & 1) * 32 + lane
            : gbeg + (int64_t)mp * BMP + (int64_t)rank * BMC + q * 32 + lane;
        const int cbase = half ? (q >> 1) * (BN / 2) : 0;
        const int ncol = half ? BN / 2 : BN;
        float* prow = a.part + (int64_t)sp * a.part_stride + row * a.part_ld + (int64_t)nt * BN + cbase;
#pragma unroll 1
        for (int c = 0; c < ncol; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          tmem_wait_ld();
          if (row < gend) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<uint4*>(prow + c)[v] =
                  make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
          }
        }
      } else if (!half) {
        const int64_t row0 = gbeg + (int64_t)mp * BMP + (int64_t)rank * BMC + q * 32;
        const int64_t nvalid64 = gend - row0;
        const int nvalid = nvalid64 < 0 ? 0 : (nvalid64 > 32 ? 32 : (int)nvalid64);
        const int n0 = swiglu ? nt * BNC : nt * BN;
        const int ncols = swiglu ? BN / 2 : BN;
#pragma unroll 1
        for (int c = 0; c < ncols && n0 + c < a.N; c += 32) {
          uint32_t gr[32];
          uint4 packed[4];
          tmem_ld32(taddr + c, gr);
          if (swiglu) {
            uint32_t ur[32];
            tmem_ld32(taddr + BN / 2 + c, ur);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                f[e] = silu_fast(__uint_as_float(gr[v * 8 + e])) * __uint_as_float(ur[v * 8 + e]);
              packed[v] = pack16(f, (const bf16*)nullptr);
            }
          } else {
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(gr[v * 8 + e]);
              packed[v] = pack16(f, (const bf16*)nullptr);
            }
          }
          store_chunk(packed, row0, nvalid, n0 + c);
        }
      } else {
        // half tile: the CTA's 64 rows; warps q and q + 2 hold the same 32
        // rows, q < 2 columns 0-127 of the tile's N, q >= 2 columns 128-255
        const int64_t row0 = gbeg + (int64_t)mp * BMP + (int64_t)rank * (BMC / 2) + (q & 1) * 32;
        const int64_t nvalid64 = gend - row0;
        const int nvalid = nvalid64 < 0 ? 0 : (nvalid64 > 32 ? 32 : (int)nvalid64);
        if (!swiglu) {
          const int n0 = nt * BN + (q >> 1) * (BN / 2);
#pragma unroll 1
          for (int c = 0; c < BN / 2 && n0 + c < a.N; c += 32) {
            uint32_t gr[32];
            uint4 packed[4];
            tmem_ld32(taddr + c, gr);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(gr[v * 8 + e]);
              packed[v] = pack16(f, (const bf16*)nullptr);
            }
            store_chunk(packed, row0, nvalid, n0 + c);
          }
        } else {
          // gate columns in lanes 0-63, the matching up columns in lanes
          // 64-127: warp q + 2 hands its up values to warp q through s_xch
          const int n0 = nt * BNC;
          float* xrow = s_xch + ((q & 1) * 32 + lane) * XCH_STRIDE;
#pragma unroll 1
          for (int c = 0; c < BNC && n0 + c < a.N; c += 32) {   // same trip count in all four warps
            uint32_t r[32];
            tmem_ld32(taddr + c, r);
            tmem_wait_ld();
            if (q >= 2) {
#pragma unroll
              for (int e = 0; e < 32; ++e) xrow[e] = __uint_as_float(r[e]);
            }
            epi_bar();
            if (q < 2) {
              uint4 packed[4];
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  f[e] = silu_fast(__uint_as_float(r[v * 8 + e])) * xrow[v * 8 + e];
                packed[v] = pack16(f, (const bf16*)nullptr);
              }
              store_chunk(packed, row0, nvalid, n0 + c);
            }
            epi_bar();   // s_xch is written again only after every read of this chunk
          }
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(map_to_rank(tempty(acc), 0));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no MMA, TMEM load or remote arrive of the pair in flight
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) set_flag(a.flags, kFlagTimeout);
}

// The K split's reduction: out[r, j] for the group rows r < offsets[G] (or
// single_rows), the splits' partial sums added in split order in fp32, then
// the epilogue (SwiGLU: silu(gate) * up, gate at column (j / 128) * 256 +
// j % 128 of the partials, up 128 further; plain: column j), rounded once.
// Nothing to do when the GEMM chose one split (it wrote out itself).
template <bool SWIGLU>
__global__ void __launch_bounds__(256) split_reduce_kernel(const float* __restrict__ part,
                                                           int64_t part_ld, int64_t part_stride,
                                                           const int32_t* ks_ptr,
                                                           const int32_t* offsets, int G,
                                                           int64_t single_rows, int64_t rows_bound,
                                                           int N,
                                                           bf16* __restrict__ out, int64_t ldo) {
  const int ks = *ks_ptr;
  if (ks <= 1) return;
  int64_t rows = offsets ? offsets[G] : single_rows;
  if (rows > rows_bound) rows = rows_bound;   // the GEMM flagged it and computed nothing
  const int per_row = N / 8;
  const int64_t items = rows * per_row;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = it / per_row;
    const int j0 = (int)(it % per_row) * 8;
    float f[8];
    if (SWIGLU) {
      const int64_t cg = (int64_t)(j0 / (BN / 2)) * BN + j0 % (BN / 2);
      float gsum[8], usum[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) gsum[e] = usum[e] = 0.0f;
      for (int sp = 0; sp < ks; ++sp) {
        const float* p = part + sp * part_stride + r * part_ld + cg;
        const float4 g0 = reinterpret_cast<const float4*>(p)[0], g1 = reinterpret_cast<const float4*>(p)[1];
        const float4 u0 = reinterpret_cast<const float4*>(p + BN / 2)[0],
                     u1 = reinterpret_cast<const float4*>(p + BN / 2)[1];
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          gsum[e] += gv[e];
          usum[e] += uv[e];
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = silu_fast(gsum[e]) * usum[e];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.0f;
      for (int sp = 0; sp < ks; ++sp) {
        const float* p = part + sp * part_stride + r * part_ld + j0;
        const float4 v0 = reinterpret_cast<const float4*>(p)[0], v1 = reinterpret_cast<const float4*>(p)[1];
        const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] += vv[e];
      }
    }
    *reinterpret_cast<uint4*>(out + r * ldo + j0) = pack16(f, (const bf16*)nullptr);
  }
}

}  // namespace tc2

cudaError_t launch_group_maps(const CUtensorMap& baseA, const CUtensorMap& baseB, void* maps,
                              const int32_t* offsets, int G, int64_t rows_bound, const void* A,
                              int64_t lda_bytes, const void* B, int64_t ldb_bytes,
                              cudaStream_t st);   // gemm_bwd.cu

cudaError_t launch_gemm_tc2(const GemmArgs& a, cudaStream_t st) {
  using namespace tc2;
  if (a.dtype != MOE_BF16 || a.mode == kStoreF32 || a.ksplit != 1 || a.gather || a.wfmt)
    return cudaErrorNotSupported;
  if ((a.K % 8) != 0 || (a.N % 8) != 0 || a.K <= 0 || a.N <= 0) return cudaErrorInvalidValue;
  cudaError_t e;
  const bool smem_sched = a.G <= MAX_SMEM_G;
  if (!smem_sched) {
    e = launch_schedule(a, BMP, st);
    if (e != cudaSuccess) return e;
  }
  const int64_t rows = a.offsets ? a.rows_bound : a.single_rows;
  if (rows <= 0) return cudaSuccess;
  CUtensorMap mA, mB0, mB1;
  CUtensorMap mA64;
  if (!tc::make_map_2d(&mA, a.A, rows, a.K, BMC)) return cudaErrorInvalidValue;
  if (!tc::make_map_2d(&mA64, a.A, rows, a.K, BMC / 2)) return cudaErrorInvalidValue;
  if (!tc::make_map_3d(&mB0, a.B0, a.N, a.K, a.G, a.bstride, BNC)) return cudaErrorInvalidValue;
  if (a.mode == kSwiGLU) {
    if (!tc::make_map_3d(&mB1, a.B1, a.N, a.K, a.G, a.bstride, BNC)) return cudaErrorInvalidValue;
  } else {
    mB1 = mB0;
  }
  Args t;
  t.mode = a.mode;
  t.N = a.N;
  t.K = a.K;
  t.G = a.G;
  t.NT = a.mode == kSwiGLU ? (a.N + BNC - 1) / BNC : (a.N + BN - 1) / BN;
  t.KB = (a.K + BK - 1) / BK;
  t.offsets = a.offsets;
  t.single_rows = a.single_rows;
  t.rows_bound = a.rows_bound;
  t.sched = smem_sched ? nullptr : a.sched;
  t.ctr = a.ctr;
  t.ksmax = kSplitPairMax;
  t.part = a.split_part;
  t.ks_out = a.split_ks;
  t.part_ld = (int64_t)t.NT * BN;
  t.part_stride = a.rows_bound * t.part_ld;
  if (t.part && !t.ks_out) return cudaErrorInvalidValue;
  t.mmajor = (int64_t)(a.mode == kSwiGLU ? 2 : 1) * a.N * a.K * 2 <= MMAJOR_WEIGHT_BYTES;
  if (a.ctr && (e = cudaMemsetAsync(a.ctr, 0, sizeof(int32_t), st)) != cudaSuccess) return e;
  t.out = a.out;
  t.ldo = a.ldo;
  t.flags = a.flags;
  t.amaps = nullptr;
  if (zero_pad_pays(a)) {
    if ((reinterpret_cast<uintptr_t>(a.amaps) & 127) != 0) return cudaErrorInvalidValue;
    e = launch_group_maps(mA, mA64, a.amaps, a.offsets, a.G, a.rows_bound, a.A, (int64_t)a.K * 2,
                          a.A, (int64_t)a.K * 2, st);
    if (e != cudaSuccess) return e;
    t.amaps = reinterpret_cast<const CUtensorMap*>(a.amaps);
  }
  int64_t mt_bound = a.offsets ? (a.rows_bound + BMP - 1) / BMP + a.G : (a.single_rows + BMP - 1) / BMP;
  if (a.offsets && mt_bound > a.rows_bound) mt_bound = a.rows_bound;
  const int64_t tiles_bound = mt_bound * t.NT;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // clusters that fit on the GPU at once (per device, queried once)
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_clusters[dev] == 0) {
    e = cudaFuncSetAttribute(tc2_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, (void*)tc2_gemm_kernel, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters[dev] = n > 0 ? n : -1;
  }
  const int mc = max_clusters[dev].load();
  if (mc < 0) return cudaErrorNotSupported;
  // a K split needs every cluster there is (it splits until they are busy);
  // a call held to max_sms SMs takes at most max_sms / 2 clusters
  t.ks_clusters = mc;
  int64_t ncl = (t.part || tiles_bound >= mc) ? mc : tiles_bound;
  if (a.max_sms > 0 && ncl > a.max_sms / 2) ncl = a.max_sms / 2 > 0 ? a.max_sms / 2 : 1;
  cfg.gridDim = dim3((unsigned)(2 * ncl));
  e = cudaLaunchKernelEx(&cfg, tc2_gemm_kernel, mA, mA64, mB0, mB1, t);
  if (e != cudaSuccess) return e;
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (t.part) {
    const int64_t items = a.rows_bound * (a.N / 8);
    int64_t blocks = (items + 255) / 256;
    const int64_t cap = (int64_t)tc_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    bf16* out = reinterpret_cast<bf16*>(a.out);
    if (a.mode == kSwiGLU)
      split_reduce_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(
          t.part, t.part_ld, t.part_stride, t.ks_out, a.offsets, a.G, a.single_rows, a.rows_bound, a.N,
          out, a.ldo);
    else
      split_reduce_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(
          t.part, t.part_ld, t.part_stride, t.ks_out, a.offsets, a.G, a.single_rows, a.rows_bound, a.N,
          out, a.ldo);
    count_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace moe
