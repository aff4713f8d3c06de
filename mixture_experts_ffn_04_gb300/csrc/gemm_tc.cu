// gemm_tc.cu -- grouped bf16 GEMM on the 5th-generation tensor cores.
//
// Same contract as the CUDA-core engine ("Fused MoE Kernel Notes",
// group_gemm_same_nk: per-expert groups of rows with shared N and K; the
// m-tile schedule comes from the real group sizes, never from the token count).
//
// Design (one CTA per SM, persistent over a device-built tile list):
//   warp 0     A producer: tile [128 rows x 64 k] of the grouped activations,
//              by TMA (2-D tensor map); or, when the rows are gathered from
//              the token matrix through a row -> token table, warps 0, 7, 8
//              and 9, one per ring slot, with 16-byte cp.async copies written
//              straight into the swizzled layout (so the grouped copy of x
//              never exists);
//   warp 6     B producer: TMA tile [256 rows x 64 k] of the expert-major
//              weights (3-D tensor map {k, n, expert}); both tiles in the
//              128-byte swizzled K-major layout the MMA reads directly.
//   warp 1     TMEM owner and MMA issuer: one thread issues
//              tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16, bf16 in,
//              fp32 accumulate in TMEM), 4 per 64-wide k-block, and commits to
//              the stage's "empty" barrier; two 256-column accumulators
//              alternate so the epilogue of tile i overlaps the MMAs of i+1.
//   warps 2-5  epilogue: tcgen05.ld of 32 columns at a time, one TMEM lane
//              (= one output row) per thread, fused SwiGLU / rounding, masked
//              stores of the rows that belong to the tile's group.
// For SwiGLU the B tile stacks 128 gate rows over the same 128 up rows, so one
// N=256 MMA produces both halves: columns 0-127 gate, 128-255 up.
//
// Every mbarrier wait is bounded (about 2 s of SM clocks); a wait that runs out
// raises the kernel's abort flag, the other roles leave their loops, in-flight
// TMA loads and MMAs are waited for (bounded), TMEM is released and the
// device status word gets the timeout bit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64;
// Two load rings: the weight tiles (B, mostly first touches in DRAM) get a
// deeper ring than the activation tiles (A, mostly re-read from L2), so more
// DRAM bytes are in flight per SM within the shared-memory budget.
constexpr int SA = 4, SB = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int RING_BYTES = SA * A_BYTES + SB * B_BYTES;
// warps: 0 A producer, 1 MMA issuer, 2-5 epilogue, 6 B producer, 7-9 the other
// three A producers when the A rows are gathered (one warp per ring slot)
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int MAX_SMEM_G = 1024;   // larger group counts use a schedule kernel
constexpr int SCHED_BYTES = (MAX_SMEM_G + 1) * 4;
constexpr int GATHER_BYTES = SA * BM * 4;   // per gathering warp: source token of each tile row
// epilogue staging: per epilogue warp 32 rows x (64 B + 16 B pad)
constexpr int OUT_ROW_BYTES = 80;
constexpr int OUT_WARP_BYTES = 32 * OUT_ROW_BYTES;
constexpr int OUT_BYTES = 4 * OUT_WARP_BYTES;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES + OUT_BYTES + SCHED_BYTES + GATHER_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (15, 16 = 0), N >> 3 at 17-22, M >> 4 at 24-28.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
static_assert(SA == 4, "one gathering warp per A ring slot: warps 0, 7, 8, 9");

struct TcArgs {
  int mode, N, K, G, NT, KB;
  const int32_t* offsets;
  int64_t single_rows;
  int64_t rows_bound;
  const int32_t* sched;   // global m-tile prefix, or NULL: built in shared memory
  void* out;
  int64_t ldo;
  uint32_t* flags;
  int ksplit;             // >1 only for fp32 outputs: partial sums per K range
  int64_t split_stride;   // floats between partial outputs
  const bf16* gA;         // gathered A: row r of the operand is gA[gather[r]]
  const int32_t* gather;  // or NULL: A through the tensor map
  int64_t a_rows;         // rows of gA (bound on gather values)
  bf16* pre;              // SwiGLU: also the pre-activations [rows, ldp] = [gate | up]
  int64_t ldp;
  // grouped calls: group g's A map at amaps[2 g], spanning only the group's
  // rows, so the rows of its last tile past the group load as zeros (less
  // power in the tensor cores; the results do not change); NULL: tmA
  const CUtensorMap* amaps;
};

// Tile -> (K split, group, m-tile, n-tile).  Within a split, tiles of one
// group are ordered n-tile major, m-tile minor, so the CTAs sharing a weight
// tile run side by side.
__device__ __forceinline__ void decode_tile(const TcArgs& a, const int32_t* sched, int64_t tile,
                                            int& ks, int& g, int& mt, int& nt) {
  const int64_t per_split = (int64_t)sched[a.G] * a.NT;
  ks = (int)(tile / per_split);
  tile -= (int64_t)ks * per_split;
  int lo = 0, hi = a.G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)sched[mid] * a.NT <= tile) lo = mid; else hi = mid;
  }
  g = lo;
  const int mtg = sched[g + 1] - sched[g];
  const int64_t local = tile - (int64_t)sched[g] * a.NT;
  nt = (int)(local / mtg);
  mt = (int)(local % mtg);
}

// m-tile prefix of the groups, built by one warp into shared memory:
// sched[g] = sum over g' < g of ceil(rows_g' / BM); sched[G] = total, or 0 when
// the offsets are inconsistent or exceed the row bound (then nothing runs and
// CTA 0 raises the device flag).
__device__ void build_schedule(const TcArgs& a, int32_t* sched, int lane) {
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < a.G; base += 32) {
    const int g = base + lane;
    int v = 0;
    if (g < a.G) {
      int64_t cnt = a.offsets ? (int64_t)a.offsets[g + 1] - a.offsets[g] : a.single_rows;
      if (cnt < 0) { bad = true; cnt = 0; }
      v = (int)((cnt + BM - 1) / BM);
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

__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  // bars: fullA[SA] emptyA[SA] fullB[SB] emptyB[SB] tfull[2] tempty[2] final
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * SA + 2 * SB + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned char* s_out = smem + RING_BYTES + BAR_BYTES;
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_out + OUT_BYTES);
  int32_t* s_rows = s_sched + (MAX_SMEM_G + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t ringA = smem_base, ringB = smem_base + SA * A_BYTES;
  auto fullA = [&](int s) { return smem_u32(&bars[s]); };
  auto emptyA = [&](int s) { return smem_u32(&bars[SA + s]); };
  auto fullB = [&](int s) { return smem_u32(&bars[2 * SA + s]); };
  auto emptyB = [&](int s) { return smem_u32(&bars[2 * SA + SB + s]); };
  auto tfull_bar = [&](int b) { return smem_u32(&bars[2 * SA + 2 * SB + b]); };
  auto tempty_bar = [&](int b) { return smem_u32(&bars[2 * SA + 2 * SB + 2 + b]); };
  const uint32_t final_bar = smem_u32(&bars[2 * SA + 2 * SB + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(fullA(s), a.gather ? 32 : 1);   // gathered: one arrival per lane
      mbar_init(emptyA(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(fullB(s), 1);
      mbar_init(emptyB(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 128);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2 && a.sched == nullptr) build_schedule(a, s_sched, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t* sched = a.sched ? a.sched : s_sched;

  const int64_t total = (int64_t)sched[a.G] * a.NT * a.ksplit;

  if (a.gather != nullptr && (warp == 0 || warp >= 7)) {
    // ---------------- A ring by row gather (warps 0, 7, 8, 9) ----------------
    // The warp of slot `slot` fills every SA-th stage.  Lane l copies 16-byte
    // chunk (l & 7) of rows (l >> 3) + 4 i of the tile to its place in the
    // 128-byte swizzle (chunk c of row r at c ^ (r & 7)).  cp.async writes are
    // generic-proxy stores: each lane waits for its own copies, fences them
    // against the async proxy the MMA reads through, and arrives (32
    // arrivals a phase).  While one warp waits for its stage to land, the
    // other slots' warps keep copies in flight.
    const int slot = warp == 0 ? 0 : warp - 6;
    int32_t* rows = s_rows + slot * BM;
    const int ck = lane & 7, rl = lane >> 3;
    uint32_t use = 0;   // fills of this slot so far (phase = use & 1)
    int64_t n = 0;      // stage number in the MMA's order
    bool ok = true, bad = false;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int ks, g, mt, nt;
      decode_tile(a, sched, tile, ks, g, mt, nt);
      const int kb0 = ks * a.KB / a.ksplit, kb1 = (ks + 1) * a.KB / a.ksplit;
      const int64_t first = n;
      n += kb1 - kb0;
      // this slot's first k-block of the tile, if any
      int kb = kb0 + (int)((slot - first % SA + SA) % SA);
      if (kb >= kb1) continue;
      const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
      const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
      const int64_t tr0 = gbeg + (int64_t)mt * BM;
      __syncwarp();   // the previous tile's table is no longer read
      for (int i = lane; i < BM; i += 32) {
        int32_t src = -1;   // rows past the group are zero-filled
        if (tr0 + i < gend) {
          src = a.gather[tr0 + i];
          if (src < 0 || src >= a.a_rows) { bad = true; src = -1; }
        }
        rows[i] = src;
      }
      __syncwarp();
      for (; kb < kb1; kb += SA) {
        int w = 0;
        if (lane == 0) w = mbar_wait(emptyA(slot), (use & 1u) ^ 1u, abort_flag) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        const uint32_t dst0 = ringA + slot * A_BYTES;
        const int k0 = kb * BK + ck * 8;
        const bool kin = k0 < a.K;
#pragma unroll 8
        for (int i = 0; i < BM / 4; ++i) {
          const int r = rl + 4 * i;
          const int32_t src = rows[r];
          const bool in = kin && src >= 0;
          const bf16* p = a.gA + (in ? (int64_t)src * a.K + k0 : 0);
          cp_async16(dst0 + r * 128 + ((ck ^ (r & 7)) << 4), p, in ? 16u : 0u);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(fullA(slot));
        ++use;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");   // no copy outlives the CTA
    if (bad) set_flag(a.flags, kFlagGather);
  } else if ((warp == 0 || warp == 6) && lane == 0) {
    // ---------------- TMA producers: warp 0 the A ring, warp 6 the B ring ----
    const bool is_a = warp == 0;
    const int S = is_a ? SA : SB;
    int s = 0;
    uint32_t ph = 0, issued = 0, par = 0;
    const CUtensorMap* acquired = nullptr;   // per-group map last made visible
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int ks, g, mt, nt;
      decode_tile(a, sched, tile, ks, g, mt, nt);
      const int64_t gbase = a.offsets ? a.offsets[g] : 0;
      int arow = (int)(gbase + (int64_t)mt * BM);
      const CUtensorMap* amap = &tmA;
      if (is_a && a.amaps) {
        amap = a.amaps + 2 * g;
        arow = mt * BM;
        if (amap != acquired) {   // written by the preceding kernel
          asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                           reinterpret_cast<uint64_t>(amap))
                       : "memory");
          acquired = amap;
        }
      }
      const int kb0 = ks * a.KB / a.ksplit, kb1 = (ks + 1) * a.KB / a.ksplit;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t fb = is_a ? fullA(s) : fullB(s);
        if (!mbar_wait(is_a ? emptyA(s) : emptyB(s), ph ^ 1u, abort_flag)) { ok = false; break; }
        if (is_a) {
          mbar_expect_tx(fb, A_BYTES);
          tma_load_2d(ringA + s * A_BYTES, amap, kb * BK, arow, fb);
        } else {
          const uint32_t sb = ringB + s * B_BYTES;
          mbar_expect_tx(fb, B_BYTES);
          if (a.mode == kSwiGLU) {
            tma_load_3d(sb, &tmB0, kb * BK, nt * (BN / 2), g, fb);
            tma_load_3d(sb + B_BYTES / 2, &tmB1, kb * BK, nt * (BN / 2), g, fb);
          } else {
            tma_load_3d(sb, &tmB0, kb * BK, nt * BN, g, fb);
          }
        }
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      // let every load still in flight land before the CTA goes away
      for (int i = 0; i < S; ++i)
        if (issued & (1u << i)) mbar_wait_quiet(is_a ? fullA(i) : fullB(i), (par >> i) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int sa = 0, sb = 0, acc = 0;
      uint32_t pha = 0, phb = 0, aph = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const int ks = (int)(tile / ((int64_t)sched[a.G] * a.NT));
        const int nkb = (ks + 1) * a.KB / a.ksplit - ks * a.KB / a.ksplit;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(fullA(sa), pha, abort_flag) || !mbar_wait(fullB(sb), phb, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = ringA + sa * A_BYTES;
          const uint32_t b_addr = ringB + sb * B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            tc_mma(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), IDESC,
                   (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(emptyA(sa));
          tc_commit(emptyB(sb));
          if (++sa == SA) { sa = 0; pha ^= 1u; }
          if (++sb == SB) { sb = 0; phb ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if (*abort_flag) {
        tc_commit(final_bar);
        mbar_wait_quiet(final_bar, 0);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue (warps 2..5) ----------------
    // Each thread owns one accumulator row (its TMEM lane).  A 32-column
    // chunk is finished in registers, staged in this warp's shared-memory
    // slice, and written back row by row with 16-byte stores, 4 or 8 lanes per
    // row, so every global write covers whole sectors.
    const int q = warp & 3;  // TMEM lanes this warp may read: 32q .. 32q+31
    unsigned char* stage = s_out + (warp - 2) * OUT_WARP_BYTES;
    unsigned char* my_row = stage + lane * OUT_ROW_BYTES;
    int acc = 0;
    uint32_t aph = 0;
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int ks, g, mt, nt;
      decode_tile(a, sched, tile, ks, g, mt, nt);
      const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
      const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
      const int64_t row0 = gbeg + (int64_t)mt * BM + q * 32;   // this warp's first row
      const int64_t nvalid64 = gend - row0;
      const int nvalid = nvalid64 < 0 ? 0 : (nvalid64 > 32 ? 32 : (int)nvalid64);
      // all 32 lanes must agree before the warp-collective tcgen05.ld
      if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, abort_flag))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * BN;
      if (a.mode != kStoreF32) {
        const bool swiglu = a.mode == kSwiGLU;
        const int n0 = swiglu ? nt * (BN / 2) : nt * BN;
        const int ncols = swiglu ? BN / 2 : BN;
        bf16* out = reinterpret_cast<bf16*>(a.out);
#pragma unroll 1
        for (int c = 0; c < ncols && n0 + c < a.N; c += 32) {
          uint32_t gr[32];
          uint4 packed[4], pg[4], pu[4];
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
            if (a.pre) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float fg[8], fu[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  fg[e] = __uint_as_float(gr[v * 8 + e]);
                  fu[e] = __uint_as_float(ur[v * 8 + e]);
                }
                pg[v] = pack16(fg, (const bf16*)nullptr);
                pu[v] = pack16(fu, (const bf16*)nullptr);
              }
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
#pragma unroll
          for (int v = 0; v < 4; ++v) reinterpret_cast<uint4*>(my_row)[v] = packed[v];
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int p = lane + 32 * i;      // 128 pieces: 32 rows x 4 x 16 B
            const int rr = p >> 2, pc = p & 3;
            const int n = n0 + c + pc * 8;
            if (rr < nvalid && n < a.N)
              *reinterpret_cast<uint4*>(out + (row0 + rr) * a.ldo + n) =
                  *reinterpret_cast<const uint4*>(stage + rr * OUT_ROW_BYTES + pc * 16);
          }
          __syncwarp();
          if (swiglu && a.pre) {
            // the gate and up pre-activations, rounded once, for the backward
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                reinterpret_cast<uint4*>(my_row)[v] = part ? pu[v] : pg[v];
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int p = lane + 32 * i;
                const int rr = p >> 2, pc = p & 3;
                const int n = n0 + c + pc * 8;
                if (rr < nvalid && n < a.N)
                  *reinterpret_cast<uint4*>(a.pre + (row0 + rr) * a.ldp + part * a.N + n) =
                      *reinterpret_cast<const uint4*>(stage + rr * OUT_ROW_BYTES + pc * 16);
              }
              __syncwarp();
            }
          }
        }
      } else {
        // fp32 rows (router logits): ldo and split_stride are multiples of 4
        const int n0 = nt * BN;
        float* out = reinterpret_cast<float*>(a.out) + ks * a.split_stride;
#pragma unroll 1
        for (int c = 0; c < BN && n0 + c < a.N; c += 32) {
          uint32_t vr[32];
          tmem_ld32(taddr + c, vr);
          tmem_wait_ld();
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {   // two 16-column halves
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<uint4*>(my_row)[v] =
                  make_uint4(vr[16 * hf + 4 * v], vr[16 * hf + 4 * v + 1], vr[16 * hf + 4 * v + 2],
                             vr[16 * hf + 4 * v + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int p = lane + 32 * i;      // 128 pieces: 32 rows x 4 x 16 B
              const int rr = p >> 2, pc = p & 3;
              const int n = n0 + c + 16 * hf + pc * 4;
              if (rr < nvalid && n < a.N) {
                float* dst = out + (row0 + rr) * a.ldo + n;
                const float* src =
                    reinterpret_cast<const float*>(stage + rr * OUT_ROW_BYTES + pc * 16);
                if (n + 3 < a.N) {
                  *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(src);
                } else {
                  for (int e = 0; e < 4 && n + e < a.N; ++e) dst[e] = src[e];
                }
              }
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) set_flag(a.flags, kFlagTimeout);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over a row-major bf16 matrix [rows, K], box 64 x box_rows.
bool make_map_2d(CUtensorMap* m, const void* ptr, int64_t rows, int K, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map {K, N, G} over G matrices [N, K] that start `gstride` elements apart.
bool make_map_3d(CUtensorMap* m, const void* ptr, int N, int K, int G, int64_t gstride,
                 int box_rows) {
  if (G == 1 && gstride == 0) gstride = (int64_t)N * K;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)gstride * 2};
  cuuint32_t box[3] = {BK, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace tc

int tc_sm_count() { return tc::sm_count(); }

int router_split(int64_t rows, int ncols, int K) {
  const int64_t base = ((rows + tc::BM - 1) / tc::BM) * ((ncols + tc::BN - 1) / tc::BN);
  const int kb = (K + tc::BK - 1) / tc::BK;
  int64_t s = base > 0 ? tc::sm_count() / base : 1;
  if (s > kMaxSplit) s = kMaxSplit;
  if (s > kb / 4) s = kb / 4;
  return s < 1 ? 1 : (int)s;
}

cudaError_t launch_group_maps(const CUtensorMap& baseA, const CUtensorMap& baseB, void* maps,
                              const int32_t* offsets, int G, int64_t rows_bound, const void* A,
                              int64_t lda_bytes, const void* B, int64_t ldb_bytes,
                              cudaStream_t st);   // gemm_bwd.cu

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st) {
  using namespace tc;
  if (a.dtype != MOE_BF16 || encode_fn() == nullptr) return cudaErrorNotSupported;
  if (a.wfmt) return cudaErrorNotSupported;   // MXFP8 weights: decode or CUDA-core engine
  // bf16 outputs are stored as 8-element vectors; fp32 outputs column by column
  if ((a.K % 8) != 0 || (a.mode != kStoreF32 && (a.N % 8) != 0) || a.K <= 0 || a.N <= 0)
    return cudaErrorInvalidValue;
  if (a.ksplit < 1 || (a.ksplit > 1 && a.mode != kStoreF32)) return cudaErrorInvalidValue;
  cudaError_t e;
  const bool smem_sched = a.G <= MAX_SMEM_G;
  if (!smem_sched) {
    e = launch_schedule(a, BM, st);
    if (e != cudaSuccess) return e;
  }
  const int64_t rows = a.offsets ? a.rows_bound : a.single_rows;
  if (rows <= 0) return cudaSuccess;
  const int brows = a.mode == kSwiGLU ? BN / 2 : BN;
  CUtensorMap mA, mB0, mB1;
  if (a.gather) {
    // the A map is unused; any valid map will do
    if (!make_map_2d(&mA, a.A, a.a_rows > 0 ? a.a_rows : 1, a.K, BM)) return cudaErrorInvalidValue;
  } else if (!make_map_2d(&mA, a.A, rows, a.K, BM)) {
    return cudaErrorInvalidValue;
  }
  if (!make_map_3d(&mB0, a.B0, a.N, a.K, a.G, a.bstride, brows)) return cudaErrorInvalidValue;
  if (a.mode == kSwiGLU) {
    if (!make_map_3d(&mB1, a.B1, a.N, a.K, a.G, a.bstride, brows)) return cudaErrorInvalidValue;
  } else {
    mB1 = mB0;
  }
  TcArgs t;
  t.mode = a.mode;
  t.N = a.N;
  t.K = a.K;
  t.G = a.G;
  t.NT = (a.N + brows - 1) / brows;
  t.KB = (a.K + BK - 1) / BK;
  t.offsets = a.offsets;
  t.single_rows = a.single_rows;
  t.rows_bound = a.rows_bound;
  t.sched = smem_sched ? nullptr : a.sched;
  t.ksplit = a.ksplit;
  t.split_stride = a.split_stride;
  t.out = a.out;
  t.ldo = a.ldo;
  t.flags = a.flags;
  t.gA = reinterpret_cast<const bf16*>(a.A);
  t.gather = a.gather;
  t.a_rows = a.a_rows;
  t.pre = reinterpret_cast<bf16*>(a.pre);
  t.ldp = a.ldp;
  if (t.pre && (a.mode != kSwiGLU || (a.ldp % 8) != 0)) return cudaErrorInvalidValue;
  t.amaps = nullptr;
  if (zero_pad_pays(a)) {
    if ((reinterpret_cast<uintptr_t>(a.amaps) & 127) != 0) return cudaErrorInvalidValue;
    e = launch_group_maps(mA, mA, a.amaps, a.offsets, a.G, a.rows_bound, a.A, (int64_t)a.K * 2,
                          a.A, (int64_t)a.K * 2, st);
    if (e != cudaSuccess) return e;
    t.amaps = reinterpret_cast<const CUtensorMap*>(a.amaps);
  }
  int64_t mt_bound = a.offsets ? (a.rows_bound + BM - 1) / BM + a.G : (a.single_rows + BM - 1) / BM;
  if (a.offsets && mt_bound > a.rows_bound) mt_bound = a.rows_bound;  // >= 1 row per tile
  const int64_t tiles_bound = mt_bound * t.NT * t.ksplit;
  static bool attr_done[64] = {false};   // the attribute is per device
  static std::mutex attr_mu;               // several host threads may launch
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_done[dev]) {
      e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      attr_done[dev] = true;
    }
  }
  const int sms = a.max_sms > 0 && a.max_sms < sm_count() ? a.max_sms : sm_count();
  int grid = (int)(tiles_bound < sms ? tiles_bound : sms);
  if (a.max_sms > 0 && tiles_bound > grid) {
    // held to max_sms SMs: the fewest CTAs that take the same rounds of tiles
    const int64_t rounds = (tiles_bound + grid - 1) / grid;
    grid = (int)((tiles_bound + rounds - 1) / rounds);
  }
  tc_gemm_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(mA, mB0, mB1, t);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
