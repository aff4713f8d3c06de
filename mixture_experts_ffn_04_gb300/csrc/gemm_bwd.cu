// gemm_bwd.cu -- the backward grouped GEMMs of the routed experts on the
// 5th-generation tensor cores ("Fused MoE Kernel Notes", Backward grouped-GEMM
// launch bound).
//
// Two shapes of grouped GEMM:
//  * dgrad (group_gemm_same_nk): groups of rows with the same N and K, the
//    m-tile schedule built on the device from the real group sizes, so a
//    group larger than the token count (duplicate routes) is covered in full
//    -- the bound is the scattered row count, never the token count.
//      out[r, n] = sum_k A[r, k] * W_g[k, n]
//    W_g is an expert's weight read in its stored [K, N] layout, i.e. the
//    operand is N-major (MN-major in tcgen05 terms).  K may come in two
//    segments with separate weights (dx = dA . W_gate + dB . W_up over the
//    concatenated [dA | dB] rows).  Epilogues: plain store (dx rows) or the
//    SwiGLU derivative (dh -> [da | db] from the saved pre-activations).
//  * wgrad (group_gemm_same_mn): every group has the same M x N output and
//    its own K = the group's row count:
//      dW_g[m, n] = sum over rows r of group g of A[r, m] * B[r, n]
//    Both operands are read in their stored [rows, M] / [rows, N] layouts
//    (MN-major), through tensor maps of the group's own rows: a small kernel
//    writes, per group, copies of the two maps whose base is the group's
//    first row and whose row extent is the group's size (tensormap.replace),
//    so the TMA zero-fills what a group's last k-block reaches past its end
//    and no row of the next group enters the sum.  A group with no rows gets
//    a zero gradient.
//
// Pipeline (one CTA per SM, persistent over the tile list): warp 0 lane 0
// issues the TMA loads of a stage (A and B on one "full" barrier), warp 1
// owns TMEM and issues tcgen05.mma (M = 128, N =
// 256, K = 16) into one of two 256-column fp32 accumulators; warps 2-9 drain
// the other accumulator (tcgen05.ld; two warps per 32-lane quarter, one per
// half of the columns), finish the values and store them through a
// shared-memory staging slice as whole-row 16-byte pieces.  The weight
// gradient's tiles carry few k-blocks (a group's rows), so its epilogue has
// to keep pace with about one tile of MMAs: hence eight epilogue warps, the
// group offsets staged in shared memory, and a last block that issues only
// the K = 16 steps holding rows of the group.
// MN-major operands sit in shared memory as 64-element-wide boxes, each box
// 64 k-rows of 128 bytes with the 128-byte swizzle; an MMA's K = 16 slice is
// two 8-row core groups of every box.
// Every wait is bounded; a wait that runs out aborts the kernel cleanly
// (loads and MMAs in flight are waited for, TMEM is freed, the device status
// word gets the timeout bit).
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace moe {
namespace tc {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();   // gemm_tc.cu
int sm_count();
}  // namespace tc

namespace tcb {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int S = 4;                              // pipeline stages
constexpr int A_BYTES = BM * BK * 2;              // 16 KB
constexpr int B_BYTES = BN * BK * 2;              // 32 KB
constexpr int BOX_BYTES = 64 * BK * 2;            // one 64-wide MN box: 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RING_BYTES = S * STAGE_BYTES;
constexpr int THREADS = 320;                      // warps 0-9
constexpr int EPI_WARPS = 8;                      // warps 2-9: two per TMEM lane quarter
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int MAX_SMEM_G = 1024;
constexpr int SCHED_BYTES = (MAX_SMEM_G + 1) * 4;
constexpr int OUT_ROW_BYTES = 80;
constexpr int OUT_WARP_BYTES = 32 * OUT_ROW_BYTES;
constexpr int OUT_BYTES = EPI_WARPS * OUT_WARP_BYTES;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES + OUT_BYTES + SCHED_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
static_assert((2 * S + 5) * 8 + 8 <= BAR_BYTES, "barrier area");

// kind::f16 instruction descriptor: D fp32, A and B bf16, N = 256, M = 128;
// bit 15: A MN-major, bit 16: B MN-major.
constexpr uint32_t IDESC_BASE = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
constexpr uint32_t IDESC_DGRAD = IDESC_BASE | (1u << 16);
constexpr uint32_t IDESC_WGRAD = IDESC_BASE | (1u << 15) | (1u << 16);

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle:
// 64-element MN blocks `lbo` bytes apart (leading byte offset), 8-row K core
// groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(lbo >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

struct Args {
  int kind;               // kBwdDgrad, kBwdDgradSwiGLU, kBwdWgrad
  int M, N;               // wgrad: output rows, columns; dgrad: N
  int K0, KB0, KB;        // dgrad: first K segment, its k-blocks, all k-blocks
  int G, MT, NT;
  const int32_t* offsets;
  int64_t rows_bound;
  const int32_t* sched;   // dgrad: global m-tile prefix, or NULL: in shared memory
  bf16* out;
  int64_t ldo, ostride;
  const bf16* pre;        // dgrad + SwiGLU: [rows, ldp] = [a | b]
  int64_t ldp;
  uint32_t* flags;
  const CUtensorMap* tmaps;   // wgrad: per group g, A's map at 2g, B's at 2g + 1
  // MN-major operands whose width is a multiple of 64 are mapped with the
  // 64-wide blocks as an outer dimension, so one TMA box brings every block
  // of a stage (wgrad: A and B; dgrad: B); otherwise one box per block
  int a_wide, b_wide;
};

// Rows of group g, 0 when the offsets are inconsistent (same answer in every
// role, so all of them skip the same tiles).  off: the offsets, staged in
// shared memory when they fit.
__device__ __forceinline__ int64_t group_rows(const Args& a, const int32_t* off, int g,
                                              int64_t& beg) {
  beg = off[g];
  const int64_t end = off[g + 1];
  if (beg < 0 || end < beg || end > a.rows_bound) return 0;
  return end - beg;
}

// dgrad tile -> (group, m-tile, n-tile); n-tile major within a group.
__device__ __forceinline__ void decode_dgrad(const Args& a, const int32_t* sched, int64_t tile,
                                             int& g, int& mt, int& nt) {
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

// wgrad tile -> (group, m-tile, n-tile): group major, so the CTAs running at
// the same time share one group's rows in L2.
__device__ __forceinline__ void decode_wgrad(const Args& a, int64_t tile, int& g, int& mt,
                                             int& nt) {
  const int64_t per = (int64_t)a.MT * a.NT;
  g = (int)(tile / per);
  const int64_t r = tile - (int64_t)g * per;
  nt = (int)(r / a.MT);
  mt = (int)(r % a.MT);
}

__device__ void build_schedule(const Args& a, int32_t* sched, int lane) {
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < a.G; base += 32) {
    const int g = base + lane;
    int v = 0;
    if (g < a.G) {
      int64_t cnt = (int64_t)a.offsets[g + 1] - a.offsets[g];
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
  if (lane == 0) bad |= a.offsets[0] != 0 || (int64_t)a.offsets[a.G] > a.rows_bound;
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sched[a.G] = bad ? 0 : carry;
    if (bad && blockIdx.x == 0) set_flag(a.flags, kFlagRows);
  }
}

// Write 32 rows x 32 columns (this warp's chunk, already packed to bf16 in
// `packed`, one row per lane) through the warp's staging slice: rows
// row_ptr(rr) for rr < nvalid, columns n .. n+31 below ncap.
template <typename RowPtr>
__device__ __forceinline__ void store_chunk(unsigned char* stage, int lane, const uint4 (&packed)[4],
                                            int nvalid, int n, int ncap, RowPtr row_ptr) {
  unsigned char* my_row = stage + lane * OUT_ROW_BYTES;
#pragma unroll
  for (int v = 0; v < 4; ++v) reinterpret_cast<uint4*>(my_row)[v] = packed[v];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = lane + 32 * i;   // 128 pieces: 32 rows x 4 x 16 B
    const int rr = p >> 2, pc = p & 3;
    const int col = n + pc * 8;
    if (rr < nvalid && col < ncap)
      *reinterpret_cast<uint4*>(row_ptr(rr) + col) =
          *reinterpret_cast<const uint4*>(stage + rr * OUT_ROW_BYTES + pc * 16);
  }
  __syncwarp();
}

__global__ void __launch_bounds__(THREADS, 1)
    bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const Args a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  // bars: full[S] empty[S] tfull[2] tempty[2] final
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned char* s_out = smem + RING_BYTES + BAR_BYTES;
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_out + OUT_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool wgrad = a.kind == kBwdWgrad;
  const uint32_t ring = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[S + s]); };
  auto tfull = [&](int b) { return smem_u32(&bars[2 * S + b]); };
  auto tempty = [&](int b) { return smem_u32(&bars[2 * S + 2 + b]); };
  const uint32_t final_bar = smem_u32(&bars[2 * S + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 32 * EPI_WARPS);
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
  if (warp == 2 && !wgrad && a.sched == nullptr) build_schedule(a, s_sched, lane);
  if (warp == 3 && wgrad && a.G <= MAX_SMEM_G)
    for (int g = lane; g <= a.G; g += 32) s_sched[g] = a.offsets[g];
  if (warp == 2 && wgrad && blockIdx.x == 0) {
    // offsets must rise from 0 to at most the row bound; a group whose own
    // range is invalid is skipped (group_rows), and the flag says so
    bool bad = lane == 0 && (a.offsets[0] != 0 || (int64_t)a.offsets[a.G] > a.rows_bound);
    for (int g = lane; g < a.G; g += 32) bad |= a.offsets[g + 1] < a.offsets[g];
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_flag(a.flags, kFlagRows);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t* sched = a.sched ? a.sched : s_sched;
  const int32_t* off = wgrad && a.G <= MAX_SMEM_G ? s_sched : a.offsets;
  const int64_t total =
      wgrad ? (int64_t)a.G * a.MT * a.NT : (int64_t)sched[a.G] * a.NT;

  // k-blocks of a tile, and for dgrad the first row of its A tile
  auto tile_kblocks = [&](int64_t tile, int& g, int& mt, int& nt, int64_t& r0) -> int {
    if (wgrad) {
      decode_wgrad(a, tile, g, mt, nt);
      const int64_t rows = group_rows(a, off, g, r0);
      return (int)((rows + BK - 1) / BK);
    }
    decode_dgrad(a, sched, tile, g, mt, nt);
    r0 = (int64_t)a.offsets[g] + (int64_t)mt * BM;
    return a.KB;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int s = 0;
      uint32_t ph = 0, issued = 0, par = 0;
      bool ok = true;
      int gmap = -1;   // wgrad: the group whose maps were last acquired
      for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int g, mt, nt;
        int64_t r0;
        const int nkb = tile_kblocks(tile, g, mt, nt, r0);
        const CUtensorMap* gA = &tmA;
        const CUtensorMap* gB = &tmB0;
        if (wgrad && nkb > 0) {
          gA = a.tmaps + 2 * g;
          gB = gA + 1;
          if (g != gmap) {   // maps written by the preceding kernel
            asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                             reinterpret_cast<uint64_t>(gA))
                         : "memory");
            asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                             reinterpret_cast<uint64_t>(gB))
                         : "memory");
            gmap = g;
          }
        }
        const int m0 = mt * BM, n0 = nt * BN;
        // boxes wholly past M or N are not loaded: they only feed outputs
        // the epilogue drops
        const int na = wgrad ? (m0 + 64 < a.M ? 2 : 1) : 1;
        int nb = (a.N - n0 + 63) / 64;
        if (nb > 4) nb = 4;
        const uint32_t bytes = (uint32_t)(wgrad && !a.a_wide ? na * BOX_BYTES : A_BYTES) +
                               (uint32_t)(a.b_wide ? B_BYTES : nb * BOX_BYTES);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty(s), ph ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t sa = ring + s * STAGE_BYTES, sb = sa + A_BYTES;
          mbar_expect_tx(full(s), bytes);
          if (wgrad) {
            const int r = kb * BK;   // row within the group's maps
            if (a.a_wide) tma_load_3d(sa, gA, 0, r, m0 / 64, full(s));
            else for (int j = 0; j < na; ++j) tma_load_2d(sa + j * BOX_BYTES, gA, m0 + 64 * j, r, full(s));
            if (a.b_wide) tma_load_3d(sb, gB, 0, r, n0 / 64, full(s));
            else for (int j = 0; j < nb; ++j) tma_load_2d(sb + j * BOX_BYTES, gB, n0 + 64 * j, r, full(s));
          } else {
            const bool seg1 = kb >= a.KB0;
            const int kk = seg1 ? kb - a.KB0 : kb;
            const int acol = seg1 ? a.K0 + kk * BK : kb * BK;
            tma_load_2d(sa, &tmA, acol, (int)r0, full(s));
            const CUtensorMap* mb = seg1 ? &tmB1 : &tmB0;
            if (a.b_wide) tma_load_4d(sb, mb, 0, kk * BK, n0 / 64, g, full(s));
            else for (int j = 0; j < nb; ++j) tma_load_3d(sb + j * BOX_BYTES, mb, n0 + 64 * j, kk * BK, g, full(s));
          }
          issued |= 1u << s;
          par = (par & ~(1u << s)) | (ph << s);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (*abort_flag) {
        for (int i = 0; i < S; ++i)
          if (issued & (1u << i)) mbar_wait_quiet(full(i), (par >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (lane 0) ----------------
    int s = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    const uint32_t idesc = wgrad ? IDESC_WGRAD : IDESC_DGRAD;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int g, mt, nt;
      int64_t r0;
      const int nkb = tile_kblocks(tile, g, mt, nt, r0);
      if (nkb == 0) continue;   // empty group: the epilogue writes zeros
      int64_t rows = 0;
      if (wgrad) rows = group_rows(a, off, g, r0);
      int w = 1;
      if (lane == 0) w = mbar_wait(tempty(acc), aph ^ 1u, abort_flag) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)acc * BN;
      for (int kb = 0; kb < nkb; ++kb) {
        w = mbar_wait(full(s), ph, abort_flag) ? 1 : 0;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        const uint32_t sa = ring + s * STAGE_BYTES, sb = sa + A_BYTES;
        const int64_t left = rows - (int64_t)kb * BK;
        const int valid = wgrad && left < BK ? (int)left : BK;
        // K = 16 steps of this block that hold rows of the group (rows past
        // the group's end arrive as zeros; later steps are not issued)
        const int ksteps = (valid + 15) / 16;
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            if (k >= ksteps) break;
            const uint64_t ad = wgrad ? sw128_mn_desc(sa + k * 2048, BOX_BYTES) : sw128_desc(sa + k * 32);
            const uint64_t bd = sw128_mn_desc(sb + k * 2048, BOX_BYTES);
            tc_mma(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        __syncwarp();
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(tfull(acc));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (lane == 0 && *abort_flag) {
      tc_commit(final_bar);
      mbar_wait_quiet(final_bar, 0);
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    // warps w and w + 4 read the same TMEM lanes (32q .. 32q+31, q = w & 3)
    // and split the 256 accumulator columns into halves
    const int q = warp & 3;
    const int c_lo = ((warp - 2) / 4) * (BN / 2), c_hi = c_lo + BN / 2;
    unsigned char* stage = s_out + (warp - 2) * OUT_WARP_BYTES;
    int acc = 0;
    uint32_t aph = 0;
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int g, mt, nt;
      int64_t r0;
      const int nkb = tile_kblocks(tile, g, mt, nt, r0);
      const int n0 = nt * BN;
      int nvalid;
      bf16* obase;          // this warp's first output row
      int64_t first_row;    // dgrad: its row index
      if (wgrad) {
        const int m = mt * BM + q * 32;
        nvalid = a.M - m <= 0 ? 0 : (a.M - m >= 32 ? 32 : a.M - m);
        obase = a.out + (int64_t)g * a.ostride + (int64_t)m * a.ldo;
        first_row = 0;
      } else {
        const int64_t gend = a.offsets[g + 1];
        first_row = r0 + q * 32;
        const int64_t left = gend - first_row;
        nvalid = left <= 0 ? 0 : (left >= 32 ? 32 : (int)left);
        obase = a.out + first_row * a.ldo;
      }
      auto row_ptr = [&](int rr) { return obase + (int64_t)rr * a.ldo; };
      if (nkb == 0) {
        // a group without rows has a zero weight gradient
        const uint4 z[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                            make_uint4(0, 0, 0, 0)};
        for (int c = c_lo; c < c_hi && n0 + c < a.N; c += 32)
          store_chunk(stage, lane, z, nvalid, n0 + c, a.N, row_ptr);
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(tfull(acc), aph, abort_flag))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * BN;
      // finish 32 accumulator columns (c .. c+31 of the tile) and store them
      auto finish = [&](const uint32_t (&v)[32], int c) {
        const int n = n0 + c;
        if (a.kind == kBwdDgradSwiGLU) {
          // dh -> da = dh * b * silu'(a), db = dh * silu(a) with the saved
          // pre-activations a = pre[r, n], b = pre[r, N + n]
          uint4 pa[4], pb[4];
          const bool live = lane < nvalid;
          const bf16* prow = a.pre + (first_row + (live ? lane : 0)) * a.ldp;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool in = live && n + 8 * j < a.N;
            pa[j] = in ? __ldg(reinterpret_cast<const uint4*>(prow + n) + j) : make_uint4(0, 0, 0, 0);
            pb[j] = in ? __ldg(reinterpret_cast<const uint4*>(prow + a.N + n) + j) : make_uint4(0, 0, 0, 0);
          }
          uint4 da[4], db[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float fa[8], fb[8], oa[8], ob[8];
            unpack16(pa[j], fa, (const bf16*)nullptr);
            unpack16(pb[j], fb, (const bf16*)nullptr);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float dh = __uint_as_float(v[8 * j + e]);
              const float sg = __fdividef(1.0f, 1.0f + __expf(-fa[e]));
              oa[e] = dh * fb[e] * sg * (1.0f + fa[e] * (1.0f - sg));
              ob[e] = dh * fa[e] * sg;
            }
            da[j] = pack16(oa, (const bf16*)nullptr);
            db[j] = pack16(ob, (const bf16*)nullptr);
          }
          store_chunk(stage, lane, da, nvalid, n, a.N, row_ptr);
          store_chunk(stage, lane, db, nvalid, n, a.N,
                      [&](int rr) { return obase + (int64_t)rr * a.ldo + a.N; });
        } else {
          uint4 pk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[8 * j + e]);
            pk[j] = pack16(f, (const bf16*)nullptr);
          }
          store_chunk(stage, lane, pk, nvalid, n, a.N, row_ptr);
        }
      };
      // two 32-column TMEM loads in flight per wait
#pragma unroll 1
      for (int c = c_lo; c < c_hi && n0 + c < a.N; c += 64) {
        uint32_t v0[32], v1[32];
        const bool two = c + 32 < c_hi && n0 + c + 32 < a.N;
        tmem_ld32(taddr + c, v0);
        if (two) tmem_ld32(taddr + c + 32, v1);
        tmem_wait_ld();
        finish(v0, c);
        if (two) finish(v1, c + 32);
      }
      tc_fence_before();
      mbar_arrive(tempty(acc));
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

// Per-group copies of two operand maps (the weight gradient's A and B; the
// forward GEMMs' A maps of two box heights): group g's maps start at its
// first row and span its rows (at least one, so the map stays valid for a
// group without rows, whose tiles load nothing).  One warp per
// group: copy the base map to shared memory, replace the base address and the
// row extent (dimension 1), and copy it out with the proxy fence that makes
// it visible to the TMA unit.
__global__ void __launch_bounds__(32) group_maps_kernel(const __grid_constant__ CUtensorMap baseA,
                                                        const __grid_constant__ CUtensorMap baseB,
                                                        CUtensorMap* maps, const int32_t* offsets,
                                                        int G, int64_t rows_bound,
                                                        const char* A, int64_t lda_bytes,
                                                        const char* B, int64_t ldb_bytes) {
  __shared__ __align__(128) CUtensorMap sm[2];
  const int lane = threadIdx.x;
  for (int g = blockIdx.x; g < G; g += gridDim.x) {
    int64_t beg = offsets[g], end = offsets[g + 1];
    if (beg < 0 || end < beg || end > rows_bound) beg = end = 0;
    const uint32_t rows = end > beg ? (uint32_t)(end - beg) : 1u;
    if (lane < 8) {
      reinterpret_cast<uint4*>(&sm[0])[lane] = reinterpret_cast<const uint4*>(&baseA)[lane];
      reinterpret_cast<uint4*>(&sm[1])[lane] = reinterpret_cast<const uint4*>(&baseB)[lane];
    }
    __syncwarp();
    if (lane == 0) {
      const uint32_t s0 = smem_u32(&sm[0]), s1 = smem_u32(&sm[1]);
      const uint64_t pa = reinterpret_cast<uint64_t>(A + beg * lda_bytes);
      const uint64_t pb = reinterpret_cast<uint64_t>(B + beg * ldb_bytes);
      asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(s0),
                   "l"(pa)
                   : "memory");
      asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], 1, %1;" ::"r"(s0),
                   "r"(rows)
                   : "memory");
      asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(s1),
                   "l"(pb)
                   : "memory");
      asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], 1, %1;" ::"r"(s1),
                   "r"(rows)
                   : "memory");
    }
    __syncwarp();
    asm volatile(
        "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned"
        " [%0], [%1], 128;" ::"l"(reinterpret_cast<uint64_t>(maps + 2 * g)),
        "r"(smem_u32(&sm[0]))
        : "memory");
    asm volatile(
        "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned"
        " [%0], [%1], 128;" ::"l"(reinterpret_cast<uint64_t>(maps + 2 * g + 1)),
        "r"(smem_u32(&sm[1]))
        : "memory");
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// 2-D map over bf16 rows: `width` elements of each row used, rows `ld`
// elements apart; box 64 x box_rows, 128-byte swizzle.
static bool map_rows(CUtensorMap* m, const void* ptr, int64_t rows, int64_t width, int64_t ld,
                     int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map {64, rows, width / 64} over the same rows: the 64-wide column blocks
// as the outer dimension, box 64 x 64 rows x `blocks`, so one box lands as
// `blocks` consecutive [64 rows][64] tiles (width a multiple of 64).
static bool map_rows_wide(CUtensorMap* m, const void* ptr, int64_t rows, int64_t width, int64_t ld,
                          int blocks) {
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(width / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
  cuuint32_t box[3] = {64, 64, (cuuint32_t)blocks};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map {64, K, N / 64, G} over G weight matrices stored [K, N], box
// 64 x 64 x 4 x 1: a stage's four 64-wide blocks in one box (N a multiple of 64).
static bool map_weights_kn_wide(CUtensorMap* m, const void* ptr, int N, int K, int G,
                                int64_t gstride) {
  if (G == 1 && gstride == 0) gstride = (int64_t)N * K;
  cuuint64_t dims[4] = {64, (cuuint64_t)K, (cuuint64_t)(N / 64), (cuuint64_t)G};
  cuuint64_t strides[3] = {(cuuint64_t)N * 2, 128, (cuuint64_t)gstride * 2};
  cuuint32_t box[4] = {64, 64, 4, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map {N, K, G} over G weight matrices stored [K, N] (N contiguous),
// `gstride` elements apart; box 64 (N) x 64 (K) x 1.
static bool map_weights_kn(CUtensorMap* m, const void* ptr, int N, int K, int G, int64_t gstride) {
  if (G == 1 && gstride == 0) gstride = (int64_t)N * K;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)K, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)gstride * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcb

// Per-group operand maps for other engines (the SM-pair forward GEMM's A
// maps): the same kernel, launched on `st`.
cudaError_t launch_group_maps(const CUtensorMap& baseA, const CUtensorMap& baseB, void* maps,
                              const int32_t* offsets, int G, int64_t rows_bound, const void* A,
                              int64_t lda_bytes, const void* B, int64_t ldb_bytes,
                              cudaStream_t st) {
  if (G <= 0) return cudaSuccess;
  const int mg = G < 1024 ? G : 1024;
  tcb::group_maps_kernel<<<mg, 32, 0, st>>>(baseA, baseB, reinterpret_cast<CUtensorMap*>(maps),
                                            offsets, G, rows_bound,
                                            reinterpret_cast<const char*>(A), lda_bytes,
                                            reinterpret_cast<const char*>(B), ldb_bytes);
  count_launch();
  return cudaGetLastError();
}

bool bwd_gemm_tc_ok(const BwdGemmArgs& a) {
  if (a.dtype != MOE_BF16 || tc::encode_fn() == nullptr) return false;
  // 16-byte TMA strides and base addresses, 8-column output pieces
  if (a.N % 8 || a.ldo % 8) return false;
  if (a.kind == kBwdWgrad) return a.M % 8 == 0 && a.lda % 8 == 0 && a.ldb % 8 == 0;
  if (a.lda % 8 || a.K0 % 8 || a.K1 % 8) return false;
  if (a.K1 > 0 && a.K0 % tcb::BK) return false;   // segment 1 starts on a k-block
  if (a.kind == kBwdDgradSwiGLU && a.ldp % 8) return false;
  return true;
}

cudaError_t launch_bwd_gemm_tc(const BwdGemmArgs& a, cudaStream_t st) {
  using namespace tcb;
  if (!bwd_gemm_tc_ok(a)) return cudaErrorNotSupported;
  cudaError_t e;
  Args t;
  t.kind = a.kind;
  t.M = a.M;
  t.N = a.N;
  t.G = a.G;
  t.offsets = a.offsets;
  t.rows_bound = a.rows_bound;
  t.out = reinterpret_cast<bf16*>(a.out);
  t.ldo = a.ldo;
  t.ostride = a.ostride;
  t.pre = reinterpret_cast<const bf16*>(a.pre);
  t.ldp = a.ldp;
  t.flags = a.flags;
  t.NT = (a.N + BN - 1) / BN;
  t.sched = nullptr;
  t.tmaps = nullptr;
  CUtensorMap mA, mB0, mB1;
  int64_t tiles_bound;
  if (a.kind == kBwdWgrad) {
    if (a.M <= 0 || a.N <= 0 || a.G <= 0) return cudaSuccess;
    t.MT = (a.M + BM - 1) / BM;
    t.K0 = t.KB0 = t.KB = 0;
    const int64_t rows = a.rows_bound > 0 ? a.rows_bound : 1;
    t.a_wide = a.M % 64 == 0;
    t.b_wide = a.N % 64 == 0;
    if (!(t.a_wide ? map_rows_wide(&mA, a.A, rows, a.M, a.lda, BM / 64)
                   : map_rows(&mA, a.A, rows, a.M, a.lda, BK)) ||
        !(t.b_wide ? map_rows_wide(&mB0, a.B0, rows, a.N, a.ldb, BN / 64)
                   : map_rows(&mB0, a.B0, rows, a.N, a.ldb, BK)))
      return cudaErrorInvalidValue;
    mB1 = mB0;
    tiles_bound = (int64_t)a.G * t.MT * t.NT;
    if (a.tmaps == nullptr) return cudaErrorInvalidValue;
    t.tmaps = reinterpret_cast<const CUtensorMap*>(a.tmaps);
    const int mg = a.G < 1024 ? a.G : 1024;
    group_maps_kernel<<<mg, 32, 0, st>>>(mA, mB0, reinterpret_cast<CUtensorMap*>(a.tmaps),
                                         a.offsets, a.G, a.rows_bound,
                                         reinterpret_cast<const char*>(a.A), a.lda * 2,
                                         reinterpret_cast<const char*>(a.B0), a.ldb * 2);
    count_launch();
  } else {
    if (a.rows_bound <= 0 || a.N <= 0) return cudaSuccess;
    t.MT = 0;
    t.K0 = a.K0;
    t.KB0 = (a.K0 + BK - 1) / BK;
    t.KB = t.KB0 + (a.K1 + BK - 1) / BK;
    if (a.G > MAX_SMEM_G) {
      GemmArgs ga;
      ga.offsets = a.offsets;
      ga.G = a.G;
      ga.single_rows = 0;
      ga.rows_bound = a.rows_bound;
      ga.sched = a.sched;
      ga.flags = a.flags;
      e = launch_schedule(ga, BM, st);
      if (e != cudaSuccess) return e;
      t.sched = a.sched;
    }
    if (!map_rows(&mA, a.A, a.rows_bound, a.K0 + a.K1, a.lda, BM)) return cudaErrorInvalidValue;
    t.a_wide = 0;
    t.b_wide = a.N % 64 == 0;
    auto map_w = [&](CUtensorMap* m, const void* p, int K) {
      return t.b_wide ? map_weights_kn_wide(m, p, a.N, K, a.G, a.bstride)
                      : map_weights_kn(m, p, a.N, K, a.G, a.bstride);
    };
    if (!map_w(&mB0, a.B0, a.K0)) return cudaErrorInvalidValue;
    if (a.K1 > 0) {
      if (!map_w(&mB1, a.B1, a.K1)) return cudaErrorInvalidValue;
    } else {
      mB1 = mB0;
    }
    int64_t mt_bound = (a.rows_bound + BM - 1) / BM + a.G;
    if (mt_bound > a.rows_bound) mt_bound = a.rows_bound;
    tiles_bound = mt_bound * t.NT;
  }
  static std::atomic<bool> attr_done[64];   // per device; several host threads may launch
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(bwd_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int grid = (int)(tiles_bound < sm_count() ? tiles_bound : sm_count());
  if (grid <= 0) return cudaSuccess;
  bwd_gemm_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(mA, mB0, mB1, t);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
