// gemm_tc_mx.cu -- grouped GEMM on the tensor cores with MXFP8 expert weights
// ("MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
// stage-marker contract": e4m3 values, one e8m0 scale per block of 8 along
// the reduced axis), bf16 activations.
//
// Same contract and tile schedule as the one-SM engine of gemm_tc.cu
// ("Fused MoE Kernel Notes", group_gemm_same_nk).  The weights cross HBM as
// 1.125 bytes a value and become bf16 only in shared memory:
//   warp 0      TMA of the activation tile [128 rows x 64 k] (as gemm_tc.cu);
//   warp 6      TMA of the weight tile's e4m3 codes [256 rows x 64 bytes] and
//               of the 16 scale bytes per row that cover this k-block and its
//               neighbour (scale rows are 16-byte aligned when K is a
//               multiple of 128);
//   warps 7-26  converters: four lanes share a weight row, each taking 16
//               codes (two blocks), so a warp reads 8 consecutive rows of the
//               staged codes without bank conflicts; each block becomes 8
//               bf16 values (e4m3 -> fp16 by the hardware conversion, times
//               the block's power of two in fp32, exact in bf16) written into
//               the
//               128-byte-swizzled K-major B stage the MMA reads; then a fence
//               against the async proxy and an arrival on the stage's "full"
//               barrier;
//   warp 1      TMEM owner and MMA issuer (tcgen05.mma kind::f16, M = 128,
//               N = 256, K = 16), two 256-column accumulators;
//   warps 2-5   epilogue (SwiGLU or plain store, staged 16-byte row stores).
// Rings: 3 stages of A (16 KB), 2 of the converted bf16 B (32 KB), 5 of codes
// (16 KB) + scales (4 KB): the weight stream keeps five stages of loads in
// flight, released as soon as they are converted, not when the MMA is done.
// Every wait is bounded; a wait that runs out aborts the kernel cleanly.
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

namespace tcm {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int SA = 3, SB = 2, SQ = 5;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_BYTES = BN * BK * 2;     // 32 KB (bf16 after conversion)
constexpr int Q_BYTES = BN * BK;         // 16 KB of e4m3 codes
constexpr int SC_BYTES = BN * 16;        // 16 scale bytes a row: two k-blocks
constexpr int RING_A = 0, RING_B = SA * A_BYTES, RING_Q = RING_B + SB * B_BYTES,
              RING_SC = RING_Q + SQ * Q_BYTES, RING_BYTES = RING_SC + SQ * SC_BYTES;
// barriers: fullA emptyA [SA], fullQ emptyQ [SQ], fullB emptyB [SB], then
// tfull[2] tempty[2] final
constexpr int NBAR = 2 * (SA + SQ + SB) + 5;
constexpr int CONV_WARP0 = 7, CONV_WARPS = 20;
constexpr int THREADS = (CONV_WARP0 + CONV_WARPS) * 32;   // warps 0-26
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int MAX_SMEM_G = 512;
constexpr int SCHED_BYTES = (MAX_SMEM_G + 1) * 4;
constexpr int OUT_ROW_BYTES = 80;
constexpr int OUT_WARP_BYTES = 32 * OUT_ROW_BYTES;
constexpr int OUT_BYTES = 4 * OUT_WARP_BYTES;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + BAR_BYTES + OUT_BYTES + SCHED_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
static_assert(NBAR * 8 + 8 <= BAR_BYTES, "barrier area");
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Args {
  int mode, N, K, G, NT, KB;
  const int32_t* offsets;
  int64_t single_rows, rows_bound;
  const int32_t* sched;
  void* out;
  int64_t ldo;
  uint32_t* flags;
};

__device__ __forceinline__ void decode_tile(const Args& a, const int32_t* sched, int64_t tile,
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

__device__ void build_schedule(const Args& a, int32_t* sched, int lane) {
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
    tc_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ0,
                 const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmS0,
                 const __grid_constant__ CUtensorMap tmS1, const Args a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned char* s_out = smem + RING_BYTES + BAR_BYTES;
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_out + OUT_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_u32(smem);
  // kinds: 0 fullA, 1 emptyA, 2 fullQ, 3 emptyQ, 4 fullB, 5 emptyB
  auto bar = [&](int kind, int s) {
    const int o = kind == 0 ? 0 : kind == 1 ? SA : kind == 2 ? 2 * SA : kind == 3 ? 2 * SA + SQ
                : kind == 4 ? 2 * SA + 2 * SQ : 2 * SA + 2 * SQ + SB;
    return smem_u32(&bars[o + s]);
  };
  const int tb = 2 * (SA + SQ + SB);
  auto tfull = [&](int b) { return smem_u32(&bars[tb + b]); };
  auto tempty = [&](int b) { return smem_u32(&bars[tb + 2 + b]); };
  const uint32_t final_bar = smem_u32(&bars[tb + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(bar(0, s), 1);
      mbar_init(bar(1, s), 1);
    }
    for (int s = 0; s < SQ; ++s) {
      mbar_init(bar(2, s), 1);
      mbar_init(bar(3, s), CONV_WARPS);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bar(4, s), CONV_WARPS);
      mbar_init(bar(5, s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 128);
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
  const int64_t total = (int64_t)sched[a.G] * a.NT;
  const bool swiglu = a.mode == kSwiGLU;

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ---------------- TMA producers: warp 0 activations, warp 6 codes+scales
    const bool is_a = warp == 0;
    const int kfull = is_a ? 0 : 2, kempty = is_a ? 1 : 3;
    const int S = is_a ? SA : SQ;
    int s = 0;
    uint32_t ph = 0, issued = 0, par = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int g, mt, nt;
      decode_tile(a, sched, tile, g, mt, nt);
      const int64_t gbase = a.offsets ? a.offsets[g] : 0;
      const int arow = (int)(gbase + (int64_t)mt * BM);
      for (int kb = 0; kb < a.KB; ++kb) {
        if (!mbar_wait(bar(kempty, s), ph ^ 1u, abort_flag)) { ok = false; break; }
        const uint32_t fb = bar(kfull, s);
        if (is_a) {
          mbar_expect_tx(fb, A_BYTES);
          tma_load_2d(base + RING_A + s * A_BYTES, &tmA, kb * BK, arow, fb);
        } else {
          const uint32_t q = base + RING_Q + s * Q_BYTES, sc = base + RING_SC + s * SC_BYTES;
          mbar_expect_tx(fb, Q_BYTES + SC_BYTES);
          const int sx = (kb >> 1) * 16;   // the 16 scale bytes of k-blocks kb & ~1, kb | 1
          if (swiglu) {
            tma_load_3d(q, &tmQ0, kb * BK, nt * (BN / 2), g, fb);
            tma_load_3d(q + Q_BYTES / 2, &tmQ1, kb * BK, nt * (BN / 2), g, fb);
            tma_load_3d(sc, &tmS0, sx, nt * (BN / 2), g, fb);
            tma_load_3d(sc + SC_BYTES / 2, &tmS1, sx, nt * (BN / 2), g, fb);
          } else {
            tma_load_3d(q, &tmQ0, kb * BK, nt * BN, g, fb);
            tma_load_3d(sc, &tmS0, sx, nt * BN, g, fb);
          }
        }
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (*abort_flag) {
      for (int i = 0; i < S; ++i)
        if (issued & (1u << i)) mbar_wait_quiet(bar(kfull, i), (par >> i) & 1u);
    }
  } else if (warp >= CONV_WARP0 && warp < CONV_WARP0 + CONV_WARPS) {
    // ---------------- converters: e4m3 + scales -> swizzled bf16 B stage ----
    const int cw = warp - CONV_WARP0;
    const int p = lane & 3;        // codes 16p .. 16p+15 of the row: blocks 2p, 2p+1
    const int rsub = lane >> 2;    // row within an 8-row step
    int sq = 0, sb = 0;
    uint32_t phq = 0, phb = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < a.KB; ++kb) {
        const bool got = mbar_wait(bar(2, sq), phq, abort_flag) &&
                         mbar_wait(bar(5, sb), phb ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const unsigned char* q = smem + RING_Q + sq * Q_BYTES;
        const unsigned char* sc = smem + RING_SC + sq * SC_BYTES + (kb & 1) * 8 + 2 * p;
        unsigned char* bst = smem + RING_B + sb * B_BYTES;
#pragma unroll 2
        for (int step = cw; step < BN / 8; step += CONV_WARPS) {
          const int r = step * 8 + rsub;
          const uint4 c = *reinterpret_cast<const uint4*>(q + r * BK + 16 * p);
          const uint32_t s2 = *reinterpret_cast<const unsigned short*>(sc + r * 16);
          float f[8];
          unpack_mx8(make_uint2(c.x, c.y), s2 & 0xFFu, f);
          *reinterpret_cast<uint4*>(bst + r * 128 + (((2 * p) ^ (r & 7)) << 4)) =
              pack16(f, (const bf16*)nullptr);
          unpack_mx8(make_uint2(c.z, c.w), s2 >> 8, f);
          *reinterpret_cast<uint4*>(bst + r * 128 + (((2 * p + 1) ^ (r & 7)) << 4)) =
              pack16(f, (const bf16*)nullptr);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(4, sb));   // B stage full
          mbar_arrive(bar(3, sq));   // staging free
        }
        if (++sq == SQ) { sq = 0; phq ^= 1u; }
        if (++sb == SB) { sb = 0; phb ^= 1u; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int sa = 0, sb = 0, acc = 0;
      uint32_t pha = 0, phb = 0, aph = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!mbar_wait(tempty(acc), aph ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)acc * BN;
        for (int kb = 0; kb < a.KB; ++kb) {
          if (!mbar_wait(bar(0, sa), pha, abort_flag) || !mbar_wait(bar(4, sb), phb, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = base + RING_A + sa * A_BYTES;
          const uint32_t b_addr = base + RING_B + sb * B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), IDESC,
                   (kb | kk) != 0 ? 1u : 0u);
          tc_commit(bar(1, sa));
          tc_commit(bar(5, sb));
          if (++sa == SA) { sa = 0; pha ^= 1u; }
          if (++sb == SB) { sb = 0; phb ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull(acc));
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if (*abort_flag) {
        tc_commit(final_bar);
        mbar_wait_quiet(final_bar, 0);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue (warps 2..5), as in gemm_tc.cu ----------------
    const int q = warp & 3;
    unsigned char* stage = s_out + (warp - 2) * OUT_WARP_BYTES;
    unsigned char* my_row = stage + lane * OUT_ROW_BYTES;
    int acc = 0;
    uint32_t aph = 0;
    bf16* out = reinterpret_cast<bf16*>(a.out);
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int g, mt, nt;
      decode_tile(a, sched, tile, g, mt, nt);
      const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
      const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
      const int64_t row0 = gbeg + (int64_t)mt * BM + q * 32;
      const int64_t nvalid64 = gend - row0;
      const int nvalid = nvalid64 < 0 ? 0 : (nvalid64 > 32 ? 32 : (int)nvalid64);
      if (!__all_sync(0xffffffffu, mbar_wait(tfull(acc), aph, abort_flag))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * BN;
      const int n0 = swiglu ? nt * (BN / 2) : nt * BN;
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
#pragma unroll
        for (int v = 0; v < 4; ++v) reinterpret_cast<uint4*>(my_row)[v] = packed[v];
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int p = lane + 32 * i;
          const int rr = p >> 2, pc = p & 3;
          const int n = n0 + c + pc * 8;
          if (rr < nvalid && n < a.N)
            *reinterpret_cast<uint4*>(out + (row0 + rr) * a.ldo + n) =
                *reinterpret_cast<const uint4*>(stage + rr * OUT_ROW_BYTES + pc * 16);
        }
        __syncwarp();
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 3-D byte map {width, N, G} over G packed matrices `gstride` bytes apart,
// rows `ld` bytes apart, box box_x x box_rows x 1, no swizzle.
static bool map_bytes(CUtensorMap* m, const void* ptr, int64_t width, int N, int G, int64_t ld,
                      int64_t gstride, int box_x, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)N, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)ld, (cuuint64_t)gstride};
  cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcm

bool gemm_tc_mx_ok(const GemmArgs& a) {
  return a.wfmt && a.dtype == MOE_BF16 && (a.mode == kSwiGLU || a.mode == kStoreAct) &&
         a.K > 0 && a.K % 128 == 0 && a.N > 0 && a.N % 8 == 0 && a.ksplit == 1 && !a.gather &&
         !a.pre && a.bstride % 16 == 0 && tc::encode_fn() != nullptr;
}

cudaError_t launch_gemm_tc_mx(const GemmArgs& a, cudaStream_t st) {
  using namespace tcm;
  if (!gemm_tc_mx_ok(a)) return cudaErrorNotSupported;
  cudaError_t e;
  const bool smem_sched = a.G <= MAX_SMEM_G;
  if (!smem_sched) {
    e = launch_schedule(a, BM, st);
    if (e != cudaSuccess) return e;
  }
  const int64_t rows = a.offsets ? a.rows_bound : a.single_rows;
  if (rows <= 0) return cudaSuccess;
  const int brows = a.mode == kSwiGLU ? BN / 2 : BN;
  // packed matrix g: codes [N, K] at B + g * bstride, scales [N, K/8] after them
  const int64_t gstride = a.G == 1 && a.bstride == 0 ? (int64_t)a.N * a.K / 8 * 9 : a.bstride;
  const char* b0 = reinterpret_cast<const char*>(a.B0);
  const char* b1 = reinterpret_cast<const char*>(a.mode == kSwiGLU ? a.B1 : a.B0);
  const int64_t nk = (int64_t)a.N * a.K;
  CUtensorMap mA, mQ0, mQ1, mS0, mS1;
  if (!make_map_2d(&mA, a.A, rows, a.K, BM)) return cudaErrorInvalidValue;
  if (!map_bytes(&mQ0, b0, a.K, a.N, a.G, a.K, gstride, BK, brows) ||
      !map_bytes(&mQ1, b1, a.K, a.N, a.G, a.K, gstride, BK, brows) ||
      !map_bytes(&mS0, b0 + nk, a.K / 8, a.N, a.G, a.K / 8, gstride, 16, brows) ||
      !map_bytes(&mS1, b1 + nk, a.K / 8, a.N, a.G, a.K / 8, gstride, 16, brows))
    return cudaErrorInvalidValue;
  Args t;
  t.mode = a.mode;
  t.N = a.N;
  t.K = a.K;
  t.G = a.G;
  t.NT = (a.N + brows - 1) / brows;
  t.KB = a.K / BK;
  t.offsets = a.offsets;
  t.single_rows = a.single_rows;
  t.rows_bound = a.rows_bound;
  t.sched = smem_sched ? nullptr : a.sched;
  t.out = a.out;
  t.ldo = a.ldo;
  t.flags = a.flags;
  int64_t mt_bound = a.offsets ? (a.rows_bound + BM - 1) / BM + a.G : (a.single_rows + BM - 1) / BM;
  if (a.offsets && mt_bound > a.rows_bound) mt_bound = a.rows_bound;
  const int64_t tiles_bound = mt_bound * t.NT;
  static std::atomic<bool> attr_done[64];   // per device; several host threads may launch
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(tc_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int grid = (int)(tiles_bound < sm_count() ? tiles_bound : sm_count());
  tc_mx_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(mA, mQ0, mQ1, mS0, mS1, t);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
