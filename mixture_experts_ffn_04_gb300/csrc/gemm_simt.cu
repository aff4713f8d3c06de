// gemm_simt.cu -- grouped GEMM on the CUDA cores (fp32 FMA), and the device
// tile schedule shared with the tensor-core engine.
//
// Grouped GEMM as in "Fused MoE Kernel Notes" (group_gemm_same_nk: same N and
// K for every expert, M varies per expert): for group g, rows r in
// [offsets[g], offsets[g+1]) of A, out[r, n] = sum_k A[r, k] * B_g[n, k].
// The m-tile schedule is built on the device from the real group sizes, so
// the launch bound never truncates a group (the max_M invariant of that page:
// a bound of `tokens` rows would miss rows of a duplicate-routed group).
//
// This engine serves the fp32 layer exactly (tensor cores would round fp32
// operands to tf32) and small bf16 problems.
#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

// sched[g] = sum over g' < g of ceil(count_g' / bm); sched[G] = total m-tiles,
// forced to 0 (nothing runs) when the offsets are inconsistent or exceed the
// caller's row bound.
__global__ void schedule_kernel(const int32_t* __restrict__ offsets, int G, int64_t single_rows,
                                int64_t rows_bound, int bm, int32_t* __restrict__ sched,
                                uint32_t* flags) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) {
    carry = 0;
    bad = 0;
    if (offsets) {
      if (offsets[0] != 0 || (int64_t)offsets[G] > rows_bound || offsets[G] < 0) bad = 1;
    } else if (single_rows > rows_bound || single_rows < 0) {
      bad = 1;
    }
  }
  __syncthreads();
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + tid;
    int v = 0;
    if (g < G) {
      int64_t cnt = offsets ? (int64_t)offsets[g + 1] - offsets[g] : single_rows;
      if (cnt < 0) {
        bad = 1;
        cnt = 0;
      }
      v = (int)((cnt + bm - 1) / bm);
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int w = lane < nw ? warp_tot[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < nw) warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    if (g < G) sched[g] = carry + warp_tot[wid] + incl - v;
    __syncthreads();
    if (tid == blockDim.x - 1) carry += warp_tot[wid] + incl;
    __syncthreads();
  }
  if (tid == 0) {
    if (bad) set_flag(flags, kFlagRows);
    sched[G] = bad ? 0 : carry;
  }
}

cudaError_t launch_schedule(const GemmArgs& a, int bm, cudaStream_t st) {
  schedule_kernel<<<1, 256, 0, st>>>(a.offsets, a.G, a.single_rows, a.rows_bound, bm, a.sched,
                                     a.flags);
  count_launch();
  return cudaGetLastError();
}

namespace {
constexpr int kBN = 64, kBK = 16, kThreads = 256;

// MX: B0/B1 hold packed MXFP8 matrices (bstride in bytes), dequantised as
// they are loaded.
template <typename T, int MODE, int BM, bool MX = false>
__global__ void __launch_bounds__(kThreads) simt_gemm_kernel(GemmArgs a) {
  constexpr int TM = BM / 16;  // rows per thread
  __shared__ __align__(16) float As[kBK][BM + 4];
  __shared__ __align__(16) float Bs[kBK][kBN + 4];
  __shared__ __align__(16) float Us[MODE == kSwiGLU ? kBK : 1][kBN + 4];
  __shared__ int64_t s_src[BM];   // source row of each tile row, -1: zeros

  const int total = a.sched[a.G];
  const int j = blockIdx.x;
  if (j >= total) return;
  const int g = find_group(a.sched, a.G, j);
  const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
  const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
  const int64_t row0 = gbeg + (int64_t)(j - a.sched[g]) * BM;
  const int n0 = blockIdx.y * kBN;
  const int K = a.K, N = a.N;

  const T* A = reinterpret_cast<const T*>(a.A);
  const T* B0 = reinterpret_cast<const T*>(a.B0) + (MX ? 0 : (int64_t)g * a.bstride);
  const T* B1 = MODE == kSwiGLU ? reinterpret_cast<const T*>(a.B1) + (MX ? 0 : (int64_t)g * a.bstride) : nullptr;
  const uint8_t* M0 = MX ? reinterpret_cast<const uint8_t*>(a.B0) + (int64_t)g * a.bstride : nullptr;
  const uint8_t* M1 = MX && MODE == kSwiGLU ? reinterpret_cast<const uint8_t*>(a.B1) + (int64_t)g * a.bstride : nullptr;

  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  for (int r = tid; r < BM; r += kThreads) {
    const int64_t row = row0 + r;
    int64_t src = -1;
    if (row < gend) {
      src = a.gather ? (int64_t)a.gather[row] : row;
      if (a.gather && (src < 0 || src >= a.a_rows)) {
        set_flag(a.flags, kFlagGather);
        src = -1;
      }
    }
    s_src[r] = src;
  }
  __syncthreads();
  float acc[TM][4], accu[MODE == kSwiGLU ? TM : 1][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[i][q] = 0.f;
      if (MODE == kSwiGLU) accu[i][q] = 0.f;
    }

  // Register double buffer: the next k-slice is fetched from global memory
  // while the current one is multiplied out of shared memory.
  constexpr int EA = BM * kBK / kThreads, EB = kBN * kBK / kThreads;
  float ra[EA], rb[EB], ru[MODE == kSwiGLU ? EB : 1];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int q = 0; q < EA; ++q) {
      const int e = tid + q * kThreads, r = e / kBK, kk = e % kBK;
      const int64_t src = s_src[r];
      ra[q] = (src >= 0 && k0 + kk < K) ? to_f(A[src * K + k0 + kk]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < EB; ++q) {
      const int e = tid + q * kThreads, n = e / kBK, kk = e % kBK;
      const bool in = n0 + n < N && k0 + kk < K;
      if (MX) {
        rb[q] = in ? mx_weight(M0, N, K, n0 + n, k0 + kk) : 0.f;
        if (MODE == kSwiGLU) ru[q] = in ? mx_weight(M1, N, K, n0 + n, k0 + kk) : 0.f;
      } else {
        rb[q] = in ? to_f(B0[(int64_t)(n0 + n) * K + k0 + kk]) : 0.f;
        if (MODE == kSwiGLU) ru[q] = in ? to_f(B1[(int64_t)(n0 + n) * K + k0 + kk]) : 0.f;
      }
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int q = 0; q < EA; ++q) {
      const int e = tid + q * kThreads;
      As[e % kBK][e / kBK] = ra[q];
    }
#pragma unroll
    for (int q = 0; q < EB; ++q) {
      const int e = tid + q * kThreads;
      Bs[e % kBK][e / kBK] = rb[q];
      if (MODE == kSwiGLU) Us[e % kBK][e / kBK] = ru[q];
    }
  };
  fetch(0);
  stash();
  __syncthreads();
  for (int k0 = 0; k0 < K; k0 += kBK) {
    const bool more = k0 + kBK < K;
    if (more) fetch(k0 + kBK);
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float av[TM], bv[4], uv[4];
#pragma unroll
      for (int i = 0; i < TM; ++i) av[i] = As[kk][ty * TM + i];
      const float4 b4 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
      if (MODE == kSwiGLU) {
        const float4 u4 = *reinterpret_cast<const float4*>(&Us[kk][tx * 4]);
        uv[0] = u4.x; uv[1] = u4.y; uv[2] = u4.z; uv[3] = u4.w;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[i][q] = fmaf(av[i], bv[q], acc[i][q]);
          if (MODE == kSwiGLU) accu[i][q] = fmaf(av[i], uv[q], accu[i][q]);
        }
    }
    __syncthreads();
    if (more) {
      stash();
      __syncthreads();
    }
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t row = row0 + ty * TM + i;
    if (row >= gend) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tx * 4 + q;
      if (n >= N) continue;
      if (MODE == kStoreF32) {
        reinterpret_cast<float*>(a.out)[row * a.ldo + n] = acc[i][q];
      } else if (MODE == kStoreAct) {
        reinterpret_cast<T*>(a.out)[row * a.ldo + n] = from_f<T>(acc[i][q]);
      } else {
        reinterpret_cast<T*>(a.out)[row * a.ldo + n] = from_f<T>(silu_f(acc[i][q]) * accu[i][q]);
        if (a.pre) {   // the pre-activations, for the backward
          T* pre = reinterpret_cast<T*>(a.pre) + row * a.ldp;
          pre[n] = from_f<T>(acc[i][q]);
          pre[N + n] = from_f<T>(accu[i][q]);
        }
      }
    }
  }
}

int64_t mtile_bound(const GemmArgs& a, int bm);

template <typename T, int BM>
cudaError_t launch_t(const GemmArgs& a, cudaStream_t st) {
  const int64_t mt_bound = mtile_bound(a, BM);
  if (mt_bound <= 0 || a.N <= 0) return cudaSuccess;
  if (mt_bound > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid((unsigned)mt_bound, (unsigned)((a.N + kBN - 1) / kBN));
  if (a.wfmt) {
    if (a.mode == kSwiGLU) simt_gemm_kernel<T, kSwiGLU, BM, true><<<grid, kThreads, 0, st>>>(a);
    else if (a.mode == kStoreAct) simt_gemm_kernel<T, kStoreAct, BM, true><<<grid, kThreads, 0, st>>>(a);
    else return cudaErrorInvalidValue;
  } else {
    switch (a.mode) {
      case kSwiGLU: simt_gemm_kernel<T, kSwiGLU, BM><<<grid, kThreads, 0, st>>>(a); break;
      case kStoreAct: simt_gemm_kernel<T, kStoreAct, BM><<<grid, kThreads, 0, st>>>(a); break;
      default: simt_gemm_kernel<T, kStoreF32, BM><<<grid, kThreads, 0, st>>>(a); break;
    }
  }
  count_launch();
  return cudaGetLastError();
}
}  // namespace

// ---------------------------------------------------------------------------
// Skinny engine for decode-sized calls (a few rows per group): the cost is
// reading each weight row once, so the engine is built to keep many weight
// loads in flight.  Each warp owns kSkC output columns of one m-tile and a
// slice of K (the block's 8 warps split K into ks = 1-8 slices per column
// group) and streams its slice of each column's weight row with 16-byte loads,
// dotting it with the m-tile's rows of A; the ks partial sums of a column are
// added in a fixed order through shared memory.  The m-tile schedule is built
// in shared memory by each block (no extra launch).
// The m-tile height R (1, 4 or 8 rows) is a template parameter: every row of
// the tile holds its accumulators in registers, and registers bound how many
// weight loads a thread keeps in flight.
// ---------------------------------------------------------------------------
namespace {
constexpr int kSkR = 8;      // largest m-tile (rows)
constexpr int kSkC = 4;      // output columns per warp
constexpr int kSkW = 8;      // warps per block (K slices)
constexpr int kSkMaxG = 1024;

// MX: the weights are packed MXFP8 matrices (bstride in bytes): per 8-value
// chunk of A a lane loads the block's 8 e4m3 bytes and its scale byte, half
// the bytes of bf16 weights, and the dequantised values are exact, so the
// sums equal those over the same weights stored in bf16.
// PAIR: a lane step covers two consecutive 8-value chunks (K a multiple of
// 16), so each weight load is 16 bytes for MXFP8 too; the chunk order per
// lane is the same with and without MX, so both give the same sums.
template <typename T, int MODE, bool MX = false, bool PAIR = false, int R = kSkR>
// One-row tiles ask for two blocks an SM (SwiGLU: the cap of 128 registers
// still holds two lane steps of weight loads in flight) or three (one weight
// matrix: a down projection's 448 blocks then fit one wave).  With MXFP8
// weights the one-row loop unpacks each column right before its use, which
// fits it under those caps (with 24-32 bytes a thread of spill stores, and
// still faster than one block an SM).
__global__ void __launch_bounds__(256, R == 1 ? (MODE == kSwiGLU ? 2 : 3) : 1)
    skinny_kernel(GemmArgs a, int smem_sched, int ks) {
  constexpr int NU = MODE == kSwiGLU ? 2 : 1;
  __shared__ int32_t s_sched[kSkMaxG + 1];
  __shared__ float red[kSkW][R * kSkC * NU];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* sched = a.sched;
  if (smem_sched) {
    if (warp == 0) block_schedule(a, R, s_sched, lane);
    __syncthreads();
    sched = s_sched;
  }
  const int total = sched[a.G];
  const int j = blockIdx.x;
  if (j >= total) return;
  const int g = find_group(sched, a.G, j);
  const int64_t gbeg = a.offsets ? a.offsets[g] : 0;
  const int64_t gend = a.offsets ? a.offsets[g + 1] : a.single_rows;
  const int64_t row0 = gbeg + (int64_t)(j - sched[g]) * R;
  const int nrows = (int)min((int64_t)R, gend - row0);
  // warp -> (column group cg, K slice sl); the block owns kSkW/ks column groups
  // of each column block by it takes (blockIdx.y, then gridDim.y apart: a
  // grid capped below the column blocks loops over them)
  const int cg = warp / ks, sl = warp % ks, ncg = kSkW / ks;
  const int nby = (a.N + ncg * kSkC - 1) / (ncg * kSkC);
  for (int by = blockIdx.y; by < nby; by += gridDim.y) {
  const int n0 = (by * ncg + cg) * kSkC;
  const int K = a.K;
  constexpr int V = 16 / sizeof(T);
  constexpr int CH = PAIR ? 2 : 1;   // chunks per lane step
  const int nv = K / V;
  const int nvp = nv / CH;
  const int c0 = (int)((int64_t)nvp * sl / ks), c1 = (int)((int64_t)nvp * (sl + 1) / ks);
  // row r of this tile reads A row arow[r] (gathered or contiguous); -1: zeros
  int64_t arow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    int64_t src = r < nrows ? row0 + r : -1;
    if (src >= 0 && a.gather) {
      src = a.gather[src];
      if (src < 0 || src >= a.a_rows) {
        if (threadIdx.x == 0) set_flag(a.flags, kFlagGather);
        src = -1;
      }
    }
    arow[r] = src;
  }
  const uint4* A = reinterpret_cast<const uint4*>(a.A);
  const T* B0 = reinterpret_cast<const T*>(a.B0) + (int64_t)g * a.bstride;
  const T* B1 = MODE == kSwiGLU ? reinterpret_cast<const T*>(a.B1) + (int64_t)g * a.bstride
                                : nullptr;
  const uint4* Bc[kSkC];
  const uint4* Uc[kSkC];
  const uint2* Bq[kSkC];
  const uint2* Uq[kSkC];
  const uint8_t* Bs[kSkC];
  const uint8_t* Us[kSkC];
#pragma unroll
  for (int q = 0; q < kSkC; ++q) {
    const int n = min(n0 + q, a.N - 1);   // clamped columns are computed, not stored
    if (MX) {
      const uint8_t* m0 = reinterpret_cast<const uint8_t*>(a.B0) + (int64_t)g * a.bstride;
      Bq[q] = reinterpret_cast<const uint2*>(m0 + (int64_t)n * K);
      Bs[q] = m0 + (int64_t)a.N * K + (int64_t)n * (K / 8);
      if (MODE == kSwiGLU) {
        const uint8_t* m1 = reinterpret_cast<const uint8_t*>(a.B1) + (int64_t)g * a.bstride;
        Uq[q] = reinterpret_cast<const uint2*>(m1 + (int64_t)n * K);
        Us[q] = m1 + (int64_t)a.N * K + (int64_t)n * (K / 8);
      }
    } else {
      Bc[q] = reinterpret_cast<const uint4*>(B0 + (int64_t)n * K);
      Uc[q] = MODE == kSwiGLU ? reinterpret_cast<const uint4*>(B1 + (int64_t)n * K) : nullptr;
    }
  }
  float acc[R][kSkC], accu[MODE == kSwiGLU ? R : 1][kSkC];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int q = 0; q < kSkC; ++q) {
      acc[r][q] = 0.f;
      if (MODE == kSwiGLU) accu[r][q] = 0.f;
    }
  if (n0 < a.N) {
#pragma unroll 2
    for (int cp = c0 + lane; cp < c1; cp += 32) {
      if constexpr (MX && PAIR && R == 1) {
        // one row: the packed weights of every column are loaded first (all
        // loads in flight), then the row's A values, then each column is
        // unpacked and used at once, so only one column's 16 values are live
        // (the same FMA order per accumulator as below)
        uint4 bq[kSkC], uq[MODE == kSwiGLU ? kSkC : 1];
        uint32_t bs[kSkC], us[MODE == kSwiGLU ? kSkC : 1];
#pragma unroll
        for (int q = 0; q < kSkC; ++q) {
          bq[q] = __ldg(reinterpret_cast<const uint4*>(Bq[q]) + cp);
          bs[q] = __ldg(reinterpret_cast<const unsigned short*>(Bs[q]) + cp);
          if (MODE == kSwiGLU) {
            uq[q] = __ldg(reinterpret_cast<const uint4*>(Uq[q]) + cp);
            us[q] = __ldg(reinterpret_cast<const unsigned short*>(Us[q]) + cp);
          }
        }
        if (arow[0] >= 0) {
          float xa[2 * V];
          unpack16(__ldg(A + arow[0] * nv + cp * 2), xa, (const T*)nullptr);
          unpack16(__ldg(A + arow[0] * nv + cp * 2 + 1), xa + V, (const T*)nullptr);
#pragma unroll
          for (int q = 0; q < kSkC; ++q) {
            float wv[2 * V];
            unpack_mx8(make_uint2(bq[q].x, bq[q].y), bs[q] & 0xFFu, wv);
            unpack_mx8(make_uint2(bq[q].z, bq[q].w), bs[q] >> 8, wv + V);
#pragma unroll
            for (int i = 0; i < 2 * V; ++i) acc[0][q] = fmaf(wv[i], xa[i], acc[0][q]);
            if (MODE == kSwiGLU) {
              unpack_mx8(make_uint2(uq[q].x, uq[q].y), us[q] & 0xFFu, wv);
              unpack_mx8(make_uint2(uq[q].z, uq[q].w), us[q] >> 8, wv + V);
#pragma unroll
              for (int i = 0; i < 2 * V; ++i) accu[0][q] = fmaf(wv[i], xa[i], accu[0][q]);
            }
          }
        }
        continue;
      }
      float w[kSkC][CH * V], u[MODE == kSwiGLU ? kSkC : 1][CH * V];
#pragma unroll
      for (int q = 0; q < kSkC; ++q) {
        if (MX && PAIR) {
          // two blocks: 16 e4m3 bytes and their two scale bytes
          const uint4 qq = __ldg(reinterpret_cast<const uint4*>(Bq[q]) + cp);
          const uint32_t ss = __ldg(reinterpret_cast<const unsigned short*>(Bs[q]) + cp);
          unpack_mx8(make_uint2(qq.x, qq.y), ss & 0xFFu, w[q]);
          unpack_mx8(make_uint2(qq.z, qq.w), ss >> 8, w[q] + V);
          if (MODE == kSwiGLU) {
            const uint4 uq = __ldg(reinterpret_cast<const uint4*>(Uq[q]) + cp);
            const uint32_t us = __ldg(reinterpret_cast<const unsigned short*>(Us[q]) + cp);
            unpack_mx8(make_uint2(uq.x, uq.y), us & 0xFFu, u[q]);
            unpack_mx8(make_uint2(uq.z, uq.w), us >> 8, u[q] + V);
          }
        } else {
#pragma unroll
          for (int h = 0; h < CH; ++h) {
            const int c = cp * CH + h;
            if (MX) {
              unpack_mx8(__ldg(Bq[q] + c), __ldg(Bs[q] + c), w[q] + h * V);
              if (MODE == kSwiGLU) unpack_mx8(__ldg(Uq[q] + c), __ldg(Us[q] + c), u[q] + h * V);
            } else {
              unpack16(__ldg(Bc[q] + c), w[q] + h * V, (const T*)nullptr);
              if (MODE == kSwiGLU) unpack16(__ldg(Uc[q] + c), u[q] + h * V, (const T*)nullptr);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (arow[r] >= 0) {
#pragma unroll
          for (int h = 0; h < CH; ++h) {
            float xa[V];
            unpack16(__ldg(A + arow[r] * nv + cp * CH + h), xa, (const T*)nullptr);
#pragma unroll
            for (int q = 0; q < kSkC; ++q)
#pragma unroll
              for (int i = 0; i < V; ++i) {
                acc[r][q] = fmaf(w[q][h * V + i], xa[i], acc[r][q]);
                if (MODE == kSwiGLU) accu[r][q] = fmaf(u[q][h * V + i], xa[i], accu[r][q]);
              }
          }
        }
      }
    }
  }
  auto store = [&](int r, int q, float sg, float su) {
    const int n = n0 + q;
    if (r >= nrows || n >= a.N) return;
    const int64_t o = (row0 + r) * a.ldo + n;
    if (MODE == kStoreF32) reinterpret_cast<float*>(a.out)[o] = sg;
    else if (MODE == kStoreAct) reinterpret_cast<T*>(a.out)[o] = from_f<T>(sg);
    else reinterpret_cast<T*>(a.out)[o] = from_f<T>(silu_f(sg) * su);
  };
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r >= nrows) break;   // uniform over the block
#pragma unroll
    for (int q = 0; q < kSkC; ++q) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        acc[r][q] += __shfl_xor_sync(0xffffffffu, acc[r][q], o);
        if (MODE == kSwiGLU) accu[r][q] += __shfl_xor_sync(0xffffffffu, accu[r][q], o);
      }
      if (lane == 0) {
        if (ks == 1) {
          store(r, q, acc[r][q], MODE == kSwiGLU ? accu[r][q] : 0.f);
        } else {
          red[warp][(r * kSkC + q) * NU] = acc[r][q];
          if (MODE == kSwiGLU) red[warp][(r * kSkC + q) * NU + 1] = accu[r][q];
        }
      }
    }
  }
  if (ks == 1) continue;
  __syncthreads();
  const int tid = threadIdx.x;
  if (tid < ncg * R * kSkC) {
    const int gi = tid / (R * kSkC), rem = tid % (R * kSkC);
    const int r = rem / kSkC, q = rem % kSkC;
    if (r < nrows) {
      float sg = 0.f, su = 0.f;
      for (int w = gi * ks; w < (gi + 1) * ks; ++w) {   // fixed order: deterministic
        sg += red[w][(r * kSkC + q) * NU];
        if (MODE == kSwiGLU) su += red[w][(r * kSkC + q) * NU + 1];
      }
      const int n = (by * ncg + gi) * kSkC + q;
      if (n < a.N) {
        const int64_t o = (row0 + r) * a.ldo + n;
        if (MODE == kStoreF32) reinterpret_cast<float*>(a.out)[o] = sg;
        else if (MODE == kStoreAct) reinterpret_cast<T*>(a.out)[o] = from_f<T>(sg);
        else reinterpret_cast<T*>(a.out)[o] = from_f<T>(silu_f(sg) * su);
      }
    }
  }
  __syncthreads();   // red is rewritten by the next column block
  }
}

// Upper bound on the m-tiles of a call: each group needs ceil(rows/bm), and a
// non-empty tile holds at least one row.
int64_t mtile_bound(const GemmArgs& a, int bm) {
  if (!a.offsets) return (a.single_rows + bm - 1) / bm;
  int64_t b = (a.rows_bound + bm - 1) / bm + a.G;
  return b < a.rows_bound ? b : a.rows_bound;
}

// m-tile height of a skinny call.  A grouped call of at most 4 rows (one
// decode token's routes) puts one row in each group when its routes are
// distinct, so one-row tiles read each weight row once with the fewest
// accumulators; a repeated route costs one more read of that expert's weights.
// One group (the shared MLP) takes all its rows in one tile.  Otherwise (MXFP8
// weights serve grouped calls of up to 512 rows here) 8 rows a tile.
int skinny_rows(const GemmArgs& a) {
  if (a.dtype != MOE_BF16 || a.mode == kStoreF32 || a.K % 16 != 0) return kSkR;
  const int64_t rows = a.offsets ? a.rows_bound : a.single_rows;
  if (a.G > 1) return rows <= 4 ? 1 : kSkR;
  return rows <= 1 ? 1 : (rows <= 4 ? 4 : kSkR);
}

template <typename T, bool MX, bool PAIR, int R>
void launch_skinny_mode(const GemmArgs& a, dim3 grid, int smem_sched, int ks, cudaStream_t st) {
  if (a.mode == kSwiGLU)
    skinny_kernel<T, kSwiGLU, MX, PAIR, R><<<grid, 256, 0, st>>>(a, smem_sched, ks);
  else if (a.mode == kStoreAct)
    skinny_kernel<T, kStoreAct, MX, PAIR, R><<<grid, 256, 0, st>>>(a, smem_sched, ks);
  else if constexpr (!MX && R == kSkR)
    skinny_kernel<T, kStoreF32, MX, PAIR, R><<<grid, 256, 0, st>>>(a, smem_sched, ks);
}

template <typename T>
cudaError_t launch_skinny_t(const GemmArgs& a, int R, int smem_sched, cudaStream_t st) {
  const int64_t mt_bound = mtile_bound(a, R);
  if (mt_bound <= 0 || a.N <= 0) return cudaSuccess;
  if (mt_bound > 0x7fffffff) return cudaErrorInvalidValue;
  // K slices per column: enough warps to keep every SM streaming weights
  const int64_t base_warps = mt_bound * ((a.N + kSkC - 1) / kSkC);
  int ks = 1;
  while (ks < kSkW && base_warps * ks < 2432) ks *= 2;
  const int cols_per_block = (kSkW / ks) * kSkC;
  dim3 grid((unsigned)mt_bound, (unsigned)((a.N + cols_per_block - 1) / cols_per_block));
  if (a.max_sms > 0) {
    // held to max_sms SMs (resident blocks an SM: the launch bounds): the
    // blocks loop over the column blocks.  (Fewer blocks taking the same
    // number of rounds measured slower here: a block's weight stream is
    // latency-bound, so fewer blocks pull less bandwidth.)
    const int per_sm = R == 1 ? (a.mode == kSwiGLU ? 2 : 3) : 1;
    const int64_t cap = (int64_t)a.max_sms * per_sm / (int64_t)grid.x;
    if (cap < (int64_t)grid.y) grid.y = (unsigned)(cap > 0 ? cap : 1);
  }
  const bool pair = a.K % (2 * (16 / (int)sizeof(T))) == 0;
  // tiles of 1 or 4 rows exist for paired bf16 chunks in the two store modes
  if (R != kSkR && (sizeof(T) != 2 || !pair || a.mode == kStoreF32)) return cudaErrorInvalidValue;
  if (a.wfmt) {
    if constexpr (sizeof(T) != 2) {
      return cudaErrorInvalidValue;   // MXFP8 blocks are one bf16 chunk
    } else {
      if (a.mode != kSwiGLU && a.mode != kStoreAct) return cudaErrorInvalidValue;
      if (!pair) launch_skinny_mode<T, true, false, kSkR>(a, grid, smem_sched, ks, st);
      else if (R == 1) launch_skinny_mode<T, true, true, 1>(a, grid, smem_sched, ks, st);
      else if (R == 4) launch_skinny_mode<T, true, true, 4>(a, grid, smem_sched, ks, st);
      else launch_skinny_mode<T, true, true, kSkR>(a, grid, smem_sched, ks, st);
    }
  } else if (!pair) {
    launch_skinny_mode<T, false, false, kSkR>(a, grid, smem_sched, ks, st);
  } else if constexpr (sizeof(T) == 2) {
    if (R == 1) launch_skinny_mode<T, false, true, 1>(a, grid, smem_sched, ks, st);
    else if (R == 4) launch_skinny_mode<T, false, true, 4>(a, grid, smem_sched, ks, st);
    else launch_skinny_mode<T, false, true, kSkR>(a, grid, smem_sched, ks, st);
  } else {
    launch_skinny_mode<T, false, true, kSkR>(a, grid, smem_sched, ks, st);
  }
  count_launch();
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t st) {
  if (a.K % (a.dtype == MOE_F32 ? 4 : 8) != 0) return cudaErrorInvalidValue;
  const int R = skinny_rows(a);
  const int smem_sched = a.G <= kSkMaxG;
  if (!smem_sched) {
    cudaError_t e = launch_schedule(a, R, st);
    if (e != cudaSuccess) return e;
  }
  return a.dtype == MOE_F32 ? launch_skinny_t<float>(a, R, smem_sched, st)
                            : launch_skinny_t<bf16>(a, R, smem_sched, st);
}

cudaError_t launch_gemm_simt(const GemmArgs& a, int bm, cudaStream_t st) {
  cudaError_t e = launch_schedule(a, bm, st);
  if (e != cudaSuccess) return e;
  if (a.dtype == MOE_F32) return bm == 16 ? launch_t<float, 16>(a, st) : launch_t<float, 64>(a, st);
  return bm == 16 ? launch_t<bf16, 16>(a, st) : launch_t<bf16, 64>(a, st);
}

}  // namespace moe
