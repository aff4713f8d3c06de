// gemm_bwd_simt.cu -- the backward grouped GEMMs on the CUDA cores (fp32
// FMA): the fp32 layer exactly, and bf16 shapes the tensor-core kernel does
// not take.  Same contracts as gemm_bwd.cu ("Fused MoE Kernel Notes",
// Backward grouped-GEMM launch bound):
//   dgrad: out[r, n] = sum_k A[r, k] * W_g[k, n] for the rows r of group g,
//          K in two segments (k < K0: B0's weights, else B1's at k - K0),
//          optionally followed by the SwiGLU derivative;
//   wgrad: dW_g[m, n] = sum over rows r of group g of A[r, m] * B[r, n].
// 64 x 64 output tiles, 16-deep k-slices staged in shared memory, a 4 x 4
// register tile per thread.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {
constexpr int kT = 64, kK = 16, kThreads = 256;

__device__ __forceinline__ int find_group_b(const int32_t* sched, int G, int j) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sched[mid] <= j) lo = mid; else hi = mid;
  }
  return lo;
}

template <typename T, int KIND>
__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(BwdGemmArgs a, int MT) {
  __shared__ __align__(16) float As[kK][kT + 4];
  __shared__ __align__(16) float Bs[kK][kT + 4];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int n0 = blockIdx.y * kT;
  const T* A = reinterpret_cast<const T*>(a.A);
  int g;
  int64_t row0 = 0, rend = 0, kbeg = 0, klen;
  int m0 = 0;
  if (KIND == kBwdWgrad) {
    g = blockIdx.x / MT;
    m0 = (blockIdx.x % MT) * kT;
    kbeg = a.offsets[g];
    const int64_t kend = a.offsets[g + 1];
    klen = (kbeg < 0 || kend < kbeg || kend > a.rows_bound) ? 0 : kend - kbeg;
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid < 32) {
      bool bad = tid == 0 && (a.offsets[0] != 0 || (int64_t)a.offsets[a.G] > a.rows_bound);
      for (int gg = tid; gg < a.G; gg += 32) bad |= a.offsets[gg + 1] < a.offsets[gg];
      if (__any_sync(0xffffffffu, bad) && tid == 0) set_flag(a.flags, kFlagRows);
    }
  } else {
    const int j = blockIdx.x;
    if (j >= a.sched[a.G]) return;
    g = find_group_b(a.sched, a.G, j);
    row0 = a.offsets[g] + (int64_t)(j - a.sched[g]) * kT;
    rend = a.offsets[g + 1];
    klen = a.K0 + a.K1;
  }
  const T* B0 = reinterpret_cast<const T*>(a.B0) + (KIND == kBwdWgrad ? 0 : (int64_t)g * a.bstride);
  const T* B1 = KIND == kBwdWgrad ? nullptr : reinterpret_cast<const T*>(a.B1) + (int64_t)g * a.bstride;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[i][q] = 0.f;

  for (int64_t k0 = 0; k0 < klen; k0 += kK) {
#pragma unroll
    for (int q = 0; q < kT * kK / kThreads; ++q) {
      const int e = tid + q * kThreads;
      if (KIND == kBwdWgrad) {
        // A[r, m] and B[r, n], m / n contiguous
        const int kk = e / kT, c = e % kT;
        const int64_t r = kbeg + k0 + kk;
        const bool kin = k0 + kk < klen;
        As[kk][c] = kin && m0 + c < a.M ? to_f(A[r * a.lda + m0 + c]) : 0.f;
        Bs[kk][c] = kin && n0 + c < a.N ? to_f(B0[r * a.ldb + n0 + c]) : 0.f;
      } else {
        // A[r, k], k contiguous; W[k, n], n contiguous
        const int r = e / kK, kk = e % kK;
        const int64_t row = row0 + r;
        const int64_t k = k0 + kk;
        As[kk][r] = row < rend && k < klen ? to_f(A[row * a.lda + k]) : 0.f;
        const int kb = e / kT, c = e % kT;
        const int64_t kw = k0 + kb;
        float bv = 0.f;
        if (kw < klen && n0 + c < a.N)
          bv = kw < a.K0 ? to_f(B0[kw * a.N + n0 + c]) : to_f(B1[(kw - a.K0) * a.N + n0 + c]);
        Bs[kb][c] = bv;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int q = 0; q < 4; ++q) bv[q] = Bs[kk][tx * 4 + q];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(av[i], bv[q], acc[i][q]);
    }
    __syncthreads();
  }

  T* out = reinterpret_cast<T*>(a.out);
  const T* pre = reinterpret_cast<const T*>(a.pre);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tx * 4 + q;
      if (n >= a.N) continue;
      if (KIND == kBwdWgrad) {
        const int m = m0 + ty * 4 + i;
        if (m < a.M) out[(int64_t)g * a.ostride + (int64_t)m * a.ldo + n] = from_f<T>(acc[i][q]);
      } else {
        const int64_t row = row0 + ty * 4 + i;
        if (row >= rend) continue;
        if (KIND == kBwdDgradSwiGLU) {
          const float av = to_f(pre[row * a.ldp + n]), bv = to_f(pre[row * a.ldp + a.N + n]);
          const float sg = 1.0f / (1.0f + expf(-av));
          out[row * a.ldo + n] = from_f<T>(acc[i][q] * bv * sg * (1.0f + av * (1.0f - sg)));
          out[row * a.ldo + a.N + n] = from_f<T>(acc[i][q] * av * sg);
        } else {
          out[row * a.ldo + n] = from_f<T>(acc[i][q]);
        }
      }
    }
  }
}

template <typename T>
cudaError_t launch_bwd_t(const BwdGemmArgs& a, cudaStream_t st) {
  const unsigned ny = (unsigned)((a.N + kT - 1) / kT);
  if (a.kind == kBwdWgrad) {
    const int MT = (a.M + kT - 1) / kT;
    const int64_t nx = (int64_t)a.G * MT;
    if (nx <= 0 || ny == 0) return cudaSuccess;
    if (nx > 0x7fffffff) return cudaErrorInvalidValue;
    simt_bwd_kernel<T, kBwdWgrad><<<dim3((unsigned)nx, ny), kThreads, 0, st>>>(a, MT);
  } else {
    // m-tiles of 64 rows: at most ceil(rows / 64) + G of them
    int64_t mt_bound = (a.rows_bound + kT - 1) / kT + a.G;
    if (mt_bound > a.rows_bound) mt_bound = a.rows_bound;
    if (mt_bound <= 0 || ny == 0) return cudaSuccess;
    if (mt_bound > 0x7fffffff) return cudaErrorInvalidValue;
    GemmArgs ga;
    ga.offsets = a.offsets;
    ga.G = a.G;
    ga.single_rows = 0;
    ga.rows_bound = a.rows_bound;
    ga.sched = a.sched;
    ga.flags = a.flags;
    cudaError_t e = launch_schedule(ga, kT, st);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)mt_bound, ny);
    if (a.kind == kBwdDgradSwiGLU)
      simt_bwd_kernel<T, kBwdDgradSwiGLU><<<grid, kThreads, 0, st>>>(a, 0);
    else
      simt_bwd_kernel<T, kBwdDgrad><<<grid, kThreads, 0, st>>>(a, 0);
  }
  count_launch();
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd_gemm_simt(const BwdGemmArgs& a, cudaStream_t st) {
  return a.dtype == MOE_F32 ? launch_bwd_t<float>(a, st) : launch_bwd_t<bf16>(a, st);
}

cudaError_t launch_bwd_gemm(const BwdGemmArgs& a, cudaStream_t st) {
  const int ov = gemm_path_override();
  if (a.dtype == MOE_BF16 && ov != 1 && bwd_gemm_tc_ok(a)) return launch_bwd_gemm_tc(a, st);
  return launch_bwd_gemm_simt(a, st);
}

}  // namespace moe
