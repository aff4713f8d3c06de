// norm.cu -- input preparation of the MoE sublayer: the input RMSNorm.
//
//   x_norm[t, h] = x[t, h] / sqrt((1/H) sum_h' x[t, h']^2 + eps) * w[h]
//
// "MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
// stage-marker contract", Group E: residual_setup covers the residual copy,
// the input RMSNorm and its norm-weight multiply ahead of the MoE FFN (the
// residual itself is x, added by the combine kernel).
//
// x_norm is stored in the activation type and feeds the router and the
// experts, so the routing is decided on it: it is computed to about 2^-44
// relative accuracy in double-float arithmetic (pairs hi + lo of floats: the
// error-free TwoSum and FMA-based TwoProduct of Knuth and Dekker) and rounded
// once, so it equals the correctly rounded value except where the exact value
// lies within that distance of a rounding midpoint.  (fp64 would do the same
// at a fraction of the speed: FP64 is slow on this GPU.)
//
// One warp per row: 16-byte loads, four in flight per lane, a (sum,
// compensation) pair per lane for the sum of squares, merged across the warp
// with TwoSum, then a second pass that scales and stores.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

struct df {
  float hi, lo;
};

__device__ __forceinline__ df two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float z = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z))};
}
__device__ __forceinline__ df fast_two_sum(float a, float b) {   // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
// Product of two activation-type values as a double-float.  Two bf16 values
// have 8 significant bits each, so their fp32 product is exact.
__device__ __forceinline__ df exact_prod(float a, float b, const bf16*) {
  return {__fmul_rn(a, b), 0.f};
}
__device__ __forceinline__ df exact_prod(float a, float b, const float*) {
  return two_prod(a, b);
}
__device__ __forceinline__ df df_add(df a, df b) {
  df s = two_sum(a.hi, b.hi);
  s.lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ df df_mul(df a, df b) {
  df p = two_prod(a.hi, b.hi);
  p.lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
  return fast_two_sum(p.hi, p.lo);
}
// a / b for a float divisor.
__device__ __forceinline__ df df_div_f(df a, float b) {
  const float q1 = __fdiv_rn(a.hi, b);
  const float r = __fadd_rn(__fmaf_rn(-q1, b, a.hi), a.lo);   // a - q1 b, nearly exact
  return fast_two_sum(q1, __fdiv_rn(r, b));
}
// 1 / sqrt(a) for a > 0: a float estimate refined by one Newton step in
// double-float (y <- y + y (1 - a y^2) / 2).
__device__ __forceinline__ df df_rsqrt(df a) {
  const float y0 = __frsqrt_rn(a.hi);
  const df y = {y0, 0.f};
  const df ay2 = df_mul(a, df_mul(y, y));
  const df e = df_add({1.f, 0.f}, {-ay2.hi, -ay2.lo});
  const df corr = df_mul(y, {__fmul_rn(0.5f, e.hi), __fmul_rn(0.5f, e.lo)});
  return df_add(y, corr);
}

// Round hi + lo (normalised: |lo| <= ulp(hi) / 2) to the output type,
// nearest-even.  bf16: the rounding of hi decides except when hi sits exactly
// on a bf16 midpoint, where the sign of lo picks the side (lo = 0: even).
__device__ __forceinline__ float round_out(df v, const float*) { return v.hi; }
__device__ __forceinline__ bf16 round_out(df v, const bf16*) {
  const uint32_t hb = __float_as_uint(v.hi);
  uint32_t r;
  if ((hb & 0xFFFFu) == 0x8000u && v.lo != 0.f) {
    const bool away = (v.lo > 0.f) == (v.hi > 0.f);
    r = (hb >> 16) + (away ? 1u : 0u);
  } else {
    r = (hb + 0x7FFFu + ((hb >> 16) & 1u)) >> 16;
  }
  const unsigned short s = (unsigned short)r;
  return *reinterpret_cast<const bf16*>(&s);
}

constexpr int kBatch = 4;   // 16-byte chunks a lane keeps in flight

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const T* __restrict__ x,
                                                      const T* __restrict__ w, float eps_hi,
                                                      float eps_lo, int64_t rows, int H,
                                                      T* __restrict__ out) {
  constexpr int V = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const int nv = H / V;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < rows;
       t += nw) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + t * H);
    df ss = {0.f, 0.f};
    // kBatch chunks a lane in flight at a time, then their products in order
    for (int c0 = lane; c0 < nv; c0 += 32 * kBatch) {
      uint4 u[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (c0 + 32 * b < nv) u[b] = __ldg(xr + c0 + 32 * b);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (c0 + 32 * b >= nv) break;
        float f[V];
        unpack16(u[b], f, (const T*)nullptr);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const df p = exact_prod(f[i], f[i], (const T*)nullptr);
          const df s = two_sum(ss.hi, p.hi);
          ss = {s.hi, __fadd_rn(ss.lo, __fadd_rn(s.lo, p.lo))};
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const df other = {__shfl_xor_sync(0xffffffffu, ss.hi, o),
                        __shfl_xor_sync(0xffffffffu, ss.lo, o)};
      ss = df_add(fast_two_sum(ss.hi, ss.lo), other);
    }
    ss = fast_two_sum(ss.hi, ss.lo);
    const df inv = df_rsqrt(df_add(df_div_f(ss, (float)H), {eps_hi, eps_lo}));
    uint4* orow = reinterpret_cast<uint4*>(out + t * H);
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    for (int c0 = lane; c0 < nv; c0 += 32 * kBatch) {
      uint4 ux[kBatch], uw[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (c0 + 32 * b < nv) {
          ux[b] = __ldg(xr + c0 + 32 * b);
          uw[b] = __ldg(wr + c0 + 32 * b);
        }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (c0 + 32 * b >= nv) break;
        float f[V], g[V];
        unpack16(ux[b], f, (const T*)nullptr);
        unpack16(uw[b], g, (const T*)nullptr);
        T o[V];
#pragma unroll
        for (int i = 0; i < V; ++i)
          o[i] = round_out(df_mul(exact_prod(f[i], g[i], (const T*)nullptr), inv),
                           (const T*)nullptr);
        orow[c0 + 32 * b] = *reinterpret_cast<const uint4*>(o);
      }
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const Shape& s, const void* x, const void* w, double eps, void* out,
                           cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const float eps_hi = (float)eps;
  const float eps_lo = (float)(eps - (double)eps_hi);
  int64_t blocks = (s.T + 7) / 8;   // 8 rows (warps) a block
  const int64_t cap = (int64_t)tc_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (s.dtype == MOE_F32)
    rmsnorm_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(
        reinterpret_cast<const float*>(x), reinterpret_cast<const float*>(w), eps_hi, eps_lo,
        s.T, s.H, reinterpret_cast<float*>(out));
  else
    rmsnorm_kernel<bf16><<<(unsigned)blocks, 256, 0, st>>>(
        reinterpret_cast<const bf16*>(x), reinterpret_cast<const bf16*>(w), eps_hi, eps_lo,
        s.T, s.H, reinterpret_cast<bf16*>(out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
