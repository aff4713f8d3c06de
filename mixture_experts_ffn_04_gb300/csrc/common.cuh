// common.cuh -- device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Bits of the device status word (first 4 bytes of every workspace).
enum : uint32_t {
  kFlagRoute = 1u << 0,    // route index outside [0, E)
  kFlagRows = 1u << 1,     // group rows exceed the stated bound
  kFlagTimeout = 1u << 2,  // a bounded pipeline wait ran out
  kFlagGather = 1u << 3,   // a gathered row's token outside [0, tokens)
};

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ void set_flag(uint32_t* flags, uint32_t bit) {
  if (flags) atomicOr(flags, bit);
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
};

// Unpack a 16-byte chunk into floats.
__device__ __forceinline__ void unpack16(const uint4& v, float* f, const float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4& v, float* f, const bf16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack16(const float* f, const float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint4 pack16(const float* f, const bf16*) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// MXFP8 expert weights ("MoE: shared experts, arbitrary V_TOPK expert
// shapes, and an enforced stage-marker contract": e4m3 values with one e8m0
// scale per block of 8 along the reduced axis).  A packed [N, K] matrix holds
// its N*K e4m3 bytes row-major, then its N*K/8 e8m0 bytes row-major.
// 2^(s - 127) for an e8m0 byte (0 -> 2^-127, a float subnormal; 255 -> NaN).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
  return s == 0u ? __uint_as_float(0x00400000u)
                 : (s == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float(s << 23));
}
// One block: 8 e4m3 bytes (element 0 in the lowest byte) and its scale byte
// -> 8 floats, exactly (e4m3 fits fp16; times a power of two).
__device__ __forceinline__ void unpack_mx8(uint2 q, uint32_t s, float* f) {
  const float x = e8m0_value(s);
  const uint32_t w[2] = {q.x, q.y};
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((w[i] >> (16 * j)) & 0xFFFFu), __NV_E4M3);
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h));
      f[4 * i + 2 * j] = v.x * x;
      f[4 * i + 2 * j + 1] = v.y * x;
    }
}
// One weight of a packed MXFP8 matrix [N, K]: element (n, k).
__device__ __forceinline__ float mx_weight(const uint8_t* m, int64_t N, int K, int64_t n, int64_t k) {
  const uint8_t q = m[n * K + k];
  const uint8_t s = m[N * K + n * (K / 8) + k / 8];
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)q, __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h)) * e8m0_value(s);
}

// silu(a) = a * sigmoid(a) = a / (1 + e^-a)
__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }
// The same with CUDA's fast exponential and division intrinsics (a few ulp in
// fp32): for results that are rounded to bf16 right after.
__device__ __forceinline__ float silu_fast(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

}  // namespace moe
