// common.cuh -- device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
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

// silu(a) = a * sigmoid(a) = a / (1 + e^-a)
__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }
// The same with CUDA's fast exponential and division intrinsics (a few ulp in
// fp32): for results that are rounded to bf16 right after.
__device__ __forceinline__ float silu_fast(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

}  // namespace moe
