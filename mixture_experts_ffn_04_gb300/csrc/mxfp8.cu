// mxfp8.cu -- quantisation of expert weights to MXFP8 ("MoE: shared experts,
// arbitrary V_TOPK expert shapes, and an enforced stage-marker contract":
// e4m3 values, one e8m0 scale per block of 8 along the reduced axis).
//
// The pages state the format and that MXFP8-representable weights quantise
// to themselves, not the rule; the rule that keeps that identity is used: a
// block's scale is the smallest power of two X with max|V| / X <= 448 (the
// largest e4m3 value), i.e. with E = floor(log2 max|V|),
//   shared = E - 8 + (max|V| > 1.75 * 2^E),  byte = shared + 127 in [0, 254],
// and each value is converted to e4m3 with round-to-nearest-even and
// saturation at 448 (the hardware conversion).  V / X is exact (a power of
// two), so the codes are those of the exact quotients.
//
// One thread per block of 8: one 16-byte load (bf16) or two (fp32), one
// 8-byte store of codes and one scale byte.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void load8(const bf16* p, float* v) {
  unpack16(*reinterpret_cast<const uint4*>(p), v, (const bf16*)nullptr);
}
__device__ __forceinline__ void load8(const float* p, float* v) {
  unpack16(*reinterpret_cast<const uint4*>(p), v, (const float*)nullptr);
  unpack16(*reinterpret_cast<const uint4*>(p + 4), v + 4, (const float*)nullptr);
}

template <typename T>
__global__ void quantize_mxfp8_kernel(const T* __restrict__ w, int64_t batch, int64_t rows, int K,
                                      int64_t src_stride, int64_t dst_stride,
                                      uint8_t* __restrict__ out) {
  const int kb = K / 8;
  const int64_t per = rows * kb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < batch * per;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per, j = i - b * per;
    const int64_t r = j / kb;
    const int c = (int)(j - r * kb);
    float v[8];
    load8(w + b * src_stride + r * K + 8 * c, v);
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      amax = fmaxf(amax, fabsf(v[e]));
      finite = finite && isfinite(v[e]);
    }
    uint8_t* dst = out + b * dst_stride;
    if (!finite) {   // a NaN or an infinity: the whole block is stored as NaN
      *reinterpret_cast<uint2*>(dst + r * K + 8 * c) = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
      dst[rows * K + r * kb + c] = 0xFF;
      continue;
    }
    int shared = 0;
    if (amax > 0.f) {
      int ex;
      frexpf(amax, &ex);                   // amax = m * 2^ex, m in [0.5, 1)
      const int E = ex - 1;                // floor(log2 amax)
      shared = E - 8 + (amax > ldexpf(1.75f, E) ? 1 : 0);
    }
    int byte = shared + 127;
    byte = byte < 0 ? 0 : (byte > 254 ? 254 : byte);
    const float inv = e8m0_value((uint32_t)(254 - byte));   // 2^(127 - byte), exact
    uint32_t word[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(v[4 * h] * inv, v[4 * h + 1] * inv), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(v[4 * h + 2] * inv, v[4 * h + 3] * inv), __NV_SATFINITE, __NV_E4M3);
      word[h] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint2*>(dst + r * K + 8 * c) = make_uint2(word[0], word[1]);
    dst[rows * K + r * kb + c] = (uint8_t)byte;
  }
}

}  // namespace

cudaError_t launch_quantize_mxfp8(int dtype, const void* w, int64_t batch, int64_t rows, int K,
                                  int64_t src_stride, int64_t dst_stride, void* out,
                                  cudaStream_t st) {
  const int64_t n = batch * rows * (K / 8);
  if (n == 0) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
  if (dtype == MOE_F32)
    quantize_mxfp8_kernel<float><<<blocks, 256, 0, st>>>(reinterpret_cast<const float*>(w), batch,
                                                         rows, K, src_stride, dst_stride,
                                                         reinterpret_cast<uint8_t*>(out));
  else
    quantize_mxfp8_kernel<bf16><<<blocks, 256, 0, st>>>(reinterpret_cast<const bf16*>(w), batch,
                                                        rows, K, src_stride, dst_stride,
                                                        reinterpret_cast<uint8_t*>(out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
