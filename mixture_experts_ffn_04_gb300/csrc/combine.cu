// combine.cu -- route-weighted gather-combine plus the shared-expert add.
//
//   y[t] = sum_s w[t, s] * y_perm[scatter_index[t, s]] + g_t * shared_out[t]
//          (+ residual[t], the sublayer input x)
//
// "Fused MoE Kernel Notes", Scatter/gather layout (moe_gather sums the routed
// expert outputs back to [tokens, hidden]); the Spyre adapter's decode path
// forms the same sum as a reduction over the K axis, and warns that a
// read-modify-write scatter-add is wrong when slots repeat an index.  So this
// is a gather: one block per token reads its k rows (and the shared row) and
// writes y[t] once; duplicate routes are just two reads of two rows.
// fp32 accumulation in slot order, one rounding at the store.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// SH: 0 no shared term, 1 shared row of T, 2 fp32 split-K partial sums.
template <typename T, int SH>
__global__ void __launch_bounds__(128) combine_kernel(const T* __restrict__ y_perm,
                                                      const int32_t* __restrict__ sidx,
                                                      const float* __restrict__ w, int k, int H,
                                                      const T* __restrict__ shared_out,
                                                      const float* __restrict__ gate,
                                                      const T* __restrict__ residual,
                                                      T* __restrict__ y,
                                                      const float* __restrict__ shared_part,
                                                      int nsplit_sh, int64_t part_stride) {
  extern __shared__ int32_t sm[];
  int32_t* rows = sm;                                    // [k]
  float* wt = reinterpret_cast<float*>(sm + k);          // [k]
  const int64_t t = blockIdx.x;
  for (int s = threadIdx.x; s < k; s += blockDim.x) {
    rows[s] = sidx[t * k + s];
    wt[s] = w ? w[t * k + s] : 1.0f;
  }
  __syncthreads();
  const float g = gate ? gate[t] : 1.0f;
  constexpr int V = 16 / sizeof(T);
  const int nvec = H / V;
  // blockIdx.y / gridDim.y: this block's slice of the row (several blocks per
  // token when there are few tokens)
  const int v0 = (int)((int64_t)nvec * blockIdx.y / gridDim.y);
  const int v1 = (int)((int64_t)nvec * (blockIdx.y + 1) / gridDim.y);
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    // up to 8 slot rows in flight at a time, then accumulate in slot order
    for (int s0 = 0; s0 < k; s0 += 8) {
      uint4 u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int s = s0 + j;
        if (s < k && rows[s] >= 0)   // rows[s] < 0: pair dropped (route out of range)
          u[j] = __ldg(reinterpret_cast<const uint4*>(y_perm + (int64_t)rows[s] * H) + v);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int s = s0 + j;
        if (s < k && rows[s] >= 0) {
          float f[V];
          unpack16(u[j], f, (const T*)nullptr);
          const float ws = wt[s];
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(ws, f[i], acc[i]);
        }
      }
    }
    if (SH == 1) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(shared_out + t * H) + v);
      float f[V];
      unpack16(u, f, (const T*)nullptr);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g, f[i], acc[i]);
    } else if (SH == 2) {
      // the shared output as split-K partial sums, added in order
      float f[V];
#pragma unroll
      for (int i = 0; i < V; ++i) f[i] = 0.f;
      for (int sp = 0; sp < nsplit_sh; ++sp) {
        const float* src = shared_part + sp * part_stride + t * H + (int64_t)v * V;
#pragma unroll
        for (int i = 0; i < V; i += 4) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(src + i));
          f[i] += q.x; f[i + 1] += q.y; f[i + 2] += q.z; f[i + 3] += q.w;
        }
      }
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g, f[i], acc[i]);
    }
    if (residual) {
      float f[V];
      unpack16(__ldg(reinterpret_cast<const uint4*>(residual + t * H) + v), f,
               (const T*)nullptr);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += f[i];
    }
    reinterpret_cast<uint4*>(y + t * H)[v] = pack16(acc, (const T*)nullptr);
  }
}

}  // namespace

cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* scatter_index,
                           const float* topk_w, const void* shared_out, const float* gate,
                           const void* residual, void* y, cudaStream_t st,
                           const float* shared_part, int nsplit_sh) {
  const int64_t part_stride = s.T * (int64_t)s.H;
  if (s.T == 0) return cudaSuccess;
  const size_t smem = (size_t)s.k * 8;
  // few tokens: split each row over several blocks (about 2 vectors a thread)
  const int nvec = s.H / (s.dtype == MOE_F32 ? 4 : 8);
  int ysplit = 1;
  if (s.T < 1024) ysplit = (nvec + 255) / 256;
  const dim3 grid((unsigned)s.T, (unsigned)ysplit);
  const int sh = shared_part ? 2 : (shared_out ? 1 : 0);
  if (s.dtype == MOE_F32) {
    const float* yp = reinterpret_cast<const float*>(y_perm);
    const float* so = reinterpret_cast<const float*>(shared_out);
    const float* rs = reinterpret_cast<const float*>(residual);
    float* yo = reinterpret_cast<float*>(y);
    if (sh == 0) combine_kernel<float, 0><<<grid, 128, smem, st>>>(yp, scatter_index, topk_w, s.k, s.H, so, gate, rs, yo, shared_part, nsplit_sh, part_stride);
    else if (sh == 1) combine_kernel<float, 1><<<grid, 128, smem, st>>>(yp, scatter_index, topk_w, s.k, s.H, so, gate, rs, yo, shared_part, nsplit_sh, part_stride);
    else combine_kernel<float, 2><<<grid, 128, smem, st>>>(yp, scatter_index, topk_w, s.k, s.H, so, gate, rs, yo, shared_part, nsplit_sh, part_stride);
  } else {
    const bf16* yp = reinterpret_cast<const bf16*>(y_perm);
    const bf16* so = reinterpret_cast<const bf16*>(shared_out);
    const bf16* rs = reinterpret_cast<const bf16*>(residual);
    bf16* yo = reinterpret_cast<bf16*>(y);
    if (sh == 0) combine_kernel<bf16, 0><<<grid, 128, smem, st>>>(yp, scatter_index, topk_w, s.k, s.H, so, gate, rs, yo, shared_part, nsplit_sh, part_stride);
    else if (sh == 1) combine_kernel<bf16, 1><<<grid, 128, smem, st>>>(yp, scatter_index, topk_w, s.k, s.H, so, gate, rs, yo, shared_part, nsplit_sh, part_stride);
    else combine_kernel<bf16, 2><<<grid, 128, smem, st>>>(yp, scatter_index, topk_w, s.k, s.H, so, gate, rs, yo, shared_part, nsplit_sh, part_stride);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
