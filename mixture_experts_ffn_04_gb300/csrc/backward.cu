// backward.cu -- the backward pass of the routed-expert FFN: the scatter of
// the output gradient with the routing-weight gradient, and the C ABI of
// include/moe_backward.h (argument checks, workspace views, the sequence of
// moe_layer_backward).  The grouped GEMMs are in gemm_bwd.cu (tensor cores)
// and gemm_bwd_simt.cu (CUDA cores); the gather is the combine kernel with
// unit weights.
//
// "Fused MoE Kernel Notes", Backward grouped-GEMM launch bound: the output
// gradient is scattered to the expert-grouped rows (grad_fc2_output =
// moe_scatter(grad_output, scatter_index)) and every grouped GEMM of the
// backward is bounded by the scattered row count, never the token count.
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "../../include/moe_backward.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSlots = 8;   // slots handled per pass over a token's row

// One block per token: the token's dy row is read once per pass of up to
// kSlots slots; for each slot the block writes w * dy to the slot's grouped
// row and accumulates <dy, y_perm row> (fp32, per thread, then across the
// block in a fixed order).
template <typename T>
__global__ void __launch_bounds__(256) scatter_grad_kernel(const T* __restrict__ dy,
                                                           const int32_t* __restrict__ sidx,
                                                           const float* __restrict__ w, int k,
                                                           int H, const T* __restrict__ y_perm,
                                                           T* __restrict__ g_fc2,
                                                           float* __restrict__ dw) {
  __shared__ int32_t rows[kSlots];
  __shared__ float wt[kSlots];
  __shared__ float red[8][kSlots];
  constexpr int V = 16 / sizeof(T);
  const int64_t t = blockIdx.x;
  const int nv = H / V;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint4* dyr = reinterpret_cast<const uint4*>(dy + t * H);
  for (int s0 = 0; s0 < k; s0 += kSlots) {
    if (threadIdx.x < kSlots) {
      const int s = s0 + threadIdx.x;
      rows[threadIdx.x] = s < k ? sidx[t * k + s] : -1;
      wt[threadIdx.x] = s < k ? w[t * k + s] : 0.f;
    }
    __syncthreads();
    float acc[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) acc[j] = 0.f;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float f[V];
      unpack16(__ldg(dyr + v), f, (const T*)nullptr);
      uint4 u[kSlots];
#pragma unroll
      for (int j = 0; j < kSlots; ++j)
        if (rows[j] >= 0) u[j] = __ldg(reinterpret_cast<const uint4*>(y_perm + (int64_t)rows[j] * H) + v);
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        if (rows[j] < 0) continue;
        float yv[V], gv[V];
        unpack16(u[j], yv, (const T*)nullptr);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          acc[j] = fmaf(f[i], yv[i], acc[j]);
          gv[i] = wt[j] * f[i];
        }
        reinterpret_cast<uint4*>(g_fc2 + (int64_t)rows[j] * H)[v] = pack16(gv, (const T*)nullptr);
      }
    }
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
      if (lane == 0) red[wid][j] = acc[j];
    }
    __syncthreads();
    if (threadIdx.x < kSlots) {
      const int j = threadIdx.x, s = s0 + j;
      float sum = 0.f;
      for (int q = 0; q < (int)(blockDim.x >> 5); ++q) sum += red[q][j];
      if (s < k) dw[t * k + s] = rows[j] >= 0 ? sum : 0.f;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_scatter_grad(const Shape& s, const void* dy, const int32_t* scatter_index,
                                const float* topk_w, const void* y_perm, void* grad_fc2,
                                float* d_topk_w, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  if (s.dtype == MOE_F32)
    scatter_grad_kernel<float><<<(unsigned)s.T, 256, 0, st>>>(
        reinterpret_cast<const float*>(dy), scatter_index, topk_w, s.k, s.H,
        reinterpret_cast<const float*>(y_perm), reinterpret_cast<float*>(grad_fc2), d_topk_w);
  else
    scatter_grad_kernel<bf16><<<(unsigned)s.T, 256, 0, st>>>(
        reinterpret_cast<const bf16*>(dy), scatter_index, topk_w, s.k, s.H,
        reinterpret_cast<const bf16*>(y_perm), reinterpret_cast<bf16*>(grad_fc2), d_topk_w);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe

using namespace moe;

namespace {

// Checks shared by the grouped calls: group count, inter, row bound, strides.
moe_status check_grouped(const Shape& s, int32_t G, int64_t rows_bound, int32_t inter,
                         int64_t stride, const int32_t* offsets) {
  if (G < 1 || (G > s.E && G != 1)) return fail(MOE_ERR_INVALID_ARG, "num_groups must be in [1, E]");
  if (!offsets) return fail(MOE_ERR_INVALID_ARG, "offsets must be non-NULL");
  if (inter <= 0 || inter % 8) return fail(MOE_ERR_INVALID_ARG, "inter must be a positive multiple of 8");
  if (rows_bound < 0 || rows_bound > 0x7fffffff) return fail(MOE_ERR_INVALID_ARG, "rows_bound out of range");
  if (stride < 0) return fail(MOE_ERR_INVALID_ARG, "expert_stride must be >= 0");
  if (G > 1 && stride == 0) return fail(MOE_ERR_INVALID_ARG, "expert_stride is 0 with several groups");
  if ((stride * s.esize) % 16) return fail(MOE_ERR_INVALID_ARG, "expert_stride must be 16-byte aligned");
  return MOE_OK;
}

BwdGemmArgs bwd_args(const Shape& s, const Layout& L, char* w, int kind, int32_t G,
                     const int32_t* offsets, int64_t rows_bound) {
  BwdGemmArgs b;
  b.kind = kind;
  b.dtype = s.dtype;
  b.A = b.B0 = b.B1 = nullptr;
  b.lda = b.ldb = b.bstride = 0;
  b.M = b.N = b.K0 = b.K1 = 0;
  b.offsets = offsets;
  b.G = G;
  b.rows_bound = rows_bound;
  b.out = nullptr;
  b.ldo = b.ostride = 0;
  b.pre = nullptr;
  b.ldp = 0;
  b.sched = reinterpret_cast<int32_t*>(w + (G > 1 ? L.sched_routed : L.sched_shared));
  b.flags = reinterpret_cast<uint32_t*>(w + L.flags);
  b.tmaps = w + L.tmaps;
  return b;
}

}  // namespace

extern "C" {

moe_status moe_backward_views(const moe_shape* shape, void* ws, moe_backward_info* v) {
  DECODE(shape, s);
  if (!ws || !v) return fail(MOE_ERR_INVALID_ARG, "ws and views must be non-NULL");
  if (!s.train) return fail(MOE_ERR_INVALID_ARG, "the backward buffers exist only when shape->train = 1");
  const Layout L = layout_for(s);
  char* w = static_cast<char*>(ws);
  v->fc1 = w + L.fc1;
  v->grad_fc2 = w + L.g_fc2;
  v->d_fc1 = w + L.d_fc1;
  v->dx_perm = w + L.dx_perm;
  return MOE_OK;
}

moe_status moe_grouped_swiglu_save(const moe_shape* shape, const void* x_perm, const void* w_gate,
                                   const void* w_up, int64_t stride, const int32_t* offsets,
                                   int32_t G, int64_t rows_bound, int32_t inter, void* h,
                                   void* fc1, void* ws, size_t ws_bytes, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  moe_status c = check_grouped(s, G, rows_bound, inter, stride, offsets);
  if (c != MOE_OK) return c;
  if (rows_bound > 0 && (!x_perm || !w_gate || !w_up || !h || !fc1))
    return fail(MOE_ERR_INVALID_ARG, "operand pointers must be non-NULL");
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h) || !aligned16(fc1))
    return fail(MOE_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  const Layout L = layout_for(s);
  c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  char* w = static_cast<char*>(ws);
  GemmArgs a;
  a.mode = kSwiGLU;
  a.dtype = s.dtype;
  a.A = x_perm;
  a.B0 = w_gate;
  a.B1 = w_up;
  a.bstride = stride;
  a.N = inter;
  a.K = s.H;
  a.offsets = offsets;
  a.G = G;
  a.single_rows = 0;
  a.rows_bound = rows_bound;
  a.out = h;
  a.ldo = inter;
  a.sched = reinterpret_cast<int32_t*>(w + (G > 1 ? L.sched_routed : L.sched_shared));
  a.flags = reinterpret_cast<uint32_t*>(w + L.flags);
  a.pre = fc1;
  a.ldp = 2 * (int64_t)inter;
  CHECK_CUDA(launch_grouped_gemm(a, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_scatter_grad(const moe_shape* shape, const void* dy, const int32_t* scatter_index,
                            const float* topk_w, const void* y_perm, void* grad_fc2,
                            float* d_topk_w, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (s.T > 0 && (!dy || !scatter_index || !topk_w || !y_perm || !grad_fc2 || !d_topk_w))
    return fail(MOE_ERR_INVALID_ARG, "dy, scatter_index, topk_w, y_perm, grad_fc2 and d_topk_w must be non-NULL");
  if (!aligned16(dy) || !aligned16(y_perm) || !aligned16(grad_fc2))
    return fail(MOE_ERR_INVALID_ARG, "dy, y_perm and grad_fc2 must be 16-byte aligned");
  CHECK_CUDA(launch_scatter_grad(s, dy, scatter_index, topk_w, y_perm, grad_fc2, d_topk_w,
                                 (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_grouped_down_dgrad(const moe_shape* shape, const void* grad_fc2,
                                  const void* w_down, int64_t stride, const void* fc1,
                                  const int32_t* offsets, int32_t G, int64_t rows_bound,
                                  int32_t inter, void* d_fc1, void* ws, size_t ws_bytes,
                                  void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  moe_status c = check_grouped(s, G, rows_bound, inter, stride, offsets);
  if (c != MOE_OK) return c;
  if (rows_bound > 0 && (!grad_fc2 || !w_down || !fc1 || !d_fc1))
    return fail(MOE_ERR_INVALID_ARG, "operand pointers must be non-NULL");
  if (!aligned16(grad_fc2) || !aligned16(w_down) || !aligned16(fc1) || !aligned16(d_fc1))
    return fail(MOE_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  const Layout L = layout_for(s);
  c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  char* w = static_cast<char*>(ws);
  BwdGemmArgs b = bwd_args(s, L, w, kBwdDgradSwiGLU, G, offsets, rows_bound);
  b.A = grad_fc2;
  b.lda = s.H;
  b.B0 = w_down;
  b.bstride = stride;
  b.N = inter;
  b.K0 = s.H;
  b.out = d_fc1;
  b.ldo = 2 * (int64_t)inter;
  b.pre = fc1;
  b.ldp = 2 * (int64_t)inter;
  CHECK_CUDA(launch_bwd_gemm(b, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_grouped_gate_up_dgrad(const moe_shape* shape, const void* d_fc1,
                                     const void* w_gate, const void* w_up, int64_t stride,
                                     const int32_t* offsets, int32_t G, int64_t rows_bound,
                                     int32_t inter, void* dx_perm, void* ws, size_t ws_bytes,
                                     void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  moe_status c = check_grouped(s, G, rows_bound, inter, stride, offsets);
  if (c != MOE_OK) return c;
  if (rows_bound > 0 && (!d_fc1 || !w_gate || !w_up || !dx_perm))
    return fail(MOE_ERR_INVALID_ARG, "operand pointers must be non-NULL");
  if (!aligned16(d_fc1) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(dx_perm))
    return fail(MOE_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  const Layout L = layout_for(s);
  c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  char* w = static_cast<char*>(ws);
  BwdGemmArgs b = bwd_args(s, L, w, kBwdDgrad, G, offsets, rows_bound);
  b.A = d_fc1;
  b.lda = 2 * (int64_t)inter;
  b.B0 = w_gate;
  b.B1 = w_up;
  b.bstride = stride;
  b.N = s.H;
  b.K0 = inter;
  b.K1 = inter;
  b.out = dx_perm;
  b.ldo = s.H;
  CHECK_CUDA(launch_bwd_gemm(b, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_grouped_wgrad(const moe_shape* shape, const void* a, int64_t lda, const void* bm,
                             int64_t ldb, const int32_t* offsets, int32_t G, int64_t rows_bound,
                             int32_t M, int32_t N, void* dw, int64_t dw_stride, void* ws,
                             size_t ws_bytes, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (G < 1 || (G > s.E && G != 1)) return fail(MOE_ERR_INVALID_ARG, "num_groups must be in [1, E]");
  if (!offsets) return fail(MOE_ERR_INVALID_ARG, "offsets must be non-NULL");
  if (M <= 0 || N <= 0 || lda < M || ldb < N)
    return fail(MOE_ERR_INVALID_ARG, "M, N must be positive with lda >= M and ldb >= N");
  if (rows_bound < 0 || rows_bound > 0x7fffffff) return fail(MOE_ERR_INVALID_ARG, "rows_bound out of range");
  if (dw_stride < (int64_t)M * N && G > 1)
    return fail(MOE_ERR_INVALID_ARG, "dw_stride smaller than one group's M x N output");
  if (!dw || (rows_bound > 0 && (!a || !bm)))
    return fail(MOE_ERR_INVALID_ARG, "a, b and dw must be non-NULL");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  char* w = static_cast<char*>(ws);
  BwdGemmArgs b = bwd_args(s, L, w, kBwdWgrad, G, offsets, rows_bound);
  b.A = a;
  b.lda = lda;
  b.B0 = bm;
  b.ldb = ldb;
  b.M = M;
  b.N = N;
  b.out = dw;
  b.ldo = N;
  b.ostride = dw_stride;
  // the tensor-core path reads through TMA maps (16-byte bases and strides)
  // and stores 16-byte pieces; other layouts take the CUDA-core path
  const bool tc_layout = aligned16(a) && aligned16(bm) && aligned16(dw) && dw_stride % 8 == 0;
  CHECK_CUDA(tc_layout ? launch_bwd_gemm(b, (cudaStream_t)stream)
                       : launch_bwd_gemm_simt(b, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_gather_grad(const moe_shape* shape, const void* dx_perm,
                           const int32_t* scatter_index, const void* residual_grad, void* dx,
                           void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (s.T > 0 && (!dx_perm || !scatter_index || !dx))
    return fail(MOE_ERR_INVALID_ARG, "dx_perm, scatter_index and dx must be non-NULL");
  if (!aligned16(dx_perm) || !aligned16(residual_grad) || !aligned16(dx))
    return fail(MOE_ERR_INVALID_ARG, "dx_perm, residual_grad and dx must be 16-byte aligned");
  CHECK_CUDA(launch_combine(s, dx_perm, scatter_index, nullptr, nullptr, nullptr, residual_grad,
                            dx, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_layer_backward(const moe_shape* shape, const moe_weights* W, const void* dy,
                              void* dx, float* d_topk_w, const moe_expert_grads* grads, void* ws,
                              size_t ws_bytes, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (!s.train) return fail(MOE_ERR_INVALID_ARG, "moe_layer_backward needs a train-mode forward (shape->train = 1)");
  if (s.I_sh) return fail(MOE_ERR_UNSUPPORTED, "the shared expert's backward is not part of the routed-expert op");
  if (s.input_norm) return fail(MOE_ERR_UNSUPPORTED, "the input RMSNorm's backward is not part of the routed-expert op");
  if (s.wfmt) return fail(MOE_ERR_UNSUPPORTED, "the backward takes expert weights in the activation type, not MXFP8");
  if (!W || !grads) return fail(MOE_ERR_INVALID_ARG, "weights and grads must be non-NULL");
  if (s.T > 0 && (!dy || !dx || !d_topk_w || !W->gate || !W->up || !W->down || !grads->gate ||
                  !grads->up || !grads->down))
    return fail(MOE_ERR_INVALID_ARG, "dy, dx, d_topk_w, the expert weights and their gradients must be non-NULL");
  if (W->gate_up_stride < (int64_t)s.I * s.H || W->down_stride < (int64_t)s.H * s.I ||
      grads->gate_up_stride < (int64_t)s.I * s.H || grads->down_stride < (int64_t)s.H * s.I)
    return fail(MOE_ERR_INVALID_ARG, "expert strides smaller than one expert matrix");
  if (!aligned16(dy) || !aligned16(dx) || !aligned16(W->gate) || !aligned16(W->up) ||
      !aligned16(W->down) || !aligned16(grads->gate) || !aligned16(grads->up) ||
      !aligned16(grads->down) || (W->gate_up_stride * s.esize) % 16 ||
      (W->down_stride * s.esize) % 16 || (grads->gate_up_stride * s.esize) % 16 ||
      (grads->down_stride * s.esize) % 16)
    return fail(MOE_ERR_INVALID_ARG, "tensors and strides must be 16-byte aligned");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.total);
  if (c != MOE_OK) return c;
  if (s.T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  char* w = static_cast<char*>(ws);
  const int32_t* offsets = reinterpret_cast<const int32_t*>(w + L.offsets);
  const int32_t* sidx = reinterpret_cast<const int32_t*>(w + L.sidx);
  const float* tw = reinterpret_cast<const float*>(w + L.topk_w);
  void* g_fc2 = w + L.g_fc2;
  void* d_fc1 = w + L.d_fc1;
  void* dx_perm = w + L.dx_perm;
  const int64_t R = s.T * (int64_t)s.k;
  const int64_t I2 = 2 * (int64_t)s.I;

  // 1. scatter of the output gradient (carrying the routing weight) and the
  //    routing-weight gradient
  CHECK_CUDA(launch_scatter_grad(s, dy, sidx, tw, w + L.y_perm, g_fc2, d_topk_w, st));
  // 2. dgrad through down, SwiGLU derivative in the epilogue
  BwdGemmArgs b = bwd_args(s, L, w, kBwdDgradSwiGLU, s.E, offsets, R);
  b.A = g_fc2;
  b.lda = s.H;
  b.B0 = W->down;
  b.bstride = W->down_stride;
  b.N = s.I;
  b.K0 = s.H;
  b.out = d_fc1;
  b.ldo = I2;
  b.pre = w + L.fc1;
  b.ldp = I2;
  CHECK_CUDA(launch_bwd_gemm(b, st));
  // 3. dW_down[e] = grad_fc2_e^T h_e
  BwdGemmArgs wg = bwd_args(s, L, w, kBwdWgrad, s.E, offsets, R);
  wg.A = g_fc2;
  wg.lda = s.H;
  wg.M = s.H;
  wg.B0 = w + L.h;
  wg.ldb = s.I;
  wg.N = s.I;
  wg.out = grads->down;
  wg.ldo = s.I;
  wg.ostride = grads->down_stride;
  CHECK_CUDA(launch_bwd_gemm(wg, st));
  // 4. dgrad through gate/up over the concatenated [da | db]
  b = bwd_args(s, L, w, kBwdDgrad, s.E, offsets, R);
  b.A = d_fc1;
  b.lda = I2;
  b.B0 = W->gate;
  b.B1 = W->up;
  b.bstride = W->gate_up_stride;
  b.N = s.H;
  b.K0 = s.I;
  b.K1 = s.I;
  b.out = dx_perm;
  b.ldo = s.H;
  CHECK_CUDA(launch_bwd_gemm(b, st));
  // 5. dW_gate[e] = da_e^T x_perm_e, dW_up[e] = db_e^T x_perm_e
  wg.A = d_fc1;
  wg.lda = I2;
  wg.M = s.I;
  wg.B0 = w + L.x_perm;
  wg.ldb = s.H;
  wg.N = s.H;
  wg.out = grads->gate;
  wg.ldo = s.H;
  wg.ostride = grads->gate_up_stride;
  CHECK_CUDA(launch_bwd_gemm(wg, st));
  wg.A = static_cast<char*>(d_fc1) + (size_t)s.I * s.esize;
  wg.out = grads->up;
  CHECK_CUDA(launch_bwd_gemm(wg, st));
  // 6. gather to the tokens (+ dy itself through the residual)
  CHECK_CUDA(launch_combine(s, dx_perm, sidx, nullptr, nullptr, nullptr, s.residual ? dy : nullptr,
                            dx, st));
  return MOE_OK;
}

}  // extern "C"
