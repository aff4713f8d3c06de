/*
 * moe_backward.h -- C ABI of libmoe's backward pass of the routed-expert FFN
 * (the fused scatter / grouped GEMM / gather op of "Fused MoE Kernel Notes":
 * Scatter/gather layout, Backward grouped-GEMM launch bound, Duplicate top-k
 * routes).  Conventions (device pointers owned by the caller, asynchronous
 * calls on `stream`, host-side validation, device status word, workspace
 * rules) are those of moe.h.
 *
 * With the routes given -- topk_idx [T, k] (duplicates allowed) and the
 * routing weights topk_w [T, k] -- the op computes, for each pair (t, s)
 * routed to expert e, with x the expert input:
 *     a = W_gate[e] x_t,  b = W_up[e] x_t,  h = silu(a) * b,
 *     o_ts = W_down[e] h,  y_t = sum_s topk_w[t, s] o_ts.
 * Given dy = dL/dy [T, H], the backward computes (chain rule, the notes'
 * grad_fc2_output = moe_scatter(grad_output, scatter_index); the scattered
 * gradient of a row is the gradient of o_ts, so it carries the routing
 * weight):
 *     grad_fc2[r]   = topk_w[t, s] dy_t              r = scatter_index[t, s]
 *     d_topk_w[t,s] = <dy_t, y_perm[r]>              (y_perm[r] = o_ts)
 *     dh[r]         = grad_fc2[r] . W_down[e]        (dgrad through down)
 *     da = dh * b * silu'(a),  db = dh * silu(a)     silu'(a) = s (1 + a (1 - s)),
 *                                                    s = sigmoid(a)
 *     dx_perm[r]    = da . W_gate[e] + db . W_up[e]  (dgrad through gate/up)
 *     dx_t          = sum_s dx_perm[scatter_index[t, s]]          (gather)
 *     dW_down[e]    = sum over rows r of e: grad_fc2[r]^T h[r]    (weight
 *     dW_gate[e]    = sum da[r]^T x_perm[r],  dW_up[e] = sum db[r]^T x_perm[r]
 *                                                     gradients, K = rows of e)
 * Every grouped GEMM covers each group in full from the device-side group
 * sizes: the launch bound is the scattered row count T*k, never T, so a
 * group larger than T (duplicate routes) is never truncated.  The router, a
 * shared expert and the input RMSNorm are dense layers around this op: their
 * gradients are the caller's (d_topk_w is what a router's backward needs).
 *
 * Precision: bf16 operands, fp32 accumulation, each output rounded once to
 * the activation type (d_topk_w fp32); the fp32 layer runs in fp32 on the
 * CUDA cores.
 */
#ifndef MOE_BACKWARD_H_
#define MOE_BACKWARD_H_

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Expert weight gradients, laid out like moe_weights' expert weights:
 * expert e's dW_gate / dW_up [I, H] at gate / up + e * gate_up_stride,
 * dW_down [H, I] at down + e * down_stride (elements, activation type). */
typedef struct {
  void *gate;
  void *up;
  int64_t gate_up_stride;
  void *down;
  int64_t down_stride;
} moe_expert_grads;

/* Pointers into a train-mode moe_layer_forward workspace (shape->train = 1)
 * where the backward's grouped buffers live: fc1 [T*k, 2I] = [a | b] kept by
 * the forward; grad_fc2 [T*k, H], d_fc1 [T*k, 2I] = [da | db] and dx_perm
 * [T*k, H] written by moe_layer_backward. */
typedef struct {
  void *fc1;
  void *grad_fc2;
  void *d_fc1;
  void *dx_perm;
} moe_backward_info;

moe_status moe_backward_views(const moe_shape *shape, void *ws, moe_backward_info *views);

/* moe_grouped_swiglu (moe.h) that also stores the pre-activations:
 * fc1[r, j] = x_perm[r] . w_gate_g[j], fc1[r, inter + j] = x_perm[r] . w_up_g[j]
 * (fp32 sums rounded once; fc1 [rows_bound, 2 * inter]).  h is bit-identical
 * to moe_grouped_swiglu's. */
moe_status moe_grouped_swiglu_save(const moe_shape *shape, const void *x_perm,
                                   const void *w_gate, const void *w_up, int64_t expert_stride,
                                   const int32_t *offsets, int32_t num_groups,
                                   int64_t rows_bound, int32_t inter, void *h, void *fc1,
                                   void *ws, size_t ws_bytes, void *stream);

/* The scatter of the output gradient ("Fused MoE Kernel Notes", Backward
 * grouped-GEMM launch bound: grad_fc2_output = moe_scatter(grad_output,
 * scatter_index)) fused with the routing-weight gradient:
 *   grad_fc2[scatter_index[t, s]] = topk_w[t, s] * dy[t]      (rounded once)
 *   d_topk_w[t, s] = sum_h dy[t, h] * y_perm[scatter_index[t, s], h]  (fp32)
 * dy [T, H]; y_perm, grad_fc2 [T*k, H]; a pair with scatter_index < 0 (a
 * dropped route) gets d_topk_w 0 and writes no row.  No workspace. */
moe_status moe_scatter_grad(const moe_shape *shape, const void *dy,
                            const int32_t *scatter_index, const float *topk_w,
                            const void *y_perm, void *grad_fc2, float *d_topk_w, void *stream);

/* Grouped dgrad through down with the SwiGLU derivative fused:
 *   dh[r, j] = sum_n grad_fc2[r, n] * w_down_g[n, j]     (w_down_g [H, inter])
 *   d_fc1[r, j] = dh * b * silu'(a),  d_fc1[r, inter + j] = dh * silu(a)
 * with a = fc1[r, j], b = fc1[r, inter + j] (moe_grouped_swiglu_save).
 * Groups as in moe_grouped_swiglu; the tile schedule comes from the device
 * group sizes (bound rows_bound, normally T*k).  grad_fc2 [rows, H], fc1 and
 * d_fc1 [rows, 2 * inter]. */
moe_status moe_grouped_down_dgrad(const moe_shape *shape, const void *grad_fc2,
                                  const void *w_down, int64_t expert_stride, const void *fc1,
                                  const int32_t *offsets, int32_t num_groups,
                                  int64_t rows_bound, int32_t inter, void *d_fc1, void *ws,
                                  size_t ws_bytes, void *stream);

/* Grouped dgrad through gate/up:
 *   dx_perm[r, n] = sum_j d_fc1[r, j] w_gate_g[j, n] + d_fc1[r, inter + j] w_up_g[j, n]
 * (w_gate_g, w_up_g [inter, H]); d_fc1 [rows, 2 * inter], dx_perm [rows, H]. */
moe_status moe_grouped_gate_up_dgrad(const moe_shape *shape, const void *d_fc1,
                                     const void *w_gate, const void *w_up,
                                     int64_t expert_stride, const int32_t *offsets,
                                     int32_t num_groups, int64_t rows_bound, int32_t inter,
                                     void *dx_perm, void *ws, size_t ws_bytes, void *stream);

/* Grouped weight gradient (the notes' group_gemm_same_mn: the same M x N
 * output for every group, K = the group's row count):
 *   dw_g[m, n] = sum over r in [offsets[g], offsets[g+1]) of a[r, m] * b[r, n]
 * a [rows, lda] (M columns used), b [rows, ldb] (N columns used); group g's
 * output [M, N] row-major at dw + g * dw_stride.  A group with no rows gets
 * zeros.  Offsets that do not rise from offsets[0] = 0 to at most rows_bound
 * set MOE_ERR_ROWS on the device, and each group whose own range is invalid
 * is treated as empty.  bf16 runs on the tensor cores when M, N, lda and ldb
 * are multiples of 8, on the CUDA cores otherwise. */
moe_status moe_grouped_wgrad(const moe_shape *shape, const void *a, int64_t lda, const void *b,
                             int64_t ldb, const int32_t *offsets, int32_t num_groups,
                             int64_t rows_bound, int32_t M, int32_t N, void *dw,
                             int64_t dw_stride, void *ws, size_t ws_bytes, void *stream);

/* The gather of the backward ("Fused MoE Kernel Notes", Scatter/gather
 * layout: moe_gather sums the routed rows back to [tokens, hidden]):
 *   dx[t] = sum_s dx_perm[scatter_index[t, s]] + residual_grad[t]
 * (residual_grad may be NULL).  fp32 sums in slot order, rounded once; each
 * dx row written once, so duplicate routes are safe.  No workspace. */
moe_status moe_gather_grad(const moe_shape *shape, const void *dx_perm,
                           const int32_t *scatter_index, const void *residual_grad, void *dx,
                           void *stream);

/* Whole backward of the routed-expert op after a train-mode
 * moe_layer_forward (shape->train = 1) on the same workspace, shape and
 * weights: scatter -> dgrad down (+SwiGLU') -> dW_down -> dgrad gate/up ->
 * dW_gate, dW_up -> gather, all on `stream`.  dx [T, H] is the gradient with
 * respect to the experts' input (x, which is the layer input since input_norm
 * must be 0), plus dy itself when shape->residual; d_topk_w [T, k] fp32.
 * Shapes with a shared expert or an input RMSNorm are MOE_ERR_UNSUPPORTED
 * (those dense layers' backward is not part of this op). */
moe_status moe_layer_backward(const moe_shape *shape, const moe_weights *weights,
                              const void *dy, void *dx, float *d_topk_w,
                              const moe_expert_grads *grads, void *ws, size_t ws_bytes,
                              void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_BACKWARD_H_ */
