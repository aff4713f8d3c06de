// internal.h -- host-side plumbing shared by the libmoe translation units:
// decoded shapes, workspace layout, and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

struct Shape {
  int64_t T;
  int H, I, I_sh, E, k;
  int gate;    // shared gate present
  int norm;    // renormalised top-k
  int dtype;   // MOE_F32 / MOE_BF16
  int esize;   // bytes per activation / weight element
  int ncols;   // router rows: E + gate
  int ldl;     // leading dimension of the fp32 logits buffer
  int input_norm, residual;
  double norm_eps;
  int train;   // the forward keeps what the backward needs (fc1 rows)
  int wfmt;    // expert weights: 0 the activation type, 1 packed MXFP8
};

// Decode and validate; on failure returns the status and sets *why.
moe_status decode_shape(const moe_shape* s, Shape* out, const char** why);

// Byte offsets of every region inside the workspace (all 256-byte aligned).
struct Layout {
  // scratch
  size_t flags, logits, hist, base, sched_routed, sched_shared, sched_router, tile_ctr, tmaps,
      scratch_end;
  int nchunks, tokens_per_chunk;
  // layer-forward intermediates
  size_t x_norm, topk_idx, topk_w, gate, counts, offsets, sidx, row_token, x_perm, h, y_perm,
      sh_h, sh_out, gemm_split,
      // training (shape.train): the gate/up pre-activations the forward keeps,
      // and the backward's grouped intermediates
      fc1, g_fc2, d_fc1, dx_perm, total;
};
Layout layout_for(const Shape& s);

// Launch accounting (per host thread).
void count_launch(int n = 1);
void reset_launch_count();

// Which GEMM engine serves bf16: 0 auto, 1 CUDA-core tiles, 2 tensor cores,
// 3 skinny (set through moe_testing.h by the tests).
int gemm_path_override();

// ----------------------------------------------------------------------------
// launchers; each returns the first CUDA error it saw
// ----------------------------------------------------------------------------
enum GemmMode { kSwiGLU = 0, kStoreAct = 1, kStoreF32 = 2 };

struct GemmArgs {
  int mode;
  int dtype;               // element type of A, B and (modes 0/1) the output
  const void* A;           // [rows, K] row-major
  const void* B0;          // group g's [N, K] at B0 + g * bstride
  const void* B1;          // SwiGLU: the "up" matrices (same stride)
  int64_t bstride;         // elements
  int N, K;
  const int32_t* offsets;  // [G + 1] device, or NULL: one group of single_rows
  int G;
  int64_t single_rows;
  int64_t rows_bound;      // caller's bound on offsets[G]
  void* out;               // [rows, ldo]
  int64_t ldo;             // elements
  int32_t* sched;          // [G + 1] scratch for the m-tile prefix
  int32_t* ctr = nullptr;  // scratch tile counter (zeroed by the launcher) of the
                           // SM-pair engine's dynamic tile order, or NULL
  float* split_part = nullptr;  // SM-pair engine K split (few-tile calls): fp32
                                // partials [kSplitPairMax][rows_bound][NT * 256]
  int32_t* split_ks = nullptr;  // the number of splits the kernel chose
  uint32_t* flags;
  int ksplit = 1;          // kStoreF32 only: partial sums over K ranges,
  int64_t split_stride = 0;  // written split_stride floats apart
  const int32_t* gather = nullptr;  // non-NULL: row r of the operand is A[gather[r]]
  int64_t a_rows = 0;               // rows of A when gathered (bound on gather values)
  void* pre = nullptr;              // SwiGLU: also store the pre-activations,
  int64_t ldp = 0;                  // gate at pre[r, n], up at pre[r, N + n]
  int wfmt = 0;                     // 1: B0/B1 are packed MXFP8 [N, K] matrices,
                                    // bstride in bytes
  void* amaps = nullptr;            // SM-pair engine, grouped calls: scratch for
                                    // 2 * G tensor maps (per-group A maps, so the
                                    // rows past a group's end load as zeros)
  int max_sms = 0;                  // > 0: the call's CTAs stay within this many
                                    // SMs' worth (decode and one-SM tensor-core
                                    // engines), leaving the rest to a concurrent
                                    // stream
};

// Per-group A maps (a.amaps: the padding rows of a group's last tile load as
// zeros instead of the next group's rows) lower the tensor cores' power; that
// pays where a call runs long enough for the power cap to set the SM clock
// and its groups are small enough for the padding to be a real share of the
// MMA work.  Layer A/B on one box: DeepSeek-V3 shape (256-row groups, 1e12
// MAC a call) -3 %; Qwen3 and Gemma-4 shapes (5e10) +2 % from the map
// launches; Zipf routing (1536 rows a group) neutral.
int zero_pad_override();   // moe_testing_set_zero_pad: 0 auto, 1 always, -1 never
inline bool zero_pad_pays(const GemmArgs& a) {
  if (a.amaps == nullptr || a.offsets == nullptr || a.gather != nullptr || a.G <= 1) return false;
  const int ov = zero_pad_override();
  if (ov != 0) return ov > 0;
  return (double)a.rows_bound * a.K * a.N >= 2.75e11 && a.rows_bound / a.G < 1024;
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_simt(const GemmArgs& a, int bm, cudaStream_t st);
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_tc2(const GemmArgs& a, cudaStream_t st);   // SM pairs
// MXFP8 weights dequantised in the tensor-core pipeline (K a multiple of 128)
bool gemm_tc_mx_ok(const GemmArgs& a);
cudaError_t launch_gemm_tc_mx(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_schedule(const GemmArgs& a, int bm, cudaStream_t st);

// Backward grouped GEMMs (gemm_bwd.cu on the tensor cores, gemm_bwd_simt.cu
// on the CUDA cores).
enum BwdKind { kBwdDgrad = 0, kBwdDgradSwiGLU = 1, kBwdWgrad = 2 };
struct BwdGemmArgs {
  int kind;
  int dtype;
  // dgrad: A [rows, lda] with K0 + K1 columns used; group g's weights
  //        B0 + g * bstride ([K0, N]) and B1 + g * bstride ([K1, N]).
  // wgrad: A [rows, lda] (M columns used), B0 [rows, ldb] (N columns used);
  //        group g's output [M, N] at out + g * ostride.
  const void* A;
  int64_t lda;
  const void* B0;
  const void* B1;
  int64_t bstride, ldb;
  int M, N, K0, K1;
  const int32_t* offsets;  // [G + 1]
  int G;
  int64_t rows_bound;
  void* out;
  int64_t ldo, ostride;
  const void* pre;         // kBwdDgradSwiGLU: [rows, ldp] = [a | b], N each
  int64_t ldp;
  int32_t* sched;          // [G + 1] scratch (dgrad)
  uint32_t* flags;
  void* tmaps = nullptr;   // wgrad on the tensor cores: 2 * G tensor maps
                           // (128 bytes each, 64-byte aligned) of scratch
};
bool bwd_gemm_tc_ok(const BwdGemmArgs& a);
cudaError_t launch_bwd_gemm(const BwdGemmArgs& a, cudaStream_t st);
cudaError_t launch_bwd_gemm_tc(const BwdGemmArgs& a, cudaStream_t st);
cudaError_t launch_bwd_gemm_simt(const BwdGemmArgs& a, cudaStream_t st);

// grad_fc2[scatter_index[t, s]] = topk_w[t, s] * dy[t];
// d_topk_w[t, s] = <dy[t], y_perm[scatter_index[t, s]]> (backward.cu).
cudaError_t launch_scatter_grad(const Shape& s, const void* dy, const int32_t* scatter_index,
                                const float* topk_w, const void* y_perm, void* grad_fc2,
                                float* d_topk_w, cudaStream_t st);

// logits: nsplit partial sums of [T, ldl] floats, T * ldl apart.
// redecided: count of tokens whose near tie was re-decided exactly.
cudaError_t launch_topk(const Shape& s, const float* logits, int nsplit, const void* x,
                        const void* w_router, int32_t* topk_idx, float* topk_w, float* gate,
                        uint32_t* redecided, cudaStream_t st);
cudaError_t launch_sum_partials(const Shape& s, const float* logits, int nsplit, float* out,
                                cudaStream_t st);
// Packed MXFP8 matrices from activation-type ones: batch matrices [rows, K]
// src_stride elements apart -> packed matrices dst_stride bytes apart.
cudaError_t launch_quantize_mxfp8(int dtype, const void* w, int64_t batch, int64_t rows, int K,
                                  int64_t src_stride, int64_t dst_stride, void* out,
                                  cudaStream_t st);
// Hash-MoE routes: idx[t, s] = table[token_ids[t] * k + s], w = 1/k.
cudaError_t launch_hash_route(const Shape& s, const int32_t* token_ids, const int32_t* table,
                              int64_t vocab, int32_t* idx, float* w, uint32_t* flags,
                              cudaStream_t st);

// Split-K factor for a tensor-core fp32-output GEMM of one group (router):
// enough CTAs to cover the SMs, at most kMaxSplit, at least 4 k-blocks each.
constexpr int kMaxSplit = 8;
// K splits of the SM-pair engine's few-tile calls (the shared MLP's gate/up
// of 65..kSplitMaxRows rows, see moe_api.cu), at most kSplitPairMax.
constexpr int kSplitPairMax = 4;
constexpr int64_t kSplitMaxRows = 2048;
int router_split(int64_t rows, int ncols, int K);

cudaError_t launch_permute(const Shape& s, const Layout& L, char* ws, const void* x,
                           const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                           int32_t* scatter_index, int32_t* row_token, void* x_perm,
                           cudaStream_t st);

cudaError_t launch_permute_scratch(const Shape& s, int nchunks, int tpc, int32_t* hist,
                                   int32_t* base, uint32_t* flags, const void* x,
                                   const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                                   int32_t* scatter_index, int32_t* row_token, void* x_perm,
                                   cudaStream_t st);

// Record why the current host call failed (read back by moe_last_error).
void set_error_message(const char* why);

// Host-side argument checks shared by the C-ABI files (moe_api.cu,
// backward.cu): every failure names its reason for moe_last_error.
inline moe_status fail(moe_status st, const char* why) {
  set_error_message(why);
  return st;
}
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline moe_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if ((uintptr_t)ws & 255u) return fail(MOE_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "workspace smaller than required");
  return MOE_OK;
}
#define CHECK_CUDA(expr)                                                          \
  do {                                                                            \
    cudaError_t e_ = (expr);                                                      \
    if (e_ != cudaSuccess) return ::moe::fail(MOE_ERR_CUDA, cudaGetErrorString(e_)); \
  } while (0)
#define DECODE(shape, s)                                         \
  ::moe::Shape s;                                                \
  do {                                                           \
    const char* why_ = "";                                       \
    moe_status st_ = ::moe::decode_shape(shape, &s, &why_);      \
    if (st_ != MOE_OK) return ::moe::fail(st_, why_);            \
  } while (0)

// topk_w == NULL: every slot weighs 1 (the backward's gather).
// shared_part/nsplit_sh: instead of shared_out, nsplit_sh fp32 partial sums
// of the shared MLP output ([T, H] each, T*H apart), added in order.
cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* scatter_index,
                           const float* topk_w, const void* shared_out, const float* gate,
                           const void* residual, void* y, cudaStream_t st,
                           const float* shared_part = nullptr, int nsplit_sh = 0);
// Input RMSNorm [T, H] -> [T, H] (norm.cu).
cudaError_t launch_rmsnorm(const Shape& s, const void* x, const void* w, double eps, void* out,
                           cudaStream_t st);

// Shared-MLP down projection split over K for at most this many tokens.
constexpr int64_t kSharedSplitMaxT = 4096;
int tc_sm_count();

}  // namespace moe
