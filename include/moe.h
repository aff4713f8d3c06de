/*
 * moe.h -- C ABI of libmoe: the forward pass of a Mixture-of-Experts FFN layer
 * on one NVIDIA GB300 GPU (sm_103a).
 *
 *     y = g(x) * shared(x) + sum_k route_weight_k * SwiGLU-expert_k(x)
 *
 * (shared expert summed unweighted, g = 1, or Qwen2-MoE's sigmoid gate:
 * "MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
 * stage-marker contract", Group C; expert-grouped scatter / grouped GEMM /
 * gather: "Fused MoE Kernel Notes", Scatter/gather layout.)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named x, w_*, h, y, ... are DEVICE pointers owned by the
 *    caller; the library never allocates, frees or retains them.  Shape and
 *    weight-table structs are read on the host during the call only.
 *  - Element types: MOE_F32 (fp32) or MOE_BF16 (bf16) for activations and
 *    weights, chosen by moe_shape.dtype; indices are int32; routing weights
 *    and the shared gate are fp32.
 *  - Layouts are row-major (last index contiguous), [out, in] for weights:
 *      x [T, H]; router [E (+1 when shared_gate), H], row E = shared-gate
 *      weight; expert gate/up [I, H] each, expert e at base + e * expert_stride
 *      elements (split fc1: stride I*H; merged fc1 [E, 2I, H]: gate = base,
 *      up = base + I*H, stride 2*I*H); expert down [H, I], expert e at
 *      base + e * expert_stride; shared gate/up [I_sh, H], shared down [H, I_sh].
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return as soon as the work is queued.  Every argument is
 *    validated on the host before anything is launched; an invalid call
 *    launches nothing and returns an error status.
 *  - Errors only visible on the device (a direct route >= E, more rows than
 *    the stated bound, a gathered row's token out of range, a pipeline wait
 *    that ran out) never trap: the kernel
 *    sets a bit in the workspace's status word and skips the offending work.
 *    moe_get_device_status() reads and clears it.
 *  - The workspace `ws` is caller-owned device memory of at least the size
 *    the matching *_bytes() function returns, 256-byte aligned.  One call
 *    sequence at a time may use a workspace (calls that overlap on the GPU
 *    and share a workspace race).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, half-specified config */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. another dtype) */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_ROUTE = 5, /* device flag: a route index outside [0, E) */
  MOE_ERR_TIMEOUT = 6,      /* device flag: a bounded pipeline wait ran out */
  MOE_ERR_ROWS = 7,         /* device flag: group rows exceed the stated bound */
  MOE_ERR_GATHER = 8        /* device flag: a row_token entry outside [0, T) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Storage of the expert weights (routed gate/up/down and the shared MLP's;
 * the router always has the activation type).  MOE_WEIGHTS_MXFP8 ("MoE:
 * shared experts, arbitrary V_TOPK expert shapes, and an enforced
 * stage-marker contract", the fusion identity: e4m3 values with one e8m0
 * scale per block of 8 along the reduced axis) stores each [N, K] matrix
 * packed: its N*K e4m3 bytes row-major, then its N*K/8 e8m0 bytes row-major
 * ([N, K/8]); value = e4m3(q) * 2^(scale - 127).  With MXFP8 the expert
 * strides of moe_weights and of the grouped calls count BYTES (at least
 * N*K*9/8, multiples of 16) and the activations are bf16.  The weights are
 * dequantised as they are loaded: on the tensor cores (calls of more than 4
 * rows with K a multiple of 128: e4m3 tiles by TMA, converted in shared
 * memory to the bf16 tile the MMA reads), by the decode engine (up to 4
 * rows; otherwise, where the tensor cores cannot take the call, grouped
 * calls of up to 512 rows and one group of up to 16) or by the CUDA-core
 * engine (the rest); results equal those of
 * the same engine on the dequantised weights stored in bf16.  The backward
 * does not take MXFP8 weights.  moe_quantize_mxfp8 makes the packed
 * matrices. */
typedef enum { MOE_WEIGHTS_ACT = 0, MOE_WEIGHTS_MXFP8 = 1 } moe_weight_format;

/* Stages of the forward pass, in execution order.  Their names (see
 * moe_stage_name) label the benchmark's per-stage timings. */
typedef enum {
  MOE_STAGE_RESIDUAL_SETUP = 0, /* input RMSNorm (compiler page, Group E:
                                   residual_setup); empty without input_norm */
  MOE_STAGE_ROUTE = 1,          /* router GEMM + top-k softmax (+ shared gate) */
  MOE_STAGE_PERMUTE = 2,        /* histogram, offsets, scatter_index, row copy */
  MOE_STAGE_GATE_UP = 3,        /* grouped GEMM gate/up with fused SwiGLU */
  MOE_STAGE_DOWN = 4,           /* grouped GEMM down */
  MOE_STAGE_SHARED = 5,         /* shared-expert MLP (one group of T rows) */
  MOE_STAGE_COMBINE = 6,        /* route-weighted gather + shared and residual add */
  MOE_NUM_STAGES = 7
} moe_stage;

/* Layer shape.  topk_shape is the packed routing-shape word
 * (num_experts << 8) | top_k of the compiler page, Group A: 1 <= E <= 16383,
 * 1 <= k <= 255; 0 means "never set" and is rejected with an error that names
 * it (simulator page, Part 2: a missing shape register must fail, never read
 * as top_k = 0).  shared_gate = 1 needs shared_inter > 0 (a half-specified
 * shared branch is rejected, as the route-trace validator of the simulator
 * page does).  norm_topk = 1: weights = softmax over the k selected logits;
 * 0: the full softmax over all E logits, taken at the k selected.
 * input_norm = 1 prepares the input as the compiler page's residual_setup
 * stage does (Group E): x_norm = x / sqrt(mean_h x^2 + norm_eps) * norm_weight
 * (stored in the activation type, computed to about 2^-44 relative accuracy
 * and rounded once), and the router, experts and shared MLP see x_norm;
 * residual = 1 adds x to the output (y = x + MoE), inside the combine.
 * train = 1: moe_layer_forward also keeps, in its workspace, what
 * moe_layer_backward (moe_backward.h) needs -- the gate/up pre-activations
 * of every grouped row and a copy of direct routes -- and the workspace
 * grows by the backward's grouped buffers. */
typedef struct {
  int64_t tokens;       /* T >= 0 */
  int32_t hidden;       /* H, multiple of 8 */
  int32_t moe_inter;    /* I, multiple of 8 */
  int32_t shared_inter; /* I_sh (fused width moe_inter * n_shared), 0 = none */
  uint32_t topk_shape;  /* (num_experts << 8) | top_k */
  int32_t shared_gate;  /* 1: y's shared term is scaled by sigmoid(x . router[E]) */
  int32_t norm_topk;    /* 1: renormalise over the selected k */
  int32_t dtype;        /* moe_dtype */
  int32_t input_norm;   /* 1: input RMSNorm before routing and experts */
  int32_t residual;     /* 1: y = x + the MoE output */
  double norm_eps;      /* RMSNorm epsilon, finite and >= 0 */
  int32_t train;        /* 1: keep what the backward needs (see above) */
  int32_t weight_format; /* moe_weight_format of the expert weights */
} moe_shape;

/* Weights for moe_layer_forward (device pointers, layouts as above). */
typedef struct {
  const void *router;    /* [E + shared_gate, H]; may be NULL with direct routes */
  const void *gate;      /* expert e's [I, H] gate at gate + e * gate_up_stride */
  const void *up;        /* expert e's [I, H] up at up + e * gate_up_stride */
  int64_t gate_up_stride;
  const void *down;      /* expert e's [H, I] at down + e * down_stride */
  int64_t down_stride;
  const void *shared_gate_proj; /* [I_sh, H] or NULL when shared_inter == 0 */
  const void *shared_up;        /* [I_sh, H] */
  const void *shared_down;      /* [H, I_sh] */
  const void *norm_weight;      /* [H] input RMSNorm weight; needed iff input_norm */
} moe_weights;

/* Device pointers into a moe_layer_forward workspace where the routing of the
 * last call lives (filled by moe_workspace_views; read after the call). */
typedef struct {
  int32_t *topk_idx;      /* [T, k] */
  float *topk_w;          /* [T, k] */
  float *gate;            /* [T] (when shared_gate) */
  int32_t *counts;        /* [E] */
  int32_t *offsets;       /* [E + 1] */
  int32_t *scatter_index; /* [T, k] */
  int32_t *row_token;     /* [T * k] */
  void *x_perm;           /* [T * k, H] */
  void *h;                /* [T * k, I] */
  void *y_perm;           /* [T * k, H] */
  void *shared_out;       /* [T, H] (when shared_inter > 0); for T <= 4096 on the
                             tensor-core engine it may hold fp32 partial sums
                             over K instead, which the combine adds */
} moe_route_info;

/* Quantise weights to packed MXFP8 matrices (see moe_weight_format): batch
 * matrices [rows, K] of `dtype` (MOE_BF16 or MOE_F32), matrix b at
 * w + b * src_stride elements, into packed matrices at packed + b * dst_stride
 * bytes (dst_stride >= rows*K*9/8).  K a multiple of 8.  A block's scale is
 * the smallest power of two X with max|V| / X <= 448 (so MXFP8-representable
 * weights come back unchanged, as the pages state), values are rounded to
 * nearest even and saturate at 448.  A block holding a NaN or an infinity is
 * stored as NaN (scale byte 0xFF, the e8m0 NaN, and eight e4m3 NaN codes
 * 0x7F), so its values, and every output they reach, are NaN.  Asynchronous
 * on `stream`; no workspace. */
moe_status moe_quantize_mxfp8(const void *w, int32_t dtype, int64_t batch, int64_t rows,
                              int32_t K, int64_t src_stride, int64_t dst_stride, void *packed,
                              void *stream);

/* Packed routing-shape word (compiler page, Group A: (num_experts << 8) |
 * top_k; the 8-bit shift keeps every shape with up to 16383 experts in a
 * 22-bit immediate and bounds top_k at 255).  Returns 0 when out of range. */
uint32_t moe_topk_pack(int32_t num_experts, int32_t top_k);

/* Inverse of moe_topk_pack.  MOE_ERR_INVALID_ARG for 0 (never set), words
 * wider than 22 bits, or a zero field; outputs untouched then. */
moe_status moe_topk_unpack(uint32_t word, int32_t *num_experts, int32_t *top_k);

/* Scratch needed by the step entry points below (status word, router logits,
 * per-chunk histograms, GEMM tile schedules).  Returns 0 for an invalid shape. */
size_t moe_scratch_bytes(const moe_shape *shape);

/* Whole workspace of moe_layer_forward: the scratch plus every intermediate
 * (routing arrays, x_perm, h, y_perm, the shared MLP's h and output).  Returns
 * 0 for an invalid shape. */
size_t moe_workspace_bytes(const moe_shape *shape);

/* Fill *views with pointers into a moe_layer_forward workspace. */
moe_status moe_workspace_views(const moe_shape *shape, void *ws, moe_route_info *views);

/* Router GEMM + top-k softmax (compiler page, Group E router logits;
 * simulator page: topk_softmax is generic in (num_experts, top_k)).
 *   logits = x . router^T in fp32 (bf16 inputs: tensor cores, fp32 sums);
 *   topk_idx[t, s] = expert with the (s+1)-th largest logit, equal logits ->
 *   lower index; a near-tie (neighbouring logits closer than the fp32 error
 *   bound) is re-decided with an error-free compensated dot product;
 *   topk_w[t, s] per norm_topk; gate[t] = sigmoid(x[t] . router[E]) when
 *   shape->shared_gate (gate must then be non-NULL, else it may be NULL).
 * x [T, H], router [E + shared_gate, H]; outputs topk_idx, topk_w [T, k]. */
moe_status moe_route(const moe_shape *shape, const void *x, const void *w_router,
                     int32_t *topk_idx, float *topk_w, float *gate, void *ws,
                     size_t ws_bytes, void *stream);

/* Hash-MoE routing ("Fused MoE Kernel Notes", Duplicate top-k routes: a
 * router whose token-to-expert lookup can send two slots of a token to the
 * same expert, as DeepSeek-V4's hash MoE does):
 *   topk_idx[t, s] = table[token_ids[t] * k + s],  topk_w[t, s] = 1/k
 * token_ids [T] int32, table [vocab, k] int32 (device).  Duplicates are kept:
 * they are what the grouped GEMMs' launch bound must cover (pass the result
 * to moe_layer_forward as direct routes).  Every slot weighs 1/k, one
 * correctly rounded fp32 division (the notes' regression pattern uses one
 * constant routing weight).  A token id outside [0, vocab) sets
 * MOE_ERR_DEVICE_ROUTE on the device and routes that token's slots to -1,
 * which moe_permute drops; a table entry outside [0, E) is dropped and
 * flagged by moe_permute.  ws: at least moe_scratch_bytes (status word). */
moe_status moe_hash_route(const moe_shape *shape, const int32_t *token_ids,
                          const int32_t *table, int64_t vocab, int32_t *topk_idx,
                          float *topk_w, void *ws, size_t ws_bytes, void *stream);

/* Expert histogram, group offsets and scatter ("Fused MoE Kernel Notes",
 * Scatter/gather layout): counts[e] = pairs routed to e (duplicates count
 * again); offsets[e] = sum of counts before e, offsets[E] = T*k;
 * scatter_index[t, s] = offsets[e] + rank of (t, s) among the pairs routed to
 * e in row-major (t, s) order; row_token[r] = token of grouped row r;
 * x_perm[scatter_index[t, s]] = x[t].  Deterministic, no global atomics.
 * topk_idx [T, k] is an input: the router's output or direct routes.  A route
 * outside [0, E) sets MOE_ERR_DEVICE_ROUTE on the device; that pair is then
 * dropped from every output.  x_perm == NULL: the routing arrays only (x may
 * then be NULL too), for moe_grouped_swiglu_gather, which reads the rows of x
 * through row_token instead of a grouped copy. */
moe_status moe_permute(const moe_shape *shape, const void *x, const int32_t *topk_idx,
                       int32_t *counts, int32_t *offsets, int32_t *scatter_index,
                       int32_t *row_token, void *x_perm, void *ws, size_t ws_bytes,
                       void *stream);

/* moe_permute without a workspace, for callers that may not allocate device
 * memory while they run (a plugin handed only its tensors, a real-time loop
 * that forbids allocation after start-up since it can synchronise the device,
 * memory already carved up by another owner).  No passage of the pages has a
 * counterpart: this is a deployment variant of moe_permute, with the same
 * arguments minus the workspace and the same outputs.
 *  - Scratch: a 2 MiB static device array inside the library (held by every
 *    GPU that loads it until exit); every valid shape fits, a shape that
 *    would not is rejected with MOE_ERR_UNSUPPORTED and a message.
 *  - Allocates nothing (no cudaMalloc/cudaFree, no allocating library call).
 *  - The first call on a device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *    The address is kept until exit: do not call it on a device after a
 *    cudaDeviceReset of that device.
 *  - x_perm may be NULL (then x may be too): only the routing arrays are
 *    written, as with moe_permute.
 *  - All calls share the array: calls that overlap on the GPU race.
 *  - No device status word: a route outside [0, E) is dropped
 *    (scatter_index -1, not counted), visible as offsets[E] < T*k. */
moe_status moe_permute_static(const moe_shape *shape, const void *x, const int32_t *topk_idx,
                              int32_t *counts, int32_t *offsets, int32_t *scatter_index,
                              int32_t *row_token, void *x_perm, void *stream);

/* Grouped GEMM gate/up with fused SwiGLU: for each group g < num_groups,
 * rows r in [offsets[g], offsets[g+1]) of x_perm [rows, H]:
 *   h[r, j] = silu(x_perm[r] . w_gate_g[j]) * (x_perm[r] . w_up_g[j]),  j < inter
 * with w_gate_g = w_gate + g * expert_stride ([inter, H]), likewise w_up.
 * silu(a) = a * sigmoid(a); fp32 accumulation, h rounded once.
 * rows_bound >= offsets[num_groups] is the caller's bound on the total row
 * count (T*k for the routed experts, T for a shared MLP given as one group
 * with offsets {0, T}); the tile schedule is built on the device from the
 * actual group sizes, so a group larger than T (duplicate routes, "Fused MoE
 * Kernel Notes", Duplicate top-k routes) is covered in full.  More rows than
 * rows_bound sets MOE_ERR_ROWS on the device.  h is [rows_bound, inter]. */
moe_status moe_grouped_swiglu(const moe_shape *shape, const void *x_perm,
                              const void *w_gate, const void *w_up, int64_t expert_stride,
                              const int32_t *offsets, int32_t num_groups, int64_t rows_bound,
                              int32_t inter, void *h, void *ws, size_t ws_bytes,
                              void *stream);

/* moe_grouped_swiglu with the rows gathered on the fly: row r of the grouped
 * operand is x[row_token[r]] (x [T, H], T = shape->tokens, row_token as
 * moe_permute writes it), so the [T*k, H] copy x_perm is never written nor
 * read back.  Same grouping, accumulation and rounding as moe_grouped_swiglu,
 * so h is bit-identical to moe_grouped_swiglu on moe_permute's x_perm.  Only
 * rows inside a group are read; a row_token entry outside [0, T) contributes
 * zeros and sets MOE_ERR_GATHER on the device.  For callers that cannot
 * spare the [T*k, H] buffer: at prefill sizes it runs slower than the copy
 * plus moe_grouped_swiglu (moe_layer_forward takes that route). */
moe_status moe_grouped_swiglu_gather(const moe_shape *shape, const void *x,
                                     const int32_t *row_token, const void *w_gate,
                                     const void *w_up, int64_t expert_stride,
                                     const int32_t *offsets, int32_t num_groups,
                                     int64_t rows_bound, int32_t inter, void *h, void *ws,
                                     size_t ws_bytes, void *stream);

/* Grouped GEMM down: y_perm[r, n] = h[r] . w_down_g[n] for the rows of group g,
 * w_down_g = w_down + g * expert_stride ([H, inter]); same grouping rules as
 * moe_grouped_swiglu.  h [rows, inter] -> y_perm [rows, H]. */
moe_status moe_grouped_down(const moe_shape *shape, const void *h, const void *w_down,
                            int64_t expert_stride, const int32_t *offsets,
                            int32_t num_groups, int64_t rows_bound, int32_t inter,
                            void *y_perm, void *ws, size_t ws_bytes, void *stream);

/* Input preparation (compiler page, Group E: residual_setup):
 *   x_norm[t, h] = x[t, h] / sqrt((1/H) sum_h x[t, h]^2 + norm_eps) * norm_weight[h]
 * x, x_norm [T, H] and norm_weight [H] in the activation type; x_norm is
 * computed to about 2^-44 relative accuracy and rounded once (nearest even).
 * Uses shape->norm_eps whatever shape->input_norm says.  No workspace. */
moe_status moe_residual_setup(const moe_shape *shape, const void *x, const void *norm_weight,
                              void *x_norm, void *stream);

/* Route-weighted gather-combine (gather of "Fused MoE Kernel Notes"; the
 * per-token K-axis sum of the Spyre adapter's decode path) with the residual:
 *   y[t] = sum_s topk_w[t, s] * y_perm[scatter_index[t, s]] + g_t * shared_out[t]
 *          + residual[t]
 * g_t = gate[t] when gate != NULL, else 1; the shared term is skipped when
 * shared_out == NULL, the residual when residual == NULL.  Each y row is
 * written once, no read-modify-write, so duplicate routes are safe.  fp32
 * sums in that order, y rounded once.  No workspace. */
moe_status moe_combine(const moe_shape *shape, const void *y_perm,
                       const int32_t *scatter_index, const float *topk_w,
                       const void *shared_out, const float *gate, const void *residual,
                       void *y, void *stream);

/* Whole layer: [residual_setup] -> route (or direct routes) -> permute ->
 * grouped gate/up+SwiGLU -> grouped down -> shared MLP -> combine (+ residual),
 * all on `stream`, no host sync.
 * routes_idx/routes_w [T, k] (device) replace the router when non-NULL
 * (duplicates allowed); weights->router may then be NULL, and shared_gate
 * must be 0.  ws_bytes >= moe_workspace_bytes(shape).
 * With a shared MLP, the shared MLP runs on a second stream of the
 * library's, forked from `stream` after the input preparation and joined back
 * before the combine (inside a stream capture this becomes a branch of the
 * graph); at decode sizes (T <= 64) its GEMMs are held to part of the SMs.
 * That stream and its two events are made on the first such call on a
 * device: make it before any capture.
 * moe_layer_forward_traced keeps every stage on `stream`. */
moe_status moe_layer_forward(const moe_shape *shape, const moe_weights *weights,
                             const void *x, const int32_t *routes_idx,
                             const float *routes_w, void *y, void *ws, size_t ws_bytes,
                             void *stream);

/* moe_layer_forward that also records `stage_events[i]` (cudaEvent_t handles
 * created by the caller) on `stream` right before stage i (moe_stage order) and
 * `stage_events[MOE_NUM_STAGES]` after the last one, so per-stage device times
 * can be read with cudaEventElapsedTime.  Stages that do not run (no router,
 * no shared expert) still get their event, giving a zero-length interval.
 * stage_events == NULL behaves exactly like moe_layer_forward. */
moe_status moe_layer_forward_traced(const moe_shape *shape, const moe_weights *weights,
                                    const void *x, const int32_t *routes_idx,
                                    const float *routes_w, void *y, void *ws, size_t ws_bytes,
                                    void *stream, void *const *stage_events);

/* Zero the device status word of a new workspace (asynchronous on `stream`).
 * Call once before the first use of a workspace; status bits then accumulate
 * until moe_get_device_status reads and clears them. */
moe_status moe_workspace_init(void *ws, void *stream);

/* Synchronise `stream`, then read and clear the device status word of `ws`:
 * MOE_OK, or the first of MOE_ERR_DEVICE_ROUTE / MOE_ERR_ROWS /
 * MOE_ERR_TIMEOUT / MOE_ERR_GATHER that is set (*bits, if non-NULL, receives
 * every bit: 1 route, 2 rows, 4 timeout, 8 gather). */
moe_status moe_get_device_status(void *ws, void *stream, uint32_t *bits);

/* Synchronise `stream`, then read and clear the workspace's count of tokens
 * whose top-k order was re-decided with the exact compensated dot product
 * (neighbouring fp32 logits closer than the error bound; see moe_route). */
moe_status moe_get_route_stats(void *ws, void *stream, uint32_t *redecided);

/* Static strings; never NULL. */
const char *moe_status_string(moe_status status);
/* Why the last call from this thread that failed host-side validation was
 * rejected (e.g. which argument); "" when none. */
const char *moe_last_error(void);
const char *moe_stage_name(int32_t stage);

/* Number of kernel launches the last successful host call queued on this
 * thread (for launch accounting in benchmarks). */
int32_t moe_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
