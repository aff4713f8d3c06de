// moe_api.cu -- the C ABI of libmoe: argument validation, workspace layout,
// engine dispatch and the whole-layer sequence.  Declarations and contracts
// are in include/moe.h.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "../../include/moe_testing.h"
#include "common.cuh"
#include "internal.h"

namespace moe {

static thread_local int tl_launches = 0;
static thread_local const char* tl_error = "";
static std::atomic<int> g_engine{0};
static std::atomic<int> g_fork_sms{0};   // moe_testing_set_fork_sms
static std::atomic<int> g_zero_pad{0};   // moe_testing_set_zero_pad

void count_launch(int n) { tl_launches += n; }
void reset_launch_count() { tl_launches = 0; }
int gemm_path_override() { return g_engine.load(); }
int zero_pad_override() { return g_zero_pad.load(); }

void set_error_message(const char* why) { tl_error = why; }

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// The layer forward's second stream (the shared MLP) and its fork/join
// events, one set per device, made on first use; the mutex is held from the
// fork to the join's enqueue so that concurrent callers never see each
// other's event records.
constexpr int64_t kForkMaxT = 64;   // decode sizes: the shared MLP held to fewer SMs
// SMs the forked shared MLP's GEMMs may fill at decode sizes.  Left to
// themselves they take every SM and the routed chain's short launches queue
// behind their CTAs; held to 96 of the 152 the two streams overlap (Qwen2-MoE
// shape, graph replay: T = 1 145 -> 133 us, T = 16 447 -> 422, T = 64 617 ->
// 584, T = 8 unchanged within noise; 32-64 SMs starve the shared MLP
// instead).  At prefill sizes the shared MLP takes whatever SMs are free:
// caps of 60-140 SMs measured slower there.
constexpr int kForkSharedSms = 96;
static int fork_shared_sms(int64_t T) {
  const int v = g_fork_sms.load();
  if (v != 0) return v < 0 ? 0 : v;
  return T <= kForkMaxT ? kForkSharedSms : 0;
}
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
static cudaError_t side_stream(SideStream** out) {
  static SideStream sides[64];
  static std::mutex init_mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SideStream& sd = sides[dev];
  std::lock_guard<std::mutex> lock(init_mu);
  if (sd.stream == nullptr) {
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if ((e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&f, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&j, cudaEventDisableTiming)) != cudaSuccess) return e;
    sd.fork = f;
    sd.join = j;
    sd.stream = st;
  }
  *out = &sd;
  return cudaSuccess;
}

moe_status decode_shape(const moe_shape* s, Shape* o, const char** why) {
  if (!s) { *why = "shape is NULL"; return MOE_ERR_INVALID_ARG; }
  if (s->topk_shape == 0) {
    *why = "topk_shape is 0: the routing shape word (num_experts << 8) | top_k was never set";
    return MOE_ERR_INVALID_ARG;
  }
  int32_t E, k;
  if (moe_topk_unpack(s->topk_shape, &E, &k) != MOE_OK) {
    *why = "topk_shape is not a valid (num_experts << 8) | top_k word";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) {
    *why = "dtype must be MOE_F32 or MOE_BF16";
    return MOE_ERR_UNSUPPORTED;
  }
  if (s->tokens < 0 || s->tokens > (int64_t)0x7fffffff / (k > 0 ? k : 1)) {
    *why = "tokens must be in [0, 2^31 / top_k)";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->hidden <= 0 || s->hidden % 8 || s->moe_inter <= 0 || s->moe_inter % 8) {
    *why = "hidden and moe_inter must be positive multiples of 8";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->shared_inter < 0 || s->shared_inter % 8) {
    *why = "shared_inter must be 0 or a positive multiple of 8";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->shared_gate != 0 && s->shared_gate != 1) {
    *why = "shared_gate must be 0 or 1";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->shared_gate && s->shared_inter == 0) {
    *why = "shared_gate is set but shared_inter is 0 (half-specified shared expert)";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->norm_topk != 0 && s->norm_topk != 1) {
    *why = "norm_topk must be 0 or 1";
    return MOE_ERR_INVALID_ARG;
  }
  if ((s->input_norm != 0 && s->input_norm != 1) || (s->residual != 0 && s->residual != 1)) {
    *why = "input_norm and residual must be 0 or 1";
    return MOE_ERR_INVALID_ARG;
  }
  if (!(s->norm_eps >= 0.0) || s->norm_eps > 1e30) {   // also rejects NaN
    *why = "norm_eps must be finite and >= 0";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->train != 0 && s->train != 1) {
    *why = "train must be 0 or 1";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->weight_format != MOE_WEIGHTS_ACT && s->weight_format != MOE_WEIGHTS_MXFP8) {
    *why = "weight_format must be MOE_WEIGHTS_ACT or MOE_WEIGHTS_MXFP8";
    return MOE_ERR_INVALID_ARG;
  }
  if (s->weight_format == MOE_WEIGHTS_MXFP8 && s->dtype != MOE_BF16) {
    *why = "MXFP8 expert weights need bf16 activations";
    return MOE_ERR_UNSUPPORTED;
  }
  o->T = s->tokens;
  o->input_norm = s->input_norm;
  o->residual = s->residual;
  o->norm_eps = s->norm_eps;
  o->train = s->train;
  o->wfmt = s->weight_format;
  o->H = s->hidden;
  o->I = s->moe_inter;
  o->I_sh = s->shared_inter;
  o->E = E;
  o->k = k;
  o->gate = s->shared_gate;
  o->norm = s->norm_topk;
  o->dtype = s->dtype;
  o->esize = s->dtype == MOE_F32 ? 4 : 2;
  o->ncols = E + s->shared_gate;
  o->ldl = (o->ncols + 3) & ~3;
  return MOE_OK;
}

// The shared MLP's gate/up takes the SM-pair engine's K split when its pair
// tiles (256-row m-tiles x 128-column n-tiles) would leave most of the SMs
// idle: bf16, no MXFP8 weights, prefill-sized (at decode sizes the shared
// MLP's weight stream is held to part of the SMs instead), at most
// kSplitMaxTiles tiles.  Routed calls do not split: their
// group sizes are known on the device only, and where they are few-tile (all
// routes on one expert at T = 128) the fp32 partials of a 2I-wide SwiGLU
// accumulator cost more than the split saves (gate/up 37 -> 48 us, measured).
constexpr int64_t kSplitMaxTiles = 48;
static bool shared_split_ok(const Shape& s) {
  if (s.dtype != MOE_BF16 || s.wfmt || s.I_sh == 0 || s.T <= kForkMaxT || s.T > kSplitMaxRows)
    return false;
  const int64_t tiles = ((s.T + 255) / 256) * ((s.I_sh + 127) / 128);
  return tiles <= kSplitMaxTiles;
}

Layout layout_for(const Shape& s) {
  Layout L;
  size_t off = 0;
  const size_t T = (size_t)s.T, k = (size_t)s.k, E = (size_t)s.E;
  L.flags = off; off += 256;
  L.logits = off; off += align256((size_t)kMaxSplit * T * (size_t)s.ldl * 4);
  int64_t nchunks = (s.T + 31) / 32;
  int64_t cap = 262144 / s.E;
  if (cap < 1) cap = 1;
  if (nchunks > cap) nchunks = cap;
  if (nchunks < 1) nchunks = 1;
  L.nchunks = (int)nchunks;
  L.tokens_per_chunk = (int)((s.T + nchunks - 1) / nchunks);
  if (L.tokens_per_chunk < 1) L.tokens_per_chunk = 1;
  L.hist = off; off += align256((size_t)nchunks * E * 4);
  L.base = off; off += align256((size_t)nchunks * E * 4);
  L.sched_routed = off; off += align256((E + 1) * 4);
  L.sched_shared = off; off += 256;
  L.sched_router = off; off += 256;
  // tile counters (routed calls at +0, one-group calls at +128) and the K
  // split the pair engine chose for a one-group call (+192)
  L.tile_ctr = off; off += 256;
  L.tmaps = off; off += align256(256 * E);   // two tensor maps per group
  L.scratch_end = off;
  L.x_norm = off; off += align256(s.input_norm ? T * (size_t)s.H * s.esize : 0);
  L.topk_idx = off; off += align256(T * k * 4);
  L.topk_w = off; off += align256(T * k * 4);
  L.gate = off; off += align256(T * 4);
  L.counts = off; off += align256(E * 4);
  L.offsets = off; off += align256((E + 1) * 4);
  L.sidx = off; off += align256(T * k * 4);
  L.row_token = off; off += align256(T * k * 4);
  L.x_perm = off; off += align256(T * k * (size_t)s.H * s.esize);
  L.h = off; off += align256(T * k * (size_t)s.I * s.esize);
  L.y_perm = off; off += align256(T * k * (size_t)s.H * s.esize);
  L.sh_h = off; off += align256(T * (size_t)s.I_sh * s.esize);
  // the shared MLP's output: bf16/fp32 rows, or (few tokens, see
  // shared_split) up to kMaxSplit fp32 partial sums over K
  size_t sh_bytes = s.I_sh ? T * (size_t)s.H * s.esize : 0;
  if (s.I_sh && s.T <= kSharedSplitMaxT)
    sh_bytes = std::max(sh_bytes, (size_t)kMaxSplit * T * (size_t)s.H * 4);
  L.sh_out = off; off += align256(sh_bytes);
  // the SM-pair engine's K-split partials (the shared MLP's gate/up when it
  // has few tiles)
  size_t split = 0;
  if (shared_split_ok(s))
    split = (size_t)kSplitPairMax * T * (size_t)(((s.I_sh + 127) / 128) * 256) * 4;
  L.gemm_split = off; off += align256(split);
  const size_t rows = s.train ? T * k : 0;
  L.fc1 = off; off += align256(rows * 2 * (size_t)s.I * s.esize);
  L.g_fc2 = off; off += align256(rows * (size_t)s.H * s.esize);
  L.d_fc1 = off; off += align256(rows * 2 * (size_t)s.I * s.esize);
  L.dx_perm = off; off += align256(rows * (size_t)s.H * s.esize);
  L.total = off;
  return L;
}

// Engine for a grouped GEMM: 1 CUDA-core tiles, 2 tensor cores, 3 skinny,
// 4 tensor cores on SM pairs.
static int engine_for(const GemmArgs& a) {
  const int ov = gemm_path_override();
  const int64_t rows = a.offsets ? a.rows_bound : a.single_rows;
  if (a.wfmt) {
    // MXFP8 weights: the decode engine (half the weight bytes), or the
    // CUDA-core engine for large calls and for the pre-activation store
    if (ov == 1 || a.pre) return 1;
    if (ov == 3) return 3;
    // the tensor cores with the weight tiles dequantised in shared memory,
    // above a few rows (as for bf16 weights)
    if (gemm_tc_mx_ok(a) && (ov == 2 || rows > 4)) return 6;
    // the decode engine re-reads the weights for every 8-row m-tile: fine for
    // many small groups, not for one big group (the shared MLP)
    return rows <= (a.G == 1 ? 16 : 512) ? 3 : 1;
  }
  if (a.dtype == MOE_F32) return ov == 3 && a.pre == nullptr ? 3 : 1;
  // the pre-activation store exists on the one-SM tensor-core and CUDA-core engines
  if (a.pre) return ov == 1 ? 1 : 2;
  const bool pair_ok = a.mode != kStoreF32 && a.ksplit == 1 && a.gather == nullptr;
  if (ov == 4) return pair_ok ? 4 : 2;
  if (ov >= 1 && ov <= 3) return ov;
  if (rows <= 4) return 3;
  // SM pairs: a 64-wide k-block needs 32 KB of operands per SM instead of
  // 48 KB (six stages instead of four) for the same MMA work, a group's last
  // tile with at most 128 rows left runs at M = 128 (half the MMA time), and
  // the tiles are handed out in one window of consecutive tile numbers (big
  // groups m-tile major).  Measured against the one-SM engine on the layer:
  // ahead for one big group (the shared MLP), for large routed groups
  // (all-to-one and Zipf routing) and for long reductions (K = 3584, 7168),
  // 5 % behind on short ones (the Qwen3- and Gemma-4-shaped layers, K <= 2816,
  // whose tiles are too short for the pair's per-tile hand-offs), and behind
  // for small grouped calls whatever K (768 rows at K = 4096, all-to-one and
  // Zipf routing at T = 128: 122 -> 120 and 414 -> 399 us a layer).
  if (pair_ok && rows >= 512 && (a.G == 1 || rows / a.G >= 1024 || (a.K >= 3072 && rows > 2048)))
    return 4;
  // a few-tile one-group gate/up the layer gives a K-split buffer: the pair
  // engine splits K until its clusters are busy
  if (pair_ok && a.split_part) return 4;
  return 2;
}

// K split of the shared MLP's down projection on the tensor cores: its N = H
// gives few output tiles when T is small, so the K range is split until the
// tiles fill the SMs in whole waves (at least 8 k-blocks per split); the
// combine kernel adds the fp32 partial sums.
static int shared_split(const Shape& s, const GemmArgs& down) {
  if (s.T > kSharedSplitMaxT || engine_for(down) != 2) return 1;
  const int64_t base = ((s.T + 127) / 128) * ((s.H + 255) / 256);
  const int kb = (s.I_sh + 63) / 64;
  const int64_t sms = tc_sm_count();
  int best = 1;
  double best_eff = 0.0;
  for (int sp = 1; sp <= kMaxSplit && kb / sp >= 8; ++sp) {
    const int64_t tiles = base * sp;
    const double eff = (double)tiles / (double)(((tiles + sms - 1) / sms) * sms);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = sp;
    }
  }
  return best;
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t st) {
  switch (engine_for(a)) {
    case 1: return launch_gemm_simt(a, 64, st);
    case 2: return launch_gemm_tc(a, st);
    case 4: return launch_gemm_tc2(a, st);
    case 6: return launch_gemm_tc_mx(a, st);
    default: return launch_gemm_skinny(a, st);
  }
}

}  // namespace moe

using namespace moe;

extern "C" {

uint32_t moe_topk_pack(int32_t num_experts, int32_t top_k) {
  if (num_experts < 1 || num_experts > 16383 || top_k < 1 || top_k > 255) return 0;
  return ((uint32_t)num_experts << 8) | (uint32_t)top_k;
}

moe_status moe_topk_unpack(uint32_t word, int32_t* num_experts, int32_t* top_k) {
  if (word == 0 || word > 0x3FFFFFu) return MOE_ERR_INVALID_ARG;
  const int32_t e = (int32_t)(word >> 8), k = (int32_t)(word & 0xFFu);
  if (e < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (num_experts) *num_experts = e;
  if (top_k) *top_k = k;
  return MOE_OK;
}

size_t moe_scratch_bytes(const moe_shape* shape) {
  Shape s;
  const char* why;
  if (decode_shape(shape, &s, &why) != MOE_OK) return 0;
  return layout_for(s).scratch_end;
}

size_t moe_workspace_bytes(const moe_shape* shape) {
  Shape s;
  const char* why;
  if (decode_shape(shape, &s, &why) != MOE_OK) return 0;
  return layout_for(s).total;
}

moe_status moe_workspace_views(const moe_shape* shape, void* ws, moe_route_info* v) {
  DECODE(shape, s);
  if (!ws || !v) return fail(MOE_ERR_INVALID_ARG, "ws and views must be non-NULL");
  const Layout L = layout_for(s);
  char* w = static_cast<char*>(ws);
  v->topk_idx = reinterpret_cast<int32_t*>(w + L.topk_idx);
  v->topk_w = reinterpret_cast<float*>(w + L.topk_w);
  v->gate = s.gate ? reinterpret_cast<float*>(w + L.gate) : nullptr;
  v->counts = reinterpret_cast<int32_t*>(w + L.counts);
  v->offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  v->scatter_index = reinterpret_cast<int32_t*>(w + L.sidx);
  v->row_token = reinterpret_cast<int32_t*>(w + L.row_token);
  v->x_perm = w + L.x_perm;
  v->h = w + L.h;
  v->y_perm = w + L.y_perm;
  v->shared_out = s.I_sh ? w + L.sh_out : nullptr;
  return MOE_OK;
}

moe_status moe_quantize_mxfp8(const void* w, int32_t dtype, int64_t batch, int64_t rows, int32_t K,
                              int64_t src_stride, int64_t dst_stride, void* packed, void* stream) {
  reset_launch_count();
  if (dtype != MOE_BF16 && dtype != MOE_F32) return fail(MOE_ERR_UNSUPPORTED, "dtype must be MOE_BF16 or MOE_F32");
  if (batch < 0 || rows < 0 || K <= 0 || K % 8) return fail(MOE_ERR_INVALID_ARG, "batch, rows >= 0 and K a positive multiple of 8");
  if (batch > 0 && rows > 0 && (!w || !packed)) return fail(MOE_ERR_INVALID_ARG, "w and packed must be non-NULL");
  if (batch > 1 && (src_stride < rows * K || dst_stride < rows * K / 8 * 9))
    return fail(MOE_ERR_INVALID_ARG, "strides smaller than one matrix");
  if (!aligned16(w) || !aligned16(packed) || (batch > 1 && (dst_stride % 16 || (src_stride * (dtype == MOE_F32 ? 4 : 2)) % 16)))
    return fail(MOE_ERR_INVALID_ARG, "w, packed and the strides must be 16-byte aligned");
  CHECK_CUDA(launch_quantize_mxfp8(dtype, w, batch, rows, K, src_stride, dst_stride, packed,
                                   (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_workspace_init(void* ws, void* stream) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  CHECK_CUDA(cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream));
  return MOE_OK;
}

// Router GEMM into the scratch logits (split-K partial sums on the tensor
// cores); returns the number of partials.
static moe_status router_gemm(const Shape& s, const Layout& L, char* w, const void* x,
                              const void* router, int* nsplit, cudaStream_t st) {
  float* logits = reinterpret_cast<float*>(w + L.logits);
  GemmArgs ra;
  ra.mode = kStoreF32;
  ra.dtype = s.dtype;
  ra.A = x;
  ra.B0 = router;
  ra.B1 = nullptr;
  ra.bstride = 0;
  ra.N = s.ncols;
  ra.K = s.H;
  ra.offsets = nullptr;
  ra.G = 1;
  ra.single_rows = s.T;
  ra.rows_bound = s.T;
  ra.out = logits;
  ra.ldo = s.ldl;
  ra.sched = reinterpret_cast<int32_t*>(w + L.sched_router);
  ra.flags = reinterpret_cast<uint32_t*>(w + L.flags);
  // On the tensor cores the router is split over K so that its few m-tiles
  // still cover the SMs; the top-k kernel adds the partial sums in order.
  ra.ksplit = engine_for(ra) == 2 ? router_split(s.T, s.ncols, s.H) : 1;
  ra.split_stride = s.T * (int64_t)s.ldl;
  CHECK_CUDA(launch_grouped_gemm(ra, st));
  *nsplit = ra.ksplit;
  return MOE_OK;
}

// Router GEMM, then top-k.
static moe_status do_route(const Shape& s, const Layout& L, char* w, const void* x,
                           const void* router, int32_t* idx, float* tw, float* gate,
                           cudaStream_t st) {
  if (s.T == 0) return MOE_OK;
  int nsplit = 1;
  moe_status r = router_gemm(s, L, w, x, router, &nsplit, st);
  if (r != MOE_OK) return r;
  float* logits = reinterpret_cast<float*>(w + L.logits);
  uint32_t* stats = reinterpret_cast<uint32_t*>(w + L.flags) + 1;
  CHECK_CUDA(launch_topk(s, logits, nsplit, x, router, idx, tw, gate, stats, st));
  return MOE_OK;
}

moe_status moe_route(const moe_shape* shape, const void* x, const void* w_router,
                     int32_t* topk_idx, float* topk_w, float* gate, void* ws, size_t ws_bytes,
                     void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (s.k > s.E) return fail(MOE_ERR_INVALID_ARG, "top_k exceeds num_experts");
  if (s.T > 0 && (!x || !w_router || !topk_idx || !topk_w))
    return fail(MOE_ERR_INVALID_ARG, "x, w_router, topk_idx and topk_w must be non-NULL");
  if (s.T > 0 && s.gate && !gate) return fail(MOE_ERR_INVALID_ARG, "shared_gate needs a gate output");
  if (!aligned16(x) || !aligned16(w_router))
    return fail(MOE_ERR_INVALID_ARG, "x and w_router must be 16-byte aligned");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  return do_route(s, L, static_cast<char*>(ws), x, w_router, topk_idx, topk_w, gate,
                  (cudaStream_t)stream);
}

moe_status moe_hash_route(const moe_shape* shape, const int32_t* token_ids, const int32_t* table,
                          int64_t vocab, int32_t* topk_idx, float* topk_w, void* ws,
                          size_t ws_bytes, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (vocab < 1) return fail(MOE_ERR_INVALID_ARG, "vocab must be >= 1");
  if (s.T > 0 && (!token_ids || !table || !topk_idx || !topk_w))
    return fail(MOE_ERR_INVALID_ARG, "token_ids, table, topk_idx and topk_w must be non-NULL");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  char* w = static_cast<char*>(ws);
  CHECK_CUDA(launch_hash_route(s, token_ids, table, vocab, topk_idx, topk_w,
                               reinterpret_cast<uint32_t*>(w + L.flags), (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_permute(const moe_shape* shape, const void* x, const int32_t* topk_idx,
                       int32_t* counts, int32_t* offsets, int32_t* scatter_index,
                       int32_t* row_token, void* x_perm, void* ws, size_t ws_bytes,
                       void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (!counts || !offsets) return fail(MOE_ERR_INVALID_ARG, "counts and offsets must be non-NULL");
  if (s.T > 0 && (!topk_idx || !scatter_index || !row_token))
    return fail(MOE_ERR_INVALID_ARG, "topk_idx, scatter_index and row_token must be non-NULL");
  if (s.T > 0 && x_perm && !x) return fail(MOE_ERR_INVALID_ARG, "x_perm needs x");
  if (!aligned16(x) || !aligned16(x_perm))
    return fail(MOE_ERR_INVALID_ARG, "x and x_perm must be 16-byte aligned");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  CHECK_CUDA(launch_permute(s, L, static_cast<char*>(ws), x, topk_idx, counts, offsets,
                            scatter_index, row_token, x_perm, (cudaStream_t)stream));
  return MOE_OK;
}

static moe_status grouped(int mode, const moe_shape* shape, const void* A, const void* B0,
                          const void* B1, int64_t stride, const int32_t* offsets, int32_t G,
                          int64_t rows_bound, int32_t inter, void* out, void* ws,
                          size_t ws_bytes, void* stream, const int32_t* gather = nullptr) {
  reset_launch_count();
  DECODE(shape, s);
  if (G < 1 || (G > s.E && G != 1)) return fail(MOE_ERR_INVALID_ARG, "num_groups must be in [1, E]");
  if (!offsets) return fail(MOE_ERR_INVALID_ARG, "offsets must be non-NULL");
  if (inter <= 0 || inter % 8) return fail(MOE_ERR_INVALID_ARG, "inter must be a positive multiple of 8");
  if (rows_bound < 0 || rows_bound > 0x7fffffff) return fail(MOE_ERR_INVALID_ARG, "rows_bound out of range");
  if (stride < 0) return fail(MOE_ERR_INVALID_ARG, "expert_stride must be >= 0");
  if (G > 1 && stride == 0) return fail(MOE_ERR_INVALID_ARG, "expert_stride is 0 with several groups");
  if (rows_bound > 0 && (!A || !B0 || !out || (mode == kSwiGLU && !B1)))
    return fail(MOE_ERR_INVALID_ARG, "operand pointers must be non-NULL");
  const int wsize = s.wfmt ? 1 : s.esize;   // MXFP8: strides in bytes
  if (!aligned16(A) || !aligned16(B0) || !aligned16(B1) || !aligned16(out) || (stride * wsize) % 16)
    return fail(MOE_ERR_INVALID_ARG, "operands and expert_stride must be 16-byte aligned");
  if (s.wfmt && G > 1) {
    const int64_t n = mode == kSwiGLU ? inter : s.H, kk = mode == kSwiGLU ? s.H : inter;
    if (stride < n * kk / 8 * 9)
      return fail(MOE_ERR_INVALID_ARG, "MXFP8 expert_stride smaller than one packed matrix");
  }
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  char* w = static_cast<char*>(ws);
  GemmArgs a;
  a.mode = mode;
  a.dtype = s.dtype;
  a.A = A;
  a.B0 = B0;
  a.B1 = B1;
  a.bstride = stride;
  a.N = mode == kSwiGLU ? inter : s.H;
  a.K = mode == kSwiGLU ? s.H : inter;
  a.offsets = offsets;
  a.G = G;
  a.single_rows = 0;
  a.rows_bound = rows_bound;
  a.out = out;
  a.ldo = a.N;
  a.sched = reinterpret_cast<int32_t*>(w + (G > 1 ? L.sched_routed : L.sched_shared));
  a.ctr = reinterpret_cast<int32_t*>(w + L.tile_ctr + (G > 1 ? 0 : 128));
  if (G > 1 && G <= s.E) a.amaps = w + L.tmaps;
  a.flags = reinterpret_cast<uint32_t*>(w + L.flags);
  a.gather = gather;
  a.a_rows = s.T;
  a.wfmt = s.wfmt;
  CHECK_CUDA(launch_grouped_gemm(a, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_grouped_swiglu(const moe_shape* shape, const void* x_perm, const void* w_gate,
                              const void* w_up, int64_t expert_stride, const int32_t* offsets,
                              int32_t num_groups, int64_t rows_bound, int32_t inter, void* h,
                              void* ws, size_t ws_bytes, void* stream) {
  return grouped(kSwiGLU, shape, x_perm, w_gate, w_up, expert_stride, offsets, num_groups,
                 rows_bound, inter, h, ws, ws_bytes, stream);
}

moe_status moe_grouped_swiglu_gather(const moe_shape* shape, const void* x,
                                     const int32_t* row_token, const void* w_gate,
                                     const void* w_up, int64_t expert_stride,
                                     const int32_t* offsets, int32_t num_groups,
                                     int64_t rows_bound, int32_t inter, void* h, void* ws,
                                     size_t ws_bytes, void* stream) {
  if (rows_bound > 0 && !row_token) {
    reset_launch_count();
    return fail(MOE_ERR_INVALID_ARG, "row_token must be non-NULL");
  }
  return grouped(kSwiGLU, shape, x, w_gate, w_up, expert_stride, offsets, num_groups,
                 rows_bound, inter, h, ws, ws_bytes, stream, row_token);
}

moe_status moe_grouped_down(const moe_shape* shape, const void* h, const void* w_down,
                            int64_t expert_stride, const int32_t* offsets, int32_t num_groups,
                            int64_t rows_bound, int32_t inter, void* y_perm, void* ws,
                            size_t ws_bytes, void* stream) {
  return grouped(kStoreAct, shape, h, w_down, nullptr, expert_stride, offsets, num_groups,
                 rows_bound, inter, y_perm, ws, ws_bytes, stream);
}

moe_status moe_residual_setup(const moe_shape* shape, const void* x, const void* norm_weight,
                              void* x_norm, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (s.T > 0 && (!x || !norm_weight || !x_norm))
    return fail(MOE_ERR_INVALID_ARG, "x, norm_weight and x_norm must be non-NULL");
  if (!aligned16(x) || !aligned16(norm_weight) || !aligned16(x_norm))
    return fail(MOE_ERR_INVALID_ARG, "x, norm_weight and x_norm must be 16-byte aligned");
  CHECK_CUDA(launch_rmsnorm(s, x, norm_weight, s.norm_eps, x_norm, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_combine(const moe_shape* shape, const void* y_perm, const int32_t* scatter_index,
                       const float* topk_w, const void* shared_out, const float* gate,
                       const void* residual, void* y, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (s.T > 0 && (!y_perm || !scatter_index || !topk_w || !y))
    return fail(MOE_ERR_INVALID_ARG, "y_perm, scatter_index, topk_w and y must be non-NULL");
  if (!aligned16(y_perm) || !aligned16(shared_out) || !aligned16(residual) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "y_perm, shared_out, residual and y must be 16-byte aligned");
  CHECK_CUDA(launch_combine(s, y_perm, scatter_index, topk_w, shared_out, gate, residual, y,
                            (cudaStream_t)stream));
  return MOE_OK;
}

// During stream capture an event record must become an external event node
// of the graph (otherwise it only orders the capture and cannot be timed).
static cudaError_t record_stage_event(void* ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), st,
                                  cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                      : cudaEventRecordDefault);
}

moe_status moe_layer_forward(const moe_shape* shape, const moe_weights* W, const void* x,
                             const int32_t* routes_idx, const float* routes_w, void* y, void* ws,
                             size_t ws_bytes, void* stream) {
  return moe_layer_forward_traced(shape, W, x, routes_idx, routes_w, y, ws, ws_bytes, stream,
                                  nullptr);
}

moe_status moe_layer_forward_traced(const moe_shape* shape, const moe_weights* W, const void* x,
                                    const int32_t* routes_idx, const float* routes_w, void* y,
                                    void* ws, size_t ws_bytes, void* stream,
                                    void* const* ev) {
  reset_launch_count();
  DECODE(shape, s);
  if (!W) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  const bool direct = routes_idx != nullptr;
  if ((routes_idx == nullptr) != (routes_w == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "routes_idx and routes_w go together");
  if (!direct && !W->router) return fail(MOE_ERR_INVALID_ARG, "no router and no direct routes");
  if (direct && s.gate) return fail(MOE_ERR_INVALID_ARG, "shared_gate needs the router");
  if (!direct && s.k > s.E) return fail(MOE_ERR_INVALID_ARG, "top_k exceeds num_experts");
  if (s.T > 0 && (!x || !y || !W->gate || !W->up || !W->down))
    return fail(MOE_ERR_INVALID_ARG, "x, y and the expert weights must be non-NULL");
  if (s.I_sh && (!W->shared_gate_proj || !W->shared_up || !W->shared_down))
    return fail(MOE_ERR_INVALID_ARG, "shared_inter > 0 needs the three shared weights");
  if (!s.I_sh && (W->shared_gate_proj || W->shared_up || W->shared_down))
    return fail(MOE_ERR_INVALID_ARG, "shared weights given but shared_inter is 0");
  // MXFP8: packed matrices, strides in bytes
  const int64_t mat = (int64_t)s.I * s.H, wsz = s.wfmt ? 1 : s.esize;
  if (W->gate_up_stride < (s.wfmt ? mat / 8 * 9 : mat) || W->down_stride < (s.wfmt ? mat / 8 * 9 : mat))
    return fail(MOE_ERR_INVALID_ARG, "expert strides smaller than one expert matrix");
  if (s.input_norm && s.T > 0 && !W->norm_weight)
    return fail(MOE_ERR_INVALID_ARG, "input_norm needs weights->norm_weight");
  if (!s.input_norm && W->norm_weight)
    return fail(MOE_ERR_INVALID_ARG, "norm_weight given but input_norm is 0");
  if (!aligned16(W->norm_weight))
    return fail(MOE_ERR_INVALID_ARG, "norm_weight must be 16-byte aligned");
  if (!aligned16(x) || !aligned16(y) || !aligned16(W->router) || !aligned16(W->gate) ||
      !aligned16(W->up) || !aligned16(W->down) || !aligned16(W->shared_gate_proj) ||
      !aligned16(W->shared_up) || !aligned16(W->shared_down) ||
      (W->gate_up_stride * wsz) % 16 || (W->down_stride * wsz) % 16)
    return fail(MOE_ERR_INVALID_ARG, "tensors and strides must be 16-byte aligned");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.total);
  if (c != MOE_OK) return c;
  if (s.T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  char* w = static_cast<char*>(ws);
  uint32_t* flags = reinterpret_cast<uint32_t*>(w + L.flags);
  int32_t* idx = reinterpret_cast<int32_t*>(w + L.topk_idx);
  float* tw = reinterpret_cast<float*>(w + L.topk_w);
  float* gate = s.gate ? reinterpret_cast<float*>(w + L.gate) : nullptr;
  const int32_t* use_idx = idx;
  const float* use_w = tw;
#define STAGE_EVENT(i) \
  if (ev) CHECK_CUDA(record_stage_event(ev[i], st))
  // the activations the FFN sees: x, or its input RMSNorm
  STAGE_EVENT(MOE_STAGE_RESIDUAL_SETUP);
  const void* xin = x;
  if (s.input_norm) {
    CHECK_CUDA(launch_rmsnorm(s, x, W->norm_weight, s.norm_eps, w + L.x_norm, st));
    xin = w + L.x_norm;
  }
  // The shared MLP depends on xin alone, so it runs on a second stream,
  // forked here and joined before the combine, beside the routing, permute
  // and routed GEMMs.  At decode sizes those are short latency-bound launches
  // that leave HBM idle; at prefill sizes the HBM-bound stages (route,
  // permute) leave power and tensor cores for the shared MLP's GEMMs under
  // the power cap (graph replay, one box: Qwen2-MoE T = 2048 1180 -> 1112
  // us, DeepSeek-V3 shape 5910 -> 5877, adversarial T = 16384 -1 to -2 %).
  // (The traced entry point keeps one stream, so its stage events time each
  // stage alone.)
  void* sh_out = nullptr;
  int sh_split = 1;
  auto launch_shared = [&](cudaStream_t ss, int max_sms) -> cudaError_t {
    sh_out = w + L.sh_out;
    GemmArgs b;
    b.max_sms = max_sms;
    b.dtype = s.dtype;
    b.offsets = nullptr;
    b.G = 1;
    b.single_rows = s.T;
    b.rows_bound = s.T;
    b.sched = reinterpret_cast<int32_t*>(w + L.sched_shared);
    b.ctr = reinterpret_cast<int32_t*>(w + L.tile_ctr + 128);
    b.flags = flags;
    b.wfmt = s.wfmt;
    b.mode = kSwiGLU;
    b.A = xin;
    b.B0 = W->shared_gate_proj;
    b.B1 = W->shared_up;
    b.bstride = 0;
    b.N = s.I_sh;
    b.K = s.H;
    b.out = w + L.sh_h;
    b.ldo = s.I_sh;
    if (shared_split_ok(s)) {
      b.split_part = reinterpret_cast<float*>(w + L.gemm_split);
      b.split_ks = reinterpret_cast<int32_t*>(w + L.tile_ctr + 192);
    }
    cudaError_t e = launch_grouped_gemm(b, ss);
    if (e != cudaSuccess) return e;
    b.split_part = nullptr;
    b.split_ks = nullptr;
    b.mode = kStoreAct;
    b.A = w + L.sh_h;
    b.B0 = W->shared_down;
    b.B1 = nullptr;
    b.N = s.H;
    b.K = s.I_sh;
    b.out = sh_out;
    b.ldo = s.H;
    sh_split = shared_split(s, b);
    if (sh_split > 1) {
      b.mode = kStoreF32;
      b.ksplit = sh_split;
      b.split_stride = s.T * (int64_t)s.H;
    }
    return launch_grouped_gemm(b, ss);
  };
  const bool fork = s.I_sh && ev == nullptr;
  SideStream* side = nullptr;
  std::unique_lock<std::mutex> side_lock;
  if (fork) {
    CHECK_CUDA(side_stream(&side));
    side_lock = std::unique_lock<std::mutex>(side->mu);
    CHECK_CUDA(cudaEventRecord(side->fork, st));
    CHECK_CUDA(cudaStreamWaitEvent(side->stream, side->fork, 0));
    CHECK_CUDA(launch_shared(side->stream, fork_shared_sms(s.T)));
    CHECK_CUDA(cudaEventRecord(side->join, side->stream));
  }
  STAGE_EVENT(MOE_STAGE_ROUTE);
  if (direct) {
    use_idx = routes_idx;
    use_w = routes_w;
    if (s.train) {   // the backward reads the routes from the workspace
      CHECK_CUDA(cudaMemcpyAsync(idx, routes_idx, (size_t)s.T * s.k * 4, cudaMemcpyDeviceToDevice, st));
      CHECK_CUDA(cudaMemcpyAsync(tw, routes_w, (size_t)s.T * s.k * 4, cudaMemcpyDeviceToDevice, st));
    }
  } else {
    moe_status r = do_route(s, L, w, xin, W->router, idx, tw, gate, st);
    if (r != MOE_OK) return r;
  }
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* sidx = reinterpret_cast<int32_t*>(w + L.sidx);
  int32_t* row_token = reinterpret_cast<int32_t*>(w + L.row_token);
  void* x_perm = w + L.x_perm;
  void* h = w + L.h;
  void* y_perm = w + L.y_perm;
  STAGE_EVENT(MOE_STAGE_PERMUTE);
  // The grouped copy x_perm is written once here and read by the gate/up GEMM
  // through a TMA tensor map: at prefill sizes that is faster than gathering
  // the rows inside the GEMM (moe_grouped_swiglu_gather), whose cp.async
  // producers cannot keep the tensor cores fed.
  CHECK_CUDA(launch_permute(s, L, w, xin, use_idx, counts, offsets, sidx, row_token, x_perm, st));
  STAGE_EVENT(MOE_STAGE_GATE_UP);

  GemmArgs a;
  a.dtype = s.dtype;
  a.offsets = offsets;
  a.G = s.E;
  a.single_rows = 0;
  a.rows_bound = s.T * s.k;
  a.sched = reinterpret_cast<int32_t*>(w + L.sched_routed);
  a.ctr = reinterpret_cast<int32_t*>(w + L.tile_ctr);
  a.amaps = w + L.tmaps;
  a.flags = flags;
  a.wfmt = s.wfmt;
  a.mode = kSwiGLU;
  a.A = x_perm;
  a.B0 = W->gate;
  a.B1 = W->up;
  a.bstride = W->gate_up_stride;
  a.N = s.I;
  a.K = s.H;
  a.out = h;
  a.ldo = s.I;
  if (s.train) {   // the backward's SwiGLU derivative needs a and b
    a.pre = w + L.fc1;
    a.ldp = 2 * (int64_t)s.I;
  }
  CHECK_CUDA(launch_grouped_gemm(a, st));
  a.pre = nullptr;
  STAGE_EVENT(MOE_STAGE_DOWN);
  a.mode = kStoreAct;
  a.A = h;
  a.gather = nullptr;
  a.B0 = W->down;
  a.B1 = nullptr;
  a.bstride = W->down_stride;
  a.N = s.H;
  a.K = s.I;
  a.out = y_perm;
  a.ldo = s.H;
  CHECK_CUDA(launch_grouped_gemm(a, st));

  STAGE_EVENT(MOE_STAGE_SHARED);
  if (s.I_sh && !fork) CHECK_CUDA(launch_shared(st, 0));
  if (fork) CHECK_CUDA(cudaStreamWaitEvent(st, side->join, 0));
  STAGE_EVENT(MOE_STAGE_COMBINE);
  const void* resid = s.residual ? x : nullptr;
  if (sh_split > 1) {
    CHECK_CUDA(launch_combine(s, y_perm, sidx, use_w, nullptr, gate, resid, y, st,
                              static_cast<const float*>(sh_out), sh_split));
  } else {
    CHECK_CUDA(launch_combine(s, y_perm, sidx, use_w, sh_out, gate, resid, y, st));
  }
  STAGE_EVENT(MOE_NUM_STAGES);
#undef STAGE_EVENT
  return MOE_OK;
}

moe_status moe_get_route_stats(void* ws, void* stream, uint32_t* redecided) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (!redecided) return fail(MOE_ERR_INVALID_ARG, "redecided is NULL");
  CHECK_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  CHECK_CUDA(cudaMemcpy(redecided, static_cast<char*>(ws) + 4, 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemset(static_cast<char*>(ws) + 4, 0, 4));
  return MOE_OK;
}

moe_status moe_testing_router_logits(const moe_shape* shape, const void* x, const void* w_router,
                                     float* logits, void* ws, size_t ws_bytes, void* stream) {
  reset_launch_count();
  DECODE(shape, s);
  if (s.T > 0 && (!x || !w_router || !logits))
    return fail(MOE_ERR_INVALID_ARG, "x, w_router and logits must be non-NULL");
  const Layout L = layout_for(s);
  moe_status c = check_ws(ws, ws_bytes, L.scratch_end);
  if (c != MOE_OK) return c;
  if (s.T == 0) return MOE_OK;
  char* w = static_cast<char*>(ws);
  int nsplit = 1;
  moe_status r = router_gemm(s, L, w, x, w_router, &nsplit, (cudaStream_t)stream);
  if (r != MOE_OK) return r;
  CHECK_CUDA(launch_sum_partials(s, reinterpret_cast<float*>(w + L.logits), nsplit, logits,
                                 (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_get_device_status(void* ws, void* stream, uint32_t* bits) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  CHECK_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  uint32_t v = 0;
  CHECK_CUDA(cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemset(ws, 0, sizeof(v)));
  if (bits) *bits = v;
  if (v & kFlagRoute) return MOE_ERR_DEVICE_ROUTE;
  if (v & kFlagRows) return MOE_ERR_ROWS;
  if (v & kFlagTimeout) return MOE_ERR_TIMEOUT;
  if (v & kFlagGather) return MOE_ERR_GATHER;
  return MOE_OK;
}

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_ROUTE: return "MOE_ERR_DEVICE_ROUTE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_ROWS: return "MOE_ERR_ROWS";
    case MOE_ERR_GATHER: return "MOE_ERR_GATHER";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error(void) { return tl_error; }

const char* moe_stage_name(int32_t stage) {
  static const char* names[MOE_NUM_STAGES] = {"residual_setup", "route", "permute", "gate_up",
                                              "down", "shared", "combine"};
  if (stage < 0 || stage >= MOE_NUM_STAGES) return "";
  return names[stage];
}

int32_t moe_last_launch_count(void) { return tl_launches; }

int32_t moe_testing_set_gemm_engine(int32_t engine) {
  if (engine < 0 || engine > 4) engine = 0;
  return g_engine.exchange(engine);
}

int32_t moe_testing_set_zero_pad(int32_t mode) {
  if (mode < -1 || mode > 1) mode = 0;
  return g_zero_pad.exchange(mode);
}

int32_t moe_testing_set_fork_sms(int32_t sms) {
  if (sms < -1) sms = 0;
  return g_fork_sms.exchange(sms);
}

}  // extern "C"
