// route.cu -- top-k softmax over router logits.
//
// "MoE: timing-replay harnesses, shared experts, parameterized V_TOPK routing"
// (C_SET_TOPK_REG section): topk_softmax is generic in (num_experts, top_k),
// so this kernel takes any E <= 16383 and k <= 255 from the packed shape word.
//
//   selection  the k largest logits, equal values resolved to the lower
//              expert index; slot s = (s+1)-th largest.  One warp per token:
//              for k + 1 <= 32 and at most 512 router columns the logits sit
//              in registers and each of the k+1 rounds is one warp
//              max-reduction of order-preserving integer keys plus one
//              min-reduction of the expert index; otherwise the rounds run
//              over shared memory with a shuffle arg-max;
//   weights    norm_topk: exp(l_s - l_max) / sum over the k selected;
//              otherwise: exp(l_s - l_max) / sum over all E;
//   gate       Qwen2-MoE shared gate sigmoid(z), z = logit column E
//              ("MoE: shared experts, arbitrary V_TOPK expert shapes, ...",
//              Group C).
//
// Near ties.  The logits arrive in fp32 (tensor-core or FMA sums), within a
// small error of the exact dot products.  When two neighbours of the sorted
// top-(k+1) list are closer than a bound tau well above that error, the
// experts within tau of the boundary are re-evaluated with an error-free
// compensated dot product (Ogita, Rump and Oishi, "Accurate Sum and Dot
// Product", SIAM J. Sci. Comput. 26(6), 2005: algorithm Dot2) and the
// selection among them is redone on those values.  The decision then matches
// exact arithmetic except for true near-ties far below the fp32 error.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxRounds = 256;  // k <= 255 plus one round for the boundary
constexpr int kMaxCand = 64;     // experts re-evaluated in a near tie
struct TopkArgs {
  const float* logits;  // nsplit partial sums, split_stride floats apart
  int ldl;
  int nsplit;
  int64_t split_stride;
  const void* x;
  const void* w;  // router [ncols, H]
  int H, E, k, norm, gated;
  int64_t T;
  float tau_scale;
  int32_t* idx;
  float* wout;
  float* gate;
  uint32_t* redecided;  // count of tokens whose order was re-decided exactly
};

struct WarpSmem {
  float* buf;        // [E] logits of this token
  uint32_t* taken;   // [ceil(E/32)]
  int* sel_i;        // [kMaxRounds]
  float* sel_v;      // [kMaxRounds]
  int* cand_i;       // [kMaxCand]
  float* cand_f;     // [kMaxCand] fp32 logits of the candidates
  float2* cand_v;    // [kMaxCand] exact values as (hi, lo) float pairs
};

__host__ __device__ inline size_t warp_smem_bytes(int E) {
  size_t b = 0;
  b += (size_t)kMaxCand * 8;            // cand_v (first: 8-byte aligned)
  b += (size_t)E * 4;                   // buf
  b += (size_t)((E + 31) / 32) * 4;     // taken
  b += (size_t)kMaxRounds * 8;          // sel_i + sel_v
  b += (size_t)kMaxCand * 8;            // cand_i + cand_f
  return (b + 15) & ~(size_t)15;
}

__device__ __forceinline__ WarpSmem warp_smem(unsigned char* base, int E) {
  WarpSmem sm;
  sm.cand_v = reinterpret_cast<float2*>(base);
  sm.buf = reinterpret_cast<float*>(base + kMaxCand * 8);
  sm.taken = reinterpret_cast<uint32_t*>(sm.buf + E);
  sm.sel_i = reinterpret_cast<int*>(sm.taken + (E + 31) / 32);
  sm.sel_v = reinterpret_cast<float*>(sm.sel_i + kMaxRounds);
  sm.cand_i = reinterpret_cast<int*>(sm.sel_v + kMaxRounds);
  sm.cand_f = reinterpret_cast<float*>(sm.cand_i + kMaxCand);
  return sm;
}

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Exact values are unevaluated pairs hi + lo with |lo| <= ulp(hi)/2, so the
// lexicographic order of (hi, lo) is the order of the values.
__device__ __forceinline__ bool better2(float2 a, int ia, float2 b, int ib) {
  return a.x > b.x || (a.x == b.x && (a.y > b.y || (a.y == b.y && ia < ib)));
}

// Warp arg-max of (v, i); every lane receives the winner.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float z = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = __fmul_rn(a, b);
  e = __fmaf_rn(a, b, -p);
}

// Dot2 of row x and router row w over H, cooperatively by the warp: each lane
// streams 16-byte chunks and keeps one (sum, compensation) pair per vector
// position, so the dependent chains are short and loads stay in flight; the
// pairs are merged with TwoSum across positions and then across lanes, and
// the result is returned as a normalised pair (hi, lo).
template <typename T>
__device__ float2 dot2(const T* x, const T* w, int H, int lane) {
  constexpr int V = 16 / sizeof(T);
  float p[V], s[V];
#pragma unroll
  for (int i = 0; i < V; ++i) p[i] = s[i] = 0.f;
  const int nv = H / V;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const uint4* wv = reinterpret_cast<const uint4*>(w);
#pragma unroll 4
  for (int c = lane; c < nv; c += 32) {
    float xf[V], wf[V];
    unpack16(__ldg(xv + c), xf, (const T*)nullptr);
    unpack16(__ldg(wv + c), wf, (const T*)nullptr);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float hp, r, q;
      two_prod(xf[i], wf[i], hp, r);
      two_sum(p[i], hp, p[i], q);
      s[i] = __fadd_rn(s[i], __fadd_rn(q, r));
    }
  }
  float P = p[0], S = s[0];
#pragma unroll
  for (int i = 1; i < V; ++i) {
    float q;
    two_sum(P, p[i], P, q);
    S = __fadd_rn(S, __fadd_rn(s[i], q));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float op = __shfl_xor_sync(0xffffffffu, P, o);
    float os = __shfl_xor_sync(0xffffffffu, S, o);
    float q;
    two_sum(P, op, P, q);
    S = __fadd_rn(__fadd_rn(S, os), q);
  }
  float hi, lo;
  two_sum(P, S, hi, lo);
  return make_float2(hi, lo);
}

__device__ __forceinline__ float tie_bound(const TopkArgs& a, float top, float boundary) {
  return a.tau_scale * (fabsf(top) + fabsf(boundary) + 1.0f);
}

// Near-tie re-decision of one token, in three steps.  sm.buf holds the E
// fp32 logits and sm.sel_i / sm.sel_v the fp32 order of the top R; vb is the
// boundary value sel_v[R-1] and tau the tie bound.
//
// 1. tie_candidates (one warp): L = every expert within tau below vb (so all
//    of the top R, plus the ones just under it) into sm.cand_i / sm.cand_v.
//    Only members of L closer than tau to another member can swap places;
//    they are marked for exact evaluation, the rest keep their fp32 value
//    (every comparison they take part in is decided by a margin of at least
//    tau).  Returns |L|; above kMaxCand the fp32 order stands.
// 2. the marked members get their exact dot product (Dot2) into sm.cand_v;
// 3. tie_reselect (one warp) redoes the R rounds among L on those keys: every
//    expert outside L lies more than tau below the boundary, so the top R are
//    all in L.  sel_v keeps the fp32 logits of the chosen experts.
__device__ int tie_candidates(const TopkArgs& a, const WarpSmem& sm, int lane, float vb,
                              float tau, unsigned long long& marked) {
  const int E = a.E;
  int nc = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    int e = e0 + lane;
    bool c = e < E && sm.buf[e] >= vb - tau;
    unsigned msk = __ballot_sync(0xffffffffu, c);
    int pos = nc + __popc(msk & ((1u << lane) - 1u));
    if (c && pos < kMaxCand) sm.cand_i[pos] = e;
    nc += __popc(msk);
  }
  __syncwarp();
  marked = 0ull;
  if (nc > kMaxCand) return nc;
  for (int c = lane; c < nc; c += 32) {
    const float vc = sm.buf[sm.cand_i[c]];
    bool mk = false;
    for (int o = 0; o < nc; ++o) mk |= (o != c) && fabsf(vc - sm.buf[sm.cand_i[o]]) < tau;
    sm.cand_f[c] = vc;
    sm.cand_v[c] = make_float2(vc, 0.f);
    if (mk) marked |= 1ull << c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) marked |= __shfl_xor_sync(0xffffffffu, marked, o);
  __syncwarp();
  return nc;
}

template <typename T>
__device__ __forceinline__ void tie_exact(const TopkArgs& a, const WarpSmem& sm, int64_t t,
                                          int c, int lane) {
  const T* xr = reinterpret_cast<const T*>(a.x) + t * a.H;
  const T* wr = reinterpret_cast<const T*>(a.w) + (int64_t)sm.cand_i[c] * a.H;
  const float2 v = dot2<T>(xr, wr, a.H, lane);
  if (lane == 0) sm.cand_v[c] = v;
}

__device__ void tie_reselect(const WarpSmem& sm, int lane, int R, int nc) {
  unsigned long long used = 0ull;
  for (int r = 0; r < R && r < nc; ++r) {
    float2 bv2 = make_float2(-INFINITY, 0.f);
    int bi2 = 0x7fffffff, bc = -1;
    for (int c = lane; c < nc; c += 32) {
      if (used & (1ull << c)) continue;
      const float2 v = sm.cand_v[c];
      const int e = sm.cand_i[c];
      if (bc < 0 || better2(v, e, bv2, bi2)) { bv2 = v; bi2 = e; bc = c; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float2 ov;
      ov.x = __shfl_xor_sync(0xffffffffu, bv2.x, o);
      ov.y = __shfl_xor_sync(0xffffffffu, bv2.y, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi2, o);
      const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
      const bool take = oc >= 0 && (bc < 0 || better2(ov, oi, bv2, bi2));
      if (take) { bv2 = ov; bi2 = oi; bc = oc; }
    }
    if (bc < 0) break;
    used |= 1ull << bc;
    if (lane == 0) {
      sm.sel_i[r] = bi2;
      sm.sel_v[r] = sm.cand_f[bc];
    }
    __syncwarp();
  }
}

// All three steps by one warp.
template <typename T>
__device__ void redecide(const TopkArgs& a, const WarpSmem& sm, int64_t t, int lane, int R,
                         float vb, float tau) {
  unsigned long long marked;
  const int nc = tie_candidates(a, sm, lane, vb, tau, marked);
  if (nc > kMaxCand) return;
  for (unsigned long long mm = marked; mm; mm &= mm - 1)
    tie_exact<T>(a, sm, t, __ffsll((long long)mm) - 1, lane);
  __syncwarp();
  tie_reselect(sm, lane, R, nc);
}

// One token, one warp, any shape (k + 1 > 32 or more than 512 router
// columns): selection rounds over shared memory, then the near-tie
// re-decision, the weights and the gate.
template <typename T>
__device__ void warp_token(const TopkArgs& a, const WarpSmem& sm, int64_t t, int lane) {
  const int E = a.E, k = a.k;
  const int R = k < E ? k + 1 : k;
  const float* row = a.logits + t * a.ldl;
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32) {
    float v = row[e];
    for (int sp = 1; sp < a.nsplit; ++sp) v += row[sp * a.split_stride + e];
    sm.buf[e] = v;
    m = fmaxf(m, v);
  }
  for (int w = lane; w < (E + 31) / 32; w += 32) sm.taken[w] = 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __syncwarp();
  for (int r = 0; r < R; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      if (sm.taken[e >> 5] & (1u << (e & 31))) continue;
      float v = sm.buf[e];
      if (bi == 0x7fffffff || better(v, e, bv, bi)) { bv = v; bi = e; }
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      sm.sel_i[r] = bi;
      sm.sel_v[r] = bv;
      sm.taken[bi >> 5] |= 1u << (bi & 31);
    }
    __syncwarp();
  }

  const float vb = sm.sel_v[R - 1];
  const float tau = tie_bound(a, sm.sel_v[0], vb);
  bool near = false;
  for (int r = lane; r + 1 < R; r += 32) near |= (sm.sel_v[r] - sm.sel_v[r + 1]) < tau;
  near = __any_sync(0xffffffffu, near);
  if (near && a.x != nullptr) {
    if (lane == 0 && a.redecided) atomicAdd(a.redecided, 1u);
    redecide<T>(a, sm, t, lane, R, vb, tau);
    __syncwarp();
  }

  float denom = 0.f;
  if (a.norm) {
    const float top = sm.sel_v[0];
    for (int s = lane; s < k; s += 32) denom += expf(sm.sel_v[s] - top);
  } else {
    for (int e = lane; e < E; e += 32) denom += expf(sm.buf[e] - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, o);
  const float ref = a.norm ? sm.sel_v[0] : m;
  for (int s = lane; s < k; s += 32) {
    a.idx[t * k + s] = sm.sel_i[s];
    a.wout[t * k + s] = expf(sm.sel_v[s] - ref) / denom;
  }
  if (a.gated && lane == 0) {
    float z = row[E];
    for (int sp = 1; sp < a.nsplit; ++sp) z += row[sp * a.split_stride + E];
    a.gate[t] = 1.0f / (1.0f + expf(-z));
  }
  __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(128) topk_warp_kernel(TopkArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const WarpSmem sm = warp_smem(smem_raw + warp_smem_bytes(a.E) * wid, a.E);
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + wid;
  if (t >= a.T) return;
  warp_token<T>(a, sm, t, lane);
}

// Order-preserving key of a logit: the unsigned order of keys is the numeric
// order of the values.  -0 is folded into +0 first so that equal values get
// equal keys.  Key 0 (reached by one NaN bit pattern only) marks a slot that
// is taken or outside [0, E).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Exact values of the marked candidates of a block's near-tie tokens.  Pair p
// = (warp pw[p], candidate pc[p]) of that warp's token.  Warp q of the block
// takes quarter q of the hidden dimension for every pair, two pairs at a
// time, so each lane keeps 8 loads of 16 bytes in flight; per pair a lane
// accumulates its products with TwoProduct / TwoSum into one (sum,
// compensation) pair, the lanes are merged with TwoSum, and the quarter's
// result goes to part[p][q].  The caller adds the four quarters in order.
constexpr int kPairs = 2;   // pairs a warp evaluates side by side

template <typename T>
__device__ void block_exact(const TopkArgs& a, const unsigned char* smem_raw, size_t per_warp,
                            int np, const uint8_t* pw, const uint8_t* pc, float2 (*part)[4],
                            int lane, int wid) {
  constexpr int V = 16 / sizeof(T);
  const int nv = a.H / V;   // 16-byte chunks in a row
  const int c0 = (int)((int64_t)nv * wid / 4), c1 = (int)((int64_t)nv * (wid + 1) / 4);
  const uint4* xb = reinterpret_cast<const uint4*>(a.x);
  const uint4* wb = reinterpret_cast<const uint4*>(a.w);
  for (int pb = 0; pb < np; pb += kPairs) {
    const uint4* xr[kPairs];
    const uint4* wr[kPairs];
    bool on[kPairs];
#pragma unroll
    for (int b = 0; b < kPairs; ++b) {
      const int p = pb + b;
      on[b] = p < np;
      const int w = on[b] ? pw[p] : 0;
      const WarpSmem smw = warp_smem(const_cast<unsigned char*>(smem_raw) + per_warp * w, a.E);
      const int e = on[b] ? smw.cand_i[pc[p]] : 0;
      xr[b] = xb + ((int64_t)blockIdx.x * 4 + w) * nv;
      wr[b] = wb + (int64_t)e * nv;
    }
    float P[kPairs], S[kPairs];
#pragma unroll
    for (int b = 0; b < kPairs; ++b) P[b] = S[b] = 0.f;
    for (int c = c0 + lane; c < c1; c += 64) {
      const bool second = c + 32 < c1;
      uint4 xv[kPairs][2], wv[kPairs][2];
#pragma unroll
      for (int b = 0; b < kPairs; ++b) {
        if (on[b]) {
          xv[b][0] = __ldg(xr[b] + c);
          wv[b][0] = __ldg(wr[b] + c);
          if (second) {
            xv[b][1] = __ldg(xr[b] + c + 32);
            wv[b][1] = __ldg(wr[b] + c + 32);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kPairs; ++b) {
        if (!on[b]) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !second) break;
          float xf[V], wf[V];
          unpack16(xv[b][h], xf, (const T*)nullptr);
          unpack16(wv[b][h], wf, (const T*)nullptr);
#pragma unroll
          for (int i = 0; i < V; ++i) {
            float hp, r, q;
            two_prod(xf[i], wf[i], hp, r);
            two_sum(P[b], hp, P[b], q);
            S[b] = __fadd_rn(S[b], __fadd_rn(q, r));
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kPairs; ++b) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float op = __shfl_xor_sync(0xffffffffu, P[b], o);
        const float os = __shfl_xor_sync(0xffffffffu, S[b], o);
        float q;
        two_sum(P[b], op, P[b], q);
        S[b] = __fadd_rn(__fadd_rn(S[b], os), q);
      }
      if (lane == 0 && on[b]) part[pb + b][wid] = make_float2(P[b], S[b]);
    }
  }
}

// One warp per token for k + 1 <= 32 and at most 128 J router columns.  Lane
// l holds columns 128 j + 4 l + c (c < 4) of every chunk j < J, read as
// 16-byte loads of each split-K partial sum and added in split order.  Round
// r takes the largest remaining key (warp max-reduction) and the lowest
// expert index that holds it (warp min-reduction); lane r keeps the r-th
// choice.  Tokens whose top-R list has two neighbours closer than the tie
// bound are re-decided in shared memory: the exact values of all marked
// candidates of the block are computed by its four warps together
// (block_exact), then each such token redoes its rounds on them.
template <typename T, int J>
__global__ void __launch_bounds__(128, 6) topk_fast_kernel(TopkArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ unsigned long long s_marked[4];
  __shared__ uint8_t s_pw[4 * kMaxCand], s_pc[4 * kMaxCand];
  __shared__ float2 s_part[4 * kMaxCand][4];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t t = (int64_t)blockIdx.x * 4 + wid;
  const bool live = t < a.T;
  const int E = a.E, k = a.k;
  const int R = k < E ? k + 1 : k;
  const float* row = a.logits + (live ? t : 0) * a.ldl;
  float v[J][4];
#pragma unroll
  for (int sp = 0; sp < kMaxSplit; ++sp) {
    if (sp < a.nsplit) {
      const float* src = row + sp * a.split_stride;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e0 = 128 * j + 4 * lane;
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && e0 < a.ldl) q = __ldg(reinterpret_cast<const float4*>(src + e0));
        if (sp == 0) {
          v[j][0] = q.x; v[j][1] = q.y; v[j][2] = q.z; v[j][3] = q.w;
        } else {
          v[j][0] += q.x; v[j][1] += q.y; v[j][2] += q.z; v[j][3] += q.w;
        }
      }
    }
  }
  if (live && a.gated) {
    // column E (the shared gate's logit) lies in one lane's registers
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (128 * j + 4 * lane + c == E) a.gate[t] = 1.0f / (1.0f + expf(-v[j][c]));
  }
  uint32_t key[J][4];
#pragma unroll
  for (int j = 0; j < J; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) key[j][c] = 128 * j + 4 * lane + c < E ? order_key(v[j][c]) : 0u;
  float my_v = -INFINITY;
  int my_i = 0x7fffffff;
  for (int r = 0; r < R; ++r) {
    uint32_t lk = 0u;
    int li = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (key[j][c] > lk) { lk = key[j][c]; li = 128 * j + 4 * lane + c; }
    const uint32_t mk = __reduce_max_sync(0xffffffffu, lk);
    const int wi = (int)__reduce_min_sync(0xffffffffu, lk == mk ? (uint32_t)li : 0xffffffffu);
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (128 * j + 4 * lane + c == wi) key[j][c] = 0u;
    if (lane == r) {
      my_v = key_value(mk);
      my_i = wi;
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_v, 0);   // the largest fp32 logit
  const float vb = __shfl_sync(0xffffffffu, my_v, R - 1);
  const float tau = tie_bound(a, m, vb);
  const float nxt = __shfl_down_sync(0xffffffffu, my_v, 1);
  const bool near = live && a.x != nullptr &&
                    __any_sync(0xffffffffu, lane + 1 < R && my_v - nxt < tau);
  const size_t per_warp = warp_smem_bytes(E);
  const WarpSmem sm = warp_smem(smem_raw + per_warp * wid, E);
  int nc = 0;
  unsigned long long marked = 0ull;
  if (near) {
    if (lane == 0 && a.redecided) atomicAdd(a.redecided, 1u);
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = 128 * j + 4 * lane + c;
        if (e < E) sm.buf[e] = v[j][c];
      }
    if (lane < R) {
      sm.sel_i[lane] = my_i;
      sm.sel_v[lane] = my_v;
    }
    __syncwarp();
    nc = tie_candidates(a, sm, lane, vb, tau, marked);
  }
  if (lane == 0) s_marked[wid] = marked;
  if (__syncthreads_or(near)) {
    // the block's pair list: warp 0's marked candidates, then warp 1's, ...
    int base = 0, np = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int cnt = __popcll(s_marked[w]);
      if (w < wid) base += cnt;
      np += cnt;
    }
    for (int c = lane; c < kMaxCand; c += 32) {
      if (marked & (1ull << c)) {
        const int p = base + __popcll(marked & ((1ull << c) - 1ull));
        s_pw[p] = (uint8_t)wid;
        s_pc[p] = (uint8_t)c;
      }
    }
    __syncthreads();
    block_exact<T>(a, smem_raw, per_warp, np, s_pw, s_pc, s_part, lane, wid);
    __syncthreads();
    if (near && nc <= kMaxCand) {
      for (int c = lane; c < nc; c += 32) {
        if (marked & (1ull << c)) {
          const int p = base + __popcll(marked & ((1ull << c) - 1ull));
          float P = s_part[p][0].x, Sc = s_part[p][0].y;
#pragma unroll
          for (int q = 1; q < 4; ++q) {
            float qq;
            two_sum(P, s_part[p][q].x, P, qq);
            Sc = __fadd_rn(__fadd_rn(Sc, s_part[p][q].y), qq);
          }
          float hi, lo;
          two_sum(P, Sc, hi, lo);
          sm.cand_v[c] = make_float2(hi, lo);
        }
      }
      __syncwarp();
      tie_reselect(sm, lane, R, nc);
      __syncwarp();
      if (lane < R) {
        my_i = sm.sel_i[lane];
        my_v = sm.sel_v[lane];
      }
    }
  }
  if (!live) return;
  // weights: norm_topk over the k chosen (reference: the top chosen value),
  // otherwise the full softmax (reference: the largest logit)
  const float ref = a.norm ? __shfl_sync(0xffffffffu, my_v, 0) : m;
  float denom = 0.f;
  if (a.norm) {
    if (lane < k) denom = expf(my_v - ref);
  } else {
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (128 * j + 4 * lane + c < E) denom += expf(v[j][c] - ref);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, o);
  if (lane < k) {
    a.idx[t * k + lane] = my_i;
    a.wout[t * k + lane] = expf(my_v - ref) / denom;
  }
}

template <typename T>
cudaError_t launch_warp(const TopkArgs& a, size_t smem, cudaStream_t st) {
  if (smem * 4 > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_warp_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(smem * 4));
    if (e != cudaSuccess) return e;
  }
  topk_warp_kernel<T><<<(unsigned)((a.T + 3) / 4), 128, smem * 4, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int J>
cudaError_t launch_fast_t(const TopkArgs& a, size_t smem, cudaStream_t st) {
  topk_fast_kernel<T, J><<<(unsigned)((a.T + 3) / 4), 128, smem * 4, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fast(const TopkArgs& a, int J, size_t smem, cudaStream_t st) {
  switch (J) {
    case 1: return launch_fast_t<T, 1>(a, smem, st);
    case 2: return launch_fast_t<T, 2>(a, smem, st);
    case 3: return launch_fast_t<T, 3>(a, smem, st);
    default: return launch_fast_t<T, 4>(a, smem, st);
  }
}

}  // namespace

cudaError_t launch_topk(const Shape& s, const float* logits, int nsplit, const void* x,
                        const void* w_router, int32_t* topk_idx, float* topk_w, float* gate,
                        uint32_t* redecided, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  if (nsplit < 1 || nsplit > kMaxSplit) return cudaErrorInvalidValue;
  TopkArgs a;
  a.logits = logits;
  a.ldl = s.ldl;
  a.nsplit = nsplit;
  a.split_stride = s.T * (int64_t)s.ldl;
  a.x = x;
  a.w = w_router;
  a.H = s.H;
  a.E = s.E;
  a.k = s.k;
  a.norm = s.norm;
  a.gated = s.gate;
  a.T = s.T;
  // tau = 2^-20 * sqrt(H) * (|l_top| + |l_boundary| + 1): measured fp32 logit
  // errors at the benchmark shapes stay below a tenth of its smallest value.
  a.tau_scale = (float)(ldexp(1.0, -20) * sqrt((double)s.H));
  a.idx = topk_idx;
  a.wout = topk_w;
  a.gate = gate;
  a.redecided = redecided;
  const int R = s.k < s.E ? s.k + 1 : s.k;
  const size_t per_warp = warp_smem_bytes(s.E);
  cudaError_t e;
  if (R <= 32 && s.ldl <= 512) {   // ldl: router columns rounded up to 4
    const int J = (s.ldl + 127) / 128;
    e = s.dtype == MOE_F32 ? launch_fast<float>(a, J, per_warp, st)
                           : launch_fast<bf16>(a, J, per_warp, st);
  } else {
    e = s.dtype == MOE_F32 ? launch_warp<float>(a, per_warp, st)
                           : launch_warp<bf16>(a, per_warp, st);
  }
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaSuccess;
}

namespace {
// Sum of the split-K partial logits, in split order (the same sum the top-k
// kernel forms), into a caller buffer [T, ncols].
__global__ void sum_partials_kernel(const float* __restrict__ part, int nsplit,
                                    int64_t split_stride, int64_t T, int ncols, int ldl,
                                    float* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < T * ncols;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / ncols;
    const int c = (int)(i % ncols);
    float v = part[t * ldl + c];
    for (int sp = 1; sp < nsplit; ++sp) v += part[sp * split_stride + t * ldl + c];
    out[i] = v;
  }
}
}  // namespace

namespace {
// Hash-MoE lookup ("Fused MoE Kernel Notes", Duplicate top-k routes): slot s
// of token t goes to table[token_ids[t], s]; every slot weighs 1/k (one
// correctly rounded fp32 division).  A token id outside the table sends its
// slots to route -1, which the permutation drops, and raises the route flag.
__global__ void hash_route_kernel(const int32_t* __restrict__ token_ids,
                                  const int32_t* __restrict__ table, int64_t vocab, int64_t T,
                                  int k, int32_t* __restrict__ idx, float* __restrict__ w,
                                  uint32_t* flags) {
  const float wk = __fdiv_rn(1.0f, (float)k);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < T * k;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / k;
    const int sl = (int)(i - t * k);
    const int64_t tok = token_ids[t];
    int32_t e = -1;
    if (tok >= 0 && tok < vocab) {
      e = table[tok * k + sl];
    } else if (sl == 0) {
      set_flag(flags, kFlagRoute);
    }
    idx[i] = e;
    w[i] = wk;
  }
}
}  // namespace

cudaError_t launch_hash_route(const Shape& s, const int32_t* token_ids, const int32_t* table,
                              int64_t vocab, int32_t* idx, float* w, uint32_t* flags,
                              cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const int64_t n = s.T * s.k;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  hash_route_kernel<<<blocks, 256, 0, st>>>(token_ids, table, vocab, s.T, s.k, idx, w, flags);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_sum_partials(const Shape& s, const float* logits, int nsplit, float* out,
                                cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const int64_t n = s.T * s.ncols;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  sum_partials_kernel<<<blocks, 256, 0, st>>>(logits, nsplit, s.T * (int64_t)s.ldl, s.T, s.ncols,
                                              s.ldl, out);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
