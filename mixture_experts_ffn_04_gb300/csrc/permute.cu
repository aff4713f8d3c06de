// permute.cu -- expert histogram, group offsets, scatter_index and the
// expert-grouped copy of the activations.
//
// "Fused MoE Kernel Notes", Scatter/gather layout: tokens are expanded by
// their top-k routes into an expert-grouped [tokens * topk, hidden] buffer and
// scatter_index maps each (token, slot) to its row there.  Rows of one expert
// keep row-major (token, slot) order, so the result is deterministic and a
// duplicate route (two slots of one token on one expert) simply adds a row.
//
// Three launches, no global atomics (rank, scan, scatter + copy; see each
// kernel below).
#include <atomic>
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// 1. rank: one warp per chunk of `tpc` tokens walks the chunk's (token, slot)
//    pairs in row-major order, 32 at a time; __match_any_sync groups the
//    lanes that route to the same expert, so each pair gets its rank among the
//    chunk's earlier pairs of that expert.  The rank is parked in
//    scatter_index (overwritten by step 3) and the chunk's per-expert count
//    goes to hist[chunk][e].
__global__ void __launch_bounds__(256) rank_kernel(const int32_t* __restrict__ idx, int64_t T,
                                                   int k, int E, int tpc, int nchunks,
                                                   int32_t* __restrict__ hist,
                                                   int32_t* __restrict__ local_rank,
                                                   uint32_t* flags) {
  extern __shared__ int32_t sm[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int c = blockIdx.x * (blockDim.x >> 5) + wid;
  if (c >= nchunks) return;
  int32_t* cnt = sm + (size_t)wid * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int64_t p0 = (int64_t)c * tpc * k;
  const int64_t p1 = min(T, (int64_t)(c + 1) * tpc) * k;
  constexpr int kBatch = 8;   // rounds of 32 pairs whose expert ids are loaded together
  for (int64_t pb = p0; pb < p1; pb += 32 * kBatch) {
    int ids[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t p = pb + 32 * b + lane;
      ids[b] = p < p1 ? idx[p] : -1;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t p = pb + 32 * b + lane;
      const bool valid = p < p1;
      const int e = ids[b];
      const bool ok = valid && e >= 0 && e < E;
      if (valid && !ok) set_flag(flags, kFlagRoute);
      const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int r = -1;
      if (ok) r = cnt[e] + rank;
      __syncwarp();
      if (ok && rank == 0) cnt[e] += __popc(peers);
      __syncwarp();
      if (valid) local_rank[p] = r;
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[(int64_t)c * E + e] = cnt[e];
}

// 2. scan: block b takes experts [32 b, 32 b + 32) (lane = expert, so every
//    load of a chunk's row of hist is one 128-byte line) and its 32 warps
//    split the chunks into 32 ranges.  The warps' column sums, their
//    exclusive prefix over the warps in shared memory, and a second pass over
//    the warp's chunks give base[chunk][e] = rows of e in earlier chunks;
//    counts[e] is the column total.  The experts' group offsets are added by
//    the scatter (each of its blocks scans the E counts), so no step here
//    waits for all experts.  T = 0 (no chunks): counts and offsets are zero.
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ hist, int nchunks,
                                                    int E, int32_t* __restrict__ base,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets) {
  __shared__ int32_t tot[32][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int c0 = (int)((int64_t)nchunks * w / 32), c1 = (int)((int64_t)nchunks * (w + 1) / 32);
  int32_t sum = 0;
  if (e < E) {
#pragma unroll 8
    for (int c = c0; c < c1; ++c) sum += hist[(int64_t)c * E + e];
  }
  tot[w][lane] = sum;
  __syncthreads();
  if (w == 0) {
    int32_t run = 0;
    for (int i = 0; i < 32; ++i) {
      const int32_t v = tot[i][lane];
      tot[i][lane] = run;
      run += v;
    }
    if (e < E) {
      counts[e] = run;
      if (nchunks == 0) offsets[e] = 0;
    }
    if (nchunks == 0 && e == E - 1) offsets[E] = 0;
  }
  __syncthreads();
  if (e < E) {
    int32_t run = tot[w][lane];
#pragma unroll 8
    for (int c = c0; c < c1; ++c) {
      const int64_t at = (int64_t)c * E + e;
      const int32_t v = hist[at];
      base[at] = run;
      run += v;
    }
  }
}

// Group offsets of the E experts in shared memory (off[E + 1], exclusive
// prefix of counts), by all threads of the block: each thread takes a run of
// consecutive experts, then the runs' totals are scanned across the block.
// Block 0 also writes them to `offsets`.
__device__ void block_offsets(const int32_t* __restrict__ counts, int E, int32_t* off,
                              int32_t* wsum, int32_t* __restrict__ offsets) {
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5, nw = blockDim.x >> 5;
  const int per = (E + blockDim.x - 1) / blockDim.x;
  int32_t loc = 0;
  for (int i = 0; i < per; ++i) {
    const int e = t * per + i;
    if (e < E) {
      const int32_t v = counts[e];
      off[e] = loc;
      loc += v;
    }
  }
  int32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int32_t v = lane < nw ? wsum[lane] : 0;
    int32_t wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    if (lane < nw) wsum[lane] = wi - v;
  }
  __syncthreads();
  const int32_t add = wsum[wid] + incl - loc;
  for (int i = 0; i < per; ++i) {
    const int e = t * per + i;
    if (e < E) off[e] += add;
  }
  if (t == blockDim.x - 1) off[E] = add + loc;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = t; e <= E; e += blockDim.x) offsets[e] = off[e];
}

// 3. scatter + copy: one warp per token (grid-stride).  The warp turns the k
//    local ranks into grouped rows (scatter_index, row_token), then copies the
//    token's row once from x to each of its rows with 16-byte vectors, four
//    loads in flight per lane.
template <typename T>
__global__ void __launch_bounds__(256) scatter_copy_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ idx, int64_t T_, int k, int E, int H,
    int tpc, const int32_t* __restrict__ base, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ scatter_index,
    int32_t* __restrict__ row_token, T* __restrict__ x_perm) {
  extern __shared__ int32_t sm[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t* off = sm;                        // [E + 1]
  int32_t* wsum = sm + E + 1;               // [32]
  int32_t* dst = wsum + 32 + (size_t)wid * k;
  block_offsets(counts, E, off, wsum, offsets);
  constexpr int V = 16 / sizeof(T);
  const int nvec = H / V;
  for (int64_t t = (int64_t)blockIdx.x * nw + wid; t < T_; t += (int64_t)gridDim.x * nw) {
    const int64_t c = t / tpc;
    for (int s = lane; s < k; s += 32) {
      const int64_t p = t * k + s;
      const int e = idx[p];
      const int r = scatter_index[p];
      int d = -1;
      if (r >= 0) {
        d = off[e] + base[c * E + e] + r;
        row_token[d] = (int32_t)t;
      }
      scatter_index[p] = d;
      dst[s] = d;
    }
    __syncwarp();
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    int v = lane;
    for (; v + 96 < nvec; v += 128) {
      uint4 val[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) val[u] = __ldg(src + v + 32 * u);
      for (int s = 0; s < k; ++s) {
        const int d = dst[s];
        if (d < 0) continue;
        uint4* o = reinterpret_cast<uint4*>(x_perm + (int64_t)d * H) + v;
#pragma unroll
        for (int u = 0; u < 4; ++u) o[32 * u] = val[u];
      }
    }
    for (; v < nvec; v += 32) {
      const uint4 val = __ldg(src + v);
      for (int s = 0; s < k; ++s) {
        const int d = dst[s];
        if (d >= 0) reinterpret_cast<uint4*>(x_perm + (int64_t)d * H)[v] = val;
      }
    }
    __syncwarp();
  }
}

// 3'. scatter only (no grouped copy of x: the gate/up GEMM gathers its rows
//     through row_token): one thread per (token, slot) pair.
__global__ void __launch_bounds__(256) scatter_index_kernel(
    const int32_t* __restrict__ idx, int64_t npairs, int k, int E, int tpc,
    const int32_t* __restrict__ base, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ scatter_index,
    int32_t* __restrict__ row_token) {
  extern __shared__ int32_t sm[];
  int32_t* off = sm;                        // [E + 1]
  block_offsets(counts, E, off, sm + E + 1, offsets);
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < npairs;
       p += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = p / k;
    const int r = scatter_index[p];
    int d = -1;
    if (r >= 0) {
      const int e = idx[p];
      d = off[e] + base[(t / tpc) * E + e] + r;
      row_token[d] = (int32_t)t;
    }
    scatter_index[p] = d;
  }
}

// All three steps in one block, for calls whose tokens fit one chunk
// (decode-sized): warp 0 ranks the pairs, the expert counts are scanned in
// shared memory, then every warp turns ranks into rows and copies its tokens.
template <typename T>
__global__ void __launch_bounds__(256) permute_small_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ idx, int T_, int k, int E, int H,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ scatter_index, int32_t* __restrict__ row_token, T* __restrict__ x_perm,
    uint32_t* flags) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;             // [E]
  int32_t* off = sm + E;         // [E + 1]
  int32_t* dst = off + E + 1;    // [T_ * k]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int np = T_ * k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  if (wid == 0) {
    for (int pb = 0; pb < np; pb += 32) {
      const int p = pb + lane;
      const bool valid = p < np;
      const int e = valid ? idx[p] : -1;
      const bool ok = valid && e >= 0 && e < E;
      if (valid && !ok) set_flag(flags, kFlagRoute);
      const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int r = -1;
      if (ok) r = cnt[e] + rank;
      __syncwarp();
      if (ok && rank == 0) cnt[e] += __popc(peers);
      __syncwarp();
      if (valid) dst[p] = r;
    }
    __syncwarp();
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int v = e < E ? cnt[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < E) {
        off[e] = carry + incl - v;
        counts[e] = v;
        offsets[e] = carry + incl - v;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      off[E] = carry;
      offsets[E] = carry;
    }
  }
  __syncthreads();
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const int r = dst[p];
    int d = -1;
    if (r >= 0) {
      d = off[idx[p]] + r;
      row_token[d] = p / k;
    }
    scatter_index[p] = d;
    dst[p] = d;
  }
  __syncthreads();
  if (x_perm == nullptr) return;   // routing arrays only
  // the copy: every thread of the block takes 16-byte vectors of the tokens'
  // rows, four loads in flight before their stores (one token's row is only
  // a few vectors a thread)
  constexpr int V = 16 / sizeof(T), U = 4;
  const int nvec = H / V;
  const int total = T_ * nvec;
  for (int i0 = threadIdx.x; i0 < total; i0 += U * blockDim.x) {
    uint4 val[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      if (i < total) val[u] = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)(i / nvec) * H) + i % nvec);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      if (i >= total) break;
      const int t = i / nvec, v = i % nvec;
      for (int s2 = 0; s2 < k; ++s2) {
        const int d = dst[t * k + s2];
        if (d >= 0) reinterpret_cast<uint4*>(x_perm + (int64_t)d * H)[v] = val[u];
      }
    }
  }
}

// SM count of the current device, cached per device (atomics: several host
// threads may launch)
int sm_count_cached() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
  if (dev >= 0) {
    const int v = cache[dev].load();
    if (v > 0) return v;
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev < 0 ? 0 : dev);
  if (n <= 0) n = 1;
  if (dev >= 0) cache[dev].store(n);
  return n;
}

}  // namespace

// The three launches with caller-chosen scratch tables (hist and base, each
// nchunks * E int32) and an optional status word.  Used with workspace
// tables by moe_permute / moe_layer_forward and with the library's static
// array by moe_permute_static.
cudaError_t launch_permute_scratch(const Shape& s, int nchunks, int tpc, int32_t* hist,
                                   int32_t* base, uint32_t* flags, const void* x,
                                   const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                                   int32_t* scatter_index, int32_t* row_token, void* x_perm,
                                   cudaStream_t st) {
  if (s.T == 0) nchunks = 0;
  cudaError_t e;
  const size_t small_smem = ((size_t)2 * s.E + 1 + (size_t)s.T * s.k) * 4;
  if (nchunks == 1 && small_smem <= 48 * 1024) {
    if (s.dtype == MOE_F32) {
      permute_small_kernel<float><<<1, 256, small_smem, st>>>(
          reinterpret_cast<const float*>(x), topk_idx, (int)s.T, s.k, s.E, s.H, counts, offsets,
          scatter_index, row_token, reinterpret_cast<float*>(x_perm), flags);
    } else {
      permute_small_kernel<bf16><<<1, 256, small_smem, st>>>(
          reinterpret_cast<const bf16*>(x), topk_idx, (int)s.T, s.k, s.E, s.H, counts, offsets,
          scatter_index, row_token, reinterpret_cast<bf16*>(x_perm), flags);
    }
    count_launch();
    return cudaGetLastError();
  }
  if (nchunks > 0) {
    int wpb = (int)((48 * 1024) / ((size_t)s.E * 4));
    if (wpb > 8) wpb = 8;
    if (wpb < 1) wpb = 1;
    const size_t rsm = (size_t)wpb * s.E * 4;
    if (rsm > 48 * 1024) {
      e = cudaFuncSetAttribute(rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm);
      if (e != cudaSuccess) return e;
    }
    rank_kernel<<<(nchunks + wpb - 1) / wpb, wpb * 32, rsm, st>>>(
        topk_idx, s.T, s.k, s.E, tpc, nchunks, hist, scatter_index, flags);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  scan_kernel<<<(unsigned)((s.E + 31) / 32), 1024, 0, st>>>(hist, nchunks, s.E, base, counts,
                                                             offsets);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nchunks == 0) return cudaSuccess;
  // the scatter kernels hold the E + 1 group offsets and 32 warp sums in
  // shared memory (the copy kernel also k rows a warp)
  const size_t osm = ((size_t)s.E + 1 + 32) * 4;
  if (x_perm == nullptr) {
    const int64_t np = s.T * s.k;
    int64_t blocks = (np + 255) / 256;
    const int64_t cap = (int64_t)sm_count_cached() * 16;
    if (blocks > cap) blocks = cap;
    if (osm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)osm);
      if (e != cudaSuccess) return e;
    }
    scatter_index_kernel<<<(unsigned)blocks, 256, osm, st>>>(topk_idx, np, s.k, s.E, tpc, base,
                                                              counts, offsets, scatter_index,
                                                              row_token);
    count_launch();
    return cudaGetLastError();
  }
  const size_t csm = osm + (size_t)8 * s.k * 4;
  int64_t blocks = (s.T + 7) / 8;
  const int64_t cap = (int64_t)sm_count_cached() * 8;
  if (blocks > cap) blocks = cap;
  if (s.dtype == MOE_F32) {
    if (csm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_copy_kernel<float>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm);
      if (e != cudaSuccess) return e;
    }
    scatter_copy_kernel<float><<<(unsigned)blocks, 256, csm, st>>>(
        reinterpret_cast<const float*>(x), topk_idx, s.T, s.k, s.E, s.H, tpc, base, counts,
        offsets, scatter_index, row_token, reinterpret_cast<float*>(x_perm));
  } else {
    if (csm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_copy_kernel<bf16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm);
      if (e != cudaSuccess) return e;
    }
    scatter_copy_kernel<bf16><<<(unsigned)blocks, 256, csm, st>>>(
        reinterpret_cast<const bf16*>(x), topk_idx, s.T, s.k, s.E, s.H, tpc, base, counts, offsets,
        scatter_index, row_token, reinterpret_cast<bf16*>(x_perm));
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_permute(const Shape& s, const Layout& L, char* ws, const void* x,
                           const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                           int32_t* scatter_index, int32_t* row_token, void* x_perm,
                           cudaStream_t st) {
  return launch_permute_scratch(s, L.nchunks, L.tokens_per_chunk,
                                reinterpret_cast<int32_t*>(ws + L.hist),
                                reinterpret_cast<int32_t*>(ws + L.base),
                                reinterpret_cast<uint32_t*>(ws + L.flags), x, topk_idx, counts,
                                offsets, scatter_index, row_token, x_perm, st);
}

}  // namespace moe
