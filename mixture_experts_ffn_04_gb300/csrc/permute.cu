// permute.cu -- expert histogram, group offsets, scatter_index and the
// expert-grouped copy of the activations.
//
// "Fused MoE Kernel Notes", Scatter/gather layout: tokens are expanded by
// their top-k routes into an expert-grouped [tokens * topk, hidden] buffer and
// scatter_index maps each (token, slot) to its row there.  Rows of one expert
// keep row-major (token, slot) order, so the result is deterministic and a
// duplicate route (two slots of one token on one expert) simply adds a row.
//
// Three launches, no global atomics:
//   1. hist     per chunk of tokens, count pairs per expert (shared memory);
//   2. scan     one block: per-expert prefix over chunks, then the exclusive
//               prefix over experts -> counts, offsets, per-(chunk, expert) base;
//   3. scatter  per chunk: one warp ranks the chunk's pairs in row-major order
//               (__match_any_sync groups equal experts within 32 pairs), then
//               all warps copy each token row once from x and write it to its
//               k destinations with 16-byte vectors.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void hist_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int tpc,
                            int32_t* __restrict__ hist, uint32_t* flags) {
  extern __shared__ int32_t cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * tpc;
  const int64_t t1 = min(T, t0 + tpc);
  for (int64_t p = t0 * k + threadIdx.x; p < t1 * k; p += blockDim.x) {
    const int e = idx[p];
    if (e < 0 || e >= E) {
      set_flag(flags, kFlagRoute);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = cnt[e];
}

// One block of 1024 threads.  Work items (e, seg): expert e, segment seg of
// the chunks (S segments when E <= 1024, else one).  smem: segsum[S*E] and
// block-scan scratch.
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ hist, int nchunks,
                                                    int E, int S, int32_t* __restrict__ base,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets) {
  extern __shared__ int32_t sm[];
  int32_t* segsum = sm;               // [S * E]
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int items = S * E;
  for (int it = tid; it < items; it += blockDim.x) {
    const int e = it % E, seg = it / E;
    const int c0 = (int)((int64_t)nchunks * seg / S), c1 = (int)((int64_t)nchunks * (seg + 1) / S);
    int32_t s = 0;
#pragma unroll 16
    for (int c = c0; c < c1; ++c) s += hist[(int64_t)c * E + e];
    segsum[seg * E + e] = s;
  }
  __syncthreads();
  // per-expert exclusive prefix over segments (in place) and the count
  for (int e = tid; e < E; e += blockDim.x) {
    int32_t run = 0;
    for (int seg = 0; seg < S; ++seg) {
      const int32_t v = segsum[seg * E + e];
      segsum[seg * E + e] = run;
      run += v;
    }
    counts[e] = run;
  }
  if (tid == 0) carry = 0;
  __syncthreads();
  // exclusive prefix of counts over experts -> offsets (chunks of 1024)
  for (int b = 0; b < E; b += blockDim.x) {
    const int e = b + tid;
    const int32_t v = e < E ? counts[e] : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int32_t w = warp_tot[lane];
      int32_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      warp_tot[lane] = wi - w;
    }
    __syncthreads();
    if (e < E) offsets[e] = carry + warp_tot[wid] + incl - v;
    __syncthreads();
    if (tid == blockDim.x - 1) carry += warp_tot[wid] + incl;
    __syncthreads();
  }
  if (tid == 0) offsets[E] = carry;
  __syncthreads();
  // per-(chunk, expert) base row
  for (int it = tid; it < items; it += blockDim.x) {
    const int e = it % E, seg = it / E;
    const int c0 = (int)((int64_t)nchunks * seg / S), c1 = (int)((int64_t)nchunks * (seg + 1) / S);
    int32_t run = offsets[e] + segsum[seg * E + e];
#pragma unroll 16
    for (int c = c0; c < c1; ++c) {
      const int64_t at = (int64_t)c * E + e;
      const int32_t v = hist[at];
      base[at] = run;
      run += v;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) scatter_kernel(const T* __restrict__ x,
                                                      const int32_t* __restrict__ idx, int64_t T_,
                                                      int k, int E, int H, int tpc,
                                                      const int32_t* __restrict__ base,
                                                      int32_t* __restrict__ scatter_index,
                                                      int32_t* __restrict__ row_token,
                                                      T* __restrict__ x_perm) {
  extern __shared__ int32_t sm[];
  int32_t* running = sm;      // [E]
  int32_t* dst = sm + E;      // [tpc * k]
  const int64_t t0 = (int64_t)blockIdx.x * tpc;
  const int64_t t1 = min(T_, t0 + tpc);
  const int npairs = (int)((t1 - t0) * k);
  for (int e = threadIdx.x; e < E; e += blockDim.x) running[e] = base[(int64_t)blockIdx.x * E + e];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int p0 = 0; p0 < npairs; p0 += 32) {
      const int pl = p0 + lane;
      const bool valid = pl < npairs;
      const int64_t p = t0 * k + pl;
      int e = valid ? idx[p] : -1;
      const bool ok = valid && e >= 0 && e < E;
      const int key = ok ? e : -1 - lane;  // invalid lanes never group
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int d = -1;
      if (ok) d = running[e] + rank;
      __syncwarp();
      if (ok && rank == 0) running[e] += __popc(peers);
      __syncwarp();
      if (valid) {
        scatter_index[p] = d;
        dst[pl] = d;
        if (ok) row_token[d] = (int32_t)(p / k);
      }
    }
  }
  __syncthreads();
  // copy: each token row read once, written to its k destinations
  const int V = 16 / (int)sizeof(T);
  const int nvec = H / V;
  const int warps = blockDim.x >> 5, wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t tl = wid; tl < t1 - t0; tl += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (t0 + tl) * H);
    for (int v = lane; v < nvec; v += 32) {
      const uint4 val = __ldg(src + v);
      for (int s = 0; s < k; ++s) {
        const int d = dst[tl * k + s];
        if (d >= 0) reinterpret_cast<uint4*>(x_perm + (int64_t)d * H)[v] = val;
      }
    }
  }
}

}  // namespace

cudaError_t launch_permute(const Shape& s, const Layout& L, char* ws, const void* x,
                           const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                           int32_t* scatter_index, int32_t* row_token, void* x_perm,
                           cudaStream_t st) {
  int32_t* hist = reinterpret_cast<int32_t*>(ws + L.hist);
  int32_t* base = reinterpret_cast<int32_t*>(ws + L.base);
  uint32_t* flags = reinterpret_cast<uint32_t*>(ws + L.flags);
  const int nchunks = s.T > 0 ? L.nchunks : 0;
  const int tpc = L.tokens_per_chunk;
  cudaError_t e;
  if (nchunks > 0) {
    const size_t hsm = (size_t)s.E * 4;
    if (hsm > 48 * 1024) {
      e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsm);
      if (e != cudaSuccess) return e;
    }
    hist_kernel<<<nchunks, 256, hsm, st>>>(topk_idx, s.T, s.k, s.E, tpc, hist, flags);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int S = s.E <= 1024 ? (nchunks > 0 ? (1024 / s.E < nchunks ? 1024 / s.E : nchunks) : 1) : 1;
  const size_t ssm = (size_t)(S > 0 ? S : 1) * s.E * 4;
  if (ssm > 48 * 1024) {
    e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return e;
  }
  scan_kernel<<<1, 1024, ssm, st>>>(hist, nchunks, s.E, S > 0 ? S : 1, base, counts, offsets);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nchunks == 0) return cudaSuccess;
  const size_t csm = ((size_t)s.E + (size_t)tpc * s.k) * 4;
  if (s.dtype == MOE_F32) {
    if (csm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)csm);
      if (e != cudaSuccess) return e;
    }
    scatter_kernel<float><<<nchunks, 256, csm, st>>>(
        reinterpret_cast<const float*>(x), topk_idx, s.T, s.k, s.E, s.H, tpc, base, scatter_index,
        row_token, reinterpret_cast<float*>(x_perm));
  } else {
    if (csm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)csm);
      if (e != cudaSuccess) return e;
    }
    scatter_kernel<bf16><<<nchunks, 256, csm, st>>>(
        reinterpret_cast<const bf16*>(x), topk_idx, s.T, s.k, s.E, s.H, tpc, base, scatter_index,
        row_token, reinterpret_cast<bf16*>(x_perm));
  }
  count_launch();
  return cudaGetLastError();
}

// Same three launches with caller-chosen scratch tables (hist and base, each
// nchunks * E int32) and an optional status word; used by the allocation-free
// entry point, whose scratch is a static device array.
cudaError_t launch_permute_scratch(const Shape& s, int nchunks, int tpc, int32_t* hist,
                                   int32_t* base, uint32_t* flags, const void* x,
                                   const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                                   int32_t* scatter_index, int32_t* row_token, void* x_perm,
                                   cudaStream_t st) {
  if (s.T == 0) nchunks = 0;
  cudaError_t e;
  if (nchunks > 0) {
    const size_t hsm = (size_t)s.E * 4;
    if (hsm > 48 * 1024) {
      e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsm);
      if (e != cudaSuccess) return e;
    }
    hist_kernel<<<nchunks, 256, hsm, st>>>(topk_idx, s.T, s.k, s.E, tpc, hist, flags);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  int S = 1;
  if (s.E <= 1024 && nchunks > 0) S = 1024 / s.E < nchunks ? 1024 / s.E : nchunks;
  const size_t ssm = (size_t)S * s.E * 4;
  if (ssm > 48 * 1024) {
    e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return e;
  }
  scan_kernel<<<1, 1024, ssm, st>>>(hist, nchunks, s.E, S, base, counts, offsets);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nchunks == 0) return cudaSuccess;
  const size_t csm = ((size_t)s.E + (size_t)tpc * s.k) * 4;
  if (s.dtype == MOE_F32) {
    if (csm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)csm);
      if (e != cudaSuccess) return e;
    }
    scatter_kernel<float><<<nchunks, 256, csm, st>>>(
        reinterpret_cast<const float*>(x), topk_idx, s.T, s.k, s.E, s.H, tpc, base, scatter_index,
        row_token, reinterpret_cast<float*>(x_perm));
  } else {
    if (csm > 48 * 1024) {
      e = cudaFuncSetAttribute(scatter_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)csm);
      if (e != cudaSuccess) return e;
    }
    scatter_kernel<bf16><<<nchunks, 256, csm, st>>>(
        reinterpret_cast<const bf16*>(x), topk_idx, s.T, s.k, s.E, s.H, tpc, base, scatter_index,
        row_token, reinterpret_cast<bf16*>(x_perm));
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
