// moe_static.cu -- moe_permute for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocating routine)
// while they run: an inference server that hands a plugin nothing but its
// input and output tensors, a real-time loop that forbids allocation after
// start-up because an allocation can synchronise the whole device, or an
// embedding whose device memory is already carved up by another owner.  Such
// a caller cannot provide the workspace that moe_permute needs for its
// per-chunk histogram tables.  moe_permute_static runs the same kernels with
// those tables in a fixed static device array owned by this library.
//
// The array is file-scope `__device__` storage, so every GPU that loads the
// library holds it until the process exits.  Its size bounds the shapes the
// entry point accepts (see kStaticScratchBytes); with the library's chunking
// (tokens per chunk chosen so that chunks * experts <= 262144) every valid
// shape fits, and the size check below only guards that invariant.
//
// In host code the symbol is only a host-side stand-in: its device address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, the first time the entry point runs on it.  That first call should
// therefore come before any stream capture.  The address is kept for the life
// of the process: after a cudaDeviceReset the module is loaded again and the
// kept address no longer names the array, so the entry point must not be used
// on a device after that device has been reset.  Every call shares the array;
// calls that overlap on the GPU (two streams, or two threads) race on it.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// hist + base tables: 2 x 262144 int32 = 2 MiB.
constexpr size_t kTableBytes = (size_t)262144 * 4;
constexpr size_t kStaticScratchBytes = 2 * kTableBytes;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static array on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_static(const moe_shape* shape, const void* x,
                                         const int32_t* topk_idx, int32_t* counts,
                                         int32_t* offsets, int32_t* scatter_index,
                                         int32_t* row_token, void* x_perm, void* stream) {
  reset_launch_count();
  Shape s;
  const char* why = "";
  moe_status st = decode_shape(shape, &s, &why);
  if (st != MOE_OK) {
    set_error_message(why);
    return st;
  }
  if (!counts || !offsets) {
    set_error_message("counts and offsets must be non-NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (s.T > 0 && (!topk_idx || !scatter_index || !row_token)) {
    set_error_message("topk_idx, scatter_index and row_token must be non-NULL");
    return MOE_ERR_INVALID_ARG;
  }
  // as moe_permute: without x_perm only the routing arrays are written
  if (s.T > 0 && x_perm && !x) {
    set_error_message("x_perm needs x");
    return MOE_ERR_INVALID_ARG;
  }
  if (((uintptr_t)x & 15u) || ((uintptr_t)x_perm & 15u)) {
    set_error_message("x and x_perm must be 16-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  const Layout L = layout_for(s);
  const size_t table = (size_t)L.nchunks * s.E * 4;
  if (table > kTableBytes) {
    set_error_message("shape needs more than the 2 MiB static scratch of moe_permute_static");
    return MOE_ERR_UNSUPPORTED;
  }
  void* base_addr = nullptr;
  cudaError_t e = scratch_address(&base_addr);
  if (e != cudaSuccess) {
    set_error_message(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  int32_t* hist = static_cast<int32_t*>(base_addr);
  int32_t* base = reinterpret_cast<int32_t*>(static_cast<char*>(base_addr) + kTableBytes);
  // Both tables are fully rewritten by every call (hist per chunk, base by the
  // scan), so nothing left over from an earlier call is read.  No status word:
  // a route outside [0, E) is dropped (scatter_index -1, not counted), which
  // the caller sees as offsets[E] < T * k.
  e = launch_permute_scratch(s, L.nchunks, L.tokens_per_chunk, hist, base, nullptr, x, topk_idx,
                             counts, offsets, scatter_index, row_token, x_perm,
                             (cudaStream_t)stream);
  if (e != cudaSuccess) {
    set_error_message(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
