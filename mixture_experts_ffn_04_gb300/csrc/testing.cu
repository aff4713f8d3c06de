// testing.cu -- test hooks (include/moe_testing.h): a bounded mbarrier wait
// that is made to run out, to check the failure path every tensor-core
// pipeline takes without faulting or hanging the GPU.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

// One warp: thread 0 initialises a barrier expecting one arrival, arrives on
// it only when `arrive` is set, and waits for its phase with the same
// try_wait loop as the pipelines, bounded by max_cycles.  A wait that runs
// out raises the timeout bit of the status word; the kernel then returns.
__global__ void wait_probe_kernel(long long max_cycles, int arrive, uint32_t* flags) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = tc::smem_u32(&bar);
  tc::mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (arrive) tc::mbar_arrive(b);
  const long long t0 = clock64();
  while (!tc::mbar_try_wait(b, 0)) {
    if (clock64() - t0 > max_cycles) {
      set_flag(flags, kFlagTimeout);
      return;
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_testing_wait_probe(void* ws, int64_t max_cycles, int32_t arrive,
                                             void* stream) {
  reset_launch_count();
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (max_cycles <= 0 || max_cycles > (int64_t)4000000000LL)
    return fail(MOE_ERR_INVALID_ARG, "max_cycles must be in (0, 4e9]");
  wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(max_cycles, arrive ? 1 : 0,
                                                      reinterpret_cast<uint32_t*>(ws));
  count_launch();
  CHECK_CUDA(cudaGetLastError());
  return MOE_OK;
}
