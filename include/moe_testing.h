/*
 * moe_testing.h -- test hooks of libmoe (not part of the layer's contract).
 *
 * The bf16 grouped GEMMs have four engines: tensor-core tiles (tcgen05,
 * 128 x 256 tiles), the same on SM pairs (256 x 256 tiles, cta_group::2, the
 * default for calls of at least 512 rows that are one group, average 1024
 * rows a group, or have more than 2048 rows and K >= 3072; a group's last
 * tile of at most 128 rows runs at M = 128), a skinny
 * weight-streaming engine (decode-sized calls, up to 4 rows) and CUDA-core
 * tiles.  Parity tests pin each engine against the oracle by
 * forcing it for a run of calls.
 */
#ifndef MOE_TESTING_H_
#define MOE_TESTING_H_

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* 0 = automatic (default), 1 = CUDA-core tiles, 2 = tensor cores, 3 = skinny,
 * 4 = tensor cores on SM pairs (256 x 256 tiles shared by the two CTAs of a
 * cluster; calls it cannot take -- fp32 outputs, split K, gathered rows -- use
 * 2).  Applies to later calls from any thread; returns the previous setting.
 * fp32 layers always use the CUDA-core engine (values other than 0 and 3 are
 * ignored for them). */
int32_t moe_testing_set_gemm_engine(int32_t engine);

/* How many SMs' worth of CTAs the shared MLP's GEMMs may take when
 * moe_layer_forward runs them on its second stream, leaving the other SMs
 * free for the routed chain on the caller's stream: 0 = the library's choice
 * (default: 96 at decode sizes, all at prefill sizes), -1 = all SMs, n > 0 =
 * n SMs.  Applies to later
 * calls from any thread; returns the previous setting.  Results do not
 * depend on it. */
int32_t moe_testing_set_fork_sms(int32_t sms);

/* Per-group A maps of the tensor-core engines' grouped calls (the rows past
 * a group's end in its last tile load as zeros, which lowers the tensor
 * cores' power; used where the call is long and its groups small): 0 = the
 * library's choice (default), 1 = every grouped call of those engines, -1 =
 * none.  Applies to later calls from any thread; returns the previous
 * setting.  Results do not depend on it. */
int32_t moe_testing_set_zero_pad(int32_t mode);

/* The router logits moe_route decides on: the router GEMM exactly as
 * moe_route runs it (same engine and K split), with the partial sums added in
 * the same order, written to logits [T, E + shared_gate] (fp32, device).
 * Lets tests measure the fp32 logit error against exact dot products. */
moe_status moe_testing_router_logits(const moe_shape *shape, const void *x, const void *w_router,
                                     float *logits, void *ws, size_t ws_bytes, void *stream);

/* The failure path of the pipelines' bounded waits, made to run out on
 * purpose without faulting: one warp waits on a shared-memory mbarrier that
 * expects one arrival, with the pipelines' try_wait loop bounded by
 * max_cycles SM clocks (at most 4e9, about 2 s).  arrive = 0: nothing
 * arrives, the wait runs out, the kernel sets the timeout bit of the
 * workspace's status word (moe_get_device_status then returns
 * MOE_ERR_TIMEOUT) and returns; arrive = 1: the arrival completes the phase
 * and no bit is set.  Needs the workspace's status word only. */
moe_status moe_testing_wait_probe(void *ws, int64_t max_cycles, int32_t arrive, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_TESTING_H_ */
