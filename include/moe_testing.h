/*
 * moe_testing.h -- test hooks of libmoe (not part of the layer's contract).
 *
 * The bf16 grouped GEMMs have three engines: tensor-core tiles (tcgen05,
 * 128 x 256 tiles, the default whenever a call may carry more than 16 rows),
 * a skinny weight-streaming engine (decode-sized calls, up to 16 rows) and
 * CUDA-core tiles.  Parity tests pin each engine against the oracle by
 * forcing it for a run of calls.
 */
#ifndef MOE_TESTING_H_
#define MOE_TESTING_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 0 = automatic (default), 1 = CUDA-core tiles, 2 = tensor cores, 3 = skinny.
 * Applies to later calls from any thread; returns the previous setting.
 * fp32 layers always use the CUDA-core engine (values other than 0 and 3 are
 * ignored for them). */
int32_t moe_testing_set_gemm_engine(int32_t engine);

#ifdef __cplusplus
}
#endif
#endif /* MOE_TESTING_H_ */
