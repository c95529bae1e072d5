// Declarations shared between the library's translation units (not part of
// the public ABI).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "../../include/bi.h"

// Device address of the status word on the current device (nullptr if the
// runtime cannot provide it).
int32_t *bi_status_ptr();

// 2-D bf16 tensor map over a row-major [outer][inner] array.
bi_status bi_make_tmap_2d_bf16(CUtensorMap *map, const void *base,
                               uint64_t inner, uint64_t outer,
                               uint64_t row_stride_bytes, uint32_t box_inner,
                               uint32_t box_outer, bool swizzle128);

// GEMM with a forced schedule, for the model driver and the schedule test:
// mode 0 = the default choice, 1 = every split in its own CTA,
// 2 = every split of a tile in one CTA.
bi_status bi_gemm_sched(const bi_bf16 *x, int M, int K, const bi_bf16 *W,
                        int N, void *out, int out_kind, void *ws,
                        size_t ws_bytes, int mode, cudaStream_t stream);
