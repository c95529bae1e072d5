// Declarations shared between the library's translation units (not part of
// the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bi.h"

// Device address of the status word on the current device (nullptr if the
// runtime cannot provide it).
int32_t *bi_status_ptr();

// Number of SMs of the current device (queried once per device).
int bi_sm_count();

// 2-D bf16 tensor map over a row-major [outer][inner] array.
bi_status bi_make_tmap_2d_bf16(CUtensorMap *map, const void *base,
                               uint64_t inner, uint64_t outer,
                               uint64_t row_stride_bytes, uint32_t box_inner,
                               uint32_t box_outer, bool swizzle128);

// 3-D tensor map over a row-major [d2][d1][d0] array of fp32 (f32) or bf16,
// box {box0, box1, box2}; with swizzle128 the 128-byte swizzle (box0 *
// element size must then be 128), else no swizzle.
bi_status bi_make_tmap_3d(CUtensorMap *map, const void *base, bool f32,
                          uint64_t d0, uint64_t d1, uint64_t d2,
                          uint32_t box0, uint32_t box1, bool swizzle128,
                          uint32_t box2 = 1);



// Attention with the KV pool size known, for the model driver.  Decode
// stages: bit 0 chunk kernels (bit 2: reuse the work list already in ws),
// bit 1 merge (nothing to do when bi_decode_whole_rows holds: the kernel
// then merges in registers and writes `out` itself).
bool bi_decode_whole_rows(int B, int Hkv, int D);
bi_status bi_decode_attn_pool(const bi_bf16 *q, const bi_bf16 *k_pool,
                              const bi_bf16 *v_pool, const int32_t *page_table,
                              int max_pages, int n_pages,
                              const int32_t *row_req, const int32_t *kv_len,
                              int B, int max_kv_len, int Hq, int Hkv, int D,
                              float scale, bi_bf16 *out, void *ws,
                              size_t ws_bytes, int stages, cudaStream_t s);
bi_status bi_prefill_attn_pool(const bi_bf16 *q, const int32_t *cu_q,
                               const int32_t *seg_req, int R, int T,
                               const int32_t *pos, int max_q, int max_kv_len,
                               const bi_bf16 *k_pool, const bi_bf16 *v_pool,
                               const int32_t *page_table, int max_pages,
                               int n_pages, int Hq, int Hkv, int D,
                               float scale, bi_bf16 *out, void *ws,
                               size_t ws_bytes, cudaStream_t stream,
                               bool reuse_list = false);
// reuse_list: ws already holds the tile list (and the split form's items)
// an earlier call with the same segments, positions and shapes built — the
// layers of one forward; the list depends on nothing else.

// Workspace with which bi_prefill_attn_pool runs the persistent tensor-core
// path (head_dim 128; without it, one CTA per query tile): its tile lists.
size_t bi_prefill_attn_ws_bytes(int T, int R, int Hq, int Hkv);
size_t bi_prefill_attn_split_ws_bytes(int T, int R, int Hq, int Hkv,
                                      int max_kv_len);

// RoPE in two parts for the model driver: the (cos, sin) table of the rows'
// positions ([T][D/2] float2), computed once per forward, and the rotation
// + KV append reading it (table == nullptr computes the same values
// in-kernel).  discard_partials: the qkv slice partials are scratch read
// here for the last time, so their L2 lines are dropped without a write-back
// (their contents are undefined afterwards); dead / dead_bytes: another
// scratch region (128-byte aligned) whose contents are dead by the time
// this runs, dropped the same way.
bi_status bi_rope_table(const int32_t *pos, int T, int D, double theta,
                        float2 *table, cudaStream_t s);
bi_status bi_rope_apply(const float *qkv, int S, const float2 *table,
                        const int32_t *pos, const int32_t *row_req, int T,
                        int Hq, int Hkv, int D, double theta,
                        bi_bf16 *q_out, bi_bf16 *k_pool, bi_bf16 *v_pool,
                        const int32_t *page_table, int max_pages, int n_pages,
                        cudaStream_t st, bool discard_partials = false,
                        const void *dead = nullptr, size_t dead_bytes = 0);

// bi_rmsnorm on a stream, with the same options for its slice partials and
// up to two dead scratch regions (H <= 4096; other widths drop nothing).
bi_status bi_rmsnorm_apply(const float *partials, int S, const bi_bf16 *x,
                           bi_bf16 *residual, const bi_bf16 *w, int T, int H,
                           float eps, bi_bf16 *y, bool discard_partials,
                           cudaStream_t s, const void *dead0 = nullptr,
                           size_t dead0_bytes = 0, const void *dead1 = nullptr,
                           size_t dead1_bytes = 0);
