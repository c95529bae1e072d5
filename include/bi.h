/*
 * bi.h - C ABI of libbi, a batch-invariant bf16 decoder library for GB300
 * (sm_103a).
 *
 * What "batch-invariant" means here (ybb.press, "LLM 推理确定性工程深度实战",
 * section 4 "Batch-Invariant Kernel"; Vosti abstract): every reduction in
 * every kernel (GEMM K-loop, RMSNorm, softmax and attention over paged KV,
 * logits argmax) runs in an order fixed by the data and by compile-time
 * constants.  The order never depends on the batch size, on a row's position
 * in the batch, on the query length, on the physical order of KV pages, nor
 * on how many SMs happen to be free.  There are no floating-point atomics.
 * A request's logits are therefore bitwise identical whatever batch it is
 * served in, and across repeated runs.
 *
 * Conventions shared by every entry point
 *   - Return value: bi_status.  BI_OK on success.  On failure nothing is
 *     launched unless stated otherwise.  A thread-local message is kept for
 *     bi_last_error().
 *   - bf16 tensors are passed as bi_bf16* (the 16-bit pattern).  Every
 *     tensor pointer is a DEVICE pointer owned by the caller unless its
 *     name starts with h_ (host memory, also caller-owned).  The library
 *     never frees caller memory, and it allocates none in any call listed
 *     here: workspaces are passed in, sized by the *_workspace_size queries.
 *   - All device work is enqueued on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and is asynchronous, except
 *     verify_commit_rollback, which synchronises `stream` to hand back its
 *     small host outputs.
 *   - Row-major layouts throughout.  "[T][H]" means T rows of H contiguous
 *     elements.
 *   - Device pointers must be 16-byte aligned; inner dimensions of bf16
 *     matrices read by the tensor-core GEMM must be multiples of 8.
 *   - A call with zero rows (M, T, B or n equal to 0) is a no-op: once its
 *     sizes pass their checks it returns BI_OK without reading its
 *     pointers, which may then be null (an empty torch tensor has a null
 *     data pointer).
 */
#ifndef BI_H
#define BI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t bi_bf16;

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad size */
    BI_ERR_UNSUPPORTED = 2,        /* shape with no compiled instantiation */
    BI_ERR_WORKSPACE_TOO_SMALL = 3,
    BI_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
    BI_ERR_BOUNDS = 5,             /* a kernel saw an out-of-range index */
    BI_ERR_TIMEOUT = 6             /* a bounded device wait ran out */
} bi_status;

/* Message for the last failing call on this thread ("" if none). */
const char *bi_last_error(void);

/* Reads and clears the device-side status word that kernels set when a
 * bounded wait runs out (BI_ERR_TIMEOUT) or an index check fails
 * (BI_ERR_BOUNDS).  Synchronises `stream`.  *h_status receives BI_OK or the
 * first error recorded since the previous call. */
bi_status bi_device_status(int32_t *h_status, void *stream);

/* Test aid for the bounded device waits (every mbarrier wait in the
 * library gives up after 2 s, records BI_ERR_TIMEOUT and lets its kernel
 * finish instead of hanging).  Launches one block whose thread waits, with
 * the library's bounded wait and a limit of limit_ns (1 us .. 100 ms, else
 * BI_ERR_INVALID_ARG), on a barrier nothing arrives at: the wait runs out,
 * BI_ERR_TIMEOUT is recorded in the status word and the kernel returns.
 * done: device int32, set to 2 when the wait ran out (1 if it completed).
 * Touches no other state; later calls run normally. */
bi_status bi_test_wait_timeout(int64_t limit_ns, int32_t *done, void *stream);

/* ------------------------------------------------------------------ GEMM --
 * y = x W^T.  ybb.press section 2.2 (GEMM heuristics switch tile shape and
 * split-K with (M, N, K); split-K with atomicAdd is run-to-run
 * nondeterministic) and section 4 (fixed tile split, a fixed split count
 * with a fixed-order second stage, no float atomics).
 *
 * x [M][K] bf16, W [N][K] bf16 (row n = output feature n, "K-major").
 * fp32 accumulation on the tcgen05 tensor cores.  The tile is 256 rows x
 * bi_gemm_tile_n(N, K) columns for every M (rows past M are zero-filled,
 * never read from memory).  The K range is cut into bi_gemm_splits(N, K)
 * fixed slices of whole 64-column blocks; each slice is an independent fp32
 * chain in ascending k.  Slices are summed in slice order 0..S-1 by the
 * consumer.
 *
 * out_kind selects what is written to `out`:
 *   BI_OUT_PARTIALS  fp32 [S][M][N]: the S slice sums, unreduced.  The
 *                    second stage is bi_rmsnorm (or bi_rope for q/k/v).
 *   BI_OUT_F32       fp32 [M][N]: slices reduced in order (needs workspace
 *                    bi_gemm_workspace_size(M, N, K) if S > 1).
 *   BI_OUT_BF16      bf16 [M][N]: as F32, rounded to nearest even.
 *   BI_OUT_SWIGLU    bf16 [M][N/2]: W holds gate and up rows interleaved
 *                    as bi_pack_gate_up writes them; out = silu(g) * u with
 *                    silu(g) = g / (1 + e^-g) in fp32 on the slice sums
 *                    (fast exponential and division: within one bf16 ulp
 *                    of bi_swiglu on the same sums).
 *                    N must be a multiple of 64; needs the workspace if
 *                    S > 1.
 */
typedef enum {
    BI_OUT_PARTIALS = 0,
    BI_OUT_F32 = 1,
    BI_OUT_BF16 = 2,
    BI_OUT_SWIGLU = 3
} bi_out_kind;

/* Fixed split count S (1..8) and tile width (128, 192 or 256) for a weight
 * of shape [N][K]: pure functions of (N, K), never of M.  They are the plan
 * a time model of a 256-row batch on a 152-SM GB300 ranks fastest (bytes
 * loaded by the busiest SM, plus the fp32 partial traffic when S > 1). */
int bi_gemm_splits(int N, int K);
int bi_gemm_tile_n(int N, int K);

/* Bytes of workspace bi_gemm needs for (M, N, K) and BI_OUT_F32, BF16 or
 * SWIGLU (S * M * N * 4 when S > 1, else 0). */
size_t bi_gemm_workspace_size(int M, int N, int K);

bi_status bi_gemm(const bi_bf16 *x, int M, int K, const bi_bf16 *W, int N,
                  void *out, int out_kind, void *ws, size_t ws_bytes,
                  void *stream);

/* Interleaves separate gate and up weights, each [F][K], into the [2F][K]
 * layout BI_OUT_SWIGLU reads, one block per GEMM tile: with
 * w0 = bi_gemm_tile_n(2F, K) / 2, block b holds features [b w0, b w0 + w),
 * w = min(w0, F - b w0), as w gate rows followed by the w up rows of the
 * same features.  F must be a multiple of 32.  A pure copy. */
bi_status bi_pack_gate_up(const bi_bf16 *wg, const bi_bf16 *wu, int F, int K,
                          bi_bf16 *wgu, void *stream);

/* --------------------------------------------------------------- RMSNorm --
 * y = x * (1 / sqrt(mean(x^2) + eps)) * w per row of length H, fused with
 * the second stage of a split GEMM and the residual add (ybb.press section
 * 4: the second stage sums partials 0..S-1 in that fixed order).
 *
 *   partials  fp32 [S][T][H] or NULL.  If given, v = sum_s partials[s] in
 *             order s = 0..S-1; then, if residual is given,
 *             residual = bf16(residual + v) and the norm reads the new
 *             residual; else the norm reads bf16(v).
 *   x         bf16 [T][H], used when partials is NULL and residual is NULL.
 *   residual  bf16 [T][H] in/out, or NULL.  With partials NULL it is only
 *             read.
 *   w         bf16 [H] norm weight.  y bf16 [T][H] output.
 * Per row: each thread sums fixed 8-element slices in order, then a fixed
 * xor-shuffle tree, then warps in fixed order. */
bi_status bi_rmsnorm(const float *partials, int S, const bi_bf16 *x,
                     bi_bf16 *residual, const bi_bf16 *w, int T, int H,
                     float eps, bi_bf16 *y, void *stream);

/* Row gather h[t] = E[tokens[t]] from the untied embedding E [V][H]. */
bi_status bi_embed(const int32_t *tokens, int T, const bi_bf16 *E, int V,
                   int H, bi_bf16 *h, void *stream);

/* ----------------------------------------------------- RoPE + KV append --
 * Half-split rotary embedding (pairs (i, i + D/2), angle
 * pos * theta^(-2i/D), no frequency scaling) of q and k, and the append of
 * k and v to the paged cache (PagedAttention pages; Vosti: KV values tied to
 * their logical positions, any physical page order).
 *
 *   qkv       fp32 [S][T][(Hq+2Hkv)D] slice partials of the QKV GEMM,
 *             summed in order s = 0..S-1 and rounded to bf16 first; rows
 *             are q heads, k heads, v heads.
 *   pos       int32 [T] absolute position of each row.
 *   row_req   int32 [T] page-table row of each row; < 0 marks a pad row
 *             (nothing appended, q written as zeros).
 *   q_out     bf16 [T][Hq][D] rotated queries.
 *   k_pool, v_pool  bf16 [n_pages][Hkv][16][D]; row t's k and v land in
 *             page page_table[row_req[t] * max_pages + pos[t] / 16], slot
 *             pos[t] % 16.  Angles in double, rotation in fp32. */
bi_status bi_rope(const float *qkv, int S, const int32_t *pos,
                  const int32_t *row_req, int T, int Hq, int Hkv, int D,
                  double theta, bi_bf16 *q_out, bi_bf16 *k_pool,
                  bi_bf16 *v_pool, const int32_t *page_table, int max_pages,
                  int n_pages, void *stream);

/* ---------------------------------------------------------------- SwiGLU --
 * out[i] = bf16(silu(g[i]) * u[i]), silu(g) = g / (1 + e^-g), fp32 inputs.
 * (The model path fuses this into the gate/up GEMM, BI_OUT_SWIGLU.) */
bi_status bi_swiglu(const float *g, const float *u, int64_t n, bi_bf16 *out,
                    void *stream);

/* ------------------------------------------------------------- attention --
 * Causal grouped-query attention over the paged cache, in fixed 256-position
 * KV chunks (Vosti: bitwise-equal outputs across batches, query lengths and
 * paged layouts; ybb.press section 4: two-stage fixed-order reduction).
 *
 * For each (query row, query head h, chunk c of absolute positions
 * [256c, 256c+256)) a partial (m, l, o) is computed from scratch:
 * s_j = (q . k_j) / sqrt(D) on the tensor cores (dims in ascending 16-steps),
 * masked past the row's context; m = max s; p_j = exp(s_j - m); l = sum p_j
 * in a fixed order; o = sum bf16(p_j) v_j in ascending 16-key steps.  The
 * chunks are then merged sequentially c = 0, 1, ...:
 * m' = max(m, m_c), o = o e^(m - m') + o_c e^(m_c - m'), likewise l, and
 * out = bf16(o / l).  Query head h reads KV head h / (Hq / Hkv).  Both
 * kernels below run the same chunk and merge code, so a (request, position)
 * gets the same bits from either.  Supported head_dim: 32 and 128;
 * Hq / Hkv in {1, 2, 4, 8, 16}. */

/* Workspace bytes for bi_paged_decode_attn with B rows and contexts of at
 * most max_kv_len positions. */
size_t bi_decode_attn_workspace_size(int B, int Hq, int D, int max_kv_len);

/* One query per row.  q bf16 [B][Hq][D]; row_req int32 [B] page-table row;
 * kv_len int32 [B] context length of each row, including its own position
 * (1 <= kv_len <= max_kv_len, max_kv_len <= 16 * max_pages).
 * out bf16 [B][Hq][D]. */
bi_status bi_paged_decode_attn(const bi_bf16 *q, const bi_bf16 *k_pool,
                               const bi_bf16 *v_pool,
                               const int32_t *page_table, int max_pages,
                               const int32_t *row_req, const int32_t *kv_len,
                               int B, int max_kv_len, int Hq, int Hkv, int D,
                               float scale, bi_bf16 *out, void *ws,
                               size_t ws_bytes, void *stream);

/* Allocation-free variant of bi_paged_decode_attn (the pages have no
 * counterpart of this entry point: it exists for callers of this library).
 *
 * For callers that cannot allocate device memory for a workspace: code whose
 * device memory is owned and handed out by another runtime that offers no
 * scratch buffer, or a latency-bound caller that must not enter an allocator
 * on the decode path.  The chunk partials go to one fixed scratch array of
 * BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES that is part of the library's device
 * module: every GPU that loads the library holds it until the process exits.
 * Arguments and results are those of bi_paged_decode_attn without ws and
 * ws_bytes; the bits of `out` are identical to it.
 *   - Calls whose bi_decode_attn_workspace_size(B, Hq, D, max_kv_len) exceeds
 *     the scratch size return BI_ERR_WORKSPACE_TOO_SMALL without launching
 *     (with D = 128 and Hq = 32: B * ceil(max_kv_len / 256) <= 992, e.g.
 *     62 rows of up to 4096 positions or 248 rows of up to 1024).
 *   - Every call made outside a stream capture looks up the array's
 *     device address (cudaGetSymbolAddress), so the variant keeps working
 *     after a cudaDeviceReset; a captured call reuses the address of the
 *     device's last uncaptured call, so make one call before capturing.
 *     No call allocates or frees device memory.
 *   - Every call uses the same array.  Nothing in it needs to start at zero
 *     (each call writes every partial it reads), but calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it and give wrong results: order them on one stream. */
#define BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

bi_status bi_paged_decode_attn_noalloc(const bi_bf16 *q,
                                       const bi_bf16 *k_pool,
                                       const bi_bf16 *v_pool,
                                       const int32_t *page_table,
                                       int max_pages, const int32_t *row_req,
                                       const int32_t *kv_len, int B,
                                       int max_kv_len, int Hq, int Hkv, int D,
                                       float scale, bi_bf16 *out,
                                       void *stream);

/* Several queries per request (prefill, verify).  Rows of segment r are
 * cu_q[r] .. cu_q[r+1]-1 (device int32 [R+1], cu_q[0] = 0,
 * cu_q[R] = T); seg_req int32 [R] is the segment's page-table row;
 * pos int32 [T] the absolute position of each row (causal: a row attends to
 * positions 0..pos).  Rows of a segment hold consecutive positions.  Rows
 * with seg_req < 0 are pad rows and get zeros.  max_q is an upper bound on
 * every segment's length, max_kv_len on every pos + 1.
 * q bf16 [T][Hq][D] -> out bf16 [T][Hq][D]. */
bi_status bi_prefill_attn(const bi_bf16 *q, const int32_t *cu_q,
                          const int32_t *seg_req, int R, int T,
                          const int32_t *pos, int max_q, int max_kv_len,
                          const bi_bf16 *k_pool, const bi_bf16 *v_pool,
                          const int32_t *page_table, int max_pages, int Hq,
                          int Hkv, int D, float scale, bi_bf16 *out,
                          void *stream);

/* Workspace bytes with which bi_prefill_attn_ws runs its persistent path:
 * the query-tile lists of T rows in R segments (0 if the shape has none). */
size_t bi_prefill_attn_workspace_size(int T, int R, int Hq, int Hkv);

/* Workspace bytes with which bi_prefill_attn_ws (head_dim 128, T <= 512:
 * verify-sized batches, LLM-42 section 4.3) spreads every query tile's
 * chunks over the SMs: one work item per (128-row tile, 256-position chunk,
 * KV head) writes the chunk's record (m, l, o) of the decode path's
 * two-stage form, and the decode merge folds the records in chunk order,
 * so the bits are those of decode.  Covers the tile list, the items, every
 * row's context and request and the records [T][Hq][ceil(max_kv_len/256)].
 * 0 when the form does not apply. */
size_t bi_prefill_attn_split_workspace_size(int T, int R, int Hq, int Hkv,
                                            int max_kv_len);

/* bi_prefill_attn with a workspace (device, caller-owned, no initial
 * contents).  For head_dim 128, T <= 512 rows (verify-sized batches),
 * R <= 4096 and ws_bytes >= bi_prefill_attn_workspace_size: one persistent
 * kernel per SM over (16 / G-token query tile, KV head) items sorted by
 * chunk count, with the decode kernel's pipeline and merge, instead of one
 * CTA per (tile, KV head).  Otherwise exactly bi_prefill_attn.  The bits of
 * `out` are the same either way. */
bi_status bi_prefill_attn_ws(const bi_bf16 *q, const int32_t *cu_q,
                             const int32_t *seg_req, int R, int T,
                             const int32_t *pos, int max_q, int max_kv_len,
                             const bi_bf16 *k_pool, const bi_bf16 *v_pool,
                             const int32_t *page_table, int max_pages, int Hq,
                             int Hkv, int D, float scale, bi_bf16 *out,
                             void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------- token selection --
 * Greedy: ids[t] = first index of the maximum of logits[t] (fp32 [T][V]).
 * NaN counts as maximal and the first NaN wins; -0 equals +0.  Exact, so the
 * result is unique (ybb.press section 1: a tiny perturbation flips argmax);
 * a row is searched by a cluster of eight CTAs, whose bests are combined in
 * this total order.  logits 16-byte aligned. */
bi_status bi_argmax_logits(const float *logits, int T, int V, int32_t *ids,
                           void *stream);

/* Temperature sampling with a counter-based generator per request (ybb.press
 * section 6, item 3): seed = (request_id * 1000003 + step) mod 2^64,
 * u = (Philox4x64-10(counter 0, key (seed, 0)) word 0 >> 40) * 2^-24,
 * p_i = exp((logits_i - max) / temperature), evaluated as
 * 2^((logits_i - max) * rn(log2(e) / temperature)) with the base-2
 * exponential (relative error about 2^-22), token = first i whose running
 * sum exceeds u * sum(p) (fixed-order blocked prefix sums over 1024
 * contiguous slices of the row; when rounding leaves none, the last i with
 * p_i > 0).  temperature 0 means greedy, temperature < 0 is refused, and
 * V must be below 2^30.  request_id, step: device uint64 [T].  The result
 * is a function of the row, request_id and step only. */
bi_status philox_sample(const float *logits, int T, int V,
                        const uint64_t *request_id, const uint64_t *step,
                        float temperature, int32_t *ids, void *stream);

/* philox_sample restricted to the top_k most likely tokens and, within
 * them, to the nucleus of mass top_p (the LLM-42 page's sampling
 * hyperparameters, fixed per request).  Tokens are ranked by logit, larger
 * first, equal logits by lower index, NaN as -inf; K = min(top_k, V).  In
 * rank order p_j = exp((l_j - l_0) / temperature) and c_j are the
 * sequential fp32 running sums; the kept tokens are the first n + 1, n the
 * first j < K with c_j >= top_p * c_{K-1} (all K when top_p = 1); the token
 * is the first kept j with c_j > u * c_n (u as in philox_sample), or, when
 * rounding leaves none, the last kept j with p_j > 0.  temperature 0 means
 * greedy.  1 <= top_k (above 1024: BI_ERR_UNSUPPORTED), 0 < top_p <= 1
 * (else BI_ERR_INVALID_ARG).  One block per row; the result is a function
 * of the row, request_id and step only. */
bi_status philox_sample_top(const float *logits, int T, int V,
                            const uint64_t *request_id, const uint64_t *step,
                            float temperature, int top_k, float top_p,
                            int32_t *ids, void *stream);

/* ------------------------------------------------------------ the model --
 * Pre-norm Llama decoder: embed, n_layers x (RMSNorm, QKV GEMM, RoPE + KV
 * append, attention, O GEMM + residual, RMSNorm, gate/up GEMM with SwiGLU,
 * down GEMM + residual), final RMSNorm, LM head with fp32 logits.  The
 * handle keeps pointers only: weights, KV pools and workspace belong to the
 * caller and must outlive it. */
typedef struct {
    int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
    float eps;
    double theta;
    int max_tokens;   /* most rows one forward call may carry */
    int max_kv_len;   /* longest context any row may attend over */
    int max_pages;    /* page-table row stride */
    int n_pages;      /* pages in each layer's pool */
} bi_model_cfg;

typedef struct {
    const bi_bf16 *embed;       /* [V][H] */
    const bi_bf16 *final_norm;  /* [H] */
    const bi_bf16 *lm_head;     /* [V][H] */
    /* host arrays of n_layers device pointers each */
    const bi_bf16 *const *attn_norm;  /* [H] */
    const bi_bf16 *const *wqkv;       /* [(Hq+2Hkv)D][H] */
    const bi_bf16 *const *wo;         /* [H][Hq D] */
    const bi_bf16 *const *ffn_norm;   /* [H] */
    const bi_bf16 *const *wgu;        /* [2F][H], bi_pack_gate_up layout */
    const bi_bf16 *const *wd;         /* [H][F] */
    bi_bf16 *const *k_pool;           /* [n_pages][Hkv][16][D] */
    bi_bf16 *const *v_pool;
} bi_model_weights;

typedef struct bi_model bi_model;

size_t bi_model_workspace_size(const bi_model_cfg *cfg);

bi_status bi_model_create(const bi_model_cfg *cfg, const bi_model_weights *w,
                          void *ws, size_t ws_bytes, bi_model **out);

void bi_model_destroy(bi_model *m);

/* Device address of the model's residual stream in its workspace: bf16
 * [T][hidden] after a bi_model_forward of T rows holds the last layer's
 * output (the hidden state before the final RMSNorm), valid until the next
 * forward.  For inspection; the library never frees it. */
bi_status bi_model_hidden(bi_model *m, void **out);

/* One forward pass over T rows.
 *   tokens, pos, row_req: device int32 [T] (row_req = page-table row,
 *   < 0 for a pad row).
 *   Decode (R == 0): every row is its own request at position pos[t] and
 *   attends to positions 0..pos[t]; max_kv_len bounds pos + 1.
 *   Prefill/verify (R > 0): rows are grouped into R segments by the device
 *   arrays cu_q [R+1] and seg_req [R]; a segment's rows are one request's
 *   consecutive positions; max_q bounds the segment length.
 *   page_table: device int32 [slots][max_pages].
 *   logits: device fp32 [T][V] (may be NULL if only ids are wanted);
 *   ids: device int32 [T] greedy tokens, or NULL. */
bi_status bi_model_forward(bi_model *m, int T, const int32_t *tokens,
                           const int32_t *pos, const int32_t *row_req,
                           int R, const int32_t *cu_q, const int32_t *seg_req,
                           int max_q, int max_kv_len,
                           const int32_t *page_table, float *logits,
                           int32_t *ids, void *stream);

/* Per-kernel-class timing of bi_model_forward for roofline accounting:
 * while enabled, every launch of a class is bracketed by CUDA events recorded
 * on the forward's stream (events are created by the library on first use
 * and reused; no device memory is allocated).  On a stream being captured
 * the events are recorded as event-record nodes of the graph
 * (cudaEventRecordExternal), so replays of that graph time each launch;
 * the pool does not grow during a capture, so run the forward once with
 * profiling enabled before capturing.  bi_model_profile(m, 1) opens
 * a new measurement window, bi_model_profile(m, 0) stops recording.
 * bi_model_profile_read waits for the recorded events and writes, per class,
 * the summed device milliseconds and the launch count into host arrays of
 * BI_PROF_CLASSES entries.  Classes: */
enum {
    BI_PROF_ATTN = 0,         /* decode chunk kernel */
    BI_PROF_ATTN_MERGE = 1,   /* decode chunk merge */
    BI_PROF_GEMM_QKV = 2,
    BI_PROF_GEMM_O = 3,
    BI_PROF_GEMM_GATE_UP = 4, /* with the SwiGLU epilogue */
    BI_PROF_GEMM_DOWN = 5,
    BI_PROF_LM_HEAD = 6,
    BI_PROF_NORM = 7,         /* RMSNorm with the fused split reduction */
    BI_PROF_ROPE = 8,         /* RoPE, QKV reduction and KV append */
    BI_PROF_OTHER = 9,        /* embedding gather, argmax */
    BI_PROF_ATTN_PREFILL = 10, /* prefill / verify attention */
    BI_PROF_CLASSES = 11
};

bi_status bi_model_profile(bi_model *m, int enable);

bi_status bi_model_profile_read(bi_model *m, double *h_ms,
                                int64_t *h_launches);

/* --------------------------------------------------- LLM-42 verification --
 * Grouped verification with commit and rollback ("LLM-42: Enabling
 * Determinism in LLM Inference with Verified Speculation", section
 * "核心方法": paper sections 4.2-4.3, Fig. 8).  Candidate windows of R
 * requests are packed first-in first-out into one fixed BI_VERIFY_ROWS-row
 * batch (pad rows after them), recomputed on the invariant path, and for
 * each request:
 *   j = first i with argmax_i != candidate_i, or w if none,
 *   commit_len = j, kv_len' = kv_len + j, fix_token = argmax_j (or -1),
 *   page-table entries at or past ceil(kv_len' / 16) become -1 and their
 *   page ids are listed in h_freed.
 * Window row i of request r sits at position h_kv_len[r] + i; its input
 * token is h_last_token[r] for i = 0 and candidate i-1 after that, so the
 * cache must hold the request's committed tokens except the last one, and
 * pages for every window position must already be in the page table.
 * Windows that do not fit after the first ones are not taken: *h_taken says
 * how many were.  Two taken windows may not name the same request
 * (BI_ERR_INVALID_ARG).
 *   h_req, h_kv_len, h_last_token, h_win_len: host int32 [R]
 *   h_candidates: host int32 [sum w], windows concatenated
 *   page_table: device int32 [slots][max_pages], updated in place
 *   kv_len: device int32 [slots], entry h_req[r] set to kv_len'
 *   h_commit_len, h_fix_token: host int32 [R] outputs
 *   h_freed: host int32 [freed_cap]; *h_n_freed receives the count
 *   logits: device fp32 [BI_VERIFY_ROWS][V] scratch, kept for inspection.
 * Synchronises `stream` before returning. */
#define BI_VERIFY_ROWS 256

bi_status verify_commit_rollback(bi_model *m, int R, const int32_t *h_req,
                                 const int32_t *h_kv_len,
                                 const int32_t *h_last_token,
                                 const int32_t *h_win_len,
                                 const int32_t *h_candidates,
                                 int32_t *page_table, int32_t *kv_len,
                                 int32_t *h_commit_len, int32_t *h_fix_token,
                                 int32_t *h_freed, int freed_cap,
                                 int32_t *h_n_freed, int32_t *h_taken,
                                 float *logits, void *stream);

/* verify_commit_rollback with its plan and results in device memory: no
 * host synchronisation and no host-dependent launch configuration, so the
 * call can sit in a captured CUDA graph beside the decode iterations (the
 * host reads the results after the replay).  The windows are packed on the
 * device, first-in first-out as above: the forward always runs the same
 * kernels over BI_VERIFY_ROWS rows in BI_VERIFY_ROWS + 1 segments (the
 * taken windows, one pad segment, empty segments).
 *   n_windows: device int32 scalar R, 1 <= R < BI_VERIFY_ROWS
 *   req, win_kv_len, last_token, win_len: device int32 [R] (as h_req,
 *     h_kv_len, h_last_token, h_win_len above)
 *   candidates: device int32, windows concatenated; only the taken
 *     windows' entries (at most BI_VERIFY_ROWS) are read
 *   page_table, kv_len: as above, updated in place
 *   commit_len, fix_token: device int32 [BI_VERIFY_ROWS] (entries of the
 *     taken windows written)
 *   freed: device int32 [freed_cap]; *n_freed (device) receives the count
 *     of pages cut (also those past freed_cap, which are cut but unlisted)
 *   taken: device int32 scalar, windows taken
 *   logits: device fp32 [BI_VERIFY_ROWS][V] scratch.
 * The plan is checked on the device with the rules above, and also
 * against two windows naming one request: a plan that fails takes no
 * window (*taken = 0, nothing committed or cut) and records BI_ERR_BOUNDS
 * in the device status word (bi_device_status).  Requests must be valid
 * page-table rows.  Returns an error before launching only for null
 * pointers or a model built for fewer than BI_VERIFY_ROWS rows. */
bi_status verify_commit_rollback_device(
    bi_model *m, const int32_t *n_windows, const int32_t *req,
    const int32_t *win_kv_len, const int32_t *last_token,
    const int32_t *win_len, const int32_t *candidates, int32_t *page_table,
    int32_t *kv_len, int32_t *commit_len, int32_t *fix_token, int32_t *freed,
    int freed_cap, int32_t *n_freed, int32_t *taken, float *logits,
    void *stream);

#ifdef __cplusplus
}
#endif
#endif /* BI_H */
