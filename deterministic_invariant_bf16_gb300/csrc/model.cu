// Model driver (bi_model_*) and LLM-42 grouped verification
// (verify_commit_rollback).
//
// The driver runs the pre-norm Llama block stack over caller-owned weights,
// KV pools and workspace.  Every launch goes to the caller's stream, so a
// caller may capture a whole forward pass in a CUDA graph.  The GEMMs write
// their fixed K slices as fp32 partials that the next kernel (RoPE, RMSNorm)
// sums in slice order; the gate/up GEMM applies SwiGLU in its epilogue.
//
// Verification follows "LLM-42: Enabling Determinism in LLM Inference with
// Verified Speculation", section "核心方法" (paper sections 4.2-4.3, Fig. 8):
// candidate windows of several requests are packed into one fixed
// 256-row batch, recomputed on the invariant path, and each request commits
// the prefix that the recomputation reproduces; at the first mismatch the
// later candidates are dropped and the KV cache is cut back to the
// committed prefix.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace {

// Per-kernel-class event timing (bi_model_profile).  Events come from a pool
// that grows on first use and is reused by later measurement windows.
struct Profiler {
    bool on = false;
    std::vector<cudaEvent_t> ev;
    size_t next = 0;
    std::vector<std::pair<int, size_t>> marks;  // (class, start index)

    int begin(cudaStream_t s) {
        if (!on) return -1;
        while (ev.size() < next + 2) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return -1;
            ev.push_back(e);
        }
        cudaEventRecord(ev[next], s);
        return (int)next;
    }
    void end(int cls, int start, cudaStream_t s) {
        if (start < 0) return;
        cudaEventRecord(ev[start + 1], s);
        marks.emplace_back(cls, (size_t)start);
        next = start + 2;
    }
    ~Profiler() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    size_t h, x, qkv, q, attn, o, f, d, gemm_ws, att_ws, kvlen, rope, vbuf,
        total;
    int S_qkv, S_o, S_d;
};

// Integer scratch of one verify call (device side), in int32 units.
struct VerifyIdx {
    static constexpr int T = BI_VERIFY_ROWS;
    static constexpr int TOK = 0, POS = T, ROWREQ = 2 * T, CAND = 3 * T,
                         CUQ = 4 * T, SEGREQ = 5 * T + 8, SEGSTART = 6 * T + 16,
                         SEGW = 7 * T + 16, SEGKV = 8 * T + 16,
                         IDS = 9 * T + 16, PACKED = 9 * T + 16,
                         OUT_COMMIT = 10 * T + 16, OUT_FIX = 11 * T + 16,
                         OUT_NFREED = 12 * T + 16, OUT_FREED = 12 * T + 32,
                         COUNT = 12 * T + 32;
};

Layout layout(const bi_model_cfg &c, int max_pages_total) {
    Layout L;
    const int T = c.max_tokens, H = c.hidden, F = c.ffn;
    const int QD = c.n_heads * c.head_dim;
    const int QKV = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    L.S_qkv = bi_gemm_splits(QKV, H);
    L.S_o = bi_gemm_splits(H, QD);
    L.S_d = bi_gemm_splits(H, F);
    size_t at = 0;
    auto take = [&](size_t bytes) {
        size_t r = at;
        at += align256(bytes);
        return r;
    };
    L.h = take((size_t)T * H * 2);
    L.x = take((size_t)T * H * 2);
    L.qkv = take((size_t)L.S_qkv * T * QKV * 4);
    L.q = take((size_t)T * QD * 2);
    L.attn = take((size_t)T * QD * 2);
    L.o = take((size_t)L.S_o * T * H * 4);
    L.f = take((size_t)T * F * 2);
    L.d = take((size_t)L.S_d * T * H * 4);
    // second-stage workspace of the gate/up and LM-head GEMMs (only for
    // shapes with more than one K slice)
    L.gemm_ws = take(std::max(bi_gemm_workspace_size(T, 2 * F, H),
                              bi_gemm_workspace_size(T, c.vocab, H)));
    L.att_ws = take(bi_decode_attn_workspace_size(T, c.n_heads, c.head_dim,
                                                  c.max_kv_len));
    L.kvlen = take((size_t)T * 4);
    L.rope = take((size_t)T * (c.head_dim / 2) * 8);
    L.vbuf = take((size_t)(VerifyIdx::COUNT + max_pages_total) * 4);
    L.total = at;
    return L;
}

__global__ void kvlen_kernel(const int32_t *pos, int T, int32_t *kvlen) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < T) kvlen[t] = pos[t] + 1;
}

// One thread per packed request: first mismatch, commit, rollback.  The
// freed-page list is laid out request after request, pages in ascending
// table index, by a sequential prefix over the requests (thread 0), so its
// order is fixed.
__global__ void commit_kernel(int R, int max_pages, int32_t *vb,
                              const int32_t *ids, int32_t *page_table,
                              int32_t *kv_len, int freed_cap) {
    __shared__ int counts[BI_VERIFY_ROWS], offs[BI_VERIFY_ROWS];
    const int r = threadIdx.x;
    int j = 0, w = 0, newlen = 0, req = -1, keep = 0;
    if (r < R) {
        const int start = vb[VerifyIdx::SEGSTART + r];
        w = vb[VerifyIdx::SEGW + r];
        req = vb[VerifyIdx::SEGREQ + r];
        j = w;
        for (int i = 0; i < w; ++i)
            if (ids[start + i] != vb[VerifyIdx::CAND + start + i]) {
                j = i;
                break;
            }
        newlen = vb[VerifyIdx::SEGKV + r] + j;
        vb[VerifyIdx::OUT_COMMIT + r] = j;
        vb[VerifyIdx::OUT_FIX + r] = j < w ? ids[start + j] : -1;
        keep = (newlen + 15) / 16;
        int cnt = 0;
        for (int p = keep; p < max_pages; ++p)
            if (page_table[(int64_t)req * max_pages + p] >= 0) ++cnt;
        counts[r] = cnt;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int i = 0; i < R; ++i) {
            offs[i] = acc;
            acc += counts[i];
        }
        vb[VerifyIdx::OUT_NFREED] = acc;
    }
    __syncthreads();
    if (r < R) {
        int at = offs[r];
        for (int p = keep; p < max_pages; ++p) {
            int32_t *e = page_table + (int64_t)req * max_pages + p;
            if (*e >= 0) {
                if (at < freed_cap) vb[VerifyIdx::OUT_FREED + at] = *e;
                ++at;
                *e = -1;
            }
        }
        kv_len[req] = newlen;
    }
}

}  // namespace

struct bi_model {
    bi_model_cfg cfg;
    Layout L;
    uint8_t *ws;
    const bi_bf16 *embed, *final_norm, *lm_head;
    std::vector<const bi_bf16 *> attn_norm, wqkv, wo, ffn_norm, wgu, wd;
    std::vector<bi_bf16 *> kpool, vpool;
    Profiler prof;
};

extern "C" bi_status bi_model_profile(bi_model *m, int enable) {
    BI_REQUIRE(m, "bi_model_profile: null model");
    m->prof.on = enable != 0;
    m->prof.next = 0;
    m->prof.marks.clear();
    return BI_OK;
}

extern "C" bi_status bi_model_profile_read(bi_model *m, double *h_ms,
                                           int64_t *h_launches) {
    BI_REQUIRE(m && h_ms && h_launches, "bi_model_profile_read: null pointer");
    for (int c = 0; c < BI_PROF_CLASSES; ++c) {
        h_ms[c] = 0.0;
        h_launches[c] = 0;
    }
    for (auto &mk : m->prof.marks) {
        cudaEvent_t a = m->prof.ev[mk.second], b = m->prof.ev[mk.second + 1];
        bi_status st = bi_cuda_check(cudaEventSynchronize(b), "profile sync");
        if (st != BI_OK) return st;
        float ms = 0.f;
        st = bi_cuda_check(cudaEventElapsedTime(&ms, a, b), "profile elapsed");
        if (st != BI_OK) return st;
        h_ms[mk.first] += ms;
        h_launches[mk.first] += 1;
    }
    return BI_OK;
}

static bi_status check_cfg(const bi_model_cfg *c) {
    BI_REQUIRE(c, "bi_model: null cfg");
    BI_REQUIRE(c->n_layers > 0 && c->hidden > 0 && c->n_heads > 0 &&
                   c->n_kv_heads > 0 && c->ffn > 0 && c->vocab > 0 &&
                   c->max_tokens > 0 && c->max_kv_len > 0 &&
                   c->max_pages > 0 && c->n_pages > 0,
               "bi_model: non-positive size in cfg");
    BI_REQUIRE(c->hidden % 64 == 0 && c->ffn % 64 == 0,
               "bi_model: hidden and ffn must be multiples of 64");
    if (c->head_dim != 32 && c->head_dim != 128)
        return bi_fail(BI_ERR_UNSUPPORTED, "bi_model: head_dim %d",
                       c->head_dim);
    BI_REQUIRE(c->n_heads % c->n_kv_heads == 0, "bi_model: GQA grouping");
    BI_REQUIRE(c->max_kv_len <= 16 * c->max_pages,
               "bi_model: max_kv_len beyond the page-table row");
    return BI_OK;
}

extern "C" size_t bi_model_workspace_size(const bi_model_cfg *cfg) {
    if (check_cfg(cfg) != BI_OK) return 0;
    return layout(*cfg, cfg->max_pages * BI_VERIFY_ROWS).total;
}

extern "C" bi_status bi_model_create(const bi_model_cfg *cfg,
                                     const bi_model_weights *w, void *ws,
                                     size_t ws_bytes, bi_model **out) {
    bi_status st = check_cfg(cfg);
    if (st != BI_OK) return st;
    BI_REQUIRE(w && out && ws, "bi_model_create: null pointer");
    const Layout L = layout(*cfg, cfg->max_pages * BI_VERIFY_ROWS);
    if (ws_bytes < L.total)
        return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                       "bi_model_create: workspace %zu < %zu", ws_bytes,
                       L.total);
    BI_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255) == 0,
               "bi_model_create: workspace must be 256-byte aligned");
    BI_REQUIRE(w->embed && w->final_norm && w->lm_head && w->attn_norm &&
                   w->wqkv && w->wo && w->ffn_norm && w->wgu && w->wd &&
                   w->k_pool && w->v_pool,
               "bi_model_create: null weight pointer");
    bi_model *m = new bi_model;
    m->cfg = *cfg;
    m->L = L;
    m->ws = static_cast<uint8_t *>(ws);
    m->embed = w->embed;
    m->final_norm = w->final_norm;
    m->lm_head = w->lm_head;
    for (int l = 0; l < cfg->n_layers; ++l) {
        const void *ptrs[] = {w->attn_norm[l], w->wqkv[l], w->wo[l],
                              w->ffn_norm[l], w->wgu[l],  w->wd[l],
                              w->k_pool[l],    w->v_pool[l]};
        for (const void *p : ptrs)
            if (!p || !bi_aligned16(p)) {
                delete m;
                return bi_fail(BI_ERR_INVALID_ARG,
                               "bi_model_create: layer %d pointer null or "
                               "misaligned",
                               l);
            }
        m->attn_norm.push_back(w->attn_norm[l]);
        m->wqkv.push_back(w->wqkv[l]);
        m->wo.push_back(w->wo[l]);
        m->ffn_norm.push_back(w->ffn_norm[l]);
        m->wgu.push_back(w->wgu[l]);
        m->wd.push_back(w->wd[l]);
        m->kpool.push_back(w->k_pool[l]);
        m->vpool.push_back(w->v_pool[l]);
    }
    *out = m;
    return BI_OK;
}

extern "C" void bi_model_destroy(bi_model *m) { delete m; }

// GEMM whose result a split-aware consumer reads: the S fp32 slice
// partials go to `out`; *slices = S.
static bi_status gemm_slices(const bi_bf16 *x, int M, int K, const bi_bf16 *W,
                             int N, float *out, int *slices,
                             cudaStream_t s) {
    *slices = bi_gemm_splits(N, K);
    return bi_gemm(x, M, K, W, N, out, BI_OUT_PARTIALS, nullptr, 0, s);
}

extern "C" bi_status bi_model_forward(bi_model *m, int T, const int32_t *tokens,
                                      const int32_t *pos,
                                      const int32_t *row_req, int R,
                                      const int32_t *cu_q,
                                      const int32_t *seg_req, int max_q,
                                      int max_kv_len,
                                      const int32_t *page_table, float *logits,
                                      int32_t *ids, void *stream) {
    BI_REQUIRE(m, "bi_model_forward: null model");
    const bi_model_cfg &c = m->cfg;
    BI_REQUIRE(T >= 0 && T <= c.max_tokens,
               "bi_model_forward: T=%d outside [0, %d]", T, c.max_tokens);
    BI_REQUIRE(max_kv_len > 0 && max_kv_len <= c.max_kv_len,
               "bi_model_forward: max_kv_len=%d outside [1, %d]", max_kv_len,
               c.max_kv_len);
    BI_REQUIRE(tokens && pos && row_req && page_table && logits,
               "bi_model_forward: null pointer");
    BI_REQUIRE(R >= 0, "bi_model_forward: R=%d", R);
    BI_REQUIRE(R == 0 || (cu_q && seg_req && max_q > 0),
               "bi_model_forward: segments need cu_q, seg_req, max_q");
    if (T == 0) return BI_OK;
    cudaStream_t s = bi_stream(stream);
    const int H = c.hidden, D = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads;
    const int QD = Hq * D, QKV = (Hq + 2 * Hkv) * D, F = c.ffn;
    const float scale = 1.0f / sqrtf((float)D);
    uint8_t *ws = m->ws;
    bi_bf16 *h = reinterpret_cast<bi_bf16 *>(ws + m->L.h);
    bi_bf16 *x = reinterpret_cast<bi_bf16 *>(ws + m->L.x);
    float *qkv = reinterpret_cast<float *>(ws + m->L.qkv);
    bi_bf16 *q = reinterpret_cast<bi_bf16 *>(ws + m->L.q);
    bi_bf16 *attn = reinterpret_cast<bi_bf16 *>(ws + m->L.attn);
    float *o = reinterpret_cast<float *>(ws + m->L.o);
    bi_bf16 *f = reinterpret_cast<bi_bf16 *>(ws + m->L.f);
    float *d = reinterpret_cast<float *>(ws + m->L.d);
    void *att_ws = ws + m->L.att_ws;
    void *gemm_ws = ws + m->L.gemm_ws;
    const size_t gemm_ws_bytes = m->L.att_ws - m->L.gemm_ws;
    int32_t *kvlen = reinterpret_cast<int32_t *>(ws + m->L.kvlen);
    float2 *rope_tab = reinterpret_cast<float2 *>(ws + m->L.rope);
    const size_t att_ws_bytes = m->L.kvlen - m->L.att_ws;

    bi_status st;
#define BI_TRY(expr)                       \
    do {                                   \
        if ((st = (expr)) != BI_OK) return st; \
    } while (0)

    Profiler &P = m->prof;
    int ev;
#define BI_TIMED(cls, expr)           \
    do {                              \
        ev = P.begin(s);              \
        BI_TRY(expr);                 \
        P.end((cls), ev, s);          \
    } while (0)

    BI_TIMED(BI_PROF_OTHER, bi_embed(tokens, T, m->embed, c.vocab, H, h, s));
    BI_TIMED(BI_PROF_ROPE, bi_rope_table(pos, T, D, c.theta, rope_tab, s));
    if (R == 0) {
        kvlen_kernel<<<(T + 255) / 256, 256, 0, s>>>(pos, T, kvlen);
        BI_LAUNCH_CHECK("kvlen launch");
    }
    int s_d = 0;
    for (int l = 0; l < c.n_layers; ++l) {
        if (l == 0)
            BI_TIMED(BI_PROF_NORM,
                     bi_rmsnorm(nullptr, 0, nullptr, h, m->attn_norm[l], T, H,
                                c.eps, x, s));
        else
            BI_TIMED(BI_PROF_NORM, bi_rmsnorm(d, s_d, nullptr, h,
                                              m->attn_norm[l], T, H, c.eps, x,
                                              s));
        int s_qkv = 0, s_o = 0;
        BI_TIMED(BI_PROF_GEMM_QKV,
                 gemm_slices(x, T, H, m->wqkv[l], QKV, qkv, &s_qkv, s));
        BI_TIMED(BI_PROF_ROPE,
                 bi_rope_apply(qkv, s_qkv, rope_tab, pos, row_req, T, Hq, Hkv,
                               D, c.theta, q, m->kpool[l], m->vpool[l],
                               page_table, c.max_pages, c.n_pages, s));
        if (R == 0) {
            BI_TIMED(BI_PROF_ATTN,
                     bi_decode_attn_pool(q, m->kpool[l], m->vpool[l],
                                         page_table, c.max_pages, c.n_pages,
                                         row_req, kvlen, T, max_kv_len, Hq,
                                         Hkv, D, scale, attn, att_ws,
                                         att_ws_bytes, l == 0 ? 1 : 1 | 4, s));
            // whole-row items: the kernel merges and writes attn itself
            if (!bi_decode_whole_rows(T, Hkv, D)) {
                BI_TIMED(BI_PROF_ATTN_MERGE,
                         bi_decode_attn_pool(q, m->kpool[l], m->vpool[l],
                                             page_table, c.max_pages,
                                             c.n_pages, row_req, kvlen, T,
                                             max_kv_len, Hq, Hkv, D, scale,
                                             attn, att_ws, att_ws_bytes, 2,
                                             s));
            }
        } else {
            BI_TIMED(BI_PROF_ATTN_PREFILL,
                     bi_prefill_attn_pool(q, cu_q, seg_req, R, T, pos, max_q,
                                          max_kv_len, m->kpool[l],
                                          m->vpool[l], page_table, c.max_pages,
                                          c.n_pages, Hq, Hkv, D, scale, attn,
                                          att_ws, att_ws_bytes, s));
        }
        BI_TIMED(BI_PROF_GEMM_O,
                 gemm_slices(attn, T, QD, m->wo[l], H, o, &s_o, s));
        BI_TIMED(BI_PROF_NORM, bi_rmsnorm(o, s_o, nullptr, h, m->ffn_norm[l],
                                          T, H, c.eps, x, s));
        BI_TIMED(BI_PROF_GEMM_GATE_UP,
                 bi_gemm(x, T, H, m->wgu[l], 2 * F, f, BI_OUT_SWIGLU,
                         gemm_ws, gemm_ws_bytes, s));
        BI_TIMED(BI_PROF_GEMM_DOWN,
                 gemm_slices(f, T, F, m->wd[l], H, d, &s_d, s));
    }
    BI_TIMED(BI_PROF_NORM, bi_rmsnorm(d, s_d, nullptr, h, m->final_norm, T, H,
                                      c.eps, x, s));
    BI_TIMED(BI_PROF_LM_HEAD,
             bi_gemm(x, T, H, m->lm_head, c.vocab, logits, BI_OUT_F32,
                     gemm_ws, gemm_ws_bytes, s));
    if (ids)
        BI_TIMED(BI_PROF_OTHER,
                 bi_argmax_logits(logits, T, c.vocab, ids, s));
#undef BI_TIMED
#undef BI_TRY
    return BI_OK;
}

extern "C" bi_status verify_commit_rollback(
    bi_model *m, int R, const int32_t *h_req, const int32_t *h_kv_len,
    const int32_t *h_last_token, const int32_t *h_win_len,
    const int32_t *h_candidates, int32_t *page_table, int32_t *kv_len,
    int32_t *h_commit_len, int32_t *h_fix_token, int32_t *h_freed,
    int freed_cap, int32_t *h_n_freed, int32_t *h_taken, float *logits,
    void *stream) {
    BI_REQUIRE(m, "verify_commit_rollback: null model");
    const bi_model_cfg &c = m->cfg;
    BI_REQUIRE(R >= 1 && R < BI_VERIFY_ROWS, "verify_commit_rollback: R=%d", R);
    BI_REQUIRE(c.max_tokens >= BI_VERIFY_ROWS,
               "verify_commit_rollback: model built for %d rows < %d",
               c.max_tokens, BI_VERIFY_ROWS);
    BI_REQUIRE(h_req && h_kv_len && h_last_token && h_win_len && h_candidates &&
                   page_table && kv_len && h_commit_len && h_fix_token &&
                   h_n_freed && h_taken && logits && (h_freed || freed_cap == 0),
               "verify_commit_rollback: null pointer");
    const int T = BI_VERIFY_ROWS;
    // ---- FIFO packing into the fixed-shape batch (host).
    std::vector<int32_t> vb(VerifyIdx::PACKED, 0);
    int used = 0, taken = 0, cand_at = 0, max_w = 1, max_kv = 1;
    for (int r = 0; r < R; ++r) {
        const int w = h_win_len[r];
        BI_REQUIRE(w >= 1, "verify_commit_rollback: window %d has length %d", r,
                   w);
        BI_REQUIRE(h_kv_len[r] >= 0 && h_req[r] >= 0,
                   "verify_commit_rollback: window %d bad kv_len/req", r);
        if (used + w > T) break;
        BI_REQUIRE(h_kv_len[r] + w <= c.max_kv_len,
                   "verify_commit_rollback: window %d reaches %d > max_kv_len",
                   r, h_kv_len[r] + w);
        for (int i = 0; i < w; ++i) {
            const int row = used + i;
            vb[VerifyIdx::TOK + row] =
                i == 0 ? h_last_token[r] : h_candidates[cand_at + i - 1];
            vb[VerifyIdx::POS + row] = h_kv_len[r] + i;
            vb[VerifyIdx::ROWREQ + row] = h_req[r];
            vb[VerifyIdx::CAND + row] = h_candidates[cand_at + i];
        }
        vb[VerifyIdx::CUQ + taken] = used;
        vb[VerifyIdx::SEGREQ + taken] = h_req[r];
        vb[VerifyIdx::SEGSTART + taken] = used;
        vb[VerifyIdx::SEGW + taken] = w;
        vb[VerifyIdx::SEGKV + taken] = h_kv_len[r];
        max_w = std::max(max_w, w);
        max_kv = std::max(max_kv, h_kv_len[r] + w);
        used += w;
        cand_at += w;
        ++taken;
    }
    BI_REQUIRE(taken >= 1, "verify_commit_rollback: first window longer than "
                           "%d rows",
               T);
    // Pad rows form one extra segment with no request.
    int nseg = taken;
    for (int row = used; row < T; ++row) {
        vb[VerifyIdx::TOK + row] = 0;
        vb[VerifyIdx::POS + row] = row - used;
        vb[VerifyIdx::ROWREQ + row] = -1;
        vb[VerifyIdx::CAND + row] = -1;
    }
    if (used < T) {
        vb[VerifyIdx::CUQ + nseg] = used;
        vb[VerifyIdx::SEGREQ + nseg] = -1;
        ++nseg;
        max_w = std::max(max_w, T - used);
        max_kv = std::max(max_kv, T - used);
    }
    vb[VerifyIdx::CUQ + nseg] = T;

    cudaStream_t s = bi_stream(stream);
    int32_t *dvb = reinterpret_cast<int32_t *>(m->ws + m->L.vbuf);
    bi_status st = bi_cuda_check(
        cudaMemcpyAsync(dvb, vb.data(), vb.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s),
        "verify: pack upload");
    if (st != BI_OK) return st;
    int32_t *ids = dvb + VerifyIdx::IDS;
    st = bi_model_forward(m, T, dvb + VerifyIdx::TOK, dvb + VerifyIdx::POS,
                          dvb + VerifyIdx::ROWREQ, nseg, dvb + VerifyIdx::CUQ,
                          dvb + VerifyIdx::SEGREQ, max_w,
                          std::min(max_kv, c.max_kv_len), page_table, logits,
                          ids, stream);
    if (st != BI_OK) return st;
    commit_kernel<<<1, BI_VERIFY_ROWS, 0, s>>>(
        taken, c.max_pages, dvb, ids, page_table, kv_len,
        c.max_pages * BI_VERIFY_ROWS);
    BI_LAUNCH_CHECK("verify commit launch");
    std::vector<int32_t> outv(VerifyIdx::OUT_FREED - VerifyIdx::OUT_COMMIT);
    st = bi_cuda_check(
        cudaMemcpyAsync(outv.data(), dvb + VerifyIdx::OUT_COMMIT,
                        outv.size() * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        s),
        "verify: result download");
    if (st != BI_OK) return st;
    st = bi_cuda_check(cudaStreamSynchronize(s), "verify: sync");
    if (st != BI_OK) return st;
    const int nfreed = outv[VerifyIdx::OUT_NFREED - VerifyIdx::OUT_COMMIT];
    for (int r = 0; r < taken; ++r) {
        h_commit_len[r] = outv[r];
        h_fix_token[r] = outv[VerifyIdx::OUT_FIX - VerifyIdx::OUT_COMMIT + r];
    }
    *h_n_freed = nfreed;
    *h_taken = taken;
    if (nfreed > 0 && freed_cap > 0) {
        st = bi_cuda_check(
            cudaMemcpy(h_freed, dvb + VerifyIdx::OUT_FREED,
                       (size_t)std::min(nfreed, freed_cap) * sizeof(int32_t),
                       cudaMemcpyDeviceToHost),
            "verify: freed pages download");
        if (st != BI_OK) return st;
    }
    if (nfreed > freed_cap)
        return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                       "verify_commit_rollback: %d pages freed, room for %d "
                       "(the rollback itself was applied)",
                       nfreed, freed_cap);
    return BI_OK;
}
