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
// that grows on first use and is reused by later measurement windows.  On
// a stream that is being captured the events become event-record nodes of
// the graph (cudaEventRecordExternal), so a replay of that graph times
// every launch without host launch latency inside the brackets; the pool
// does not grow during a capture (such launches go untimed).
struct Profiler {
    bool on = false;
    std::vector<cudaEvent_t> ev;
    size_t next = 0;
    std::vector<std::pair<int, size_t>> marks;  // (class, start index)

    static bool capturing(cudaStream_t s) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        return cudaStreamIsCapturing(s, &cs) == cudaSuccess &&
               cs == cudaStreamCaptureStatusActive;
    }
    static void record(cudaEvent_t e, cudaStream_t s) {
        if (capturing(s))
            cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
        else
            cudaEventRecord(e, s);
    }
    int begin(cudaStream_t s) {
        if (!on) return -1;
        while (ev.size() < next + 2) {
            if (capturing(s)) return -1;
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return -1;
            ev.push_back(e);
        }
        record(ev[next], s);
        return (int)next;
    }
    void end(int cls, int start, cudaStream_t s) {
        if (start < 0) return;
        record(ev[start + 1], s);
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

// Integer scratch of one verify call (device side), in int32 units: the
// packed rows and segments of the fixed batch, the argmax ids, the plan of
// the host entry point (uploaded there) and its outputs (downloaded there).
struct VerifyIdx {
    static constexpr int T = BI_VERIFY_ROWS;
    // segments of the forward: the taken windows, one pad segment, then
    // empty segments up to this fixed count, so that the forward's launch
    // configuration never depends on the plan
    static constexpr int NSEG = T + 1;
    static constexpr int TOK = 0, POS = T, ROWREQ = 2 * T, CAND = 3 * T,
                         CUQ = 4 * T, SEGREQ = 5 * T + 8, SEGSTART = 6 * T + 16,
                         SEGW = 7 * T + 16, SEGKV = 8 * T + 16,
                         IDS = 9 * T + 16, TAKEN = 10 * T + 16,
                         PLAN = 10 * T + 24, PLAN_R = PLAN,
                         PLAN_REQ = PLAN + 8, PLAN_KV = PLAN_REQ + T,
                         PLAN_LAST = PLAN_KV + T, PLAN_WIN = PLAN_LAST + T,
                         PLAN_CAND = PLAN_WIN + T, OUT = PLAN_CAND + T,
                         OUT_TAKEN = OUT, OUT_NFREED = OUT + 1,
                         OUT_COMMIT = OUT + 8, OUT_FIX = OUT_COMMIT + T,
                         OUT_FREED = OUT_FIX + T, COUNT = OUT_FREED;
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
    // decode records of T rows, or the split form of a verify-sized batch
    // (its segments: the taken windows, a pad segment, empty ones)
    L.att_ws = take(std::max(
        bi_decode_attn_workspace_size(T, c.n_heads, c.head_dim, c.max_kv_len),
        bi_prefill_attn_split_ws_bytes(std::min(T, BI_VERIFY_ROWS),
                                       BI_VERIFY_ROWS + 1, c.n_heads,
                                       c.n_kv_heads, c.max_kv_len)));
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

// Packs a verify plan into the fixed batch (LLM-42 section 4.3: windows
// taken first-in first-out while their rows fit).  One block of
// BI_VERIFY_ROWS threads.  The windows' fields are staged in shared memory
// and thread 0 walks them in order, with exactly the checks of the host
// entry point: every window up to the first that does not fit must have
// w >= 1, kv_len >= 0 and req >= 0; every taken window must end within
// max_kv_len and name a request no earlier taken window names.  A plan that
// fails a check (or has R outside [1, BI_VERIFY_ROWS)) takes no window and
// records BI_ERR_BOUNDS; the batch is then all pad rows.  Then thread i
// fills row i: window row k of request r sits at position kv_len_r + k with
// input token last_r (k = 0) or candidate k - 1, compared with candidate k;
// rows after the taken windows are pad rows (token 0, no request).
__global__ void pack_kernel(const int32_t *__restrict__ n_windows,
                            const int32_t *__restrict__ req,
                            const int32_t *__restrict__ kvl,
                            const int32_t *__restrict__ last,
                            const int32_t *__restrict__ win,
                            const int32_t *__restrict__ cand, int max_kv_len,
                            int32_t *__restrict__ vb, int32_t *status) {
    constexpr int T = BI_VERIFY_ROWS;
    __shared__ int s_req[T], s_kv[T], s_w[T], s_start[T];
    __shared__ int s_taken, s_used;
    const int t = threadIdx.x;
    const int R = *n_windows;
    const bool r_ok = R >= 1 && R < T;
    if (r_ok && t < R) {
        s_req[t] = req[t];
        s_kv[t] = kvl[t];
        s_w[t] = win[t];
    }
    __syncthreads();
    if (t == 0) {
        int used = 0, taken = 0;
        bool bad = !r_ok;
        for (int r = 0; !bad && r < R; ++r) {
            const int w = s_w[r];
            if (w < 1 || s_kv[r] < 0 || s_req[r] < 0) {
                bad = true;
                break;
            }
            if (used + w > T) break;
            if (s_kv[r] + w > max_kv_len) {
                bad = true;
                break;
            }
            s_start[r] = used;
            used += w;
            ++taken;
        }
        if (taken == 0) bad = true;
        s_taken = bad ? 0 : taken;
        s_used = bad ? 0 : used;
        if (bad) bi_record_error(status, BI_ERR_BOUNDS);
    }
    __syncthreads();
    int taken = s_taken;
    // a request named by two taken windows would have both write its KV
    // and both commit kernels cut its page-table row: refuse the plan
    bool dup = false;
    if (t < taken)
        for (int i = 0; i < t; ++i) dup |= s_req[i] == s_req[t];
    if (__syncthreads_or(dup)) {
        taken = 0;
        if (t == 0) bi_record_error(status, BI_ERR_BOUNDS);
    }
    const int used = taken > 0 ? s_used : 0;
    // row t
    if (t < used) {
        int lo = 0, hi = taken - 1;  // the last window starting at or before t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_start[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int k = t - s_start[lo];
        vb[VerifyIdx::TOK + t] = k == 0 ? last[lo] : cand[t - 1];
        vb[VerifyIdx::POS + t] = s_kv[lo] + k;
        vb[VerifyIdx::ROWREQ + t] = s_req[lo];
        vb[VerifyIdx::CAND + t] = cand[t];
    } else {
        vb[VerifyIdx::TOK + t] = 0;
        vb[VerifyIdx::POS + t] = t - used;
        vb[VerifyIdx::ROWREQ + t] = -1;
        vb[VerifyIdx::CAND + t] = -1;
    }
    // segments: taken windows, the pad segment, then empty segments
    for (int i = t; i <= VerifyIdx::NSEG; i += T) {
        int cu, sr;
        if (i < taken) {
            cu = s_start[i];
            sr = s_req[i];
        } else if (i == taken) {
            cu = used;
            sr = -1;
        } else {
            cu = T;
            sr = -1;
        }
        vb[VerifyIdx::CUQ + i] = cu;
        if (i < VerifyIdx::NSEG) vb[VerifyIdx::SEGREQ + i] = sr;
    }
    if (t < taken) {
        vb[VerifyIdx::SEGSTART + t] = s_start[t];
        vb[VerifyIdx::SEGW + t] = s_w[t];
        vb[VerifyIdx::SEGKV + t] = s_kv[t];
    }
    if (t == 0) vb[VerifyIdx::TAKEN] = taken;
}

// One thread per taken window: first mismatch, commit, rollback.  The
// freed-page list is laid out request after request, pages in ascending
// table index, by a sequential prefix over the requests (thread 0), so its
// order is fixed.  Pages past freed_cap are cut from the table but not
// listed; *n_freed counts them all.
__global__ void commit_kernel(int max_pages, const int32_t *__restrict__ vb,
                              const int32_t *__restrict__ ids,
                              int32_t *page_table, int32_t *kv_len,
                              int32_t *commit_len, int32_t *fix_token,
                              int32_t *freed, int freed_cap, int32_t *n_freed,
                              int32_t *taken_out) {
    __shared__ int counts[BI_VERIFY_ROWS], offs[BI_VERIFY_ROWS];
    const int r = threadIdx.x;
    const int R = vb[VerifyIdx::TAKEN];
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
        commit_len[r] = j;
        fix_token[r] = j < w ? ids[start + j] : -1;
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
        *n_freed = acc;
        *taken_out = R;
    }
    __syncthreads();
    if (r < R) {
        int at = offs[r];
        for (int p = keep; p < max_pages; ++p) {
            int32_t *e = page_table + (int64_t)req * max_pages + p;
            if (*e >= 0) {
                if (at < freed_cap) freed[at] = *e;
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
            // (the previous layer's SwiGLU output has had its last read)
            BI_TIMED(BI_PROF_NORM,
                     bi_rmsnorm_apply(d, s_d, nullptr, h, m->attn_norm[l], T,
                                      H, c.eps, x, true, s, f,
                                      (size_t)T * F * 2));
        int s_qkv = 0, s_o = 0;
        BI_TIMED(BI_PROF_GEMM_QKV,
                 gemm_slices(x, T, H, m->wqkv[l], QKV, qkv, &s_qkv, s));
        BI_TIMED(BI_PROF_ROPE,
                 bi_rope_apply(qkv, s_qkv, rope_tab, pos, row_req, T, Hq, Hkv,
                               D, c.theta, q, m->kpool[l], m->vpool[l],
                               page_table, c.max_pages, c.n_pages, s, true,
                               x, (size_t)T * H * 2));  // x: QKV's input
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
                                          att_ws, att_ws_bytes, s,
                                          /* list of layer 0 */ l > 0));
        }
        BI_TIMED(BI_PROF_GEMM_O,
                 gemm_slices(attn, T, QD, m->wo[l], H, o, &s_o, s));
        // (the queries and the attention output have had their last reads)
        BI_TIMED(BI_PROF_NORM,
                 bi_rmsnorm_apply(o, s_o, nullptr, h, m->ffn_norm[l], T, H,
                                  c.eps, x, true, s, attn,
                                  (size_t)T * QD * 2, q, (size_t)T * QD * 2));
        BI_TIMED(BI_PROF_GEMM_GATE_UP,
                 bi_gemm(x, T, H, m->wgu[l], 2 * F, f, BI_OUT_SWIGLU,
                         gemm_ws, gemm_ws_bytes, s));
        BI_TIMED(BI_PROF_GEMM_DOWN,
                 gemm_slices(f, T, F, m->wd[l], H, d, &s_d, s));
    }
    BI_TIMED(BI_PROF_NORM,
             bi_rmsnorm_apply(d, s_d, nullptr, h, m->final_norm, T, H, c.eps,
                              x, true, s, f, (size_t)T * F * 2));
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

extern "C" bi_status bi_model_hidden(bi_model *m, void **out) {
    BI_REQUIRE(m && out, "bi_model_hidden: null pointer");
    *out = m->ws + m->L.h;
    return BI_OK;
}

extern "C" bi_status verify_commit_rollback_device(
    bi_model *m, const int32_t *n_windows, const int32_t *req,
    const int32_t *win_kv_len, const int32_t *last_token,
    const int32_t *win_len, const int32_t *candidates, int32_t *page_table,
    int32_t *kv_len, int32_t *commit_len, int32_t *fix_token, int32_t *freed,
    int freed_cap, int32_t *n_freed, int32_t *taken, float *logits,
    void *stream) {
    BI_REQUIRE(m, "verify_commit_rollback: null model");
    const bi_model_cfg &c = m->cfg;
    BI_REQUIRE(c.max_tokens >= BI_VERIFY_ROWS,
               "verify_commit_rollback: model built for %d rows < %d",
               c.max_tokens, BI_VERIFY_ROWS);
    BI_REQUIRE(n_windows && req && win_kv_len && last_token && win_len &&
                   candidates && page_table && kv_len && commit_len &&
                   fix_token && n_freed && taken && logits &&
                   (freed || freed_cap == 0) && freed_cap >= 0,
               "verify_commit_rollback: null pointer");
    const int T = BI_VERIFY_ROWS;
    cudaStream_t s = bi_stream(stream);
    int32_t *dvb = reinterpret_cast<int32_t *>(m->ws + m->L.vbuf);
    pack_kernel<<<1, T, 0, s>>>(n_windows, req, win_kv_len, last_token,
                                win_len, candidates, c.max_kv_len, dvb,
                                bi_status_ptr());
    BI_LAUNCH_CHECK("verify pack launch");
    int32_t *ids = dvb + VerifyIdx::IDS;
    bi_status st = bi_model_forward(
        m, T, dvb + VerifyIdx::TOK, dvb + VerifyIdx::POS,
        dvb + VerifyIdx::ROWREQ, VerifyIdx::NSEG, dvb + VerifyIdx::CUQ,
        dvb + VerifyIdx::SEGREQ, T, c.max_kv_len, page_table, logits, ids,
        stream);
    if (st != BI_OK) return st;
    commit_kernel<<<1, T, 0, s>>>(c.max_pages, dvb, ids, page_table, kv_len,
                                  commit_len, fix_token, freed, freed_cap,
                                  n_freed, taken);
    BI_LAUNCH_CHECK("verify commit launch");
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
                   h_n_freed && h_taken && logits &&
                   (h_freed || freed_cap == 0) && freed_cap >= 0,
               "verify_commit_rollback: null pointer");
    const int T = BI_VERIFY_ROWS;
    // The checks of the device-side packing, made here first so that a bad
    // plan is refused before anything is launched.
    int used = 0, taken = 0;
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
        for (int i = 0; i < taken; ++i)
            BI_REQUIRE(h_req[i] != h_req[r],
                       "verify_commit_rollback: windows %d and %d both name "
                       "request %d",
                       i, r, h_req[r]);
        used += w;
        ++taken;
    }
    BI_REQUIRE(taken >= 1, "verify_commit_rollback: first window longer than "
                           "%d rows",
               T);
    // Plan upload: the windows (the device packs only the taken ones, whose
    // candidates are the first `used` entries).
    std::vector<int32_t> plan(VerifyIdx::OUT - VerifyIdx::PLAN, 0);
    plan[VerifyIdx::PLAN_R - VerifyIdx::PLAN] = R;
    for (int r = 0; r < R; ++r) {
        plan[VerifyIdx::PLAN_REQ - VerifyIdx::PLAN + r] = h_req[r];
        plan[VerifyIdx::PLAN_KV - VerifyIdx::PLAN + r] = h_kv_len[r];
        plan[VerifyIdx::PLAN_LAST - VerifyIdx::PLAN + r] = h_last_token[r];
        plan[VerifyIdx::PLAN_WIN - VerifyIdx::PLAN + r] = h_win_len[r];
    }
    for (int i = 0; i < used; ++i)
        plan[VerifyIdx::PLAN_CAND - VerifyIdx::PLAN + i] = h_candidates[i];
    cudaStream_t s = bi_stream(stream);
    int32_t *dvb = reinterpret_cast<int32_t *>(m->ws + m->L.vbuf);
    bi_status st = bi_cuda_check(
        cudaMemcpyAsync(dvb + VerifyIdx::PLAN, plan.data(),
                        plan.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                        s),
        "verify: plan upload");
    if (st != BI_OK) return st;
    const int cap = c.max_pages * BI_VERIFY_ROWS;
    st = verify_commit_rollback_device(
        m, dvb + VerifyIdx::PLAN_R, dvb + VerifyIdx::PLAN_REQ,
        dvb + VerifyIdx::PLAN_KV, dvb + VerifyIdx::PLAN_LAST,
        dvb + VerifyIdx::PLAN_WIN, dvb + VerifyIdx::PLAN_CAND, page_table,
        kv_len, dvb + VerifyIdx::OUT_COMMIT, dvb + VerifyIdx::OUT_FIX,
        dvb + VerifyIdx::OUT_FREED, cap, dvb + VerifyIdx::OUT_NFREED,
        dvb + VerifyIdx::OUT_TAKEN, logits, stream);
    if (st != BI_OK) return st;
    std::vector<int32_t> outv(VerifyIdx::OUT_FREED - VerifyIdx::OUT);
    st = bi_cuda_check(
        cudaMemcpyAsync(outv.data(), dvb + VerifyIdx::OUT,
                        outv.size() * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        s),
        "verify: result download");
    if (st != BI_OK) return st;
    st = bi_cuda_check(cudaStreamSynchronize(s), "verify: sync");
    if (st != BI_OK) return st;
    const int nfreed = outv[VerifyIdx::OUT_NFREED - VerifyIdx::OUT];
    const int got = outv[VerifyIdx::OUT_TAKEN - VerifyIdx::OUT];
    if (got != taken)
        return bi_fail(BI_ERR_CUDA,
                       "verify_commit_rollback: device packed %d windows, "
                       "host %d",
                       got, taken);
    for (int r = 0; r < taken; ++r) {
        h_commit_len[r] = outv[VerifyIdx::OUT_COMMIT - VerifyIdx::OUT + r];
        h_fix_token[r] = outv[VerifyIdx::OUT_FIX - VerifyIdx::OUT + r];
    }
    *h_n_freed = nfreed;
    *h_taken = taken;
    const int listed = std::min(std::min(nfreed, freed_cap), cap);
    if (listed > 0) {
        st = bi_cuda_check(
            cudaMemcpyAsync(h_freed, dvb + VerifyIdx::OUT_FREED,
                            (size_t)listed * sizeof(int32_t),
                            cudaMemcpyDeviceToHost, s),
            "verify: freed pages download");
        if (st != BI_OK) return st;
        st = bi_cuda_check(cudaStreamSynchronize(s), "verify: sync");
        if (st != BI_OK) return st;
    }
    if (nfreed > freed_cap)
        return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                       "verify_commit_rollback: %d pages freed, room for %d "
                       "(the rollback itself was applied)",
                       nfreed, freed_cap);
    return BI_OK;
}
