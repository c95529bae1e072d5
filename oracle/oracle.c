/*
 * Oracle for the batch-invariant bf16 decoder and the LLM-42 commit rule.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, sequential CPU
 * statement of what the GPU library computes.  Only the test suite, the
 * package smoke check and the CPU-baseline leg of the benchmark may load it;
 * the product path never does, and it shares no code, header or table with
 * the CUDA library.
 *
 * Rules followed throughout:
 *   - every reduction runs sequentially in index order with an fp32
 *     accumulator ("Batch-Invariant Kernel" section of the ybb.press article on
 *     inference determinism: the reduction order depends only on the data);
 *   - parallelism (OpenMP) is used only across independent outputs, so the
 *     result of any output never depends on the thread count;
 *   - built with -O2 -fno-fast-math -ffp-contract=off, so every fp32 multiply
 *     and add is separately rounded (IEEE-754 round to nearest even).
 *
 * bf16 values travel as uint16 bit patterns; fp32 everywhere else.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
static inline float bf16_bits_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even (bfloat16 keeps 8 mantissa
 * bits; ybb.press article, section 2.1).  NaN becomes the canonical quiet
 * NaN 0x7FC0. */
static inline uint16_t f32_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)0x7fc0u;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

void orc_f32_to_bf16(const float *x, int64_t n, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_bits(x[i]);
}

void orc_bf16_to_f32(const uint16_t *x, int64_t n, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_bits_to_f32(x[i]);
}

/* ------------------------------------------------- non-associativity -- */

/* The fp32 example of the ybb.press article, section 2.1: with a = 1e8,
 * b = -1e8, c = 1 the left grouping gives 1 and the right grouping 0. */
void orc_nonassoc_demo(float a, float b, float c, float *left, float *right)
{
    volatile float ab = a + b;
    volatile float bc = b + c;
    *left = ab + c;
    *right = a + bc;
}

/* -------------------------------------------------------------- GEMM -- */

/* y[m][n] = sum_{k=0}^{K-1} x[m][k] * W[n][k], W stored [N][K] (row n is
 * output feature n).  One sequential fp32 sum per output, k ascending. */
void orc_gemm_bf16(const uint16_t *x, int M, int K, const uint16_t *W, int N,
                   float *y)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            const uint16_t *xr = x + (int64_t)m * K;
            const uint16_t *wr = W + (int64_t)n * K;
            float acc = 0.0f;
            for (int k = 0; k < K; ++k)
                acc += bf16_bits_to_f32(xr[k]) * bf16_bits_to_f32(wr[k]);
            y[(int64_t)m * N + n] = acc;
        }
}

/* ----------------------------------------------------------- RMSNorm -- */

/* y = x * (1 / sqrt(mean(x^2) + eps)) * w, per row of length H. */
void orc_rmsnorm(const float *x, int T, int H, const uint16_t *w, float eps,
                 float *y)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *xr = x + (int64_t)t * H;
        float *yr = y + (int64_t)t * H;
        float ss = 0.0f;
        for (int i = 0; i < H; ++i)
            ss += xr[i] * xr[i];
        float r = 1.0f / sqrtf(ss / (float)H + eps);
        for (int i = 0; i < H; ++i)
            yr[i] = (xr[i] * r) * bf16_bits_to_f32(w[i]);
    }
}

/* -------------------------------------------------------------- RoPE -- */

/* Rotary embedding, half-split pairing: element i pairs with i + D/2 and
 * turns by angle pos * theta^(-2i/D).  The angle and its cosine and sine are
 * taken in double and then rounded to fp32; the rotation itself is fp32.
 * x is [T][nh][D], rotated in place; pos[t] is the absolute position. */
void orc_rope(float *x, int T, int nh, int D, const int32_t *pos, double theta)
{
    const int half = D / 2;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < half; ++i) {
            double inv_freq = pow(theta, -(2.0 * (double)i) / (double)D);
            double ang = (double)pos[t] * inv_freq;
            float c = (float)cos(ang);
            float s = (float)sin(ang);
            for (int h = 0; h < nh; ++h) {
                float *v = x + ((int64_t)t * nh + h) * D;
                float x0 = v[i], x1 = v[i + half];
                v[i] = x0 * c - x1 * s;
                v[i + half] = x1 * c + x0 * s;
            }
        }
    }
}

/* --------------------------------------------------------- attention -- */

/* Causal grouped-query attention for rows that sit at absolute positions.
 *   q      [T][Hq][D]
 *   kc, vc [R][L][Hkv][D]   cache of request r in logical position order
 *   row_req[t], row_pos[t]  request and absolute position of row t
 * out[t][h] = sum_{j<=pos} softmax_j(q.k_j * scale) v_j, with query head h
 * reading kv head h / (Hq / Hkv) (contiguous groups).  The softmax takes the
 * maximum out first; the sums run in ascending j. */
void orc_attention(const float *q, int T, int Hq, int Hkv, int D,
                   const float *kc, const float *vc, int L,
                   const int32_t *row_req, const int32_t *row_pos, float scale,
                   float *s_scratch /* [T*Hq][L] */, float *out)
{
    const int group = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < Hq; ++h) {
            const int g = h / group;
            const int r = row_req[t];
            const int n = row_pos[t] + 1;
            const float *qv = q + ((int64_t)t * Hq + h) * D;
            float *s = s_scratch + ((int64_t)t * Hq + h) * L;
            float m = -INFINITY;
            for (int j = 0; j < n; ++j) {
                const float *kv = kc + (((int64_t)r * L + j) * Hkv + g) * D;
                float dot = 0.0f;
                for (int d = 0; d < D; ++d)
                    dot += qv[d] * kv[d];
                s[j] = dot * scale;
                if (s[j] > m)
                    m = s[j];
            }
            float l = 0.0f;
            for (int j = 0; j < n; ++j) {
                s[j] = expf(s[j] - m);
                l += s[j];
            }
            float *o = out + ((int64_t)t * Hq + h) * D;
            for (int d = 0; d < D; ++d) {
                float acc = 0.0f;
                for (int j = 0; j < n; ++j)
                    acc += s[j] * vc[(((int64_t)r * L + j) * Hkv + g) * D + d];
                o[d] = acc / l;
            }
        }
}

/* ------------------------------------------------------------ SwiGLU -- */

/* out = silu(g) * u with silu(g) = g / (1 + e^-g). */
void orc_swiglu(const float *g, const float *u, int64_t n, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (g[i] / (1.0f + expf(-g[i]))) * u[i];
}

/* ------------------------------------------------------------ argmax -- */

/* First index of the maximum of each row.  NaN counts as larger than any
 * number and the first NaN wins; -0 and +0 compare equal, so the earlier
 * one is kept. */
void orc_argmax(const float *x, int T, int V, int32_t *ids)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *row = x + (int64_t)t * V;
        int best = 0;
        float bv = row[0];
        for (int i = 1; i < V && !isnan(bv); ++i) {
            float v = row[i];
            if (isnan(v) || v > bv) {
                bv = v;
                best = i;
            }
        }
        ids[t] = best;
    }
}

/* ------------------------------------------------------------ Philox -- */

/* Philox4x64 with 10 rounds, from its published definition (Salmon, Moraes,
 * Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11): each
 * round takes the two 64x64->128 products of counter words 0 and 2 with the
 * round multipliers, mixes the high halves with counter words 1 and 3 and
 * the key, and the key is bumped by the Weyl constants between rounds. */
static inline void mulhilo64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *lo = (uint64_t)p;
    *hi = (uint64_t)(p >> 64);
}

void orc_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2],
                       uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        uint64_t hi0, lo0, hi1, lo1;
        mulhilo64(M0, c0, &hi0, &lo0);
        mulhilo64(M1, c2, &hi1, &lo1);
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n1 = lo1;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        uint64_t n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Per-request sampling seed of the ybb.press article, section 6, item 3:
 * (request_id * 1000003 + step) mod 2^64. */
uint64_t orc_sample_seed(uint64_t request_id, uint64_t step)
{
    return request_id * 1000003ull + step;
}

/* Uniform in [0,1) from the top 24 bits of Philox4x64-10 word 0 for key
 * (seed, 0) and counter 0.  Exact in fp32. */
float orc_sample_uniform(uint64_t seed)
{
    const uint64_t ctr[4] = {0, 0, 0, 0};
    const uint64_t key[2] = {seed, 0};
    uint64_t o[4];
    orc_philox4x64_10(ctr, key, o);
    return (float)(o[0] >> 40) * 0x1.0p-24f;
}

/* Temperature sampling by inverse CDF: p_i = exp((l_i - max)/tau), the token
 * is the first i whose running sum exceeds u * sum(p).  All sums sequential.
 * tau == 0 means greedy (argmax).  Rows whose running sum never exceeds the
 * target because of rounding take the last index with p_i > 0. */
void orc_philox_sample(const float *logits, int T, int V,
                       const uint64_t *request_id, const uint64_t *step,
                       float tau, float *p_scratch /* [T][V] */, int32_t *ids)
{
    if (tau == 0.0f) {
        orc_argmax(logits, T, V, ids);
        return;
    }
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *row = logits + (int64_t)t * V;
        float *p = p_scratch + (int64_t)t * V;
        float m = -INFINITY;
        for (int i = 0; i < V; ++i)
            if (row[i] > m)
                m = row[i];
        float total = 0.0f;
        for (int i = 0; i < V; ++i) {
            p[i] = expf((row[i] - m) / tau);
            total += p[i];
        }
        float u = orc_sample_uniform(orc_sample_seed(request_id[t], step[t]));
        float target = u * total;
        float cdf = 0.0f;
        int chosen = -1, last_pos = 0;
        for (int i = 0; i < V; ++i) {
            if (p[i] > 0.0f)
                last_pos = i;
            cdf += p[i];
            if (chosen < 0 && cdf > target)
                chosen = i;
        }
        ids[t] = chosen >= 0 ? chosen : last_pos;
    }
}

/* ------------------------------------------------------ top-k / top-p -- */

/* Order of tokens for top-k / top-p: larger logit first, equal logits by
 * lower index; NaN ranks as -inf and -0 as +0. */
static float rank_value(float v)
{
    if (isnan(v))
        return -INFINITY;
    return v == 0.0f ? 0.0f : v;
}

static const float *g_sort_row; /* row being sorted (one thread per call) */

static int by_rank(const void *a, const void *b)
{
    const int32_t i = *(const int32_t *)a, j = *(const int32_t *)b;
    const float x = rank_value(g_sort_row[i]), y = rank_value(g_sort_row[j]);
    if (x != y)
        return x > y ? -1 : 1;
    return i < j ? -1 : (i > j ? 1 : 0);
}

/* Temperature sampling over the K = min(top_k, V) highest-ranked tokens
 * and, within them, the nucleus of mass top_p: with the tokens in rank
 * order and p_j = exp((l_j - l_0) / tau) (l_0 the largest logit), c_j the
 * sequential fp32 running sums, the kept tokens are the first n + 1 where
 * n is the first j < K with c_j >= top_p * c_{K-1} (all K when top_p = 1);
 * the token is the first kept j (in rank order) with c_j > u * c_{n},
 * u the request's Philox uniform.  Rounding that leaves no such j takes the
 * last kept j with p_j > 0; a row whose largest logit is -inf (or NaN)
 * takes the first-ranked token.  tau == 0 is greedy (orc_argmax).
 * Sequential per row (the qsort order is a total order, so the result does
 * not depend on the sort algorithm). */
void orc_philox_sample_top(const float *logits, int T, int V,
                           const uint64_t *request_id, const uint64_t *step,
                           float tau, int top_k, float top_p,
                           int32_t *order_scratch /* [V] */,
                           float *c_scratch /* [V] */, int32_t *ids)
{
    if (tau == 0.0f) {
        orc_argmax(logits, T, V, ids);
        return;
    }
    const int K = top_k < V ? top_k : V;
    for (int t = 0; t < T; ++t) {
        const float *row = logits + (int64_t)t * V;
        for (int i = 0; i < V; ++i)
            order_scratch[i] = i;
        g_sort_row = row;
        qsort(order_scratch, (size_t)V, sizeof(int32_t), by_rank);
        const float l0 = rank_value(row[order_scratch[0]]);
        if (l0 == -INFINITY) {
            ids[t] = order_scratch[0];
            continue;
        }
        float c = 0.0f;
        for (int j = 0; j < K; ++j) {
            const float p = expf((rank_value(row[order_scratch[j]]) - l0) / tau);
            c += p;
            c_scratch[j] = c;
        }
        int n = K - 1;
        if (top_p < 1.0f) {
            const float cut = top_p * c_scratch[K - 1];
            for (int j = 0; j < K; ++j)
                if (c_scratch[j] >= cut) {
                    n = j;
                    break;
                }
        }
        const float u = orc_sample_uniform(orc_sample_seed(request_id[t],
                                                           step[t]));
        const float target = u * c_scratch[n];
        int chosen = -1, last_pos = 0;
        for (int j = 0; j <= n; ++j) {
            const float p = expf((rank_value(row[order_scratch[j]]) - l0) / tau);
            if (p > 0.0f)
                last_pos = j;
            if (chosen < 0 && c_scratch[j] > target)
                chosen = j;
        }
        ids[t] = order_scratch[chosen >= 0 ? chosen : last_pos];
    }
}
