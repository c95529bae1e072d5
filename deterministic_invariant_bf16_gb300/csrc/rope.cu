// bi_rope: second stage of the QKV GEMM (slice partials summed in slice
// order, rounded to bf16), rotary embedding of q and k, and the append of
// k and v to the paged KV cache.
//
// Rotation: half-split pairs (i, i + D/2) turn by angle pos * theta^(-2i/D).
// The angle and its cosine and sine are computed in double and rounded to
// fp32 once per (row, i); the rotation itself is fp32 with every multiply
// and add rounded separately:
//   x'_i       = x_i * cos - x_{i+D/2} * sin
//   x'_{i+D/2} = x_{i+D/2} * cos + x_i * sin
// Pages: PagedAttention-style pools [n_pages][Hkv][16][D]; the page of a
// position is looked up in the request's page-table row, so any physical
// page order gives the same logical cache (Vosti: KV tied to its logical
// prefix).
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int ROPE_THREADS = 256;

// Slices summed in slice order and rounded to bf16.  S is a template
// argument so that all S loads are in flight before the adds.
template <int S>
__device__ __forceinline__ float qkv_value(const float *__restrict__ qkv,
                                           int64_t TQ, int64_t off) {
    float p[S];
#pragma unroll
    for (int s = 0; s < S; ++s) p[s] = __ldcs(qkv + s * TQ + off);
    float v = p[0];
#pragma unroll
    for (int s = 1; s < S; ++s) v = __fadd_rn(v, p[s]);
    return bf16_to_f32(f32_to_bf16(v));
}

template <int S>
__global__ void __launch_bounds__(ROPE_THREADS)
    rope_kernel(const float *__restrict__ qkv,
                const int32_t *__restrict__ pos,
                const int32_t *__restrict__ row_req, int T, int Hq, int Hkv,
                int D, double theta, uint16_t *__restrict__ q_out,
                uint16_t *__restrict__ k_pool, uint16_t *__restrict__ v_pool,
                const int32_t *__restrict__ page_table, int max_pages,
                int n_pages, int32_t *status) {
    __shared__ float cs[64], sn[64];
    const int t = blockIdx.x;
    const int half = D / 2;
    const int QKV = (Hq + 2 * Hkv) * D;
    const int64_t TQ = (int64_t)T * QKV;
    const int64_t rowoff = (int64_t)t * QKV;
    const int p = pos[t];
    const int req = row_req[t];

    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double inv_freq = pow(theta, -(2.0 * (double)i) / (double)D);
        const double ang = (double)p * inv_freq;
        cs[i] = (float)cos(ang);
        sn[i] = (float)sin(ang);
    }
    int64_t page = -1;
    if (req >= 0) {
        const int pi = p / 16;
        if (p < 0 || pi >= max_pages) {
            if (threadIdx.x == 0) bi_record_error(status, BI_ERR_BOUNDS);
        } else {
            const int pg = page_table[(int64_t)req * max_pages + pi];
            if (pg < 0 || pg >= n_pages) {
                if (threadIdx.x == 0) bi_record_error(status, BI_ERR_BOUNDS);
            } else {
                page = pg;
            }
        }
    }
    __syncthreads();
    const int slot = p & 15;

    // q and k heads: one pair (i, i + D/2) per work item.
    const int pairs = (Hq + Hkv) * half;
    for (int e = threadIdx.x; e < pairs; e += blockDim.x) {
        const int head = e / half, i = e % half;
        const int64_t c0 = rowoff + (int64_t)head * D + i;
        const float x0 = qkv_value<S>(qkv, TQ, c0);
        const float x1 = qkv_value<S>(qkv, TQ, c0 + half);
        const float c = cs[i], s = sn[i];
        const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
        const float y1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
        if (head < Hq) {
            uint16_t *qd = q_out + ((int64_t)t * Hq + head) * D;
            const bool live = req >= 0;
            qd[i] = live ? f32_to_bf16(y0) : 0;
            qd[i + half] = live ? f32_to_bf16(y1) : 0;
        } else if (page >= 0) {
            uint16_t *kd = k_pool +
                           ((page * Hkv + (head - Hq)) * 16 + slot) * (int64_t)D;
            kd[i] = f32_to_bf16(y0);
            kd[i + half] = f32_to_bf16(y1);
        }
    }
    // v heads: copied as rounded.
    if (page >= 0) {
        for (int e = threadIdx.x; e < Hkv * D; e += blockDim.x) {
            const int head = e / D, d = e % D;
            const float v = qkv_value<S>(qkv, TQ,
                                      rowoff + (int64_t)(Hq + Hkv) * D + e);
            v_pool[((page * Hkv + head) * 16 + slot) * (int64_t)D + d] =
                f32_to_bf16(v);
        }
    }
}

}  // namespace

extern "C" bi_status bi_rope(const float *qkv, int S, const int32_t *pos,
                             const int32_t *row_req, int T, int Hq, int Hkv,
                             int D, double theta, bi_bf16 *q_out,
                             bi_bf16 *k_pool, bi_bf16 *v_pool,
                             const int32_t *page_table, int max_pages,
                             int n_pages, void *stream) {
    BI_REQUIRE(T >= 0 && S >= 1 && S <= 8 && Hq > 0 && Hkv > 0 &&
                   Hq % Hkv == 0,
               "bi_rope: bad shape T=%d S=%d Hq=%d Hkv=%d", T, S, Hq, Hkv);
    BI_REQUIRE(D % 2 == 0 && D <= 128 && D > 0, "bi_rope: D=%d", D);
    BI_REQUIRE(qkv && pos && row_req && q_out && k_pool && v_pool && page_table,
               "bi_rope: null pointer");
    BI_REQUIRE(max_pages > 0 && n_pages > 0, "bi_rope: empty page table/pool");
    if (T == 0) return BI_OK;
    cudaStream_t st = bi_stream(stream);
    int32_t *status = bi_status_ptr();
    switch (S) {
#define BI_ROPE_CASE(n)                                                       \
    case n:                                                                   \
        rope_kernel<n><<<T, ROPE_THREADS, 0, st>>>(                           \
            qkv, pos, row_req, T, Hq, Hkv, D, theta, q_out, k_pool, v_pool,   \
            page_table, max_pages, n_pages, status);                          \
        break;
        BI_ROPE_CASE(1) BI_ROPE_CASE(2) BI_ROPE_CASE(3) BI_ROPE_CASE(4)
        BI_ROPE_CASE(5) BI_ROPE_CASE(6) BI_ROPE_CASE(7) BI_ROPE_CASE(8)
#undef BI_ROPE_CASE
    }
    BI_LAUNCH_CHECK("rope launch");
    return BI_OK;
}
