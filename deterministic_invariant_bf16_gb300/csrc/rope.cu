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
// The model driver computes the (cos, sin) table of a forward pass once
// (rope_table_kernel) and every layer reads it; the stand-alone entry point
// computes the same values inside each block.  Either way the fp32 values
// come from the same double-precision expressions, so the bits agree.
// Pages: PagedAttention-style pools [n_pages][Hkv][16][D]; the page of a
// position is looked up in the request's page-table row, so any physical
// page order gives the same logical cache (Vosti: KV tied to its logical
// prefix).
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int ROPE_THREADS = 128;

// (cos, sin) of angle pos * theta^(-2i/D), in double, rounded to fp32.
__device__ __forceinline__ float2 rope_cs(int p, int i, int D, double theta) {
    const double inv_freq = pow(theta, -(2.0 * (double)i) / (double)D);
    const double ang = (double)p * inv_freq;
    return make_float2((float)cos(ang), (float)sin(ang));
}

__global__ void rope_table_kernel(const int32_t *__restrict__ pos, int T,
                                  int D, double theta,
                                  float2 *__restrict__ table) {
    const int half = D / 2;
    const int64_t n = (int64_t)T * half;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(e / half), i = (int)(e % half);
        table[e] = rope_cs(pos[t], i, D, theta);
    }
}

// Slices summed in slice order and rounded to bf16, for PAIRS consecutive
// elements (one float4 per slice when PAIRS = 4).  S is a template argument
// so that all S loads are in flight before the adds.
template <int S, int PAIRS>
__device__ __forceinline__ void qkv_values(const float *__restrict__ qkv,
                                           int64_t TQ, int64_t off,
                                           float *out) {
    float p[S][PAIRS];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        if constexpr (PAIRS == 4) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(
                qkv + s * TQ + off));
            p[s][0] = v.x;
            p[s][1] = v.y;
            p[s][2] = v.z;
            p[s][3] = v.w;
        } else {
            p[s][0] = __ldcs(qkv + s * TQ + off);
        }
    }
#pragma unroll
    for (int k = 0; k < PAIRS; ++k) {
        float v = p[0][k];
#pragma unroll
        for (int s = 1; s < S; ++s) v = __fadd_rn(v, p[s][k]);
        out[k] = bf16_to_f32(f32_to_bf16(v));
    }
}

// PAIRS bf16 values to 2 * PAIRS bytes of memory (one 8-byte store for 4).
template <int PAIRS>
__device__ __forceinline__ void store_bf16(uint16_t *dst, const float *v,
                                           bool zero) {
    if constexpr (PAIRS == 4) {
        *reinterpret_cast<uint2 *>(dst) =
            zero ? make_uint2(0, 0)
                 : make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
    } else {
        dst[0] = zero ? 0 : f32_to_bf16(v[0]);
    }
}

// Block (t, y) handles row t, heads [y * HPB, (y + 1) * HPB) with
// HPB = ROPE_THREADS / (D / (2 PAIRS)); thread -> (head, pairs i .. i +
// PAIRS - 1).  Heads are q heads, then k heads (rotated and appended), then
// v heads (appended as rounded).  128-thread blocks measured slightly
// faster in the decode step than 256 (512 slower); each thread's
// arithmetic does not depend on the block shape.
template <int S, int PAIRS>
__global__ void __launch_bounds__(ROPE_THREADS)
    rope_kernel(const float *__restrict__ qkv, const float2 *__restrict__ table,
                const int32_t *__restrict__ pos,
                const int32_t *__restrict__ row_req, int T, int Hq, int Hkv,
                int D, double theta, uint16_t *__restrict__ q_out,
                uint16_t *__restrict__ k_pool, uint16_t *__restrict__ v_pool,
                const int32_t *__restrict__ page_table, int max_pages,
                int n_pages, int32_t *status, int discard, DeadRegion dead) {
    discard_region(dead);
    __shared__ float2 cs_s[64];
    const int t = blockIdx.x;
    const int half = D / 2;
    const int tph = half / PAIRS;  // threads per head
    const int hpb = ROPE_THREADS / tph;
    const int QKV = (Hq + 2 * Hkv) * D;
    const int64_t TQ = (int64_t)T * QKV;
    const int64_t rowoff = (int64_t)t * QKV;
    const int p = pos[t];
    const int req = row_req[t];
    const int i = (threadIdx.x % tph) * PAIRS;
    const int head = blockIdx.y * hpb + threadIdx.x / tph;

    if (!table) {
        if (threadIdx.x < half) cs_s[threadIdx.x] = rope_cs(p, threadIdx.x, D, theta);
        __syncthreads();
    }
    if (head >= Hq + 2 * Hkv) return;
    // The slice partials and the (cos, sin) pairs are read before the
    // page lookup, so that their loads and the page-table load are in
    // flight together.
    const int64_t c0 = rowoff + (int64_t)head * D + i;
    float x0[PAIRS], x1[PAIRS];
    qkv_values<S, PAIRS>(qkv, TQ, c0, x0);
    qkv_values<S, PAIRS>(qkv, TQ, c0 + half, x1);
    if (PAIRS == 4 && discard) {
        // The slice partials have had their only read: drop their lines from
        // L2 without writing them back.  A 128-byte line holds the pairs of
        // eight consecutive threads of one warp (i = 0 .. 28 or 32 .. 60).
        __syncwarp(__activemask());
        if ((i & 31) == 0) {
#pragma unroll
            for (int s = 0; s < S; ++s) {
                discard_l2_line(qkv + s * TQ + c0);
                discard_l2_line(qkv + s * TQ + c0 + half);
            }
        }
    }
    float2 cs[PAIRS];
    if (head < Hq + Hkv) {
#pragma unroll
        for (int k = 0; k < PAIRS; ++k)
            cs[k] = table ? table[(int64_t)t * half + i + k] : cs_s[i + k];
    }
    int64_t page = -1;
    if (req >= 0 && head >= Hq) {
        const int pi = p / 16;
        if (p < 0 || pi >= max_pages) {
            if (i == 0) bi_record_error(status, BI_ERR_BOUNDS);
        } else {
            const int pg = page_table[(int64_t)req * max_pages + pi];
            if (pg < 0 || pg >= n_pages) {
                if (i == 0) bi_record_error(status, BI_ERR_BOUNDS);
            } else {
                page = pg;
            }
        }
    }
    const int slot = p & 15;
    if (head < Hq + Hkv) {
        float y0[PAIRS], y1[PAIRS];
#pragma unroll
        for (int k = 0; k < PAIRS; ++k) {
            const float c = cs[k].x, s = cs[k].y;
            y0[k] = __fsub_rn(__fmul_rn(x0[k], c), __fmul_rn(x1[k], s));
            y1[k] = __fadd_rn(__fmul_rn(x1[k], c), __fmul_rn(x0[k], s));
        }
        if (head < Hq) {
            uint16_t *qd = q_out + ((int64_t)t * Hq + head) * D;
            const bool pad = req < 0;
            store_bf16<PAIRS>(qd + i, y0, pad);
            store_bf16<PAIRS>(qd + i + half, y1, pad);
        } else if (page >= 0) {
            uint16_t *kd = k_pool +
                           ((page * Hkv + (head - Hq)) * 16 + slot) * (int64_t)D;
            store_bf16<PAIRS>(kd + i, y0, false);
            store_bf16<PAIRS>(kd + i + half, y1, false);
        }
    } else if (page >= 0) {
        uint16_t *vd = v_pool +
                       ((page * Hkv + (head - Hq - Hkv)) * 16 + slot) * (int64_t)D;
        store_bf16<PAIRS>(vd + i, x0, false);
        store_bf16<PAIRS>(vd + i + half, x1, false);
    }
}

}  // namespace

bi_status bi_rope_table(const int32_t *pos, int T, int D, double theta,
                        float2 *table, cudaStream_t s) {
    if (T == 0) return BI_OK;
    // 64-thread blocks: the double-precision power, cosine and sine of a
    // 256-row table then run on every SM instead of a quarter of them
    const int64_t n = (int64_t)T * (D / 2);
    const int blocks = (int)((n + 63) / 64);
    rope_table_kernel<<<blocks, 64, 0, s>>>(pos, T, D, theta, table);
    BI_LAUNCH_CHECK("rope table launch");
    return BI_OK;
}

bi_status bi_rope_apply(const float *qkv, int S, const float2 *table,
                        const int32_t *pos, const int32_t *row_req, int T,
                        int Hq, int Hkv, int D, double theta,
                        bi_bf16 *q_out, bi_bf16 *k_pool, bi_bf16 *v_pool,
                        const int32_t *page_table, int max_pages, int n_pages,
                        cudaStream_t st, bool discard_partials,
                        const void *dead, size_t dead_bytes) {
    BI_REQUIRE(T >= 0 && S >= 1 && S <= 8 && Hq > 0 && Hkv > 0 &&
                   Hq % Hkv == 0,
               "bi_rope: bad shape T=%d S=%d Hq=%d Hkv=%d", T, S, Hq, Hkv);
    BI_REQUIRE(D % 2 == 0 && D <= 128 && D >= 4 && ROPE_THREADS % (D / 2) == 0,
               "bi_rope: D=%d", D);
    if (T == 0) return BI_OK;
    BI_REQUIRE(qkv && pos && row_req && q_out && k_pool && v_pool && page_table,
               "bi_rope: null pointer");
    BI_REQUIRE(max_pages > 0 && n_pages > 0, "bi_rope: empty page table/pool");
    BI_REQUIRE(bi_aligned16(qkv) && bi_aligned16(q_out) &&
                   bi_aligned16(k_pool) && bi_aligned16(v_pool),
               "bi_rope: pointers must be 16-byte aligned");
    int32_t *status = bi_status_ptr();
    // four pairs per thread (16-byte loads) when D / 2 is a multiple of 4
    const bool vec = (D / 2) % 4 == 0;
    const int tph = vec ? D / 8 : D / 2;
    const int hpb = ROPE_THREADS / tph;
    dim3 grid(T, (Hq + 2 * Hkv + hpb - 1) / hpb);
    // the discard needs whole 128-byte lines per head: D = 128, 16-byte
    // loads, the planes on 128-byte boundaries
    const int dis = discard_partials && vec && D == 128 &&
                            (reinterpret_cast<uintptr_t>(qkv) & 127) == 0
                        ? 1
                        : 0;
    const DeadRegion dr{dead, dead_bytes};
    switch (S) {
#define BI_ROPE_CASE(n)                                                       \
    case n:                                                                   \
        if (vec)                                                              \
            rope_kernel<n, 4><<<grid, ROPE_THREADS, 0, st>>>(                 \
                qkv, table, pos, row_req, T, Hq, Hkv, D, theta, q_out,        \
                k_pool, v_pool, page_table, max_pages, n_pages, status, dis,  \
                dr);                                                          \
        else                                                                  \
            rope_kernel<n, 1><<<grid, ROPE_THREADS, 0, st>>>(                 \
                qkv, table, pos, row_req, T, Hq, Hkv, D, theta, q_out,        \
                k_pool, v_pool, page_table, max_pages, n_pages, status, 0,    \
                dr);                                                          \
        break;
        BI_ROPE_CASE(1) BI_ROPE_CASE(2) BI_ROPE_CASE(3) BI_ROPE_CASE(4)
        BI_ROPE_CASE(5) BI_ROPE_CASE(6) BI_ROPE_CASE(7) BI_ROPE_CASE(8)
#undef BI_ROPE_CASE
    }
    BI_LAUNCH_CHECK("rope launch");
    return BI_OK;
}

extern "C" bi_status bi_rope(const float *qkv, int S, const int32_t *pos,
                             const int32_t *row_req, int T, int Hq, int Hkv,
                             int D, double theta, bi_bf16 *q_out,
                             bi_bf16 *k_pool, bi_bf16 *v_pool,
                             const int32_t *page_table, int max_pages,
                             int n_pages, void *stream) {
    return bi_rope_apply(qkv, S, nullptr, pos, row_req, T, Hq, Hkv, D, theta,
                         q_out, k_pool, v_pool, page_table, max_pages, n_pages,
                         bi_stream(stream), false, nullptr, 0);
}
