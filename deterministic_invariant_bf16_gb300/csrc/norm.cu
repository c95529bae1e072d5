// bi_rmsnorm (fused with the split-GEMM second stage and the residual add),
// bi_embed and bi_swiglu.
//
// RMSNorm reduction order for one row (fixed by H and the constants below,
// never by T or the row's index): thread i owns the 8-element slices
// i, i + 256, i + 512, ... and sums their squares in ascending order; the 32
// lanes of a warp combine with an xor-shuffle tree (16, 8, 4, 2, 1); the 8
// warp totals are added in warp order.  Split partials are summed in slice
// order 0..S-1 before anything else (ybb.press section 4, second stage).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int NORM_THREADS = 256;
constexpr int NORM_MAX_VEC = 8;  // H <= 8 * 8 * 256 = 16384

// S (the number of split slices, 0 = no partials) is a template argument so
// that all S loads of a slice group are issued before the in-order adds.
template <int S>
__global__ void __launch_bounds__(NORM_THREADS)
    rmsnorm_kernel(const float *__restrict__ partials,
                   const uint16_t *__restrict__ x, uint16_t *residual,
                   const uint16_t *__restrict__ w, int T, int H, float eps,
                   uint16_t *__restrict__ y) {
    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const int nvec = H / 8;
    const int64_t row = (int64_t)t * H;
    const int64_t TH = (int64_t)T * H;
    float v[NORM_MAX_VEC][8];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < NORM_MAX_VEC; ++k) {
        const int vi = tid + k * NORM_THREADS;
        if (vi >= nvec) break;
        const int64_t off = row + (int64_t)vi * 8;
        if (S > 0) {
            float4 pa[S > 0 ? S : 1][2];
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const float4 *ps =
                    reinterpret_cast<const float4 *>(partials + s * TH + off);
                pa[s][0] = __ldcs(ps);
                pa[s][1] = __ldcs(ps + 1);
            }
            float acc[8] = {pa[0][0].x, pa[0][0].y, pa[0][0].z, pa[0][0].w,
                            pa[0][1].x, pa[0][1].y, pa[0][1].z, pa[0][1].w};
#pragma unroll
            for (int s = 1; s < S; ++s) {
                const float4 c = pa[s][0], d = pa[s][1];
                acc[0] = __fadd_rn(acc[0], c.x);
                acc[1] = __fadd_rn(acc[1], c.y);
                acc[2] = __fadd_rn(acc[2], c.z);
                acc[3] = __fadd_rn(acc[3], c.w);
                acc[4] = __fadd_rn(acc[4], d.x);
                acc[5] = __fadd_rn(acc[5], d.y);
                acc[6] = __fadd_rn(acc[6], d.z);
                acc[7] = __fadd_rn(acc[7], d.w);
            }
            if (residual) {
                uint4 r = *reinterpret_cast<const uint4 *>(residual + off);
                const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float lo = bf16_to_f32(f32_to_bf16(
                        __fadd_rn(bf16_lo(rr[j]), acc[2 * j])));
                    float hi = bf16_to_f32(f32_to_bf16(
                        __fadd_rn(bf16_hi(rr[j]), acc[2 * j + 1])));
                    v[k][2 * j] = lo;
                    v[k][2 * j + 1] = hi;
                    o[j] = pack_bf16x2(lo, hi);
                }
                *reinterpret_cast<uint4 *>(residual + off) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[k][j] = bf16_to_f32(f32_to_bf16(acc[j]));
            }
        } else {
            const uint16_t *src = residual ? residual : x;
            uint4 r = *reinterpret_cast<const uint4 *>(src + off);
            const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[k][2 * j] = bf16_lo(rr[j]);
                v[k][2 * j + 1] = bf16_hi(rr[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = __fadd_rn(ss, __fmul_rn(v[k][j], v[k][j]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    __shared__ float warp_ss[NORM_THREADS / 32];
    if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
    __syncthreads();
    float tot = warp_ss[0];
#pragma unroll
    for (int i = 1; i < NORM_THREADS / 32; ++i) tot = __fadd_rn(tot, warp_ss[i]);
    const float r = __fdiv_rn(
        1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), eps)));
#pragma unroll
    for (int k = 0; k < NORM_MAX_VEC; ++k) {
        const int vi = tid + k * NORM_THREADS;
        if (vi >= nvec) break;
        const int64_t off = row + (int64_t)vi * 8;
        uint4 wv = *reinterpret_cast<const uint4 *>(w + (int64_t)vi * 8);
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = pack_bf16x2(
                __fmul_rn(__fmul_rn(v[k][2 * j], r), bf16_lo(ww[j])),
                __fmul_rn(__fmul_rn(v[k][2 * j + 1], r), bf16_hi(ww[j])));
        *reinterpret_cast<uint4 *>(y + off) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void embed_kernel(const int32_t *__restrict__ tokens,
                             const uint4 *__restrict__ E, int V, int H8,
                             uint4 *__restrict__ h, int32_t *status) {
    const int t = blockIdx.x;
    const int id = tokens[t];
    const bool ok = id >= 0 && id < V;
    if (!ok && threadIdx.x == 0) bi_record_error(status, BI_ERR_BOUNDS);
    for (int i = threadIdx.x; i < H8; i += blockDim.x)
        h[(int64_t)t * H8 + i] =
            ok ? E[(int64_t)id * H8 + i] : make_uint4(0, 0, 0, 0);
}

__global__ void swiglu_kernel(const float *__restrict__ g,
                              const float *__restrict__ u, int64_t n,
                              uint16_t *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float gv = g[i];
        out[i] = f32_to_bf16(
            __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv))), u[i]));
    }
}

}  // namespace

// The same computation for H <= VEC * 8 * NORM_THREADS with every load
// (the slice partials, the residual or x, the weights) issued before the
// first use: one round of memory latency instead of one per slice group
// and another for the weights.  The arithmetic and its order are those of
// rmsnorm_kernel, so the bits are the same.
template <int S, int VEC>
__global__ void __launch_bounds__(NORM_THREADS)
    rmsnorm_fast_kernel(const float *__restrict__ partials,
                        const uint16_t *__restrict__ x, uint16_t *residual,
                        const uint16_t *__restrict__ w, int T, int H, float eps,
                        uint16_t *__restrict__ y, int discard,
                        DeadRegion dead0, DeadRegion dead1) {
    discard_region(dead0);
    discard_region(dead1);
    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const int nvec = H / 8;
    const int64_t row = (int64_t)t * H;
    const int64_t TH = (int64_t)T * H;
    constexpr int SP = S > 0 ? S : 1;
    float4 pa[VEC][SP][2];
    uint4 rv[VEC], wv[VEC];
    bool act[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int vi = tid + k * NORM_THREADS;
        act[k] = vi < nvec;
        rv[k] = make_uint4(0, 0, 0, 0);
        if (!act[k]) continue;
        const int64_t off = row + (int64_t)vi * 8;
        if (S > 0) {
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const float4 *ps =
                    reinterpret_cast<const float4 *>(partials + s * TH + off);
                pa[k][s][0] = __ldcs(ps);
                pa[k][s][1] = __ldcs(ps + 1);
            }
        }
        const uint16_t *src = residual ? residual : x;
        if (S == 0 || residual)
            rv[k] = *reinterpret_cast<const uint4 *>(src + off);
        wv[k] = *reinterpret_cast<const uint4 *>(w + (int64_t)vi * 8);
    }
    float v[VEC][8];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        if (!act[k]) continue;
        const int64_t off = row + (int64_t)(tid + k * NORM_THREADS) * 8;
        const uint32_t rr[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
        if (S > 0) {
            float acc[8] = {pa[k][0][0].x, pa[k][0][0].y, pa[k][0][0].z,
                            pa[k][0][0].w, pa[k][0][1].x, pa[k][0][1].y,
                            pa[k][0][1].z, pa[k][0][1].w};
#pragma unroll
            for (int s = 1; s < S; ++s) {
                const float4 c = pa[k][s][0], d = pa[k][s][1];
                acc[0] = __fadd_rn(acc[0], c.x);
                acc[1] = __fadd_rn(acc[1], c.y);
                acc[2] = __fadd_rn(acc[2], c.z);
                acc[3] = __fadd_rn(acc[3], c.w);
                acc[4] = __fadd_rn(acc[4], d.x);
                acc[5] = __fadd_rn(acc[5], d.y);
                acc[6] = __fadd_rn(acc[6], d.z);
                acc[7] = __fadd_rn(acc[7], d.w);
            }
            if (residual) {
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float lo = bf16_to_f32(f32_to_bf16(
                        __fadd_rn(bf16_lo(rr[j]), acc[2 * j])));
                    const float hi = bf16_to_f32(f32_to_bf16(
                        __fadd_rn(bf16_hi(rr[j]), acc[2 * j + 1])));
                    v[k][2 * j] = lo;
                    v[k][2 * j + 1] = hi;
                    o[j] = pack_bf16x2(lo, hi);
                }
                *reinterpret_cast<uint4 *>(residual + off) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[k][j] = bf16_to_f32(f32_to_bf16(acc[j]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[k][2 * j] = bf16_lo(rr[j]);
                v[k][2 * j + 1] = bf16_hi(rr[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            ss = __fadd_rn(ss, __fmul_rn(v[k][j], v[k][j]));
    }
    if (S > 0 && discard) {
        // The partial planes have had their only read: drop their lines from
        // L2 without writing them back.  A 128-byte line holds the 8-element
        // slices of four consecutive threads of one warp, all read by now.
        __syncwarp();
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
            const int vi = tid + k * NORM_THREADS;
            if (!act[k] || (vi & 3)) continue;
#pragma unroll
            for (int s = 0; s < SP; ++s)
                discard_l2_line(partials + s * TH + row + (int64_t)vi * 8);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    __shared__ float warp_ss[NORM_THREADS / 32];
    if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
    __syncthreads();
    float tot = warp_ss[0];
#pragma unroll
    for (int i = 1; i < NORM_THREADS / 32; ++i) tot = __fadd_rn(tot, warp_ss[i]);
    const float r = __fdiv_rn(
        1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), eps)));
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        if (!act[k]) continue;
        const int64_t off = row + (int64_t)(tid + k * NORM_THREADS) * 8;
        const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = pack_bf16x2(
                __fmul_rn(__fmul_rn(v[k][2 * j], r), bf16_lo(ww[j])),
                __fmul_rn(__fmul_rn(v[k][2 * j + 1], r), bf16_hi(ww[j])));
        *reinterpret_cast<uint4 *>(y + off) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

bi_status bi_rmsnorm_apply(const float *partials, int S, const bi_bf16 *x,
                           bi_bf16 *residual, const bi_bf16 *w, int T, int H,
                           float eps, bi_bf16 *y, bool discard_partials,
                           cudaStream_t s, const void *dead0,
                           size_t dead0_bytes, const void *dead1,
                           size_t dead1_bytes) {
    BI_REQUIRE(T >= 0 && H > 0 && H % 8 == 0 &&
                   H <= NORM_MAX_VEC * 8 * NORM_THREADS,
               "bi_rmsnorm: H=%d must be a positive multiple of 8, <= 16384",
               H);
    if (T == 0) return BI_OK;
    BI_REQUIRE(w && y, "bi_rmsnorm: null w or y");
    BI_REQUIRE(partials || x || residual,
               "bi_rmsnorm: need partials, x or residual");
    BI_REQUIRE(!partials || (S >= 1 && S <= 8), "bi_rmsnorm: S=%d not in 1..8",
               S);
    BI_REQUIRE((!partials || bi_aligned16(partials)) && (!x || bi_aligned16(x)) &&
                   (!residual || bi_aligned16(residual)) && bi_aligned16(w) &&
                   bi_aligned16(y),
               "bi_rmsnorm: pointers must be 16-byte aligned");
    // the partials' lines are dropped only where each 128-byte line holds
    // four slices of one row (rows of a multiple of 32 elements, planes on
    // 128-byte boundaries)
    const int dis = discard_partials && partials && H % 32 == 0 &&
                            (reinterpret_cast<uintptr_t>(partials) & 127) == 0
                        ? 1
                        : 0;
    const DeadRegion d0{dead0, dead0_bytes}, d1{dead1, dead1_bytes};
    // up to two 8-element slices per thread (H <= 4096): all loads first
    const int vec = (H / 8 + NORM_THREADS - 1) / NORM_THREADS;
    switch (partials ? S : 0) {
#define BI_NORM_CASE(n)                                                      \
    case n:                                                                  \
        if (vec == 1)                                                        \
            rmsnorm_fast_kernel<n, 1><<<T, NORM_THREADS, 0, s>>>(            \
                partials, x, residual, w, T, H, eps, y, dis, d0, d1);        \
        else if (vec == 2)                                                   \
            rmsnorm_fast_kernel<n, 2><<<T, NORM_THREADS, 0, s>>>(            \
                partials, x, residual, w, T, H, eps, y, dis, d0, d1);        \
        else                                                                 \
            rmsnorm_kernel<n><<<T, NORM_THREADS, 0, s>>>(partials, x,        \
                                                         residual, w, T, H,  \
                                                         eps, y);            \
        break;
        BI_NORM_CASE(0) BI_NORM_CASE(1) BI_NORM_CASE(2) BI_NORM_CASE(3)
        BI_NORM_CASE(4) BI_NORM_CASE(5) BI_NORM_CASE(6) BI_NORM_CASE(7)
        BI_NORM_CASE(8)
#undef BI_NORM_CASE
    }
    BI_LAUNCH_CHECK("rmsnorm launch");
    return BI_OK;
}

extern "C" bi_status bi_rmsnorm(const float *partials, int S,
                                const bi_bf16 *x, bi_bf16 *residual,
                                const bi_bf16 *w, int T, int H, float eps,
                                bi_bf16 *y, void *stream) {
    return bi_rmsnorm_apply(partials, S, x, residual, w, T, H, eps, y, false,
                            bi_stream(stream), nullptr, 0, nullptr, 0);
}

extern "C" bi_status bi_embed(const int32_t *tokens, int T, const bi_bf16 *E,
                              int V, int H, bi_bf16 *h, void *stream) {
    BI_REQUIRE(T >= 0 && V > 0 && H > 0 && H % 8 == 0,
               "bi_embed: bad shape T=%d V=%d H=%d", T, V, H);
    if (T == 0) return BI_OK;
    BI_REQUIRE(tokens && E && h, "bi_embed: null pointer");
    BI_REQUIRE(bi_aligned16(E) && bi_aligned16(h),
               "bi_embed: pointers must be 16-byte aligned");
    embed_kernel<<<T, 128, 0, bi_stream(stream)>>>(
        tokens, reinterpret_cast<const uint4 *>(E), V, H / 8,
        reinterpret_cast<uint4 *>(h), bi_status_ptr());
    BI_LAUNCH_CHECK("embed launch");
    return BI_OK;
}

extern "C" bi_status bi_swiglu(const float *g, const float *u, int64_t n,
                               bi_bf16 *out, void *stream) {
    BI_REQUIRE(n >= 0, "bi_swiglu: n=%lld", (long long)n);
    if (n == 0) return BI_OK;
    BI_REQUIRE(g && u && out, "bi_swiglu: null pointer");
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 152 * 16);
    swiglu_kernel<<<blocks, 256, 0, bi_stream(stream)>>>(g, u, n, out);
    BI_LAUNCH_CHECK("swiglu launch");
    return BI_OK;
}
