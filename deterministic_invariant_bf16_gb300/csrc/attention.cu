// bi_paged_decode_attn and bi_prefill_attn: causal grouped-query attention
// over the paged KV cache in fixed 256-position chunks.
//
// Invariance (Vosti abstract: bitwise-equal kernel outputs across batches,
// query lengths and paged KV layouts; ybb.press section 4: two-stage
// fixed-order reductions).  The arithmetic applied to one (query row, head)
// depends only on its query vector, its position and the logical KV prefix:
//
//   chunk c covers absolute positions [256c, 256c + 256).  For each chunk a
//   partial (m, l, o) is computed FROM SCRATCH by chunk_partial() below:
//     s_j = (q . k_j) * scale   mma.sync m16n8k16, dims in ascending 16-steps
//     s_j = -inf past the row's context
//     m   = max_j s_j
//     p_j = exp(s_j - m)
//     l   = sum_j p_j           fixed order: per thread 16 values in key
//                               order, quad xor-tree (1, 2), 4 warps in order
//     o   = sum_j bf16(p_j) v_j mma.sync, keys in ascending 16-steps
//   chunks are merged in ascending c by merge_step():
//     m' = max(m, m_c); a = exp(m - m'); b = exp(m_c - m')
//     l  = l a + l_c b;  o = o a + o_c b;   out = bf16(o / l)
//
// Decode computes each chunk in its own CTA, stores the partials and merges
// them in a second kernel; prefill loops over the chunks inside one CTA and
// merges in registers.  Both run the same two functions with the same warp
// and lane mapping, and every floating-point operation outside the MMAs is an
// explicit round-to-nearest intrinsic, so no contraction can differ.  A row
// sits in a 16-row MMA tile (decode: the G query heads of one KV head;
// prefill: 16/G queries x G heads); the tensor core treats rows
// independently, so the other rows of the tile do not matter.
//
// KV pages are read with 16-byte cp.async copies into an XOR-swizzled shared
// tile; positions past the context are zero-filled (stale pages may hold
// NaN, and 0 * NaN would poison the PV product).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int CHUNK = 256;
constexpr int ATT_THREADS = 128;  // 4 warps

// Shared-memory pieces common to both kernels ("misc"): the 16-row query
// tile, the bf16 P tile, the cross-warp reduction slots and the per-row
// visible key counts.
template <int D>
struct Misc {
    static constexpr int Q_OFF = 0;
    static constexpr int P_OFF = Q_OFF + 16 * D * 2;
    static constexpr int RED_OFF = P_OFF + 16 * CHUNK * 2;   // float [128]
    static constexpr int LEN_OFF = RED_OFF + 128 * 4;        // int [16]
    static constexpr int BYTES = LEN_OFF + 16 * 4;
};

// One K or V tile of a chunk: 256 positions x D, bf16.
template <int D>
constexpr int tile_bytes() { return CHUNK * D * 2; }

// Prefill layout: K tile, V tile, misc.
template <int D>
constexpr int prefill_smem() { return 2 * tile_bytes<D>() + Misc<D>::BYTES; }

// Decode layout: a ring of three tile slots, misc.
template <int D>
constexpr int decode_smem() { return 3 * tile_bytes<D>() + Misc<D>::BYTES; }

// Byte offset of 16-byte piece `ch` of row `row` in a tile of rows of
// `nch` pieces, XOR-swizzled so that ldmatrix row groups hit distinct banks.
__device__ __forceinline__ uint32_t swz(int row, int ch, int nch) {
    const int m = nch >= 8 ? 7 : nch - 1;
    return (uint32_t)(row * nch * 16 + ((ch ^ (row & m)) * 16));
}

// Issue (not commit) the cp.async copies of chunk c of KV head g of the
// page-table row pt_row from `pool` into the tile at shared address `base`.
// Positions >= valid_max are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t base,
                                          const uint16_t *__restrict__ pool,
                                          const int32_t *__restrict__ pt_row,
                                          int max_pages, int n_pages, int Hkv,
                                          int g, int c, int valid_max,
                                          int32_t *status) {
    constexpr int NCH = D / 8;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < CHUNK * NCH; idx += ATT_THREADS) {
        const int key = idx / NCH, ch = idx % NCH;
        const int p = c * CHUNK + key;
        const uint16_t *src = pool;
        uint32_t bytes = 0;
        if (p < valid_max) {
            const int pi = p >> 4;
            const int pg = pi < max_pages ? pt_row[pi] : -1;
            if (pg >= 0 && pg < n_pages) {
                src = pool + (((int64_t)pg * Hkv + g) * 16 + (p & 15)) * D +
                      ch * 8;
                bytes = 16;
            } else {
                bi_record_error(status, BI_ERR_BOUNDS);
            }
        }
        cp_async16(base + swz(key, ch, NCH), src, bytes);
    }
}

// Store the 16-row query tile: row r <- q + row_off[r] (row_off < 0 ->
// zeros).
template <int D>
__device__ __forceinline__ void store_q(uint8_t *misc, const uint16_t *q,
                                        const int64_t *row_off /* [16] */) {
    constexpr int NCH = D / 8;
    for (int idx = threadIdx.x; idx < 16 * NCH; idx += ATT_THREADS) {
        const int r = idx / NCH, ch = idx % NCH;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row_off[r] >= 0)
            v = *reinterpret_cast<const uint4 *>(q + row_off[r] + ch * 8);
        *reinterpret_cast<uint4 *>(misc + Misc<D>::Q_OFF + swz(r, ch, NCH)) = v;
    }
}

// ---------------------------------------------------------------------------
// The partial (m, l, o) of the 16-row query tile against one chunk, in two
// phases so that the caller can overlap the V copy with phase 1.
//
// Phase 1 (needs the Q tile, valid_len and the K tile visible): scores
// s = (q . k) * scale with mma.sync m16n8k16 (warp w takes keys
// [64w, 64w + 64), dims in ascending 16-steps), masked past each row's
// visible count, the row maximum m, p = exp(s - m), the bf16 P tile and the
// per-warp partial row sums (each thread adds its 16 values in key order,
// then a quad xor-tree over lanes 1, 2).  Every thread returns m for its
// rows rg = lane/4 and rg + 8.  Ends after writing shared memory; the caller
// must __syncthreads before phase 2.
template <int D>
__device__ __forceinline__ void chunk_phase1(uint32_t ktile, uint8_t *misc,
                                             float scale, float m[2]) {
    constexpr int NCH = D / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2, tq = lane & 3;
    const uint32_t qbase = smem_u32(misc + Misc<D>::Q_OFF);
    float *red = reinterpret_cast<float *>(misc + Misc<D>::RED_OFF);
    const int *valid_len = reinterpret_cast<const int *>(misc + Misc<D>::LEN_OFF);

    float sc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        {
            const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int ch = 2 * ks + (lane >> 4);
            ldsm_x4(qbase + swz(r, ch, NCH), a0, a1, a2, a3);
        }
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            const int key = 64 * warp + 16 * np + (lane & 7) + 8 * (lane >> 4);
            const int ch = 2 * ks + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ktile + swz(key, ch, NCH), b0, b1, b2, b3);
            mma_16816(sc[2 * np], a0, a1, a2, a3, b0, b1);
            mma_16816(sc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
    const int len0 = valid_len[rg], len1 = valid_len[rg + 8];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int key = 64 * warp + 8 * nt + 2 * tq + e;
            float s0 = __fmul_rn(sc[nt][e], scale);
            float s1 = __fmul_rn(sc[nt][2 + e], scale);
            s0 = key < len0 ? s0 : -INFINITY;
            s1 = key < len1 ? s1 : -INFINITY;
            sc[nt][e] = s0;
            sc[nt][2 + e] = s1;
            mx0 = fmaxf(mx0, s0);
            mx1 = fmaxf(mx1, s1);
        }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (tq == 0) {
        red[warp * 16 + rg] = mx0;
        red[warp * 16 + rg + 8] = mx1;
    }
    __syncthreads();
    const float m0 = fmaxf(fmaxf(red[rg], red[16 + rg]),
                           fmaxf(red[32 + rg], red[48 + rg]));
    const float m1 = fmaxf(fmaxf(red[8 + rg], red[24 + rg]),
                           fmaxf(red[40 + rg], red[56 + rg]));
    const float mu0 = m0 == -INFINITY ? 0.f : m0;
    const float mu1 = m1 == -INFINITY ? 0.f : m1;

    float l0 = 0.f, l1 = 0.f;
    uint8_t *P = misc + Misc<D>::P_OFF;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const float p00 = expf(__fsub_rn(sc[nt][0], mu0));
        const float p01 = expf(__fsub_rn(sc[nt][1], mu0));
        const float p10 = expf(__fsub_rn(sc[nt][2], mu1));
        const float p11 = expf(__fsub_rn(sc[nt][3], mu1));
        l0 = __fadd_rn(__fadd_rn(l0, p00), p01);
        l1 = __fadd_rn(__fadd_rn(l1, p10), p11);
        const int key = 64 * warp + 8 * nt + 2 * tq;  // even: a 4-byte pair
        const int ch = key >> 3, within = (key & 7) * 2;
        *reinterpret_cast<uint32_t *>(P + swz(rg, ch, 32) + within) =
            pack_bf16x2(p00, p01);
        *reinterpret_cast<uint32_t *>(P + swz(rg + 8, ch, 32) + within) =
            pack_bf16x2(p10, p11);
    }
    l0 = __fadd_rn(l0, __shfl_xor_sync(0xffffffffu, l0, 1));
    l0 = __fadd_rn(l0, __shfl_xor_sync(0xffffffffu, l0, 2));
    l1 = __fadd_rn(l1, __shfl_xor_sync(0xffffffffu, l1, 1));
    l1 = __fadd_rn(l1, __shfl_xor_sync(0xffffffffu, l1, 2));
    if (tq == 0) {
        red[64 + warp * 16 + rg] = l0;
        red[64 + warp * 16 + rg + 8] = l1;
    }
    m[0] = m0;
    m[1] = m1;
}

// Phase 2 (after a __syncthreads that follows phase 1 and the V copy): the
// row sums l = ((w0 + w1) + w2) + w3 over the per-warp partials and
// o = P V with mma.sync (warp w takes dims [w*D/4, (w+1)*D/4), keys in
// ascending 16-steps).  Each thread gets o[nt][0..1] for row rg and
// o[nt][2..3] for row rg + 8, dims w*D/4 + 8*nt + 2*(lane%4) + {0,1}.
template <int D>
__device__ __forceinline__ void chunk_phase2(uint32_t vtile, uint8_t *misc,
                                             float l[2], float o[D / 32][4]) {
    constexpr int NCH = D / 8;
    constexpr int NTV = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2;
    const uint32_t pbase = smem_u32(misc + Misc<D>::P_OFF);
    const float *red = reinterpret_cast<const float *>(misc + Misc<D>::RED_OFF);
    l[0] = __fadd_rn(__fadd_rn(__fadd_rn(red[64 + rg], red[80 + rg]),
                               red[96 + rg]),
                     red[112 + rg]);
    l[1] = __fadd_rn(__fadd_rn(__fadd_rn(red[72 + rg], red[88 + rg]),
                               red[104 + rg]),
                     red[120 + rg]);
#pragma unroll
    for (int nt = 0; nt < NTV; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < CHUNK / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        {
            const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int ch = 2 * kk + (lane >> 4);
            ldsm_x4(pbase + swz(r, ch, 32), a0, a1, a2, a3);
        }
        const int key = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
        if constexpr (NTV >= 2) {
#pragma unroll
            for (int np = 0; np < NTV / 2; ++np) {
                const int dim = warp * (D / 4) + 16 * np + 8 * (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vtile + swz(key, dim >> 3, NCH), b0, b1, b2, b3);
                mma_16816(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        } else {
            const int dim = warp * (D / 4);
            uint32_t b0, b1;
            ldsm_x2_t(vtile + swz(key, dim >> 3, NCH), b0, b1);
            mma_16816(o[0], a0, a1, a2, a3, b0, b1);
        }
    }
}

// One step of the fixed-order chunk merge.
__device__ __forceinline__ void merge_scalars(float &M, float &L, float m,
                                              float l, float &a, float &b) {
    const float Mn = fmaxf(M, m);
    a = expf(__fsub_rn(M, Mn));
    b = expf(__fsub_rn(m, Mn));
    L = __fadd_rn(__fmul_rn(L, a), __fmul_rn(l, b));
    M = Mn;
}
__device__ __forceinline__ float merge_value(float O, float o, float a,
                                             float b) {
    return __fadd_rn(__fmul_rn(O, a), __fmul_rn(o, b));
}

// Record layout of one decode chunk partial: m, l, 2 pad, o[D] (fp32).
template <int D>
constexpr int rec_floats() { return D + 4; }

// Number of chunks of each decode row (0 for pad rows), as an exclusive
// prefix: prefix[b] = sum of the counts of rows 0..b-1, prefix[B] = total.
// One block; the integer scan is exact, so its order does not matter.
__global__ void chunk_prefix_kernel(const int32_t *__restrict__ kv_len,
                                    const int32_t *__restrict__ row_req, int B,
                                    int Cmax, int32_t *__restrict__ prefix) {
    __shared__ int carry, wsum[32];
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int base = 0; base < B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int cnt = 0;
        if (b < B && row_req[b] >= 0) {
            const int L = kv_len[b];
            if (L > 0 && L <= Cmax * CHUNK) cnt = (L + CHUNK - 1) / CHUNK;
        }
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
        }
        if (lane == 31) wsum[w] = inc;
        __syncthreads();
        if (w == 0) {
            int x = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += n;
            }
            wsum[lane] = x;
        }
        __syncthreads();
        const int before = carry + (w > 0 ? wsum[w - 1] : 0);
        if (b < B) prefix[b] = before + inc - cnt;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = before + inc;
        __syncthreads();
    }
    if (threadIdx.x == 0) prefix[B] = carry;
}

// Decode chunk partials, persistent: CTA k takes work items k, k + grid,
// k + 2 grid, ...; item i is KV head i % Hkv of chunk j = i / Hkv in the
// row-major list of (row, chunk) pairs.  K and V tiles stream through a ring
// of three shared-memory slots (item n: K in slot 2n mod 3, V in slot
// 2n + 1 mod 3), so the copies of item n + 1 are in flight while item n is
// computed.  The arithmetic of each item is chunk_phase1 + chunk_phase2,
// exactly as in the prefill kernel.
template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    decode_chunks_kernel(const uint16_t *__restrict__ q,
                         const uint16_t *__restrict__ kp,
                         const uint16_t *__restrict__ vp,
                         const int32_t *__restrict__ page_table, int max_pages,
                         int n_pages, const int32_t *__restrict__ row_req,
                         const int32_t *__restrict__ kv_len, int B, int Hq,
                         int Hkv, int G, float scale, float *__restrict__ ws,
                         int Cmax, const int32_t *__restrict__ prefix,
                         int32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int64_t row_off[16];
    constexpr int TB = tile_bytes<D>();
    uint8_t *misc = smem + 3 * TB;
    const uint32_t slot0 = smem_u32(smem);
    const int total = prefix[B] * Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2, tq = lane & 3;

    // item n of this CTA -> (row b, head g, chunk c); false past the end
    auto item = [&](int n, int &b, int &g, int &c) -> bool {
        const int i = blockIdx.x + n * gridDim.x;
        if (i >= total) return false;
        g = i % Hkv;
        const int j = i / Hkv;
        int lo = 0, hi = B;  // largest b with prefix[b] <= j
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= j) lo = mid; else hi = mid;
        }
        b = lo;
        c = j - prefix[b];
        return true;
    };
    auto issue = [&](int n, bool is_v, int slot) {
        int b, g, c;
        if (item(n, b, g, c))
            load_tile<D>(slot0 + slot * TB, is_v ? vp : kp,
                         page_table + (int64_t)row_req[b] * max_pages,
                         max_pages, n_pages, Hkv, g, c, kv_len[b], status);
        cp_async_commit();
    };

    issue(0, false, 0);
    issue(0, true, 1);
    issue(1, false, 2);
    int b, g, c;
    for (int n = 0; item(n, b, g, c); ++n) {
        const int L = kv_len[b];
        int *valid_len = reinterpret_cast<int *>(misc + Misc<D>::LEN_OFF);
        if (threadIdx.x < 16) {
            valid_len[threadIdx.x] =
                threadIdx.x < G ? min(CHUNK, L - c * CHUNK) : 0;
            row_off[threadIdx.x] =
                threadIdx.x < G ? ((int64_t)b * Hq + g * G + threadIdx.x) * D
                                : -1;
        }
        __syncthreads();
        store_q<D>(misc, q, row_off);
        cp_async_wait<2>();  // K of item n
        __syncthreads();
        float m[2], l[2], o[D / 32][4];
        chunk_phase1<D>(slot0 + ((2 * n) % 3) * TB, misc, scale, m);
        __syncthreads();     // K slot free, P and row sums visible
        issue(n + 1, true, (2 * n) % 3);
        cp_async_wait<2>();  // V of item n
        __syncthreads();
        chunk_phase2<D>(slot0 + ((2 * n + 1) % 3) * TB, misc, l, o);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = rg + 8 * half;
            if (r >= G) continue;
            float *rec = ws + (((int64_t)b * Hq + g * G + r) * Cmax + c) *
                                  rec_floats<D>();
            if (warp == 0 && tq == 0) {
                rec[0] = m[half];
                rec[1] = l[half];
            }
#pragma unroll
            for (int nt = 0; nt < D / 32; ++nt) {
                const int dim = warp * (D / 4) + 8 * nt + 2 * tq;
                *reinterpret_cast<float2 *>(rec + 4 + dim) =
                    make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
            }
        }
        __syncthreads();     // V slot free
        issue(n + 2, false, (2 * n + 1) % 3);
    }
    cp_async_wait<0>();
}

// Second stage of decode: one warp per (row, head) merges chunks 0..C-1.
template <int D>
__global__ void decode_merge_kernel(const float *__restrict__ ws,
                                    const int32_t *__restrict__ kv_len,
                                    const int32_t *__restrict__ row_req, int B,
                                    int Hq, int Cmax,
                                    uint16_t *__restrict__ out) {
    constexpr int PER = D / 32;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= B * Hq) return;
    const int b = wid / Hq;
    uint16_t *dst = out + (int64_t)wid * D;
    const int L = kv_len[b];
    if (row_req[b] < 0 || L <= 0 || L > Cmax * CHUNK) {
        for (int i = 0; i < PER; ++i) dst[lane * PER + i] = 0;
        return;
    }
    const int C = (L + CHUNK - 1) / CHUNK;
    const float *rec = ws + (int64_t)wid * Cmax * rec_floats<D>();
    float M = rec[0], Ls = rec[1], O[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) O[i] = rec[4 + lane * PER + i];
    for (int c = 1; c < C; ++c) {
        const float *rc = rec + (int64_t)c * rec_floats<D>();
        float a, bb;
        merge_scalars(M, Ls, rc[0], rc[1], a, bb);
#pragma unroll
        for (int i = 0; i < PER; ++i)
            O[i] = merge_value(O[i], rc[4 + lane * PER + i], a, bb);
    }
#pragma unroll
    for (int i = 0; i < PER; ++i)
        dst[lane * PER + i] = f32_to_bf16(__fdiv_rn(O[i], Ls));
}

// Prefill / verify: CTA = (16-row tile of one segment, KV head g); loops
// over the chunks and merges in registers with the same functions.
template <int D>
__global__ void __launch_bounds__(ATT_THREADS)
    prefill_kernel(const uint16_t *__restrict__ q,
                   const int32_t *__restrict__ cu_q,
                   const int32_t *__restrict__ seg_req, int R,
                   const int32_t *__restrict__ pos,
                   const uint16_t *__restrict__ kp,
                   const uint16_t *__restrict__ vp,
                   const int32_t *__restrict__ page_table, int max_pages,
                   int n_pages, int Hq, int Hkv, int G, float scale,
                   int max_kv_len, uint16_t *__restrict__ out,
                   int32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int64_t row_off[16];
    __shared__ int s_info[4];  // t0, nq, req, valid_max
    constexpr int TB = tile_bytes<D>();
    const uint32_t ktile = smem_u32(smem), vtile = ktile + TB;
    uint8_t *misc = smem + 2 * TB;
    const int g = blockIdx.y;
    const int QPT = 16 / G;
    if (threadIdx.x == 0) {
        // Find the segment and the tile inside it.
        int tile = blockIdx.x, r = 0, t0 = -1, nq = 0;
        for (; r < R; ++r) {
            const int len = cu_q[r + 1] - cu_q[r];
            const int nt = (len + QPT - 1) / QPT;
            if (tile < nt) {
                t0 = cu_q[r] + tile * QPT;
                nq = min(QPT, len - tile * QPT);
                break;
            }
            tile -= nt;
        }
        s_info[0] = t0;
        s_info[1] = nq;
        s_info[2] = t0 >= 0 ? seg_req[r] : -1;
        s_info[3] = t0 >= 0 ? pos[t0 + nq - 1] + 1 : 0;
    }
    __syncthreads();
    const int t0 = s_info[0], nq = s_info[1], req = s_info[2];
    const int vmax = s_info[3];
    if (t0 < 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2, tq = lane & 3;
    if (req < 0 || vmax > max_kv_len) {
        if (req >= 0 && threadIdx.x == 0) bi_record_error(status, BI_ERR_BOUNDS);
        for (int idx = threadIdx.x; idx < nq * G * D; idx += ATT_THREADS) {
            const int qi = idx / (G * D), rem = idx % (G * D);
            out[((int64_t)(t0 + qi) * Hq + g * G) * D + rem] = 0;
        }
        return;
    }
    if (threadIdx.x < 16) {
        const int qi = threadIdx.x / G, hh = threadIdx.x % G;
        row_off[threadIdx.x] =
            qi < nq ? ((int64_t)(t0 + qi) * Hq + g * G + hh) * D : -1;
    }
    const int32_t *pt_row = page_table + (int64_t)req * max_pages;
    int *valid_len = reinterpret_cast<int *>(misc + Misc<D>::LEN_OFF);
    const int p_r0 = (rg / G) < nq ? pos[t0 + rg / G] : -1;
    const int p_r1 = ((rg + 8) / G) < nq ? pos[t0 + (rg + 8) / G] : -1;
    const int C = (vmax + CHUNK - 1) / CHUNK;

    float M[2] = {0.f, 0.f}, Ls[2] = {0.f, 0.f}, O[D / 32][4];
    for (int c = 0; c < C; ++c) {
        __syncthreads();  // previous chunk fully consumed
        if (threadIdx.x < 16) {
            const int qi = threadIdx.x / G;
            const int pr = qi < nq ? pos[t0 + qi] : -1;
            valid_len[threadIdx.x] = max(0, min(CHUNK, pr + 1 - c * CHUNK));
        }
        load_tile<D>(ktile, kp, pt_row, max_pages, n_pages, Hkv, g, c, vmax,
                     status);
        cp_async_commit();
        load_tile<D>(vtile, vp, pt_row, max_pages, n_pages, Hkv, g, c, vmax,
                     status);
        cp_async_commit();
        if (c == 0) {
            __syncthreads();
            store_q<D>(misc, q, row_off);
        }
        cp_async_wait<1>();
        __syncthreads();
        float m[2], l[2], o[D / 32][4];
        chunk_phase1<D>(ktile, misc, scale, m);
        cp_async_wait<0>();
        __syncthreads();
        chunk_phase2<D>(vtile, misc, l, o);
        const int pr[2] = {p_r0, p_r1};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (pr[half] + 1 - c * CHUNK <= 0) continue;  // chunk not visible
            if (c == 0) {
                M[half] = m[half];
                Ls[half] = l[half];
#pragma unroll
                for (int nt = 0; nt < D / 32; ++nt) {
                    O[nt][2 * half] = o[nt][2 * half];
                    O[nt][2 * half + 1] = o[nt][2 * half + 1];
                }
            } else {
                float a, bb;
                merge_scalars(M[half], Ls[half], m[half], l[half], a, bb);
#pragma unroll
                for (int nt = 0; nt < D / 32; ++nt) {
                    O[nt][2 * half] = merge_value(O[nt][2 * half],
                                                  o[nt][2 * half], a, bb);
                    O[nt][2 * half + 1] = merge_value(
                        O[nt][2 * half + 1], o[nt][2 * half + 1], a, bb);
                }
            }
        }
    }
    const int pr[2] = {p_r0, p_r1};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        if (pr[half] < 0) continue;
        const int r = rg + 8 * half;
        const int qi = r / G, hh = r % G;
        uint16_t *dst = out + ((int64_t)(t0 + qi) * Hq + g * G + hh) * D;
#pragma unroll
        for (int nt = 0; nt < D / 32; ++nt) {
            const int dim = warp * (D / 4) + 8 * nt + 2 * tq;
            *reinterpret_cast<uint32_t *>(dst + dim) =
                pack_bf16x2(__fdiv_rn(O[nt][2 * half], Ls[half]),
                            __fdiv_rn(O[nt][2 * half + 1], Ls[half]));
        }
    }
}

template <typename K>
bi_status set_attr(K kernel, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return bi_cuda_check(e, "attention smem attribute");
}

bool group_ok(int Hq, int Hkv) {
    if (Hkv <= 0 || Hq % Hkv) return false;
    const int G = Hq / Hkv;
    return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

size_t records_bytes(int B, int Hq, int D, int max_kv_len) {
    const int C = (max_kv_len + CHUNK - 1) / CHUNK;
    return ((size_t)B * Hq * C * (D + 4) * sizeof(float) + 255) & ~size_t(255);
}

}  // namespace

extern "C" size_t bi_decode_attn_workspace_size(int B, int Hq, int D,
                                                int max_kv_len) {
    if (B <= 0 || Hq <= 0 || D <= 0 || max_kv_len <= 0) return 0;
    return records_bytes(B, Hq, D, max_kv_len) +
           (((size_t)(B + 1) * sizeof(int32_t) + 255) & ~size_t(255));
}

// Decode attention with the pool size known (page ids are range-checked
// against it).  stages: bit 0 runs the chunk kernels, bit 1 the merge.
bi_status bi_decode_attn_pool(const bi_bf16 *q, const bi_bf16 *k_pool,
                              const bi_bf16 *v_pool, const int32_t *page_table,
                              int max_pages, int n_pages,
                              const int32_t *row_req, const int32_t *kv_len,
                              int B, int max_kv_len, int Hq, int Hkv, int D,
                              float scale, bi_bf16 *out, void *ws,
                              size_t ws_bytes, int stages,
                              cudaStream_t s) {
    BI_REQUIRE(B >= 0 && max_kv_len > 0 && max_kv_len <= 16 * max_pages,
               "bi_paged_decode_attn: B=%d max_kv_len=%d max_pages=%d", B,
               max_kv_len, max_pages);
    if (D != 32 && D != 128)
        return bi_fail(BI_ERR_UNSUPPORTED, "bi_paged_decode_attn: D=%d", D);
    if (!group_ok(Hq, Hkv))
        return bi_fail(BI_ERR_UNSUPPORTED,
                       "bi_paged_decode_attn: Hq=%d Hkv=%d", Hq, Hkv);
    BI_REQUIRE(q && k_pool && v_pool && page_table && row_req && kv_len && out,
               "bi_paged_decode_attn: null pointer");
    BI_REQUIRE(bi_aligned16(q) && bi_aligned16(k_pool) && bi_aligned16(v_pool) &&
                   bi_aligned16(out) && bi_aligned16(ws),
               "bi_paged_decode_attn: pointers must be 16-byte aligned");
    if (B == 0) return BI_OK;
    const size_t need = bi_decode_attn_workspace_size(B, Hq, D, max_kv_len);
    if (!ws || ws_bytes < need)
        return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                       "bi_paged_decode_attn: workspace %zu < %zu", ws_bytes,
                       need);
    const int Cmax = (max_kv_len + CHUNK - 1) / CHUNK;
    const int G = Hq / Hkv;
    float *rec = static_cast<float *>(ws);
    int32_t *prefix = reinterpret_cast<int32_t *>(
        static_cast<uint8_t *>(ws) + records_bytes(B, Hq, D, max_kv_len));
    int32_t *status = bi_status_ptr();
    if (stages & 1) {
        chunk_prefix_kernel<<<1, 1024, 0, s>>>(kv_len, row_req, B, Cmax,
                                               prefix);
        BI_LAUNCH_CHECK("decode chunk prefix launch");
        const int grid = bi_sm_count();
        if (D == 128) {
            static std::once_flag f;
            static bi_status fs;
            std::call_once(f, [] {
                fs = set_attr(decode_chunks_kernel<128>, decode_smem<128>());
            });
            if (fs != BI_OK) return fs;
            decode_chunks_kernel<128><<<grid, ATT_THREADS, decode_smem<128>(),
                                        s>>>(
                q, k_pool, v_pool, page_table, max_pages, n_pages, row_req,
                kv_len, B, Hq, Hkv, G, scale, rec, Cmax, prefix, status);
        } else {
            static std::once_flag f;
            static bi_status fs;
            std::call_once(f, [] {
                fs = set_attr(decode_chunks_kernel<32>, decode_smem<32>());
            });
            if (fs != BI_OK) return fs;
            decode_chunks_kernel<32><<<grid, ATT_THREADS, decode_smem<32>(),
                                       s>>>(
                q, k_pool, v_pool, page_table, max_pages, n_pages, row_req,
                kv_len, B, Hq, Hkv, G, scale, rec, Cmax, prefix, status);
        }
        BI_LAUNCH_CHECK("decode attention launch");
    }
    if (stages & 2) {
        const int warps = B * Hq;
        const int blocks = (warps * 32 + 255) / 256;
        if (D == 128)
            decode_merge_kernel<128><<<blocks, 256, 0, s>>>(
                rec, kv_len, row_req, B, Hq, Cmax, out);
        else
            decode_merge_kernel<32><<<blocks, 256, 0, s>>>(
                rec, kv_len, row_req, B, Hq, Cmax, out);
        BI_LAUNCH_CHECK("decode merge launch");
    }
    return BI_OK;
}

extern "C" bi_status bi_paged_decode_attn(
    const bi_bf16 *q, const bi_bf16 *k_pool, const bi_bf16 *v_pool,
    const int32_t *page_table, int max_pages, const int32_t *row_req,
    const int32_t *kv_len, int B, int max_kv_len, int Hq, int Hkv, int D,
    float scale, bi_bf16 *out, void *ws, size_t ws_bytes, void *stream) {
    // The pool size is not an argument of this entry point, so page ids are
    // range-checked against INT32_MAX only; the model driver passes the
    // real pool size.
    return bi_decode_attn_pool(q, k_pool, v_pool, page_table, max_pages,
                               0x7fffffff, row_req, kv_len, B, max_kv_len, Hq,
                               Hkv, D, scale, out, ws, ws_bytes, 3,
                               bi_stream(stream));
}

// ------------------------------------------- allocation-free decode variant --
//
// Scratch of bi_paged_decode_attn_noalloc: the chunk partials live in this
// fixed array instead of a caller-supplied workspace.  It is part of the
// module, so every GPU that loads the library holds these bytes until the
// process exits.  Host code cannot use the array's name as a device address;
// its address is looked up once per device below.
static __device__ __align__(256) uint8_t
    g_decode_noalloc_scratch[BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up with
// cudaGetSymbolAddress the first time the variant runs on that device.
static bi_status noalloc_scratch(void **out) {
    static std::mutex mu;
    static void *ptrs[64] = {nullptr};
    int dev = 0;
    bi_status st = bi_cuda_check(cudaGetDevice(&dev), "noalloc: cudaGetDevice");
    if (st != BI_OK) return st;
    if (dev < 0 || dev >= 64)
        return bi_fail(BI_ERR_UNSUPPORTED, "noalloc: device %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        st = bi_cuda_check(cudaGetSymbolAddress(&p, g_decode_noalloc_scratch),
                           "noalloc: cudaGetSymbolAddress");
        if (st != BI_OK) return st;
        ptrs[dev] = p;
    }
    *out = ptrs[dev];
    return BI_OK;
}

extern "C" bi_status bi_paged_decode_attn_noalloc(
    const bi_bf16 *q, const bi_bf16 *k_pool, const bi_bf16 *v_pool,
    const int32_t *page_table, int max_pages, const int32_t *row_req,
    const int32_t *kv_len, int B, int max_kv_len, int Hq, int Hkv, int D,
    float scale, bi_bf16 *out, void *stream) {
    const size_t need = bi_decode_attn_workspace_size(B, Hq, D, max_kv_len);
    if (need > (size_t)BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES)
        return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                       "bi_paged_decode_attn_noalloc: B=%d Hq=%d D=%d "
                       "max_kv_len=%d needs %zu bytes of scratch, more than "
                       "the fixed %d; use bi_paged_decode_attn with a "
                       "workspace",
                       B, Hq, D, max_kv_len, need,
                       (int)BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES);
    void *ws = nullptr;
    bi_status st = noalloc_scratch(&ws);
    if (st != BI_OK) return st;
    // The chunk kernel writes every partial the merge kernel reads, so
    // nothing left in the array by an earlier call is ever read.
    return bi_decode_attn_pool(q, k_pool, v_pool, page_table, max_pages,
                               0x7fffffff, row_req, kv_len, B, max_kv_len, Hq,
                               Hkv, D, scale, out, ws,
                               BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES, 3,
                               bi_stream(stream));
}

bi_status bi_prefill_attn_pool(const bi_bf16 *q, const int32_t *cu_q,
                               const int32_t *seg_req, int R, int T,
                               const int32_t *pos, int max_q, int max_kv_len,
                               const bi_bf16 *k_pool, const bi_bf16 *v_pool,
                               const int32_t *page_table, int max_pages,
                               int n_pages, int Hq, int Hkv, int D,
                               float scale, bi_bf16 *out,
                               cudaStream_t stream) {
    BI_REQUIRE(R >= 0 && T >= 0 && max_q >= 0 && max_kv_len > 0 &&
                   max_kv_len <= 16 * max_pages,
               "bi_prefill_attn: R=%d T=%d max_q=%d max_kv_len=%d", R, T,
               max_q, max_kv_len);
    if (D != 32 && D != 128)
        return bi_fail(BI_ERR_UNSUPPORTED, "bi_prefill_attn: D=%d", D);
    if (!group_ok(Hq, Hkv))
        return bi_fail(BI_ERR_UNSUPPORTED, "bi_prefill_attn: Hq=%d Hkv=%d", Hq,
                       Hkv);
    BI_REQUIRE(q && cu_q && seg_req && pos && k_pool && v_pool && page_table &&
                   out,
               "bi_prefill_attn: null pointer");
    BI_REQUIRE(bi_aligned16(q) && bi_aligned16(k_pool) && bi_aligned16(v_pool) &&
                   bi_aligned16(out),
               "bi_prefill_attn: pointers must be 16-byte aligned");
    if (T == 0 || R == 0) return BI_OK;
    const int G = Hq / Hkv;
    const int QPT = 16 / G;
    const int tiles = (T + QPT - 1) / QPT + R;
    int32_t *status = bi_status_ptr();
    dim3 grid(tiles, Hkv);
    if (D == 128) {
        static std::once_flag f;
        static bi_status fs;
        std::call_once(f, [] {
            fs = set_attr(prefill_kernel<128>, prefill_smem<128>());
        });
        if (fs != BI_OK) return fs;
        prefill_kernel<128><<<grid, ATT_THREADS, prefill_smem<128>(), stream>>>(
            q, cu_q, seg_req, R, pos, k_pool, v_pool, page_table, max_pages,
            n_pages, Hq, Hkv, G, scale, max_kv_len, out, status);
    } else {
        prefill_kernel<32><<<grid, ATT_THREADS, prefill_smem<32>(), stream>>>(
            q, cu_q, seg_req, R, pos, k_pool, v_pool, page_table, max_pages,
            n_pages, Hq, Hkv, G, scale, max_kv_len, out, status);
    }
    BI_LAUNCH_CHECK("prefill attention launch");
    return BI_OK;
}

extern "C" bi_status bi_prefill_attn(
    const bi_bf16 *q, const int32_t *cu_q, const int32_t *seg_req, int R,
    int T, const int32_t *pos, int max_q, int max_kv_len,
    const bi_bf16 *k_pool, const bi_bf16 *v_pool, const int32_t *page_table,
    int max_pages, int Hq, int Hkv, int D, float scale, bi_bf16 *out,
    void *stream) {
    return bi_prefill_attn_pool(q, cu_q, seg_req, R, T, pos, max_q, max_kv_len,
                                k_pool, v_pool, page_table, max_pages,
                                0x7fffffff, Hq, Hkv, D, scale, out,
                                bi_stream(stream));
}
