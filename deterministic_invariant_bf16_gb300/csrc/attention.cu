// bi_paged_decode_attn and bi_prefill_attn: causal grouped-query attention
// over the paged KV cache in fixed 256-position chunks.
//
// Invariance (Vosti abstract: bitwise-equal kernel outputs across batches,
// query lengths and paged KV layouts; ybb.press section 4: two-stage
// fixed-order reductions).  The arithmetic applied to one (query row, head)
// depends only on its query vector, its position and the logical KV prefix:
//
//   chunk c covers absolute positions [256c, 256c + 256).  For each chunk a
//   partial (m, l, o) is computed FROM SCRATCH:
//     s_j = (q . k_j) * scale   MMA over the head dims in ascending 16-steps
//     s_j = -inf past the row's context
//     m   = max_j s_j
//     p_j = exp(s_j - m)        head_dim 128: p_of, 2^(s c1 - m log2 e)
//     l   = sum_j p_j           fixed order: each 32-key group by an xor
//                               tree, the eight groups in order
//     o   = sum_j bf16(p_j) v_j MMA over the keys in ascending 16-steps
//   chunks are merged in ascending c by merge_scalars/merge_value:
//     m' = max(m, m_c); a = exp(m - m'); b = exp(m_c - m')
//     l  = l a + l_c b;  o = o a + o_c b;   out = bf16(o / l)
//
// Kernels.  Head_dim 128 runs on tcgen05 with TMA page boxes:
//   attn_tc_kernel       decode, persistent over whole (row, KV head) items
//                        (S^T = K Q^T and O^T = V^T P^T, N = 16 query rows),
//                        chunks merged in registers;
//   decode_tc_chunks_kernel  the same over (row, chunk) items for small
//                        batches, writing fp32 records that
//                        decode_merge_kernel merges in chunk order;
//   attn_rows_kernel     prefill and verify, 128-row query tiles with one
//                        thread per query row (S = Q K^T, O = P V, N = 256
//                        keys / 128 dims); in-kernel over a tile's chunks, or
//                        in split form, one item per (tile, chunk, KV head)
//                        writing the same records for decode_merge_kernel;
//   prefill_tc_kernel    prefill without a workspace, 16-row tiles.
// Head_dim 32 runs the mma.sync forms (decode_chunks_kernel + merge,
// prefill_kernel).  All forms share the phase and merge functions, every
// floating-point operation outside the MMAs is an explicit round-to-nearest
// intrinsic, and the tensor core's per-element results do not depend on N
// or on which operand holds the row, so a row's bits are the same in every
// kernel and batch.
//
// Positions past a row's context never contribute: their scores are
// replaced by -inf (a select, so stale or NaN keys cannot leak) and their
// p is 0 without evaluating exp (exp(-inf) is 0 as well), and the V rows past
// the visible part of a chunk are zero-filled (0 * NaN would poison the PV
// product).
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int CHUNK = 256;
constexpr int RING = 3;               // decode tile slots

// Compute warps per chunk: 16 for head_dim 128 (each warp 16 keys in the
// score phase, 8 dims in the PV phase), 4 for head_dim 32.
template <int D>
constexpr int nwarps() { return D == 128 ? 16 : 4; }
template <int D>
constexpr int cthreads() { return nwarps<D>() * 32; }

// Byte offset of 16-byte piece `ch` (0 .. D/8 - 1) of row `row` in a K, V
// or Q tile of ROWS rows.  D = 128: two 64-column halves, each [ROWS][128 B]
// laid out as the TMA 128-byte swizzle writes it (piece XOR row % 8), so
// ldmatrix row groups hit distinct banks.  D = 32: plain [ROWS][64 B].
template <int D, int ROWS>
__device__ __forceinline__ uint32_t toff(int row, int ch) {
    if constexpr (D == 128) {
        return (uint32_t)((ch >> 3) * (ROWS * 128) + row * 128 +
                          (((ch & 7) ^ (row & 7)) << 4));
    } else {
        return (uint32_t)(row * (D * 2) + ch * 16);
    }
}

// P tile (bf16 [16][256]) offset: 32 pieces per row, XOR-swizzled.
__device__ __forceinline__ uint32_t poff(int row, int ch) {
    return (uint32_t)(row * 512 + ((ch ^ (row & 7)) << 4));
}

template <int D>
constexpr int tile_bytes() { return CHUNK * D * 2; }
template <int D>
constexpr int qtile_bytes() { return 16 * D * 2; }
constexpr int P_BYTES = 16 * CHUNK * 2;
// cross-warp slots: row maxima [NW][16], then row sums [NW][16]
template <int D>
constexpr int red_bytes() { return 2 * nwarps<D>() * 16 * 4; }

// Barrier among the compute threads: the whole CTA (BAR = 0) or the compute
// warps of the decode kernel (named barrier BAR).
template <int D, int BAR>
__device__ __forceinline__ void compute_sync() {
    if constexpr (BAR == 0)
        __syncthreads();
    else
        asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(cthreads<D>())
                     : "memory");
}

// ---------------------------------------------------------------------------
// The partial (m, l, o) of a 16-row query tile against one chunk, in two
// phases so that loads can overlap phase 1.
//
// Phase 1 (Q and K tiles visible): scores s = (q . k) * scale with
// mma.sync m16n8k16 (warp w takes keys [w*KPW, (w+1)*KPW)); the dims are
// summed as two independent chains, the low and the high half of the dims
// each in ascending 16-steps, added low + high (two chains halve the
// dependent MMA latency), masked past len0 (row rg = lane/4) and len1 (row
// rg + 8), the
// row maximum m, p = exp(s - m), the bf16 P tile and the per-warp partial row
// sums (each thread adds its values in key order, then a quad xor-tree over
// lanes 1, 2).  Returns m for rows rg and rg + 8.  Ends after writing shared
// memory; the caller must synchronise the compute threads before phase 2.
// low8: only tile rows 0-7 are used (decode with G <= 8); rows 8-15 of Q
// are then not loaded (their MMA rows come out as don't-care values, the
// tensor core keeps rows independent) and their p is neither computed nor
// stored, which halves the shared-memory reads of Q and P.
template <int D, int BAR>
__device__ __forceinline__ void chunk_phase1(uint32_t ktile, uint32_t qtile,
                                             uint32_t ptile, float *red,
                                             float scale, int len0, int len1,
                                             float m[2], bool low8) {
    constexpr int NW = nwarps<D>();
    constexpr int KPW = CHUNK / NW;   // keys per warp
    constexpr int NT = KPW / 8;       // score n-tiles per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2, tq = lane & 3;

    constexpr int KS = D / 16;        // 16-dim steps
    static_assert(KS % 2 == 0, "two chains over the dims");
    float sc[NT][4], sh[NT][4];       // low-half and high-half chains
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[i][e] = sh[i][e] = 0.f;
#pragma unroll
    for (int step = 0; step < KS; ++step) {
        // interleave the chains: low step j, then high step j
        const int ks = (step >> 1) + (step & 1) * (KS / 2);
        float(*acc)[4] = (step & 1) ? sh : sc;
        uint32_t a0, a1 = 0, a2, a3 = 0;
        if (low8) {
            const int r = lane & 7;
            const int ch = 2 * ks + ((lane >> 3) & 1);
            ldsm_x2(qtile + toff<D, 16>(r, ch), a0, a2);
        } else {
            const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int ch = 2 * ks + (lane >> 4);
            ldsm_x4(qtile + toff<D, 16>(r, ch), a0, a1, a2, a3);
        }
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            const int key = KPW * warp + 16 * np + (lane & 7) + 8 * (lane >> 4);
            const int ch = 2 * ks + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ktile + toff<D, CHUNK>(key, ch), b0, b1, b2, b3);
            mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
            mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[i][e] = __fadd_rn(sc[i][e], sh[i][e]);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int key = KPW * warp + 8 * nt + 2 * tq + e;
            float s0 = __fmul_rn(sc[nt][e], scale);
            s0 = key < len0 ? s0 : -INFINITY;
            sc[nt][e] = s0;
            mx0 = fmaxf(mx0, s0);
            if (!low8) {
                float s1 = __fmul_rn(sc[nt][2 + e], scale);
                s1 = key < len1 ? s1 : -INFINITY;
                sc[nt][2 + e] = s1;
                mx1 = fmaxf(mx1, s1);
            }
        }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    if (!low8) {
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    }
    if (tq == 0) {
        red[warp * 16 + rg] = mx0;
        red[warp * 16 + rg + 8] = mx1;
    }
    compute_sync<D, BAR>();
    // block maxima: lane tq of a quad reads warps tq, tq + 4, ..., then the
    // quad combines (a maximum does not depend on the order)
    float m0 = red[tq * 16 + rg], m1 = -INFINITY;
#pragma unroll
    for (int w = tq + 4; w < NW; w += 4) m0 = fmaxf(m0, red[w * 16 + rg]);
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    if (!low8) {
        m1 = red[tq * 16 + 8 + rg];
#pragma unroll
        for (int w = tq + 4; w < NW; w += 4)
            m1 = fmaxf(m1, red[w * 16 + 8 + rg]);
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    }
    const float mu0 = m0 == -INFINITY ? 0.f : m0;
    const float mu1 = m1 == -INFINITY ? 0.f : m1;

    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int key = KPW * warp + 8 * nt + 2 * tq;  // even: a 4-byte pair
        const float p00 = key < len0 ? expf(__fsub_rn(sc[nt][0], mu0)) : 0.f;
        const float p01 = key + 1 < len0 ? expf(__fsub_rn(sc[nt][1], mu0)) : 0.f;
        l0 = __fadd_rn(__fadd_rn(l0, p00), p01);
        const int ch = key >> 3, within = (key & 7) * 2;
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(ptile + poff(rg, ch) +
                                                       within),
                     "r"(pack_bf16x2(p00, p01))
                     : "memory");
        if (!low8) {
            const float p10 =
                key < len1 ? expf(__fsub_rn(sc[nt][2], mu1)) : 0.f;
            const float p11 =
                key + 1 < len1 ? expf(__fsub_rn(sc[nt][3], mu1)) : 0.f;
            l1 = __fadd_rn(__fadd_rn(l1, p10), p11);
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(
                             ptile + poff(rg + 8, ch) + within),
                         "r"(pack_bf16x2(p10, p11))
                         : "memory");
        }
    }
    l0 = __fadd_rn(l0, __shfl_xor_sync(0xffffffffu, l0, 1));
    l0 = __fadd_rn(l0, __shfl_xor_sync(0xffffffffu, l0, 2));
    l1 = __fadd_rn(l1, __shfl_xor_sync(0xffffffffu, l1, 1));
    l1 = __fadd_rn(l1, __shfl_xor_sync(0xffffffffu, l1, 2));
    if (tq == 0) {
        red[NW * 16 + warp * 16 + rg] = l0;
        red[NW * 16 + warp * 16 + rg + 8] = l1;
    }
    m[0] = m0;
    m[1] = m1;
}

// Phase 2 (after a compute-thread barrier that follows phase 1 and the V
// copy): the row sums l = (..((w0 + w1) + w2) ..) + w_{NW-1} over the
// per-warp partials, and o = P V with mma.sync (warp w takes dims
// [w*DPW, (w+1)*DPW)); the 16 key steps form four independent chains,
// chain j taking steps j, j + 4, j + 8, j + 12 in that order, and
// o = (c0 + c1) + (c2 + c3).  Each thread gets
// o[nt][0..1] for row rg and o[nt][2..3] for row rg + 8, dims
// w*DPW + 8*nt + 2*(lane%4) + {0,1}.
// need_l: this thread uses l (else l is left 0 and the sums are skipped).
template <int D>
__device__ __forceinline__ void chunk_phase2(uint32_t vtile, uint32_t ptile,
                                             const float *red, float l[2],
                                             float o[][4], bool low8,
                                             bool need_l) {
    constexpr int NW = nwarps<D>();
    constexpr int DPW = D / NW;       // dims per warp
    constexpr int NTV = DPW / 8;      // PV n-tiles per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = lane >> 2;
    l[0] = l[1] = 0.f;
    if (need_l) {
        float la = red[NW * 16 + rg];
#pragma unroll
        for (int w = 1; w < NW; ++w)
            la = __fadd_rn(la, red[NW * 16 + w * 16 + rg]);
        l[0] = la;
        if (!low8) {
            float lb = red[NW * 16 + 8 + rg];
#pragma unroll
            for (int w = 1; w < NW; ++w)
                lb = __fadd_rn(lb, red[NW * 16 + w * 16 + 8 + rg]);
            l[1] = lb;
        }
    }
    float oc[4][NTV][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int nt = 0; nt < NTV; ++nt)
            oc[j][nt][0] = oc[j][nt][1] = oc[j][nt][2] = oc[j][nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < CHUNK / 16; ++kk) {
        float(*acc)[4] = oc[kk & 3];
        uint32_t a0, a1 = 0, a2, a3 = 0;
        if (low8) {  // P rows 8-15 unused (see chunk_phase1)
            const int r = lane & 7;
            const int ch = 2 * kk + ((lane >> 3) & 1);
            ldsm_x2(ptile + poff(r, ch), a0, a2);
        } else {
            const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int ch = 2 * kk + (lane >> 4);
            ldsm_x4(ptile + poff(r, ch), a0, a1, a2, a3);
        }
        const int key = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
        if constexpr (NTV >= 2) {
#pragma unroll
            for (int np = 0; np < NTV / 2; ++np) {
                const int dim = warp * DPW + 16 * np + 8 * (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vtile + toff<D, CHUNK>(key, dim >> 3), b0, b1, b2,
                          b3);
                mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
                mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        } else {
            const int dim = warp * DPW;
            uint32_t b0, b1;
            ldsm_x2_t(vtile + toff<D, CHUNK>(key, dim >> 3), b0, b1);
            mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NTV; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[nt][e] = __fadd_rn(__fadd_rn(oc[0][nt][e], oc[1][nt][e]),
                                 __fadd_rn(oc[2][nt][e], oc[3][nt][e]));
}

// 2^y by the PTX base-2 exponential ex2.approx.ftz (relative error about
// 2^-22; results below 2^-126 flush to zero).  e^x is taken as
// 2^rn(x log2 e) (change of base) by the merge below and, with the
// argument from one fma, for the softmax's p (p_of).
constexpr float LOG2E = 1.4426950408889634f;
__device__ __forceinline__ float exp2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// One step of the fixed-order chunk merge: the new maximum, the factors
// a = e^(M - M'), b = e^(m - M') (each 2^rn(rn(x - M') log2 e)), and the
// running sum.  Every path's merge goes through this one function.
__device__ __forceinline__ void merge_scalars(float &M, float &L, float m,
                                              float l, float &a, float &b) {
    const float Mn = fmaxf(M, m);
    a = exp2_approx(__fmul_rn(__fsub_rn(M, Mn), LOG2E));
    b = exp2_approx(__fmul_rn(__fsub_rn(m, Mn), LOG2E));
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

// Zero the 16-byte pieces of rows [from, 256) of a tile (compute threads).
template <int D>
__device__ __forceinline__ void zero_rows(uint32_t tile, int from) {
    constexpr int NCH = D / 8;
    for (int idx = threadIdx.x; idx < (CHUNK - from) * NCH;
         idx += cthreads<D>()) {
        const int row = from + idx / NCH, ch = idx % NCH;
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                         tile + toff<D, CHUNK>(row, ch)),
                     "r"(0)
                     : "memory");
    }
}

// ------------------------------------------------------------------ decode --

// Work list of the decode kernels: for each row b with row_req >= 0 and a
// context within bounds, C_b = ceil(kv_len / 256) chunks.  prefix[b] is the
// exclusive prefix of C_b (prefix[B] = total) and items[prefix[b] + c] =
// (b, c).  One block; integer scans are exact, so their order is free.
__global__ void build_items_kernel(const int32_t *__restrict__ kv_len,
                                   const int32_t *__restrict__ row_req, int B,
                                   int Cmax, int32_t *__restrict__ prefix,
                                   int2 *__restrict__ items) {
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
        const int before = carry + (w > 0 ? wsum[w - 1] : 0) + inc - cnt;
        if (b < B) {
            prefix[b] = before;
            for (int c = 0; c < cnt; ++c) items[before + c] = make_int2(b, c);
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = before + cnt;
        __syncthreads();
    }
    if (threadIdx.x == 0) prefix[B] = carry;
}

// Shared-memory layout of the decode kernel (offsets from a 1024-aligned
// base): RING tile slots, RING query slots, the P tile, the reduction slots,
// then the mbarriers.
template <int D>
struct DecSmem {
    static constexpr int SLOT = 0;
    static constexpr int QSLOT = SLOT + RING * tile_bytes<D>();
    static constexpr int P = QSLOT + RING * qtile_bytes<D>();
    static constexpr int RED = P + P_BYTES;
    static constexpr int BAR = RED + red_bytes<D>();     // full[], empty[]
    static constexpr int BYTES = BAR + 2 * RING * 8;
    static constexpr int ALLOC = BYTES + 1024;           // alignment slack
};

// Items a CTA's prefetch warp may run ahead of its producer.
constexpr int PF_AHEAD = 2;

// Persistent decode chunk kernel.  CTA k takes work items k, k + grid,
// k + 2 grid, ...; item i is KV head i % Hkv of list entry i / Hkv.  Item n
// of a CTA loads K (with the Q rows) into slot 2n mod RING and V into slot
// 2n + 1 mod RING.  Warp NW is the producer: it waits for a slot to be
// freed, reads the chunk's page ids (one lane per page) and issues one TMA
// box per page and 64-column half.  Warp NW + 1 walks the same items up to
// PF_AHEAD ahead of the producer and asks L2 for their K and V pages, so
// that DRAM reads start before a shared-memory slot is free for them.  The
// compute warps wait for the tiles, run the two phases and store the
// partial record.
template <int D>
__global__ void __launch_bounds__(cthreads<D>() + 64, 1)
    decode_chunks_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap,
                         const __grid_constant__ CUtensorMap qmap,
                         const int32_t *__restrict__ page_table, int max_pages,
                         int n_pages, const int32_t *__restrict__ row_req,
                         const int32_t *__restrict__ kv_len, int Hq, int Hkv,
                         int G, float scale, float *__restrict__ ws, int Cmax,
                         const int32_t *__restrict__ prefix, int B,
                         const int2 *__restrict__ items,
                         const bi_bf16 *__restrict__ k_pool,
                         const bi_bf16 *__restrict__ v_pool, int32_t *status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_progress;  // items the producer has issued
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = DecSmem<D>;
    constexpr int NW = nwarps<D>();
    constexpr int DPW = D / NW;
    constexpr int TB = tile_bytes<D>(), QB = qtile_bytes<D>();
    constexpr int HALVES = D == 128 ? 2 : 1;
    constexpr int BOX_W = D == 128 ? 64 : D;            // columns per box
    constexpr int PAGE_BYTES = 16 * BOX_W * 2;          // one box
    constexpr int HALF_TILE = CHUNK * BOX_W * 2;        // one half of a tile
    constexpr int HALF_Q = 16 * BOX_W * 2;
    const uint32_t base = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR);
    uint64_t *empty = full + RING;
    float *red = reinterpret_cast<float *>(smem + L::RED);
    const uint32_t ptile = base + L::P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = prefix[B] * Hkv;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RING; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        mbar_fence_init();
        s_progress = 0;
    }
    __syncthreads();
    volatile int *progress = &s_progress;

    if (warp == NW + 1) {
        // ------------------------------------------------------ prefetch --
        constexpr uint32_t PAGE_KV = 16 * D * 2;  // one (page, head) of K
        for (int n = 0;; ++n) {
            const int i = blockIdx.x + n * gridDim.x;
            if (i >= total) break;
            bool go = true;
            if (lane == 0 && *progress + PF_AHEAD < n) {
                const uint64_t t0 = bi_globaltimer();
                while (*progress + PF_AHEAD < n) {
                    __nanosleep(256);
                    if (bi_globaltimer() - t0 > BI_WAIT_LIMIT_NS) {
                        go = false;  // the producer stopped; nothing to do
                        break;
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) break;
            const int g = i % Hkv;
            const int2 bc = items[i / Hkv];
            const int vl = min(CHUNK, kv_len[bc.x] - bc.y * CHUNK);
            const int npg = (vl + 15) >> 4;
            if (lane < npg) {
                const int pi = bc.y * 16 + lane;
                const int pg = pi < max_pages
                                   ? page_table[(int64_t)row_req[bc.x] *
                                                    max_pages + pi]
                                   : -1;
                if (pg >= 0 && pg < n_pages) {
                    const int64_t off = ((int64_t)pg * Hkv + g) * 16 * D;
                    prefetch_l2_bulk(k_pool + off, PAGE_KV);
                    prefetch_l2_bulk(v_pool + off, PAGE_KV);
                }
            }
        }
        return;
    }

    if (warp == NW) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            tma_prefetch_desc(&qmap);
        }
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int i = blockIdx.x + n * gridDim.x;
            if (i >= total) break;
            const int g = i % Hkv;
            const int2 bc = items[i / Hkv];
            const int b = bc.x, c = bc.y;
            const int Lb = kv_len[b];
            const int vl = min(CHUNK, Lb - c * CHUNK);
            const int npg = (vl + 15) >> 4;
            const int32_t *pt_row = page_table + (int64_t)row_req[b] * max_pages;
            int pg = -1;
            if (lane < npg) {
                const int pi = c * 16 + lane;
                pg = pi < max_pages ? pt_row[pi] : -1;
                if (pg < 0 || pg >= n_pages) {
                    bi_record_error(status, BI_ERR_BOUNDS);
                    pg = -1;
                }
            }
            const unsigned have = __ballot_sync(0xffffffffu, pg >= 0);
            const int nvalid = __popc(have);
            for (int kv = 0; kv < 2 && ok; ++kv) {
                const int j = 2 * n + kv;
                const int slot = j % RING;
                const int use = j / RING;
                bool w_ok = true;
                if (lane == 0 && use > 0)
                    w_ok = mbar_wait(&empty[slot], (use - 1) & 1, status);
                ok = __shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (lane == 0)
                    mbar_arrive_expect_tx(
                        &full[slot],
                        nvalid * HALVES * PAGE_BYTES +
                            (kv == 0 ? HALVES * HALF_Q : 0));
                __syncwarp();
                const CUtensorMap *map = kv == 0 ? &kmap : &vmap;
                if (pg >= 0) {
                    const int row = (pg * Hkv + g) * 16;
#pragma unroll
                    for (int h = 0; h < HALVES; ++h)
                        tma_load_2d(smem + L::SLOT + slot * TB + h * HALF_TILE +
                                        lane * PAGE_BYTES,
                                    map, h * BOX_W, row, &full[slot]);
                }
                if (kv == 0 && lane == 0) {
#pragma unroll
                    for (int h = 0; h < HALVES; ++h)
                        tma_load_2d(smem + L::QSLOT + slot * QB + h * HALF_Q,
                                    &qmap, h * BOX_W, b * Hq + g * G,
                                    &full[slot]);
                }
            }
            if (lane == 0) *progress = n + 1;
        }
        if (lane == 0) *progress = 0x3fffffff;  // release the prefetch warp
        return;
    }

    // ------------------------------------------------------- compute --
    const int rg = lane >> 2, tq = lane & 3;
    // (row, chunk, visible length) of the next item, loaded one item ahead
    int nb = 0, nc = 0, nvl = 0;
    if (blockIdx.x < total) {
        const int2 bc = items[blockIdx.x / Hkv];
        nb = bc.x;
        nc = bc.y;
        nvl = min(CHUNK, kv_len[nb] - nc * CHUNK);
    }
    for (int n = 0;; ++n) {
        const int i = blockIdx.x + n * gridDim.x;
        if (i >= total) break;
        const int g = i % Hkv;
        const int b = nb, c = nc, vl = nvl;
        if (i + (int)gridDim.x < total) {
            const int2 bc = items[(i + gridDim.x) / Hkv];
            nb = bc.x;
            nc = bc.y;
            nvl = min(CHUNK, kv_len[nb] - nc * CHUNK);
        }
        const int len0 = rg < G ? vl : 0, len1 = rg + 8 < G ? vl : 0;
        const int sk = (2 * n) % RING, sv = (2 * n + 1) % RING;
        if (!mbar_wait(&full[sk], ((2 * n) / RING) & 1, status)) break;
        float m[2], l[2], o[DPW / 8][4];
        chunk_phase1<D, 1>(base + L::SLOT + sk * TB, base + L::QSLOT + sk * QB,
                           ptile, red, scale, len0, len1, m, G <= 8);
        // the K slot was only read: the barrier alone orders the next copy
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sk]);
        if (!mbar_wait(&full[sv], ((2 * n + 1) / RING) & 1, status)) break;
        const uint32_t vtile = base + L::SLOT + sv * TB;
        if (vl < CHUNK) zero_rows<D>(vtile, vl);
        compute_sync<D, 1>();
        // only warp 0 stores (m, l)
        chunk_phase2<D>(vtile, ptile, red, l, o, G <= 8, warp == 0);
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
            for (int nt = 0; nt < DPW / 8; ++nt) {
                const int dim = warp * DPW + 8 * nt + 2 * tq;
                *reinterpret_cast<float2 *>(rec + 4 + dim) =
                    make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
            }
        }
        // rows zeroed by these threads must be ordered before the next copy
        // into the slot (a different proxy); a slot only read needs no fence
        if (vl < CHUNK) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sv]);
    }
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
    // Records are loaded four at a time (independent loads in flight), then
    // merged strictly in chunk order.
    constexpr int BATCH = 4;
    for (int c0 = 1; c0 < C; c0 += BATCH) {
        float mb[BATCH], lb[BATCH], ob[BATCH][PER];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int c = c0 + j;
            if (c < C) {
                const float *rc = rec + (int64_t)c * rec_floats<D>();
                mb[j] = rc[0];
                lb[j] = rc[1];
#pragma unroll
                for (int i = 0; i < PER; ++i) ob[j][i] = rc[4 + lane * PER + i];
            }
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            if (c0 + j >= C) break;
            float a, bb;
            merge_scalars(M, Ls, mb[j], lb[j], a, bb);
#pragma unroll
            for (int i = 0; i < PER; ++i)
                O[i] = merge_value(O[i], ob[j][i], a, bb);
        }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i)
        dst[lane * PER + i] = f32_to_bf16(__fdiv_rn(O[i], Ls));
}

// ----------------------------------------------------------------- prefill --

// Issue (not commit) cp.async copies of chunk c of KV head g of page-table
// row pt_row into a tile.  Positions >= valid_max are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t tile,
                                          const uint16_t *__restrict__ pool,
                                          const int32_t *__restrict__ pt_row,
                                          int max_pages, int n_pages, int Hkv,
                                          int g, int c, int valid_max,
                                          int32_t *status, int nthreads) {
    constexpr int NCH = D / 8;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < CHUNK * NCH; idx += nthreads) {
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
        cp_async16(tile + toff<D, CHUNK>(key, ch), src, bytes);
    }
}

template <int D>
constexpr int prefill_smem() {
    return 2 * tile_bytes<D>() + qtile_bytes<D>() + P_BYTES + red_bytes<D>();
}

// Prefill / verify: CTA = (16-row tile of one segment, KV head g); loops
// over the chunks and merges in registers with the same functions.
template <int D>
__global__ void __launch_bounds__(cthreads<D>())
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
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int s_info[4];  // t0, nq, req, valid_max
    constexpr int TB = tile_bytes<D>();
    constexpr int NCH = D / 8;
    constexpr int NT = cthreads<D>();
    constexpr int DPW = D / nwarps<D>();
    const uint32_t ktile = smem_u32(smem), vtile = ktile + TB;
    const uint32_t qtile = vtile + TB;
    const uint32_t ptile = qtile + qtile_bytes<D>();
    float *red = reinterpret_cast<float *>(smem + 2 * TB + qtile_bytes<D>() +
                                           P_BYTES);
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
        for (int idx = threadIdx.x; idx < nq * G * D; idx += NT) {
            const int qi = idx / (G * D), rem = idx % (G * D);
            out[((int64_t)(t0 + qi) * Hq + g * G) * D + rem] = 0;
        }
        return;
    }
    // query tile: row r = (query qi, head hh) with r = qi * G + hh
    for (int idx = threadIdx.x; idx < 16 * NCH; idx += NT) {
        const int r = idx / NCH, ch = idx % NCH;
        const int qi = r / G, hh = r % G;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (qi < nq)
            v = *reinterpret_cast<const uint4 *>(
                q + ((int64_t)(t0 + qi) * Hq + g * G + hh) * D + ch * 8);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         qtile + toff<D, 16>(r, ch)),
                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
    }
    const int32_t *pt_row = page_table + (int64_t)req * max_pages;
    const int p_r0 = (rg / G) < nq ? pos[t0 + rg / G] : -1;
    const int p_r1 = ((rg + 8) / G) < nq ? pos[t0 + (rg + 8) / G] : -1;
    const int C = (vmax + CHUNK - 1) / CHUNK;

    float M[2] = {0.f, 0.f}, Ls[2] = {0.f, 0.f}, O[DPW / 8][4];
    for (int c = 0; c < C; ++c) {
        __syncthreads();  // previous chunk fully consumed
        load_tile<D>(ktile, kp, pt_row, max_pages, n_pages, Hkv, g, c, vmax,
                     status, NT);
        cp_async_commit();
        load_tile<D>(vtile, vp, pt_row, max_pages, n_pages, Hkv, g, c, vmax,
                     status, NT);
        cp_async_commit();
        const int len0 = max(0, min(CHUNK, p_r0 + 1 - c * CHUNK));
        const int len1 = max(0, min(CHUNK, p_r1 + 1 - c * CHUNK));
        cp_async_wait<1>();
        __syncthreads();
        float m[2], l[2], o[DPW / 8][4];
        chunk_phase1<D, 0>(ktile, qtile, ptile, red, scale, len0, len1, m,
                           false);
        cp_async_wait<0>();
        __syncthreads();
        chunk_phase2<D>(vtile, ptile, red, l, o, false, true);
        const int pr[2] = {p_r0, p_r1};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (pr[half] + 1 - c * CHUNK <= 0) continue;  // chunk not visible
            if (c == 0) {
                M[half] = m[half];
                Ls[half] = l[half];
#pragma unroll
                for (int nt = 0; nt < DPW / 8; ++nt) {
                    O[nt][2 * half] = o[nt][2 * half];
                    O[nt][2 * half + 1] = o[nt][2 * half + 1];
                }
            } else {
                float a, bb;
                merge_scalars(M[half], Ls[half], m[half], l[half], a, bb);
#pragma unroll
                for (int nt = 0; nt < DPW / 8; ++nt) {
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
        for (int nt = 0; nt < DPW / 8; ++nt) {
            const int dim = warp * DPW + 8 * nt + 2 * tq;
            *reinterpret_cast<uint32_t *>(dst + dim) =
                pack_bf16x2(__fdiv_rn(O[nt][2 * half], Ls[half]),
                            __fdiv_rn(O[nt][2 * half + 1], Ls[half]));
        }
    }
}

// ------------------------------------------- tensor-core chunk (head_dim 128) --
//
// For head_dim 128 the chunk partial runs on the tcgen05 tensor cores; decode
// and prefill both use the functions below, so their bits agree.  Per
// 16-row query tile and 256-key chunk:
//   S^T[key][row] = sum_d K[key][d] Q[row][d]: two MMA chains (keys 0-127
//     and 128-255; M = 128 keys, N = 16 rows), each over the dims in
//     ascending 16-steps, fp32 in tensor memory;
//   s = S^T * scale, -inf past the row's visible length; m = block maximum;
//   p = p_of(raw score, rn(scale log2 e), rn(m log2 e)) = 2^(s log2 e -
//   m log2 e) (0 when masked); l = per-warp xor-tree sums over 32 keys
//   (16, 8, 4, 2, 1), then (((w0 + w1) + w2) .. + w7) over the 8 warps;
//   O^T[dim][row] = sum_key V[key][dim] bf16(p)[row][key]: one MMA chain
//   (M = 128 dims, N = 16 rows) over the keys in ascending 16-steps, with V
//   read in place as an MN-major operand.
// V rows past a chunk's visible part are zero when the PV MMAs read them
// (0 * NaN would poison the sum); K rows there are never used (masked).
namespace tca {

// p = e^(s scale - mu) for a raw score s (QK product) of a chunk whose
// scaled maximum is mu, by the change of base e^x = 2^(x log2 e):
// 2^(s c1 - mu2) with c1 = rn(scale log2 e) and mu2 = rn(mu log2 e), the
// argument from one fma, then exp2_approx.  The
// argument's error is a few fp32 ulp of |s scale|, far below the bf16
// rounding P gets next.  Every head_dim-128 path (decode, prefill, verify)
// takes p from this one function, so they agree bit for bit; it is two
// instructions per score.
__device__ __forceinline__ float p_of(float s, float c1, float mu2) {
    return exp2_approx(__fmaf_rn(s, c1, -mu2));
}

constexpr int SW = 8;                         // softmax warps, thread = key
constexpr int STHREADS = SW * 32;
constexpr uint32_t IDESC_QK = make_idesc_bf16(128, 16);
constexpr uint32_t IDESC_PV = make_idesc_bf16(128, 16) | (1u << 15);
constexpr int P_TILE = 16 * CHUNK * 2;        // bf16 [16][256], 8 KB
constexpr int RED_FLOATS = 2 * SW * 16;       // maxima then sums, [8][16] each

// P tile, the B operand of the PV MMAs (K-major, 128-byte swizzle): keys in
// groups of 64 (2 KB each), row r at r * 128 B, 16-byte unit j at j ^ (r % 8).
__device__ __forceinline__ uint32_t poff(int row, int key) {
    return (uint32_t)((key >> 6) * 2048 + row * 128 +
                      ((((key & 63) >> 3) ^ (row & 7)) << 4) + (key & 7) * 2);
}

// S^T into TMEM columns d .. d + 31 (keys 0-127 in d .. d + 15, keys
// 128-255 in d + 16 .. d + 31; lane = key % 128).  K tile: the 2-half
// [256][128 B] layout the TMA writes; Q tile: 2 halves of [16][128 B].
__device__ __forceinline__ void issue_qk(uint32_t d, uint32_t ktile,
                                         uint32_t qtile) {
    // the two chains' steps alternate, so each step's MMA has the other
    // chain's to overlap with (each chain's own k order is unchanged)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t a = ktile + (kk >> 2) * (CHUNK * 128) +
                               h * (128 * 128) + (kk & 3) * 32;
            const uint32_t b = qtile + (kk >> 2) * (16 * 128) + (kk & 3) * 32;
            tc_mma_bf16(d + h * 16, make_sw128_desc(a), make_sw128_desc(b),
                        IDESC_QK, kk > 0 ? 1u : 0u);
        }
}

// O^T into TMEM columns d .. d + 15 (lane = dim).  The V tile's two 64-dim
// halves are the MN atoms (32 KB apart), 8-key row groups the K atoms.
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t vtile,
                                         uint32_t ptile) {
#pragma unroll
    for (int kk = 0; kk < CHUNK / 16; ++kk) {
        const uint32_t a = vtile + kk * 2048;
        const uint32_t b = ptile + (kk >> 2) * 2048 + (kk & 3) * 32;
        tc_mma_bf16(d, make_sw128_desc_mn(a, CHUNK * 128, 1024),
                    make_sw128_desc(b), IDESC_PV, kk > 0 ? 1u : 0u);
    }
}

__device__ __forceinline__ void sync_softmax() {
    asm volatile("bar.sync 1, %0;" ::"n"(STHREADS) : "memory");
}

// Softmax of one chunk by the 256 softmax threads (thread t <-> key t), for
// rows 0 .. NR-1 of the tile: reads S^T at s_tmem, applies scale and the
// per-row visible lengths, writes m[r] (every thread), the warp sums to
// red + 128 and bf16(p) to the P tile.  Rows >= NR are not touched.  The
// reductions of the NR rows run stage by stage across the rows (independent
// shuffle chains side by side); each row's own operations and their order
// do not depend on NR.
template <int NR, int NA>
__device__ __forceinline__ void softmax(uint32_t s_tmem, float scale,
                                        const int (&len)[NA], uint32_t ptile,
                                        float *red, float (&m)[NA]) {
    static_assert(NR <= NA, "rows");
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int key = (w >> 2) * 128 + (w & 3) * 32 + lane;
    const float c1 = __fmul_rn(scale, LOG2E);
    float v[16], x[NR];   // v: raw scores
    tmem_ld_16cols(s_tmem + ((uint32_t)((w & 3) * 32) << 16) + (w >> 2) * 16,
                   v);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float s = __fmul_rn(v[r], scale);
        x[r] = key < len[r] ? s : -INFINITY;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int r = 0; r < NR; ++r)
            x[r] = fmaxf(x[r], __shfl_xor_sync(0xffffffffu, x[r], o));
    if (lane == 0)
#pragma unroll
        for (int r = 0; r < NR; ++r) red[w * 16 + r] = x[r];
    sync_softmax();
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        float mm = red[r];
#pragma unroll
        for (int k = 1; k < SW; ++k) mm = fmaxf(mm, red[k * 16 + r]);
        m[r] = mm;
        const float mu = mm == -INFINITY ? 0.f : mm;
        const float p =
            key < len[r] ? p_of(v[r], c1, __fmul_rn(mu, LOG2E)) : 0.f;
        v[r] = p;
        x[r] = p;
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(ptile + poff(r, key)),
                     "h"(f32_to_bf16(p))
                     : "memory");
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int r = 0; r < NR; ++r)
            x[r] = __fadd_rn(x[r], __shfl_xor_sync(0xffffffffu, x[r], o));
    if (lane == 0)
#pragma unroll
        for (int r = 0; r < NR; ++r) red[SW * 16 + w * 16 + r] = x[r];
}

// Block row sum of row r from the warp sums (fixed warp order).
__device__ __forceinline__ float row_sum(const float *red, int r) {
    float l = red[SW * 16 + r];
#pragma unroll
    for (int x = 1; x < SW; ++x) l = __fadd_rn(l, red[SW * 16 + x * 16 + r]);
    return l;
}

// Rows [from, to) of both 64-dim halves of a V tile set to zero.
__device__ __forceinline__ void zero_v_rows(uint8_t *vtile, int from, int to,
                                            int tid, int nthreads) {
    for (int idx = tid; idx < (to - from) * 16; idx += nthreads) {
        const int row = from + (idx >> 4), u = idx & 15;
        *reinterpret_cast<uint4 *>(vtile + (u >> 3) * (CHUNK * 128) +
                                   row * 128 + (u & 7) * 16) =
            make_uint4(0, 0, 0, 0);
    }
}

// Decode kernel shared-memory layout (offsets from a 1024-aligned base).
struct DecL {
    static constexpr int TB = CHUNK * 128 * 2;          // K or V tile, 64 KB
    static constexpr int QB = 16 * 128 * 2;             // Q tile, 4 KB
    static constexpr int SLOT = 0;
    static constexpr int QSLOT = SLOT + RING * TB;
    static constexpr int P = QSLOT + RING * QB;          // 2 P tiles
    static constexpr int RED = P + 2 * P_TILE;           // 2 x [2][8][16] f32
    static constexpr int BAR = RED + 2 * RED_FLOATS * 4;
    // full[RING], empty[RING], s_full[2], p_full[2], p_empty[2], o_full[2],
    // o_empty[2], then the TMEM address
    static constexpr int BYTES = BAR + (2 * RING + 10) * 8 + 16;
    static constexpr int ALLOC = BYTES + 1024;
};
constexpr int DEC_THREADS = (SW + 4) * 32;  // softmax, MMA, K, prefetch, V
// the whole-row decode kernel: two K and two V producer warps
constexpr int DEC_ROW_THREADS = (SW + 6) * 32;

// Position of the K and V loads of item n in the ring's load sequence.
__device__ __forceinline__ int k_load(int n) { return 2 * n; }
__device__ __forceinline__ int v_load(int n) { return 2 * n + 1; }

}  // namespace tca

// Exclusive prefix of v over the block (blockDim.x a multiple of 32, at most
// 1024); *total gets the sum.  Uses wsum[32]; all threads must call it.
__device__ __forceinline__ int block_excl_scan_int(int v, int *wsum,
                                                   int *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int inc = v;
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
    const int before = (w > 0 ? wsum[w - 1] : 0) + inc - v;
    *total = wsum[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

// Work list of the tensor-core prefill path: the segments' query tiles of
// QPT = 16 / G tokens as (first token, context L = last token's position +
// 1, tokens, page-table row).  A tile is valid when its request is >= 0,
// L <= max_kv_len and its positions are consecutive (as the segments of a
// prefill or a verify are); valid tiles come first, sorted by chunk count
// (most first, ties by tile index), the others after them with L = 0 (a
// tile with a request but out of range also records BI_ERR_BOUNDS).
// cnt = {valid tiles, all tiles}; tmp holds the unsorted list.  One block,
// R <= MAX_SEGS (checked by the caller).
constexpr int MAX_SEGS = 4096;
__global__ void build_tiles_kernel(const int32_t *__restrict__ cu_q,
                                   const int32_t *__restrict__ seg_req,
                                   const int32_t *__restrict__ pos, int R,
                                   int QPT, int max_kv_len,
                                   int4 *__restrict__ tmp,
                                   int4 *__restrict__ tiles,
                                   int32_t *__restrict__ cnt,
                                   int32_t *status, int T = 0,
                                   int2 *__restrict__ sitems = nullptr,
                                   int32_t *__restrict__ kvl_tok = nullptr,
                                   int32_t *__restrict__ req_tok = nullptr) {
    constexpr int TILE = 2048;
    __shared__ int soff[MAX_SEGS + 1];  // first tile of each segment
    __shared__ int skey[TILE];
    __shared__ int wsum[32];
    __shared__ int nvalid;
    const int tid = threadIdx.x;
    int carry = 0;
    for (int r0 = 0; r0 < R; r0 += blockDim.x) {
        const int r = r0 + tid;
        const int n = r < R ? cu_q[r + 1] - cu_q[r] : 0;
        int tot;
        const int before = block_excl_scan_int((n + QPT - 1) / QPT, wsum, &tot);
        if (r < R) soff[r] = carry + before;
        carry += tot;
    }
    if (tid == 0) {
        soff[R] = carry;
        nvalid = 0;
    }
    __syncthreads();
    const int ntiles = carry;
    for (int j = tid; j < ntiles; j += blockDim.x) {
        int lo = 0, hi = R - 1;  // the last segment starting at or before j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (soff[mid] <= j)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int k = j - soff[lo];
        const int s0 = cu_q[lo], n = cu_q[lo + 1] - s0;
        const int t0 = s0 + k * QPT, nt = min(QPT, n - k * QPT);
        const int p0 = pos[t0];
        bool consec = true;
        for (int i = 1; i < nt; ++i) consec &= pos[t0 + i] == p0 + i;
        const int req = seg_req[lo];
        const int L = p0 + nt;
        const bool valid = req >= 0 && consec && L >= 1 && L <= max_kv_len;
        if (req >= 0 && !valid) bi_record_error(status, BI_ERR_BOUNDS);
        tmp[j] = make_int4(t0, valid ? L : 0, nt, req);
    }
    __syncthreads();
    for (int j0 = 0; j0 < ntiles; j0 += blockDim.x) {
        const int j = j0 + tid;
        const int Lj = j < ntiles ? tmp[j].y : 0;
        const int kj = j < ntiles ? (Lj + CHUNK - 1) / CHUNK : -1;
        int rank = 0;
        for (int t0 = 0; t0 < ntiles; t0 += TILE) {
            const int n = min(TILE, ntiles - t0);
            __syncthreads();
            for (int i = tid; i < n; i += blockDim.x)
                skey[i] = (tmp[t0 + i].y + CHUNK - 1) / CHUNK;
            __syncthreads();
            if (j < ntiles)
                for (int i = 0; i < n; ++i) {
                    const int kk = skey[i];
                    rank += kk > kj || (kk == kj && t0 + i < j);
                }
        }
        if (j < ntiles) {
            tiles[rank] = tmp[j];
            if (kj > 0) atomicAdd(&nvalid, 1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        cnt[0] = nvalid;
        cnt[1] = ntiles;
    }
    if (sitems) {
        // split form: one item per (valid entry, chunk), the entries in list
        // order, cnt[2] items; every token's context and request (no
        // request for tokens of invalid entries or of no entry)
        const int nv = nvalid;
        int carry2 = 0;
        for (int j0 = 0; j0 < nv; j0 += blockDim.x) {
            const int j = j0 + tid;
            const int Cj = j < nv ? (tiles[j].y + CHUNK - 1) / CHUNK : 0;
            int tot;
            __syncthreads();
            const int before = block_excl_scan_int(Cj, wsum, &tot);
            for (int c = 0; c < Cj; ++c)
                sitems[carry2 + before + c] = make_int2(j, c);
            carry2 += tot;
        }
        for (int t = tid; t < T; t += blockDim.x) {
            kvl_tok[t] = 0;
            req_tok[t] = -1;
        }
        __syncthreads();
        for (int j = tid; j < ntiles; j += blockDim.x) {
            const int4 e = tiles[j];
            const bool valid = j < nv;
            for (int i = 0; i < e.z; ++i) {
                kvl_tok[e.x + i] = valid ? e.y - e.z + i + 1 : 0;
                req_tok[e.x + i] = valid ? e.w : -1;
            }
        }
        if (tid == 0) cnt[2] = carry2;
    }
}

// Work list of the tensor-core decode kernel: the valid rows (row_req >= 0,
// 0 < kv_len <= Cmax * 256) as (row, kv_len), most chunks first (ties by
// row), then the other rows as (row, 0); prefix[B] = number of valid rows.
// One block; every thread ranks its rows against all rows (keys compared in
// shared-memory tiles), an exact and order-free computation.
__global__ void build_rows_kernel(const int32_t *__restrict__ kv_len,
                                  const int32_t *__restrict__ row_req, int B,
                                  int Cmax, int32_t *__restrict__ prefix,
                                  int2 *__restrict__ rows) {
    constexpr int TILE = 2048;
    __shared__ int skey[TILE];
    __shared__ int nvalid;
    const int tid = threadIdx.x;
    auto key_of = [&](int b) {
        const int L = kv_len[b];
        return row_req[b] >= 0 && L > 0 && L <= Cmax * CHUNK
                   ? (L + CHUNK - 1) / CHUNK
                   : 0;
    };
    if (tid == 0) nvalid = 0;
    for (int b0 = 0; b0 < B; b0 += blockDim.x) {
        const int b = b0 + tid;
        const int kb = b < B ? key_of(b) : -1;
        int rank = 0;
        for (int t0 = 0; t0 < B; t0 += TILE) {
            const int n = min(TILE, B - t0);
            __syncthreads();
            for (int i = tid; i < n; i += blockDim.x) skey[i] = key_of(t0 + i);
            __syncthreads();
            if (b < B)
                for (int i = 0; i < n; ++i) {
                    const int k = skey[i];
                    rank += k > kb || (k == kb && t0 + i < b);
                }
        }
        if (b < B) {
            rows[rank] = make_int2(b, kb > 0 ? kv_len[b] : 0);
            if (kb > 0) atomicAdd(&nvalid, 1);
        }
    }
    __syncthreads();
    if (tid == 0) prefix[B] = nvalid;
}

namespace tca {

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Item n (0, 1, ...) of CTA k out of `grid`: the item list is walked in
// rounds of `grid` items, the CTA order reversed every other round, so the
// long rows at the front spread evenly over the CTAs.
__device__ __forceinline__ int item_of(int n, int k, int grid) {
    return n * grid + ((n & 1) ? grid - 1 - k : k);
}

// The units (chunks) of this CTA in order: item r of the CTA is KV head
// j % Hkv of sorted entry j / Hkv (j = item_of(r)); its units are chunks
// 0 .. C - 1, C = ceil(L / 256).  Decode entries are (row, kv_len); prefill
// entries (first token, tile's context = last token's position + 1, tokens,
// page-table row).  Every role walks the same sequence; the next item's
// entry is loaded one item ahead.
template <bool PRE>
struct UnitWalk {
    using E = typename std::conditional<PRE, int4, int2>::type;
    const E *rows;
    int total, Hkv;
    int r, c, C, b, L, g, ntok, req;  // current unit
    int nb, nL, ng, nntok, nreq;      // next item
    bool nok;

    __device__ bool load(int rr, int &b_, int &L_, int &g_, int &nt_,
                         int &rq_) const {
        const int j = item_of(rr, blockIdx.x, gridDim.x);
        if (j >= total) return false;
        const E e = rows[j / Hkv];
        b_ = e.x;
        L_ = e.y;
        g_ = j % Hkv;
        if constexpr (PRE) {
            nt_ = e.z;
            rq_ = e.w;
        } else {
            nt_ = 1;
            rq_ = -1;
        }
        return true;
    }
    __device__ bool begin() {
        r = c = 0;
        if (!load(0, b, L, g, ntok, req)) return false;
        C = (L + CHUNK - 1) / CHUNK;
        nok = load(1, nb, nL, ng, nntok, nreq);
        return true;
    }
    __device__ bool next() {
        if (++c < C) return true;
        if (!nok) return false;
        ++r;
        c = 0;
        b = nb;
        L = nL;
        g = ng;
        ntok = nntok;
        req = nreq;
        C = (L + CHUNK - 1) / CHUNK;
        nok = load(r + 1, nb, nL, ng, nntok, nreq);
        return true;
    }
    __device__ int vl() const { return min(CHUNK, L - c * CHUNK); }
};

}  // namespace tca

// Persistent decode kernel on the tensor cores (head_dim 128).  CTA k takes
// whole (row, KV head) items (UnitWalk) and streams their 256-position
// chunks through the pipeline in order; the chunk partials are merged in
// registers in chunk order with the merge functions of the two-stage path,
// as the prefill kernel does, and the last chunk of an item writes the
// item's G output rows.  The ring loads K0 V0 K1 V1 ... over the units,
// load j in slot j mod RING (k_load / v_load).
//   warps 0-7   softmax (thread t <-> key t of the chunk); warps 0-3 also
//               keep the running (m, l, o) of the item's rows for their dim
//               and write the output;
//   warp 8      owns the tensor memory; lane 0 issues the MMAs: S^T of unit
//               n + 2 is issued as soon as unit n's softmax has read S^T
//               (two S buffers), O^T of unit n once its P tile is written
//               (two P tiles, two O buffers);
//   warp 9      producer: page ids -> TMA boxes (K and V of the visible pages;
//               the V rows past them are zeroed by the softmax warps);
//   warp 10     asks L2 for the K/V pages of the unit after the one the
//               producer loads next (one ahead: 1% faster than two, 9%
//               faster than four or none).
// Rows outside the work list (no request, or a context out of range) get
// zero outputs.
//
// PRE: the same kernel over prefill / verify tiles (16 / G consecutive
// tokens of one segment, whose positions are consecutive) as items: the
// query tile is the tokens x G heads (a 3-D TMA box), each row masked at
// its own position, all 16 rows merged and written.  The chunk partials and
// their merge are the same computation as decode's, so a (request,
// position) gets the same bits either way.
template <bool PRE, int NR>
__global__ void __launch_bounds__(tca::DEC_ROW_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap,
                   const int32_t *__restrict__ page_table, int max_pages,
                   int n_pages, const int32_t *__restrict__ row_req, int Hq,
                   int Hkv, int G, float scale,
                   const int32_t *__restrict__ cnt, int B,
                   const void *__restrict__ list,
                   const bi_bf16 *__restrict__ k_pool,
                   const bi_bf16 *__restrict__ v_pool,
                   uint16_t *__restrict__ out, int32_t *status) {
    using namespace tca;
    using Walk = UnitWalk<PRE>;
    using E = typename Walk::E;
    const E *rows = static_cast<const E *>(list);
    constexpr int D = 128;
    constexpr int PAGE_BYTES = 16 * 64 * 2;   // one box: 16 rows x 64 dims
    constexpr int HALF_TILE = CHUNK * 128;
    constexpr int HALF_Q = 16 * 128;
    extern __shared__ uint8_t smem_raw[];
    // units whose K (s_progress, s_kprog2) / V (s_vprog[2]) each of the
    // producer warps has issued
    __shared__ int s_progress, s_kprog2;
    __shared__ int s_vprog[2];
    __shared__ int s_units;     // units of this CTA
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + DecL::BAR);
    uint64_t *empty = full + RING;
    uint64_t *s_full = empty + RING;
    uint64_t *p_full = s_full + 2;
    uint64_t *p_empty = p_full + 2;
    uint64_t *o_full = p_empty + 2;
    uint64_t *o_empty = o_full + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(o_empty + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_valid = cnt[0];
    const int n_all = PRE ? cnt[1] : B;  // entries, the invalid ones last
    const int total = n_valid * Hkv;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RING; ++i) {
            mbar_init(&full[i], 2);  // the two producer warps of the load
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], SW);
            mbar_init(&p_empty[i], 1);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 4);
        }
        mbar_fence_init();
        s_progress = 0;
        s_kprog2 = 0;
        s_vprog[0] = s_vprog[1] = 0;
    }
    if (warp < SW) {
        // both P tiles start at zero: rows >= G are never written again
        for (int i = threadIdx.x; i < 2 * P_TILE / 16; i += STHREADS)
            reinterpret_cast<uint4 *>(smem + DecL::P)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == SW + 2) {
        // units of this CTA: the chunk counts of its items, one round per
        // lane (round r's item index is at least r * grid)
        int sum = 0;
        for (int r0 = 0; r0 * (int)gridDim.x < total; r0 += 32) {
            const int j = item_of(r0 + lane, blockIdx.x, gridDim.x);
            const int C = j < total ? (rows[j / Hkv].y + CHUNK - 1) / CHUNK : 0;
            sum += warp_sum_int(C);
        }
        if (lane == 0) s_units = sum;
    }
    if (warp == SW) tmem_alloc(tslot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    volatile int *progress = &s_progress;
    const int n_units = s_units;

    // Warp SW + 2 counted the CTA's units above and has no further role:
    // the K and V pages are streamed with the L2 evict-first policy and not
    // prefetched (an L2 prefetch of the next unit's pages made the
    // evict-first reads slower, and without the policy it gained nothing).
    if (warp == SW + 2) return;

    if (warp == SW + 1 || warp >= SW + 3) {
        // ----------------------------------------------------- producers --
        // Warps SW + 1 and SW + 3 issue K (+ Q), warps SW + 4 and SW + 5
        // issue V, each for half of a unit's 16 pages (lanes 0-7: pages
        // 8 hf + lane): a TMA box costs its issuing warp about 70 cycles,
        // so a tile's boxes go out from two warps at once.  Load t = 2n + kv
        // goes to slot t % RING after the consumer of load t - RING has
        // released it; t - RING is always the other pair's, so before load t
        // a warp also waits until both warps of the other pair have issued
        // t - RING (their progress counters): every slot's loads are then
        // issued in order and each empty-barrier wait names an unambiguous
        // phase.  full[] takes one arrival (with its bytes) from each warp
        // of the pair.
        const int kv = warp == SW + 1 || warp == SW + 3 ? 0 : 1;
        const int hf = warp == SW + 1 || warp == SW + 4 ? 0 : 1;
        // each page is read once per forward: evict it from L2 first, so
        // that the next kernels' inputs stay
        const uint64_t pol = l2_evict_first_policy();
        volatile int *kp[2] = {progress, (volatile int *)&s_kprog2};
        volatile int *vp[2] = {(volatile int *)&s_vprog[0],
                               (volatile int *)&s_vprog[1]};
        volatile int *mine = kv == 0 ? kp[hf] : vp[hf];
        volatile int *const *other = kv == 0 ? vp : kp;
        if (lane == 0 && hf == 0) {
            if (kv == 0) {
                tma_prefetch_desc(&kmap);
                tma_prefetch_desc(&qmap);
            } else {
                tma_prefetch_desc(&vmap);
            }
        }
        bool ok = true;
        Walk w{rows, total, Hkv};
        if (w.begin()) {
            // page-table rows of the current and the next item
            int req = PRE ? w.req : row_req[w.b];
            int nreq = PRE ? 0 : (w.nok ? row_req[w.nb] : 0);
            for (int n = 0; ok; ++n) {
                const int b = w.b, c = w.c, g = w.g;
                const int npg = (w.vl() + 15) >> 4;
                const int32_t *pt_row = page_table + (int64_t)req * max_pages;
                const int pl = 8 * hf + lane;   // this lane's page of the chunk
                int pg = -1;
                if (lane < 8 && pl < npg) {
                    const int pi = c * 16 + pl;
                    pg = pi < max_pages ? pt_row[pi] : -1;
                    if (pg < 0 || pg >= n_pages) {
                        bi_record_error(status, BI_ERR_BOUNDS);
                        pg = -1;
                    }
                }
                const int nvalid = __popc(__ballot_sync(0xffffffffu, pg >= 0));
                // K (+ Q) and V: the visible pages only; the V rows past
                // them are zeroed in shared memory by the softmax warps
                // (a TMA box each would cost the producer as much as a
                // page of data).
                {
                    const int t = 2 * n + kv;
                    const int slot = t % RING;
                    const int use = t / RING;
                    bool w_ok = true;
                    if (lane == 0 && use > 0) {
                        // load t - RING = 2 m + (1 - kv) issued by both
                        // warps of the other pair: their counts passed m
                        const int need = (t - RING - (1 - kv)) / 2 + 1;
                        if (*other[0] < need || *other[1] < need) {
                            const uint64_t t0 = bi_globaltimer();
                            while (*other[0] < need || *other[1] < need) {
                                __nanosleep(64);
                                if (bi_globaltimer() - t0 > BI_WAIT_LIMIT_NS) {
                                    bi_record_error(status, BI_ERR_TIMEOUT);
                                    w_ok = false;
                                    break;
                                }
                            }
                        }
                        if (w_ok)
                            w_ok = mbar_wait(&empty[slot], (use - 1) & 1,
                                             status);
                    }
                    ok = __shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (lane == 0)
                        mbar_arrive_expect_tx(
                            &full[slot],
                            nvalid * 2 * PAGE_BYTES +
                                (kv == 0 && hf == 0 ? 2 * HALF_Q : 0));
                    __syncwarp();
                    uint8_t *tile = smem + DecL::SLOT + slot * DecL::TB;
                    if (pg >= 0) {
                        const int row = (pg * Hkv + g) * 16;
                        const CUtensorMap *map = kv == 0 ? &kmap : &vmap;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d_hint(tile + h * HALF_TILE +
                                                 pl * PAGE_BYTES,
                                             map, h * 64, row, &full[slot],
                                             pol);
                    }
                    if (kv == 0 && hf == 0 && lane == 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint8_t *qdst = smem + DecL::QSLOT +
                                            slot * DecL::QB + h * HALF_Q;
                            if constexpr (PRE)  // tokens b .. x heads g G ..
                                tma_load_3d(qdst, &qmap, h * 64, g * G, b,
                                            &full[slot]);
                            else
                                tma_load_2d(qdst, &qmap, h * 64, b * Hq + g * G,
                                            &full[slot]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence_block();
                        *mine = n + 1;
                    }
                }
                if (!ok || !w.next()) break;
                if (w.c == 0) {
                    if constexpr (PRE) {
                        req = w.req;
                    } else {
                        req = nreq;
                        nreq = w.nok ? row_req[w.nb] : 0;
                    }
                }
            }
        }
        // every load issued: release the other pair.
        // After a failed wait the count stays where it is, so the other
        // pair's wait for it runs out too and nothing is issued into a slot
        // out of order.
        if (lane == 0 && ok) *mine = 0x3fffffff;
        return;
    }

    if (warp == SW) {
        // ----------------------------------------------------------- MMA --
        // Event loop: the S^T MMAs of unit nq (once its K tile has landed
        // and S^T buffer nq % 2 is free, i.e. the PV MMAs of unit nq - 2 are
        // issued) and the PV MMAs of unit np (once its P tile is written and
        // O^T buffer np % 2 has been read), whichever is ready first, each
        // in unit order.  Gives up after a stall of the wait limit.
        if (lane == 0) {
            int nq = 0, np = 0;
            uint64_t t0 = bi_globaltimer();
            while (np < n_units) {
                bool did = false;
                if (nq < n_units && nq < np + 2) {
                    const int jk = k_load(nq), sk = jk % RING;
                    if (mbar_try_wait(&full[sk], (jk / RING) & 1)) {
                        tc_fence_after();
                        issue_qk(tmem + (nq & 1) * 32,
                                 base + DecL::SLOT + sk * DecL::TB,
                                 base + DecL::QSLOT + sk * DecL::QB);
                        tc_commit(&s_full[nq & 1]);
                        tc_commit(&empty[sk]);
                        ++nq;
                        did = true;
                    }
                }
                if (np < nq) {
                    const int bf = np & 1;
                    if (mbar_try_wait(&p_full[bf], (np >> 1) & 1) &&
                        (np < 2 ||
                         mbar_try_wait(&o_empty[bf], ((np - 2) >> 1) & 1))) {
                        const int sv = v_load(np) % RING;
                        tc_fence_after();
                        issue_pv(tmem + 64 + bf * 16,
                                 base + DecL::SLOT + sv * DecL::TB,
                                 base + DecL::P + bf * P_TILE);
                        tc_commit(&o_full[bf]);
                        tc_commit(&p_empty[bf]);
                        tc_commit(&empty[sv]);
                        ++np;
                        did = true;
                    }
                }
                if (did) {
                    t0 = bi_globaltimer();
                } else if (bi_globaltimer() - t0 > BI_WAIT_LIMIT_NS) {
                    bi_record_error(status, BI_ERR_TIMEOUT);
                    break;
                }
            }
            // the last epilogues have read O^T before the memory is freed
            for (int n = max(0, np - 2); n < np; ++n)
                mbar_wait(&o_empty[n & 1], (n >> 1) & 1, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 128);
        return;
    }

    // ------------------------------------------------ softmax + epilogue --
    const int tid = threadIdx.x;  // 0 .. 255
    // entries outside the work list: zero outputs for their tokens
    for (int i = blockIdx.x; i < n_all - n_valid; i += gridDim.x) {
        const E e = rows[n_valid + i];
        int nt = 1;
        if constexpr (PRE) nt = e.z;
        uint4 *dst = reinterpret_cast<uint4 *>(out + (int64_t)e.x * Hq * D);
        for (int k = tid; k < nt * Hq * D / 8; k += STHREADS)
            dst[k] = make_uint4(0, 0, 0, 0);
    }
    float m[NR], m_prev[NR];
    // running (max, sum, output) of the item's rows for this thread's dim
    // (warps 0-3), merged chunk by chunk in order
    float Mr[NR], Lr[NR], Or[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) m_prev[r] = Mr[r] = Lr[r] = Or[r] = 0.f;
    // previous unit: row (first token), chunk, head, chunks, tokens, and
    // the position of its first token relative to the chunk (PRE)
    int pb = 0, pc = 0, pg_ = 0, pC = 1, pnt = 1, pp0 = 0;
    // epilogue of unit e (buffer e & 1): merge its partial into the running
    // state; the item's last chunk writes the outputs
    auto epilogue = [&](int e) -> bool {
        const int bf = e & 1;
        const float *red = reinterpret_cast<const float *>(
            smem + DecL::RED + bf * RED_FLOATS * 4);
        if (warp < 4) {
            if (!mbar_wait(&o_full[bf], (e >> 1) & 1, status)) return false;
            tc_fence_after();
            float o[16];
            tmem_ld_16cols(tmem + 64 + bf * 16 + ((uint32_t)(warp * 32) << 16),
                           o);
            const int dim = warp * 32 + lane;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (!PRE && r >= G) break;
                const int qi = PRE ? r / G : 0;  // token of row r
                if (qi >= pnt) continue;
                // the chunk is visible to the row (always, for decode)
                if (!PRE || pp0 + qi + 1 > 0) {
                    const float l = row_sum(red, r);
                    if (pc == 0) {
                        Mr[r] = m_prev[r];
                        Lr[r] = l;
                        Or[r] = o[r];
                    } else {
                        float a, bb;
                        merge_scalars(Mr[r], Lr[r], m_prev[r], l, a, bb);
                        Or[r] = merge_value(Or[r], o[r], a, bb);
                    }
                }
                if (pc == pC - 1)
                    out[((int64_t)(pb + qi) * Hq + pg_ * G + (r - qi * G)) * D +
                        dim] = f32_to_bf16(__fdiv_rn(Or[r], Lr[r]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[bf]);
        }
        return true;
    };
    bool ok = true;
    int n = 0;
    Walk w{rows, total, Hkv};
    if (w.begin()) {
        do {
            const int vl = w.vl();
            const int bf = n & 1;
            float *red = reinterpret_cast<float *>(smem + DecL::RED +
                                                   bf * RED_FLOATS * 4);
            const uint32_t ptile = base + DecL::P + bf * P_TILE;
            if (!mbar_wait(&s_full[bf], (n >> 1) & 1, status) ||
                (n >= 2 &&
                 !mbar_wait(&p_empty[bf], ((n - 2) >> 1) & 1, status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            int len[NR];
            if constexpr (PRE) {
                // row r: token r / G at position (L - ntok) + r / G
                const int p0 = w.L - w.ntok - w.c * CHUNK;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const int qi = r / G;
                    len[r] = qi < w.ntok ? max(0, min(CHUNK, p0 + qi + 1)) : 0;
                }
            } else {
#pragma unroll
                for (int r = 0; r < NR; ++r) len[r] = r < G ? vl : 0;
            }
            softmax<NR>(tmem + bf * 32, scale, len, ptile, red, m);
            // V rows past the context: the rest of the tile
            const int jv = v_load(n), sv = jv % RING;
            if (!mbar_wait(&full[sv], (jv / RING) & 1, status)) {
                ok = false;
                break;
            }
            if (vl < CHUNK)
                zero_v_rows(smem + DecL::SLOT + sv * DecL::TB, vl, CHUNK, tid,
                            STHREADS);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[bf]);
            if (n > 0) ok = epilogue(n - 1);
#pragma unroll
            for (int r = 0; r < NR; ++r) m_prev[r] = m[r];
            pp0 = w.L - w.ntok - w.c * CHUNK;
            pb = w.b;
            pc = w.c;
            pg_ = w.g;
            pC = w.C;
            pnt = w.ntok;
            ++n;
        } while (ok && w.next());
    }
    if (ok && n > 0) {
        sync_softmax();  // every warp's row sums of the last unit are in
        epilogue(n - 1);
    }
}

// Per-chunk form of the tensor-core decode kernel, for small batches (too
// few (row, KV head) items to fill the SMs): CTA k takes chunk items k,
// k + grid, ...; item i is KV head i % Hkv of list entry i / Hkv (a (row,
// chunk) of build_items_kernel), and writes the chunk's (m, l, o) record;
// decode_merge_kernel merges the records in chunk order with the same
// functions, so the bits equal the whole-row kernel's.  The ring loads K0
// V0 K1 V1 ..., load j in slot j mod RING (k_load / v_load below).
//   warps 0-7   softmax and epilogue (thread t <-> key t of the chunk);
//   warp 8      owns the tensor memory; lane 0 issues the MMAs: S^T of item
//               n + 2 is issued as soon as item n's softmax has read S^T
//               (two S buffers), O^T of item n once its P tile is written
//               (two P tiles, two O buffers);
//   warp 9      producer: page ids -> TMA boxes (K and V of the visible pages;
//               the V rows past them are zeroed by the softmax warps);
//   warp 10     asks L2 for the K/V pages of the item after the one the
//               producer loads next (one item ahead: 1% faster than two,
//               9% faster than four or none).
__global__ void __launch_bounds__(tca::DEC_THREADS, 1)
    decode_tc_chunks_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ CUtensorMap qmap,
                            const int32_t *__restrict__ page_table,
                            int max_pages, int n_pages,
                            const int32_t *__restrict__ row_req,
                            const int32_t *__restrict__ kv_len, int Hq,
                            int Hkv, int G, float scale,
                            float *__restrict__ ws, int Cmax,
                            const int32_t *__restrict__ prefix, int B,
                            const int2 *__restrict__ items,
                            const bi_bf16 *__restrict__ k_pool,
                            const bi_bf16 *__restrict__ v_pool,
                            int32_t *status) {
    using namespace tca;
    constexpr int D = 128;
    constexpr int PAGE_BYTES = 16 * 64 * 2;   // one box: 16 rows x 64 dims
    constexpr int HALF_TILE = CHUNK * 128;
    constexpr int HALF_Q = 16 * 128;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_progress;  // items the producer has issued
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + DecL::BAR);
    uint64_t *empty = full + RING;
    uint64_t *s_full = empty + RING;
    uint64_t *p_full = s_full + 2;
    uint64_t *p_empty = p_full + 2;
    uint64_t *o_full = p_empty + 2;
    uint64_t *o_empty = o_full + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(o_empty + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = prefix[B] * Hkv;
    int n_items = 0;  // items of this CTA
    if ((int)blockIdx.x < total)
        n_items = (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RING; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], SW);
            mbar_init(&p_empty[i], 1);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 4);
        }
        mbar_fence_init();
        s_progress = 0;
    }
    if (warp < SW) {
        // both P tiles start at zero: rows >= G are never written again
        for (int i = threadIdx.x; i < 2 * P_TILE / 16; i += STHREADS)
            reinterpret_cast<uint4 *>(smem + DecL::P)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == SW) tmem_alloc(tslot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (warp > SW + 2) return;  // one producer here
    volatile int *progress = &s_progress;

    if (warp == SW + 2) {
        // ------------------------------------------------------ prefetch --
        constexpr uint32_t PAGE_KV = 16 * D * 2;
        for (int n = 0; n < n_items; ++n) {
            const int i = blockIdx.x + n * gridDim.x;
            bool go = true;
            if (lane == 0 && *progress + 1 < n) {
                const uint64_t t0 = bi_globaltimer();
                while (*progress + 1 < n) {
                    __nanosleep(256);
                    if (bi_globaltimer() - t0 > BI_WAIT_LIMIT_NS) {
                        go = false;
                        break;
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) break;
            const int g = i % Hkv;
            const int2 bc = items[i / Hkv];
            const int vl = min(CHUNK, kv_len[bc.x] - bc.y * CHUNK);
            if (lane < ((vl + 15) >> 4)) {
                const int pi = bc.y * 16 + lane;
                const int pg = pi < max_pages
                                   ? page_table[(int64_t)row_req[bc.x] *
                                                    max_pages + pi]
                                   : -1;
                if (pg >= 0 && pg < n_pages) {
                    const int64_t off = ((int64_t)pg * Hkv + g) * 16 * D;
                    prefetch_l2_bulk(k_pool + off, PAGE_KV);
                    prefetch_l2_bulk(v_pool + off, PAGE_KV);
                }
            }
        }
        return;
    }

    if (warp == SW + 1) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            tma_prefetch_desc(&qmap);
        }
        bool ok = true;
        // load t of the sequence: the K (t even) or V (t odd) of item t / 2
        for (int t = 0; t < 2 * n_items && ok; ++t) {
            const bool is_k = (t & 1) == 0;
            const int n = t >> 1;
            const int i = blockIdx.x + n * gridDim.x;
            const int g = i % Hkv;
            const int2 bc = items[i / Hkv];
            const int b = bc.x, c = bc.y;
            const int vl = min(CHUNK, kv_len[b] - c * CHUNK);
            const int npg = (vl + 15) >> 4;
            const int32_t *pt_row = page_table + (int64_t)row_req[b] * max_pages;
            int pg = -1;
            if (lane < npg) {
                const int pi = c * 16 + lane;
                pg = pi < max_pages ? pt_row[pi] : -1;
                if (pg < 0 || pg >= n_pages) {
                    if (is_k) bi_record_error(status, BI_ERR_BOUNDS);
                    pg = -1;
                }
            }
            const int nvalid = __popc(__ballot_sync(0xffffffffu, pg >= 0));
            const int slot = t % RING;
            const int use = t / RING;
            bool w_ok = true;
            if (lane == 0 && use > 0)
                w_ok = mbar_wait(&empty[slot], (use - 1) & 1, status);
            ok = __shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            // K (+ Q) and V: the visible pages only; the V rows past them
            // are zeroed in shared memory by the softmax warps.
            if (lane == 0)
                mbar_arrive_expect_tx(&full[slot],
                                      nvalid * 2 * PAGE_BYTES +
                                          (is_k ? 2 * HALF_Q : 0));
            __syncwarp();
            uint8_t *tile = smem + DecL::SLOT + slot * DecL::TB;
            if (lane < 16 && pg >= 0) {
                const int row = (pg * Hkv + g) * 16;
                const CUtensorMap *map = is_k ? &kmap : &vmap;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tma_load_2d(tile + h * HALF_TILE + lane * PAGE_BYTES, map,
                                h * 64, row, &full[slot]);
            }
            if (is_k && lane == 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tma_load_2d(smem + DecL::QSLOT + slot * DecL::QB + h * HALF_Q,
                                &qmap, h * 64, b * Hq + g * G, &full[slot]);
                *progress = n + 1;
            }
        }
        if (lane == 0) *progress = 0x3fffffff;  // release the prefetch warp
        return;
    }

    if (warp == SW) {
        // ----------------------------------------------------------- MMA --
        // Event loop: the S^T MMAs of item nq (once its K tile has landed
        // and S^T buffer nq % 2 is free, i.e. the PV MMAs of item nq - 2 are
        // issued) and the PV MMAs of item np (once its P tile is written and
        // O^T buffer np % 2 has been read), whichever is ready first, each
        // in item order.  Gives up after a stall of the wait limit.
        if (lane == 0) {
            int nq = 0, np = 0;
            uint64_t t0 = bi_globaltimer();
            while (np < n_items) {
                bool did = false;
                if (nq < n_items && nq < np + 2) {
                    const int jk = k_load(nq), sk = jk % RING;
                    if (mbar_try_wait(&full[sk], (jk / RING) & 1)) {
                        tc_fence_after();
                        issue_qk(tmem + (nq & 1) * 32,
                                 base + DecL::SLOT + sk * DecL::TB,
                                 base + DecL::QSLOT + sk * DecL::QB);
                        tc_commit(&s_full[nq & 1]);
                        tc_commit(&empty[sk]);
                        ++nq;
                        did = true;
                    }
                }
                if (np < nq) {
                    const int bf = np & 1;
                    if (mbar_try_wait(&p_full[bf], (np >> 1) & 1) &&
                        (np < 2 ||
                         mbar_try_wait(&o_empty[bf], ((np - 2) >> 1) & 1))) {
                        const int sv = v_load(np) % RING;
                        tc_fence_after();
                        issue_pv(tmem + 64 + bf * 16,
                                 base + DecL::SLOT + sv * DecL::TB,
                                 base + DecL::P + bf * P_TILE);
                        tc_commit(&o_full[bf]);
                        tc_commit(&p_empty[bf]);
                        tc_commit(&empty[sv]);
                        ++np;
                        did = true;
                    }
                }
                if (did) {
                    t0 = bi_globaltimer();
                } else if (bi_globaltimer() - t0 > BI_WAIT_LIMIT_NS) {
                    bi_record_error(status, BI_ERR_TIMEOUT);
                    break;
                }
            }
            // the last epilogues have read O^T before the memory is freed
            for (int n = max(0, np - 2); n < np; ++n)
                mbar_wait(&o_empty[n & 1], (n >> 1) & 1, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 128);
        return;
    }

    // ------------------------------------------------ softmax + epilogue --
    const int tid = threadIdx.x;  // 0 .. 255
    float m[16], m_prev[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) m_prev[r] = 0.f;
    int pb = 0, pc = 0, pg_ = 0;  // previous item: row, chunk, KV head
    // (row, chunk, visible length) of the next item, loaded one item ahead
    int nb = 0, nc = 0, nvl = 0;
    if (n_items > 0) {
        const int2 bc = items[blockIdx.x / Hkv];
        nb = bc.x;
        nc = bc.y;
        nvl = min(CHUNK, kv_len[nb] - nc * CHUNK);
    }
    // epilogue of item e (buffer e & 1): records of rows < G
    auto epilogue = [&](int e) -> bool {
        const int bf = e & 1;
        const float *red = reinterpret_cast<const float *>(
            smem + DecL::RED + bf * RED_FLOATS * 4);
        if (warp == 4 && lane < G) {
            float *rec = ws + (((int64_t)pb * Hq + pg_ * G + lane) * Cmax +
                               pc) * rec_floats<D>();
            float mm = m_prev[0];
#pragma unroll
            for (int r = 1; r < 16; ++r)
                if (r == lane) mm = m_prev[r];
            rec[0] = mm;
            rec[1] = row_sum(red, lane);
        }
        if (warp < 4) {
            if (!mbar_wait(&o_full[bf], (e >> 1) & 1, status)) return false;
            tc_fence_after();
            float o[16];
            tmem_ld_16cols(tmem + 64 + bf * 16 + ((uint32_t)(warp * 32) << 16),
                           o);
            const int dim = warp * 32 + lane;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                if (r >= G) break;
                ws[(((int64_t)pb * Hq + pg_ * G + r) * Cmax + pc) *
                       rec_floats<D>() + 4 + dim] = o[r];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[bf]);
        }
        return true;
    };
    bool ok = true;
    for (int n = 0; n < n_items && ok; ++n) {
        const int i = blockIdx.x + n * gridDim.x;
        const int g = i % Hkv;
        const int b = nb, c = nc, vl = nvl;
        if (n + 1 < n_items) {
            const int2 bc = items[(i + gridDim.x) / Hkv];
            nb = bc.x;
            nc = bc.y;
            nvl = min(CHUNK, kv_len[nb] - nc * CHUNK);
        }
        const int bf = n & 1;
        float *red = reinterpret_cast<float *>(smem + DecL::RED +
                                               bf * RED_FLOATS * 4);
        const uint32_t ptile = base + DecL::P + bf * P_TILE;
        if (!mbar_wait(&s_full[bf], (n >> 1) & 1, status) ||
            (n >= 2 && !mbar_wait(&p_empty[bf], ((n - 2) >> 1) & 1, status))) {
            ok = false;
            break;
        }
        tc_fence_after();
        int len[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) len[r] = r < G ? vl : 0;
        if (G <= 4)
            softmax<4>(tmem + bf * 32, scale, len, ptile, red, m);
        else
            softmax<16>(tmem + bf * 32, scale, len, ptile, red, m);
        // V rows past the context: the rest of the tile
        const int jv = v_load(n), sv = jv % RING;
        if (!mbar_wait(&full[sv], (jv / RING) & 1, status)) {
            ok = false;
            break;
        }
        if (vl < CHUNK)
            zero_v_rows(smem + DecL::SLOT + sv * DecL::TB, vl, CHUNK, tid,
                        STHREADS);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[bf]);
        if (n > 0) ok = epilogue(n - 1);
#pragma unroll
        for (int r = 0; r < 16; ++r) m_prev[r] = m[r];
        pb = b;
        pc = c;
        pg_ = g;
    }
    if (ok && n_items > 0) {
        sync_softmax();  // every warp's row sums of the last item are in
        epilogue(n_items - 1);
    }
}

// Prefill / verify on the tensor cores (head_dim 128): CTA = (16-row tile of
// one segment, KV head g); loops over the chunks with the functions above and
// merges the chunk partials in registers in chunk order, as the decode merge
// kernel does, so prefill and decode rows agree bit for bit.  Warp 8 issues
// the TMA page loads (the tile layouts decode uses) and the MMAs: chunk c + 1's
// K is loaded once chunk c's scores are done, its V once chunk c's PV
// products are done, so the loads overlap the softmax and the merge.
namespace tca {
struct PreL {
    static constexpr int TB = CHUNK * 128 * 2;
    static constexpr int K = 0, V = TB, Q = 2 * TB, P = Q + 16 * 128 * 2;
    static constexpr int RED = P + P_TILE;
    // k_full, v_full, s_full, p_full, o_full, then the TMEM address
    static constexpr int BAR = RED + RED_FLOATS * 4;
    static constexpr int BYTES = BAR + 5 * 8 + 16;
    static constexpr int ALLOC = BYTES + 1024;
};
constexpr int PRE_THREADS = STHREADS + 32;
}  // namespace tca

__global__ void __launch_bounds__(tca::PRE_THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const uint16_t *__restrict__ q,
                      const int32_t *__restrict__ cu_q,
                      const int32_t *__restrict__ seg_req, int R,
                      const int32_t *__restrict__ pos,
                      const int32_t *__restrict__ page_table, int max_pages,
                      int n_pages, int Hq, int Hkv, int G, float scale,
                      int max_kv_len, uint16_t *__restrict__ out,
                      int32_t *status) {
    using namespace tca;
    constexpr int D = 128;
    constexpr int NCH = D / 8;
    constexpr int PAGE_BYTES = 16 * 64 * 2;   // one box: 16 rows x 64 dims
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_info[4];  // t0, nq, req, valid_max
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    const uint32_t ktile = base + PreL::K, vtile = base + PreL::V;
    const uint32_t qtile = base + PreL::Q, ptile = base + PreL::P;
    float *red = reinterpret_cast<float *>(smem + PreL::RED);
    uint64_t *k_full = reinterpret_cast<uint64_t *>(smem + PreL::BAR);
    uint64_t *v_full = k_full + 1, *s_full = k_full + 2, *p_full = k_full + 3;
    uint64_t *o_full = k_full + 4;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(k_full + 5);
    const int g = blockIdx.y;
    const int QPT = 16 / G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
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
        mbar_init(k_full, 1);
        mbar_init(v_full, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, SW);
        mbar_init(o_full, 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int t0 = s_info[0], nq = s_info[1], req = s_info[2];
    const int vmax = s_info[3];
    if (t0 < 0) return;
    if (req < 0 || vmax > max_kv_len) {
        if (req >= 0 && threadIdx.x == 0) bi_record_error(status, BI_ERR_BOUNDS);
        for (int idx = threadIdx.x; idx < nq * G * D; idx += PRE_THREADS) {
            const int qi = idx / (G * D), rem = idx % (G * D);
            out[((int64_t)(t0 + qi) * Hq + g * G) * D + rem] = 0;
        }
        return;
    }
    // query tile: row r = (query r / G, head r % G)
    for (int idx = threadIdx.x; idx < 16 * NCH; idx += PRE_THREADS) {
        const int r = idx / NCH, ch = idx % NCH;
        const int qi = r / G, hh = r % G;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (qi < nq)
            v = *reinterpret_cast<const uint4 *>(
                q + ((int64_t)(t0 + qi) * Hq + g * G + hh) * D + ch * 8);
        *reinterpret_cast<uint4 *>(smem + PreL::Q + toff<D, 16>(r, ch)) = v;
    }
    fence_proxy_async_smem();
    if (warp == SW) tmem_alloc(tslot, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int32_t *pt_row = page_table + (int64_t)req * max_pages;
    const int C = (vmax + CHUNK - 1) / CHUNK;

    if (warp == SW) {
        // ------------------------------------------------ loads and MMAs --
        // Pages of chunk c: lane p < 16 loads page 16c + p (a zero-filled box
        // past the tile's last visible position or for a missing page).
        auto load = [&](int c, bool is_k) {
            int pg = -1;
            if (lane < 16) {
                const int pi = c * 16 + lane;
                if (c * CHUNK + lane * 16 < vmax && pi < max_pages) {
                    pg = pt_row[pi];
                    if (pg < 0 || pg >= n_pages) {
                        if (is_k) bi_record_error(status, BI_ERR_BOUNDS);
                        pg = -1;
                    }
                }
            }
            uint64_t *bar = is_k ? k_full : v_full;
            if (lane == 0) mbar_arrive_expect_tx(bar, 16 * 2 * PAGE_BYTES);
            __syncwarp();
            if (lane < 16) {
                const int row = pg >= 0 ? (pg * Hkv + g) * 16 : -16;
                uint8_t *tile = smem + (is_k ? PreL::K : PreL::V);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tma_load_2d(tile + h * (CHUNK * 128) + lane * PAGE_BYTES,
                                is_k ? &kmap : &vmap, h * 64, row, bar);
            }
        };
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        load(0, true);
        load(0, false);
        for (int c = 0; c < C; ++c) {
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(k_full, c & 1, status);
                if (ok) {
                    tc_fence_after();
                    issue_qk(tmem, ktile, qtile);
                    tc_commit(s_full);
                    ok = mbar_wait(s_full, c & 1, status);  // K read
                }
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (c + 1 < C) load(c + 1, true);
            if (lane == 0) {
                ok = mbar_wait(p_full, c & 1, status);  // P written, V zeroed
                if (ok) {
                    tc_fence_after();
                    issue_pv(tmem + 32, vtile, ptile);
                    tc_commit(o_full);
                    ok = mbar_wait(o_full, c & 1, status);  // V, P read
                }
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (c + 1 < C) load(c + 1, false);
        }
    } else {
        // -------------------------------------------- softmax and merge --
        int prow[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            prow[r] = (r / G) < nq ? pos[t0 + r / G] : -1;
        float M[16], L[16], O[16], m[16];
        for (int c = 0; c < C; ++c) {
            int len[16];
#pragma unroll
            for (int r = 0; r < 16; ++r)
                len[r] = max(0, min(CHUNK, prow[r] + 1 - c * CHUNK));
            // the previous chunk's PV products are done with P
            if (c > 0 && !mbar_wait(o_full, (c - 1) & 1, status)) break;
            if (!mbar_wait(s_full, c & 1, status)) break;
            tc_fence_after();
            softmax<16>(tmem, scale, len, ptile, red, m);
            // V rows past the tile's last visible position in the last page
            if (!mbar_wait(v_full, c & 1, status)) break;
            const int vl = min(CHUNK, vmax - c * CHUNK);
            if (vl & 15)
                zero_v_rows(smem + PreL::V, vl, (vl + 15) & ~15, threadIdx.x,
                            STHREADS);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            if (warp < 4) {
                if (!mbar_wait(o_full, c & 1, status)) break;
                tc_fence_after();
                float o[16];
                tmem_ld_16cols(tmem + 32 + ((uint32_t)(warp * 32) << 16), o);
                sync_softmax();  // every warp's row sums are in
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    if (len[r] <= 0) continue;  // chunk not visible to the row
                    const float l = row_sum(red, r);
                    if (c == 0) {
                        M[r] = m[r];
                        L[r] = l;
                        O[r] = o[r];
                    } else {
                        float a, bb;
                        merge_scalars(M[r], L[r], m[r], l, a, bb);
                        O[r] = merge_value(O[r], o[r], a, bb);
                    }
                }
                tc_fence_before();
            } else {
                sync_softmax();
            }
        }
        if (warp < 4) {
            const int dim = warp * 32 + lane;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int qi = r / G, hh = r % G;
                if (qi >= nq) continue;
                out[((int64_t)(t0 + qi) * Hq + g * G + hh) * D + dim] =
                    f32_to_bf16(__fdiv_rn(O[r], L[r]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == SW) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// ------------------------------------------------- prefill, row per thread --
// Attention of query tiles of 128 rows (128 / G consecutive tokens x the G
// query heads of KV head g; row r = token r / G, head r % G) with one thread
// per row.  The tensor core computes the chunk's scores untransposed,
// S[row][key] = Q K^T (M = 128 rows, N = 256 keys, K = 128 dims in 8 steps
// of 16), and the chunk's values O[row][dim] = P V (M = 128 rows, N = 128
// dims, K = 256 keys in 16 steps).  The other kernels compute the same
// elements as S^T = K Q^T and O^T = V^T P^T over 16-row tiles; the tensor
// core's result for an element does not depend on N nor on which operand
// holds the row (checked bit for bit on GB300 for both products over
// N = 16 .. 256), so each element keeps its bits.  Thread r then runs the
// decode softmax of its row alone: the exact maximum of the scaled, masked
// scores (for scale > 0 taken on the raw scores and scaled once: rounding is
// monotone, so the maximum is the same number), p = p_of(s, c1, mu2),
// bf16(p) into the P tile, the row sum as the xor tree over each 32-key
// group (16, 8, 4, 2, 1) and the eight groups in order, then merge_scalars /
// merge_value against the row's running (M, L, O) in chunk order and
// bf16(O / L) at the end.  No value crosses threads, so no shuffle, shared
// score buffer or barrier sits between a row's operations.
//   warps 0-3   rows 32 w + lane (TMEM lane quarter w); per chunk n: the
//               maximum (pass 1), the merge of chunk n - 1 into the running
//               O held in registers (its values arrive while pass 1 runs),
//               the exponentials, P and the row sum (pass 2);
//   warp 4      one lane issues the MMAs: S of chunk n + 1 into the other
//               tensor-memory slot once the merge of chunk n - 1 has read
//               it (so it runs under pass 2 of chunk n), then the values of
//               chunk n into the first 128 columns of chunk n's own slot
//               (its scores are consumed) once P and V are in;
//   warp 5      the query tile (once per item) and K of each chunk by TMA;
//   warp 6      V of each chunk by TMA, then zeroes the rows past the last
//               visible position in the chunk's last page (0 * NaN would
//               poison the sums).
// Tensor memory (512 columns): two slots of 256, chunk n in slot n % 2 (S,
// then its values).  Items (tile, KV head) are walked by persistent CTAs in
// list order (most chunks first); chunks are counted over the CTA's walk.
// Waits are bounded as in the other kernels, and each role waits (bounded)
// for its own copies and products in flight before the CTA leaves.
namespace tca {
struct RowL {
    static constexpr int TB = CHUNK * 128 * 2;   // K or V tile, 64 KB
    static constexpr int QH = 128 * 128;         // a 64-dim half of Q, 16 KB
    static constexpr int PG = 128 * 128;         // a 64-key group of P, 16 KB
    static constexpr int Q = 0, K = 2 * QH, V = K + TB, P = V + TB;
    static constexpr int BAR = P + 4 * PG;
    // k_full, k_free, v_full, v_ready, v_free, p_full, o_full, done,
    // s_full[2], slot_free[2]; then the TMEM address and the failure flag
    static constexpr int NBAR = 12;
    static constexpr int BYTES = BAR + NBAR * 8 + 8;
    static constexpr int ALLOC = BYTES + 1024;
};
constexpr int ROW_THREADS = 128 + 3 * 32;
constexpr uint32_t ROW_TMEM = 512;
constexpr uint32_t IDESC_S = make_idesc_bf16(128, 256);
constexpr uint32_t IDESC_O = make_idesc_bf16(128, 128) | (1u << 16);

// S = Q K^T of one chunk into TMEM columns d .. d + 255 (lane = row).
__device__ __forceinline__ void issue_rows_s(uint32_t d, uint32_t qt,
                                             uint32_t kt) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = qt + (kk >> 2) * RowL::QH + (kk & 3) * 32;
        const uint32_t b = kt + (kk >> 2) * (CHUNK * 128) + (kk & 3) * 32;
        tc_mma_bf16(d, make_sw128_desc(a), make_sw128_desc(b), IDESC_S,
                    kk > 0 ? 1u : 0u);
    }
}

// O = P V of one chunk into TMEM columns d .. d + 127 (lane = row); V read
// in place as the MN-major operand (its two 64-dim halves are the atoms).
__device__ __forceinline__ void issue_rows_o(uint32_t d, uint32_t pt,
                                             uint32_t vt) {
#pragma unroll
    for (int kk = 0; kk < CHUNK / 16; ++kk) {
        const uint32_t a = pt + (kk >> 2) * RowL::PG + (kk & 3) * 32;
        const uint32_t b = vt + kk * 2048;
        tc_mma_bf16(d, make_sw128_desc(a),
                    make_sw128_desc_mn(b, CHUNK * 128, 1024), IDESC_O,
                    kk > 0 ? 1u : 0u);
    }
}

// Exact maximum of 32 values (any order gives the same number).
__device__ __forceinline__ float max32(const float *v) {
    float m[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) m[j] = fmaxf(v[j], v[j + 16]);
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], m[j + 8]);
#pragma unroll
    for (int j = 0; j < 4; ++j) m[j] = fmaxf(m[j], m[j + 4]);
    return fmaxf(fmaxf(m[0], m[2]), fmaxf(m[1], m[3]));
}

// The decode path's sum of one 32-key group: lane 0's xor tree, levels 16,
// 8, 4, 2, 1 pairing key i with i + 16, i + 8, ...
__device__ __forceinline__ float xor_tree32(const float *x) {
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = __fadd_rn(x[i], x[i + 16]);
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __fadd_rn(a[i], a[i + 8]);
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = __fadd_rn(a[i], a[i + 4]);
#pragma unroll
    for (int i = 0; i < 2; ++i) a[i] = __fadd_rn(a[i], a[i + 2]);
    return __fadd_rn(a[0], a[1]);
}
}  // namespace tca

template <bool SPLIT>
__global__ void __launch_bounds__(tca::ROW_THREADS, 1)
    attn_rows_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap qmap,
                     const int4 *__restrict__ list,
                     const int32_t *__restrict__ cnt,
                     const int32_t *__restrict__ page_table, int max_pages,
                     int n_pages, int Hq, int Hkv, int G, float scale,
                     uint16_t *__restrict__ out, int32_t *status,
                     const int2 *__restrict__ sitems, float *__restrict__ rec,
                     int Cmax) {
    using namespace tca;
    constexpr int D = 128;
    constexpr int PAGE_BYTES = 16 * 64 * 2;   // one box: 16 rows x 64 dims
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RowL::BAR);
    uint64_t *k_full = bars, *k_free = bars + 1, *v_full = bars + 2,
             *v_ready = bars + 3, *v_free = bars + 4, *p_full = bars + 5,
             *o_full = bars + 6, *done = bars + 7, *s_full = bars + 8,
             *slot_free = bars + 10;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + RowL::NBAR);
    volatile int *fail = reinterpret_cast<volatile int *>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_valid = cnt[0], n_all = cnt[1];
    // item it: KV head it % Hkv of list entry it / Hkv, chunks 0 .. C - 1;
    // split form: of split item it / Hkv = (entry, chunk c0), that chunk
    const int items = (SPLIT ? cnt[2] : n_valid) * Hkv;
    auto item = [&](int it, int4 &e, int &g, int &c0, int &Cn) {
        g = it % Hkv;
        if constexpr (SPLIT) {
            const int2 si = sitems[it / Hkv];
            e = list[si.x];
            c0 = si.y;
            Cn = 1;
        } else {
            e = list[it / Hkv];
            c0 = 0;
            Cn = (e.y + CHUNK - 1) / CHUNK;
        }
    };

    // Bounded wait; once any wait of the CTA has run out, returns at once.
    auto gw = [&](uint64_t *bar, uint32_t parity) {
        if (*fail) return;
        if (mbar_try_wait(bar, parity)) return;
        const uint64_t t0 = bi_globaltimer();
        uint32_t n = 0;
        while (!mbar_try_wait(bar, parity)) {
            if ((++n & 1023u) == 0) {
                if (*fail) return;
                if (bi_globaltimer() - t0 > BI_WAIT_LIMIT_NS) {
                    bi_record_error(status, BI_ERR_TIMEOUT);
                    *fail = 1;
                    return;
                }
            }
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(k_full, 1);
        mbar_init(k_free, 1);
        mbar_init(v_full, 1);
        mbar_init(v_ready, 1);
        mbar_init(v_free, 1);
        mbar_init(p_full, 4);
        mbar_init(o_full, 1);
        mbar_init(done, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&slot_free[b], 4);
        }
        mbar_fence_init();
        *fail = 0;
    }
    if (warp == 4) tmem_alloc(tslot, ROW_TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp >= 5) {
        // ------------------------------------------------ K and V loads --
        const bool is_k = warp == 5;
        if (lane == 0) {
            tma_prefetch_desc(is_k ? &kmap : &vmap);
            if (is_k) tma_prefetch_desc(&qmap);
        }
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *freed = is_k ? k_free : v_free;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        uint8_t *tile = smem + (is_k ? RowL::K : RowL::V);
        uint32_t n = 0;   // loads so far
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            int4 e;
            int g, c0, C;
            item(it, e, g, c0, C);
            const int L = e.y, req = e.w;
            const int32_t *pt_row = page_table + (int64_t)req * max_pages;
            for (int cl = 0; cl < C; ++cl, ++n) {
                const int c = c0 + cl;   // the chunk
                // the buffer is free once the previous chunk's products
                // that read it have completed
                if (lane == 0 && n > 0) gw(freed, (n - 1) & 1);
                __syncwarp();
                int pg = -1;
                if (lane < 16) {
                    const int pi = c * 16 + lane;
                    if (c * CHUNK + lane * 16 < L && pi < max_pages) {
                        pg = pt_row[pi];
                        if (pg < 0 || pg >= n_pages) {
                            if (is_k) bi_record_error(status, BI_ERR_BOUNDS);
                            pg = -1;
                        }
                    }
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(
                        full, 16 * 2 * PAGE_BYTES +
                                  (is_k && cl == 0 ? 2 * RowL::QH : 0));
                __syncwarp();
                if (lane < 16) {
                    const int row = pg >= 0 ? (pg * Hkv + g) * 16 : -16;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tma_load_2d(tile + h * (CHUNK * 128) + lane * PAGE_BYTES,
                                    map, h * 64, row, full);
                }
                if (is_k && cl == 0 && lane == 0) {
                    // rows = 128 / G tokens from e.x x the G heads of g
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(smem + RowL::Q + h * RowL::QH, &qmap,
                                    h * 64, g * G, e.x, full);
                }
                if (!is_k) {
                    gw(v_full, n & 1);
                    const int vl = min(CHUNK, L - c * CHUNK);
                    if (vl & 15)
                        zero_v_rows(tile, vl, (vl + 15) & ~15, lane, 32);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(v_ready);
                }
            }
        }
        // own copies in flight have landed before the CTA leaves (after a
        // wait gave up, the last load may not have been waited on)
        if (lane == 0 && n > 0)
            mbar_wait_for(full, (n - 1) & 1, status, BI_WAIT_LIMIT_NS);
    } else if (warp == 4) {
        // ---------------------------------------------------------- MMAs --
        if (lane == 0) {
            const uint32_t qt = base + RowL::Q, kt = base + RowL::K,
                           vt = base + RowL::V, pt = base + RowL::P;
            // S of chunk n into slot n % 2: the slot's previous chunk
            // (n - 2) has been merged, K of chunk n is in
            auto qk = [&](uint32_t n) {
                const uint32_t b = n & 1;
                if (n >= 2) gw(&slot_free[b], ((n - 2) >> 1) & 1);
                gw(k_full, n & 1);
                tc_fence_after();
                issue_rows_s(tmem + 256 * b, qt, kt);
                tc_commit(&s_full[b]);
                tc_commit(k_free);
            };
            uint32_t n = 0;
            const int it0 = blockIdx.x;
            if (it0 < items) qk(0);
            for (int it = it0; it < items; it += gridDim.x) {
                int4 e;
                int g, c0, C;
                item(it, e, g, c0, C);
                for (int c = 0; c < C; ++c, ++n) {
                    // the next chunk (of this item or the next one) first
                    if (c + 1 < C || it + (int)gridDim.x < items) qk(n + 1);
                    gw(p_full, n & 1);   // pass 2 of chunk n wrote P
                    gw(v_ready, n & 1);
                    tc_fence_after();
                    issue_rows_o(tmem + 256 * (n & 1), pt, vt);
                    tc_commit(o_full);
                    tc_commit(v_free);
                }
            }
            // the products in flight have completed before the CTA leaves
            tc_commit(done);
            mbar_wait_for(done, 0, status, BI_WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else {
        // ------------------------------------- rows: softmax and merges --
        const int r = threadIdx.x;   // 0..127
        const uint32_t lq = (uint32_t)(warp * 32) << 16;
        const uint32_t prow_smem = base + RowL::P + r * 128;
        const bool pos_scale = scale > 0.f;
        const float c1 = __fmul_rn(scale, LOG2E);
        uint32_t n = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            int4 e;
            int g, c0, C;
            item(it, e, g, c0, C);
            const int t0 = e.x, L = e.y, ntok = e.z;
            const int tk = r / G, hh = r % G;
            // position of the row's token (tokens of a tile are consecutive
            // positions ending at L - 1), -1 past the tile's tokens
            const int prow = tk < ntok ? L - ntok + tk : -1;
            float O[D];                      // running values
            float M = -INFINITY, Ls = 0.f;   // running max and sum
            float pm = 0.f, pl = 0.f;        // chunk n - 1
            int plen = 0;
            // merge of the previous chunk (index np, first of the item if
            // first): its values from its slot into O, then the slot is free
            auto merge = [&](uint32_t np, bool first) {
                gw(o_full, np & 1);
                tc_fence_after();
                const uint32_t o_t = tmem + 256 * (np & 1) + lq;
                const bool part = plen > 0;
                if (first) {
                    if (part) {
                        M = pm;
                        Ls = pl;
                    }
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk)
                        tmem_ld_32cols(o_t + 32 * blk, O + 32 * blk);
                } else {
                    float a = 0.f, b = 0.f;
                    if (part) merge_scalars(M, Ls, pm, pl, a, b);
                    if (__any_sync(0xffffffffu, part)) {
#pragma unroll
                        for (int blk = 0; blk < 4; ++blk) {
                            float o[32];
                            tmem_ld_32cols(o_t + 32 * blk, o);
                            if (part)
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    O[32 * blk + i] = merge_value(
                                        O[32 * blk + i], o[i], a, b);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&slot_free[np & 1]);
            };
            for (int c = 0; c < C; ++c, ++n) {
                const uint32_t s_t = tmem + 256 * (n & 1) + lq;
                gw(&s_full[n & 1], (n >> 1) & 1);
                tc_fence_after();
                const int len = prow + 1 - (c0 + c) * CHUNK;   // visible keys
                const bool any = __any_sync(0xffffffffu, len > 0);
                // pass 1: the exact maximum of the row's visible scores
                float m = -INFINITY;
                if (any) {
#pragma unroll 1
                    for (int gq = 0; gq < 8; ++gq) {
                        float v[32];
                        tmem_ld_32cols(s_t + 32 * gq, v);
                        if (!pos_scale)
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __fmul_rn(v[j], scale);
                        if (len < CHUNK)
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (32 * gq + j >= len) v[j] = -INFINITY;
                        m = fmaxf(m, max32(v));
                    }
                    if (pos_scale) m = __fmul_rn(m, scale);
                }
                const float mu2 =
                    __fmul_rn(m == -INFINITY ? 0.f : m, LOG2E);
                // the previous chunk's values (its products also finished
                // reading P)
                if (c > 0) merge(n - 1, c == 1);
                // pass 2: p, bf16(p) into P, the row sum in the decode order
                float l = 0.f;
#pragma unroll 1
                for (int gq = 0; gq < 8; ++gq) {
                    float x[32];
                    if (any) {
                        tmem_ld_32cols(s_t + 32 * gq, x);
                        if (len >= CHUNK) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                x[j] = p_of(x[j], c1, mu2);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                x[j] = 32 * gq + j < len ? p_of(x[j], c1, mu2)
                                                         : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) x[j] = 0.f;
                    }
                    const uint32_t pg_base =
                        prow_smem + (gq >> 1) * RowL::PG;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int u = ((gq & 1) * 4 + q4) ^ (r & 7);
                        asm volatile(
                            "st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                pg_base + (u << 4)),
                            "r"(pack_bf16x2(x[8 * q4 + 0], x[8 * q4 + 1])),
                            "r"(pack_bf16x2(x[8 * q4 + 2], x[8 * q4 + 3])),
                            "r"(pack_bf16x2(x[8 * q4 + 4], x[8 * q4 + 5])),
                            "r"(pack_bf16x2(x[8 * q4 + 6], x[8 * q4 + 7]))
                            : "memory");
                    }
                    const float W = xor_tree32(x);
                    l = gq == 0 ? W : __fadd_rn(l, W);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
                pm = m;
                pl = l;
                plen = len;
            }
            // the last chunk's values, then the rows out
            merge(n - 1, C == 1);
            if constexpr (SPLIT) {
                // the chunk's record (m, l, 2 pad, o[D]) of the decode
                // path's two-stage form, for rows that see the chunk
                if (prow >= 0 && plen > 0) {
                    float4 *dst = reinterpret_cast<float4 *>(
                        rec + (((int64_t)(t0 + tk) * Hq + g * G + hh) * Cmax +
                               c0) * rec_floats<D>());
                    dst[0] = make_float4(M, Ls, 0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < D / 4; ++i)
                        dst[1 + i] = make_float4(O[4 * i], O[4 * i + 1],
                                                 O[4 * i + 2], O[4 * i + 3]);
                }
            } else if (prow >= 0) {
                uint16_t *dst =
                    out + ((int64_t)(t0 + tk) * Hq + g * G + hh) * D;
#pragma unroll
                for (int q8 = 0; q8 < D / 8; ++q8) {
                    uint4 w;
                    w.x = pack_bf16x2(__fdiv_rn(O[8 * q8 + 0], Ls),
                                      __fdiv_rn(O[8 * q8 + 1], Ls));
                    w.y = pack_bf16x2(__fdiv_rn(O[8 * q8 + 2], Ls),
                                      __fdiv_rn(O[8 * q8 + 3], Ls));
                    w.z = pack_bf16x2(__fdiv_rn(O[8 * q8 + 4], Ls),
                                      __fdiv_rn(O[8 * q8 + 5], Ls));
                    w.w = pack_bf16x2(__fdiv_rn(O[8 * q8 + 6], Ls),
                                      __fdiv_rn(O[8 * q8 + 7], Ls));
                    *reinterpret_cast<uint4 *>(dst + 8 * q8) = w;
                }
            }
        }
    }
    // entries with no valid context: zero outputs (split form: the merge
    // writes every row)
    for (int j = n_valid + blockIdx.x; !SPLIT && j < n_all; j += gridDim.x) {
        const int4 e = list[j];
        const int64_t n = (int64_t)e.z * Hq * D;
        for (int64_t idx = threadIdx.x; idx < n; idx += ROW_THREADS)
            out[(int64_t)e.x * Hq * D + idx] = 0;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, ROW_TMEM);
    }
}

// ------------------------------------------------------------------- host --

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

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

size_t records_bytes(int B, int Hq, int D, int max_kv_len) {
    const int C = (max_kv_len + CHUNK - 1) / CHUNK;
    return up256((size_t)B * Hq * C * (D + 4) * sizeof(float));
}

}  // namespace

// Whole (row, KV head) items when there are at least 8 per SM; below that
// the per-chunk kernel spreads a row's chunks over the SMs.  Measured at 8
// KV heads: batches of 8-128 rows 2-6% faster per chunk, 256 rows 4.6%
// faster as whole rows.  Both forms give the same bits.
bool bi_decode_whole_rows(int B, int Hkv, int D) {
    return D == 128 && (int64_t)B * Hkv >= 8 * (int64_t)bi_sm_count();
}

namespace {

template <int D>
bi_status launch_decode_chunks(bool whole_rows, const CUtensorMap &km,
                               const CUtensorMap &vm,
                               const CUtensorMap &qm,
                               const int32_t *page_table, int max_pages,
                               int n_pages, const int32_t *row_req,
                               const int32_t *kv_len, int Hq, int Hkv, int G,
                               float scale, float *rec, int Cmax,
                               const int32_t *prefix, int B,
                               const int2 *items, const bi_bf16 *k_pool,
                               const bi_bf16 *v_pool, bi_bf16 *out,
                               int32_t *status, cudaStream_t s) {
    static std::once_flag f, f2;
    static bi_status fs, fs2;
    if (D == 128 && !whole_rows) {
        std::call_once(f2, [] {
            fs2 = set_attr(decode_tc_chunks_kernel, tca::DecL::ALLOC);
        });
        if (fs2 != BI_OK) return fs2;
        decode_tc_chunks_kernel<<<bi_sm_count(), tca::DEC_THREADS,
                                  tca::DecL::ALLOC, s>>>(
            km, vm, qm, page_table, max_pages, n_pages, row_req, kv_len, Hq,
            Hkv, G, scale, rec, Cmax, prefix, B, items, k_pool, v_pool,
            status);
    } else if constexpr (D == 128) {
        std::call_once(f, [] {
            fs = set_attr(attn_tc_kernel<false, 4>, tca::DecL::ALLOC);
            if (fs == BI_OK)
                fs = set_attr(attn_tc_kernel<false, 16>, tca::DecL::ALLOC);
        });
        if (fs != BI_OK) return fs;
        // rows per item: G query heads (the arrays of the row state)
        auto kern = G <= 4 ? attn_tc_kernel<false, 4> : attn_tc_kernel<false, 16>;
        kern<<<bi_sm_count(), tca::DEC_ROW_THREADS, tca::DecL::ALLOC, s>>>(
            km, vm, qm, page_table, max_pages, n_pages, row_req, Hq, Hkv, G,
            scale, prefix + B, B, items, k_pool, v_pool,
            reinterpret_cast<uint16_t *>(out), status);
    } else {
        std::call_once(f, [] {
            fs = set_attr(decode_chunks_kernel<D>, DecSmem<D>::ALLOC);
        });
        if (fs != BI_OK) return fs;
        decode_chunks_kernel<D>
            <<<bi_sm_count(), cthreads<D>() + 64, DecSmem<D>::ALLOC, s>>>(
                km, vm, qm, page_table, max_pages, n_pages, row_req, kv_len,
                Hq, Hkv, G, scale, rec, Cmax, prefix, B, items, k_pool, v_pool,
                status);
    }
    BI_LAUNCH_CHECK("decode attention launch");
    return BI_OK;
}

}  // namespace

extern "C" size_t bi_decode_attn_workspace_size(int B, int Hq, int D,
                                                int max_kv_len) {
    if (B <= 0 || Hq <= 0 || D <= 0 || max_kv_len <= 0) return 0;
    const int C = (max_kv_len + CHUNK - 1) / CHUNK;
    return records_bytes(B, Hq, D, max_kv_len) +
           up256((size_t)(B + 1) * sizeof(int32_t)) +
           up256((size_t)B * C * sizeof(int2));
}

// Decode attention with the pool size known (page ids are range-checked
// against it).  stages: bit 0 runs the chunk kernels (after building the
// work list, unless bit 2 says the list in `ws` is already built for these
// kv_len and row_req), bit 1 the merge.  With whole-row items (head_dim 128,
// bi_decode_whole_rows) the kernel merges in registers and writes `out`
// itself (bit 1 does nothing); its work list is the sorted row list of
// build_rows_kernel.  Otherwise the work list holds (row, chunk) items and
// bit 1 merges the chunk records.
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
    if (B == 0) return BI_OK;
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
    BI_REQUIRE(n_pages > 0, "bi_paged_decode_attn: n_pages=%d", n_pages);
    const size_t need = bi_decode_attn_workspace_size(B, Hq, D, max_kv_len);
    if (!ws || ws_bytes < need)
        return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                       "bi_paged_decode_attn: workspace %zu < %zu", ws_bytes,
                       need);
    const int Cmax = (max_kv_len + CHUNK - 1) / CHUNK;
    const int G = Hq / Hkv;
    float *rec = static_cast<float *>(ws);
    uint8_t *after = static_cast<uint8_t *>(ws) +
                     records_bytes(B, Hq, D, max_kv_len);
    int32_t *prefix = reinterpret_cast<int32_t *>(after);
    int2 *items = reinterpret_cast<int2 *>(
        after + up256((size_t)(B + 1) * sizeof(int32_t)));
    int32_t *status = bi_status_ptr();
    if (stages & 1) {
        // Pools as 2-D [rows][D] bf16, rows = (page * Hkv + head) * 16 + slot;
        // queries as [B * Hq][D].  Boxes of 16 rows x 64 columns (D = 128,
        // 128-byte swizzle) or 16 x 32 (D = 32, no swizzle).
        const uint64_t pool_rows = (uint64_t)n_pages * Hkv * 16;
        const uint32_t bw = D == 128 ? 64 : D;
        CUtensorMap km, vm, qm;
        bi_status st;
        if ((st = bi_make_tmap_2d_bf16(&km, k_pool, D, pool_rows, D * 2, bw, 16,
                                       D == 128)) != BI_OK)
            return st;
        if ((st = bi_make_tmap_2d_bf16(&vm, v_pool, D, pool_rows, D * 2, bw, 16,
                                       D == 128)) != BI_OK)
            return st;
        if ((st = bi_make_tmap_2d_bf16(&qm, q, D, (uint64_t)B * Hq, D * 2, bw,
                                       16, D == 128)) != BI_OK)
            return st;
        const bool rows = bi_decode_whole_rows(B, Hkv, D);
        if (!(stages & 4)) {
            if (rows)
                build_rows_kernel<<<1, 1024, 0, s>>>(kv_len, row_req, B, Cmax,
                                                     prefix, items);
            else
                build_items_kernel<<<1, 1024, 0, s>>>(kv_len, row_req, B,
                                                      Cmax, prefix, items);
            BI_LAUNCH_CHECK("decode item list launch");
        }
        if (D == 128)
            st = launch_decode_chunks<128>(rows, km, vm, qm, page_table,
                                           max_pages,
                                           n_pages, row_req, kv_len, Hq, Hkv,
                                           G, scale, rec, Cmax, prefix, B,
                                           items, k_pool, v_pool, out, status,
                                           s);
        else
            st = launch_decode_chunks<32>(false, km, vm, qm, page_table,
                                          max_pages,
                                          n_pages, row_req, kv_len, Hq, Hkv, G,
                                          scale, rec, Cmax, prefix, B, items,
                                          k_pool, v_pool, out, status, s);
        if (st != BI_OK) return st;
    }
    if ((stages & 2) && !bi_decode_whole_rows(B, Hkv, D)) {
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

// Without the pool size the 2-D maps of the pools are given the largest row
// count a page id (int32) can address; page ids are trusted below it.
static int unbounded_pages(int Hkv) { return 0x7fffffff / (Hkv * 16); }

extern "C" bi_status bi_paged_decode_attn(
    const bi_bf16 *q, const bi_bf16 *k_pool, const bi_bf16 *v_pool,
    const int32_t *page_table, int max_pages, const int32_t *row_req,
    const int32_t *kv_len, int B, int max_kv_len, int Hq, int Hkv, int D,
    float scale, bi_bf16 *out, void *ws, size_t ws_bytes, void *stream) {
    BI_REQUIRE(Hkv > 0, "bi_paged_decode_attn: Hkv=%d", Hkv);
    return bi_decode_attn_pool(q, k_pool, v_pool, page_table, max_pages,
                               unbounded_pages(Hkv), row_req, kv_len, B,
                               max_kv_len, Hq, Hkv, D, scale, out, ws,
                               ws_bytes, 3, bi_stream(stream));
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

// Device address of the scratch array on the current device.  Every call
// made outside a stream capture looks it up again (cudaGetSymbolAddress, a
// host-side lookup), so a device reset that reloads the module, and may move
// the array, is followed; a call being captured reuses the address of the
// device's last uncaptured call (and looks it up only if there was none).
static bi_status noalloc_scratch(cudaStream_t s, void **out) {
    static std::mutex mu;
    static void *ptrs[64] = {nullptr};
    int dev = 0;
    bi_status st = bi_cuda_check(cudaGetDevice(&dev), "noalloc: cudaGetDevice");
    if (st != BI_OK) return st;
    if (dev < 0 || dev >= 64)
        return bi_fail(BI_ERR_UNSUPPORTED, "noalloc: device %d", dev);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    st = bi_cuda_check(cudaStreamIsCapturing(s, &cs),
                       "noalloc: cudaStreamIsCapturing");
    if (st != BI_OK) return st;
    std::lock_guard<std::mutex> lock(mu);
    if (cs == cudaStreamCaptureStatusNone || !ptrs[dev]) {
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
    BI_REQUIRE(Hkv > 0, "bi_paged_decode_attn_noalloc: Hkv=%d", Hkv);
    void *ws = nullptr;
    bi_status st = noalloc_scratch(bi_stream(stream), &ws);
    if (st != BI_OK) return st;
    // The chunk kernel writes every partial the merge kernel reads, and the
    // item list is rebuilt by every call, so nothing left in the array by an
    // earlier call is ever read.
    return bi_decode_attn_pool(q, k_pool, v_pool, page_table, max_pages,
                               unbounded_pages(Hkv), row_req, kv_len, B,
                               max_kv_len, Hq, Hkv, D, scale, out, ws,
                               BI_DECODE_ATTN_NOALLOC_SCRATCH_BYTES, 3,
                               bi_stream(stream));
}

size_t bi_prefill_attn_ws_bytes(int T, int R, int Hq, int Hkv) {
    if (T <= 0 || R <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
    const int QPT = 16 / (Hq / Hkv);
    const size_t tiles = (size_t)(T + QPT - 1) / QPT + R;
    return up256(2 * tiles * sizeof(int4) + 2 * sizeof(int32_t));
}

// Split form (head_dim 128, T <= SPLIT_MAX_T): the tile list and counts,
// the (entry, chunk) items, every token's context and request, and the
// chunk records [T][Hq][Cmax] of the decode path's two-stage form.
constexpr int SPLIT_MAX_T = 512;
size_t bi_prefill_attn_split_ws_bytes(int T, int R, int Hq, int Hkv,
                                      int max_kv_len) {
    if (T <= 0 || T > SPLIT_MAX_T || R <= 0 || Hkv <= 0 || Hq % Hkv ||
        !group_ok(Hq, Hkv) || max_kv_len <= 0)
        return 0;
    const int QPT = 16 / (Hq / Hkv);
    const size_t tiles = (size_t)(T + QPT - 1) / QPT + R;
    const size_t Cmax = (size_t)(max_kv_len + CHUNK - 1) / CHUNK;
    return up256(2 * tiles * sizeof(int4) + 4 * sizeof(int32_t)) +
           up256(tiles * Cmax * sizeof(int2)) +
           up256(2 * (size_t)T * sizeof(int32_t)) +
           up256((size_t)T * Hq * Cmax * rec_floats<128>() * sizeof(float));
}

bi_status bi_prefill_attn_pool(const bi_bf16 *q, const int32_t *cu_q,
                               const int32_t *seg_req, int R, int T,
                               const int32_t *pos, int max_q, int max_kv_len,
                               const bi_bf16 *k_pool, const bi_bf16 *v_pool,
                               const int32_t *page_table, int max_pages,
                               int n_pages, int Hq, int Hkv, int D,
                               float scale, bi_bf16 *out, void *ws,
                               size_t ws_bytes, cudaStream_t stream,
                               bool reuse_list) {
    BI_REQUIRE(R >= 0 && T >= 0 && max_q >= 0 && max_kv_len > 0 &&
                   max_kv_len <= 16 * max_pages,
               "bi_prefill_attn: R=%d T=%d max_q=%d max_kv_len=%d", R, T,
               max_q, max_kv_len);
    if (T == 0 || R == 0) return BI_OK;
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
    const int G = Hq / Hkv;
    const int QPT = 16 / G;
    const int tiles = (T + QPT - 1) / QPT + R;
    int32_t *status = bi_status_ptr();
    dim3 grid(tiles, Hkv);
    // With a workspace, head_dim 128: the row-per-thread kernel over a
    // sorted list of 128-row tiles (one K / V chunk load per tile of
    // 128 / G tokens).  Without a workspace, one CTA per 16-row tile.  Both
    // give the bits of decode.
    const size_t split_need =
        D == 128 ? bi_prefill_attn_split_ws_bytes(T, R, Hq, Hkv, max_kv_len)
                 : 0;
    if (D == 128 && ws && R <= MAX_SEGS && split_need &&
        ws_bytes >= split_need) {
        // verify-sized batches: every (tile, chunk) its own item, the
        // records merged in chunk order by the decode merge
        const int QPR = 128 / G;
        static std::once_flag f;
        static bi_status fs;
        std::call_once(f, [] {
            fs = set_attr(attn_rows_kernel<true>, tca::RowL::ALLOC);
        });
        if (fs != BI_OK) return fs;
        const uint64_t pool_rows = (uint64_t)n_pages * Hkv * 16;
        CUtensorMap km, vm, qm;
        bi_status st;
        if ((st = bi_make_tmap_2d_bf16(&km, k_pool, D, pool_rows, D * 2, 64, 16,
                                       true)) != BI_OK)
            return st;
        if ((st = bi_make_tmap_2d_bf16(&vm, v_pool, D, pool_rows, D * 2, 64, 16,
                                       true)) != BI_OK)
            return st;
        if ((st = bi_make_tmap_3d(&qm, q, false, D, Hq, T, 64, G, true,
                                  QPR)) != BI_OK)
            return st;
        const int Cmax = (max_kv_len + CHUNK - 1) / CHUNK;
        int4 *tmp = static_cast<int4 *>(ws);
        int4 *list = tmp + tiles;
        int32_t *cnt = reinterpret_cast<int32_t *>(list + tiles);
        uint8_t *p = static_cast<uint8_t *>(ws) +
                     up256(2 * (size_t)tiles * sizeof(int4) +
                           4 * sizeof(int32_t));
        int2 *sitems = reinterpret_cast<int2 *>(p);
        p += up256((size_t)tiles * Cmax * sizeof(int2));
        int32_t *kvl_tok = reinterpret_cast<int32_t *>(p);
        int32_t *req_tok = kvl_tok + T;
        p += up256(2 * (size_t)T * sizeof(int32_t));
        float *rec = reinterpret_cast<float *>(p);
        if (!reuse_list) {
            build_tiles_kernel<<<1, 1024, 0, stream>>>(
                cu_q, seg_req, pos, R, QPR, max_kv_len, tmp, list, cnt, status,
                T, sitems, kvl_tok, req_tok);
            BI_LAUNCH_CHECK("prefill split list launch");
        }
        attn_rows_kernel<true>
            <<<bi_sm_count(), tca::ROW_THREADS, tca::RowL::ALLOC, stream>>>(
                km, vm, qm, list, cnt, page_table, max_pages, n_pages, Hq, Hkv,
                G, scale, reinterpret_cast<uint16_t *>(out), status, sitems,
                rec, Cmax);
        BI_LAUNCH_CHECK("prefill split attention launch");
        const int warps = T * Hq;
        decode_merge_kernel<128><<<(warps * 32 + 255) / 256, 256, 0, stream>>>(
            rec, kvl_tok, req_tok, T, Hq, Cmax,
            reinterpret_cast<uint16_t *>(out));
    } else if (D == 128 && ws && R <= MAX_SEGS &&
               ws_bytes >= bi_prefill_attn_ws_bytes(T, R, Hq, Hkv)) {
        const int QPR = 128 / G;   // tokens per 128-row tile
        static std::once_flag f;
        static bi_status fs;
        std::call_once(f, [] {
            fs = set_attr(attn_rows_kernel<false>, tca::RowL::ALLOC);
        });
        if (fs != BI_OK) return fs;
        const uint64_t pool_rows = (uint64_t)n_pages * Hkv * 16;
        CUtensorMap km, vm, qm;
        bi_status st;
        if ((st = bi_make_tmap_2d_bf16(&km, k_pool, D, pool_rows, D * 2, 64, 16,
                                       true)) != BI_OK)
            return st;
        if ((st = bi_make_tmap_2d_bf16(&vm, v_pool, D, pool_rows, D * 2, 64, 16,
                                       true)) != BI_OK)
            return st;
        // queries as [T][Hq][D]: boxes of 64 dims x G heads x QPR tokens
        if ((st = bi_make_tmap_3d(&qm, q, false, D, Hq, T, 64, G, true,
                                  QPR)) != BI_OK)
            return st;
        const int tiles128 = (T + QPR - 1) / QPR + R;
        int4 *tmp = static_cast<int4 *>(ws);
        int4 *list = tmp + tiles128;
        int32_t *cnt = reinterpret_cast<int32_t *>(list + tiles128);
        if (!reuse_list) {
            build_tiles_kernel<<<1, 1024, 0, stream>>>(cu_q, seg_req, pos, R,
                                                       QPR, max_kv_len, tmp,
                                                       list, cnt, status);
            BI_LAUNCH_CHECK("prefill row-tile list launch");
        }
        const int grid =
            (int)std::min<int64_t>((int64_t)tiles128 * Hkv, bi_sm_count());
        attn_rows_kernel<false><<<grid, tca::ROW_THREADS, tca::RowL::ALLOC,
                                  stream>>>(
            km, vm, qm, list, cnt, page_table, max_pages, n_pages, Hq, Hkv, G,
            scale, reinterpret_cast<uint16_t *>(out), status, nullptr, nullptr,
            0);
    } else if (D == 128) {
        static std::once_flag f;
        static bi_status fs;
        std::call_once(f, [] {
            fs = set_attr(prefill_tc_kernel, tca::PreL::ALLOC);
        });
        if (fs != BI_OK) return fs;
        const uint64_t pool_rows = (uint64_t)n_pages * Hkv * 16;
        CUtensorMap km, vm;
        bi_status st;
        if ((st = bi_make_tmap_2d_bf16(&km, k_pool, D, pool_rows, D * 2, 64, 16,
                                       true)) != BI_OK)
            return st;
        if ((st = bi_make_tmap_2d_bf16(&vm, v_pool, D, pool_rows, D * 2, 64, 16,
                                       true)) != BI_OK)
            return st;
        prefill_tc_kernel<<<grid, tca::PRE_THREADS, tca::PreL::ALLOC,
                            stream>>>(
            km, vm, q, cu_q, seg_req, R, pos, page_table, max_pages, n_pages,
            Hq, Hkv, G, scale, max_kv_len, out, status);
    } else {
        static std::once_flag f;
        static bi_status fs;
        std::call_once(f, [] {
            fs = set_attr(prefill_kernel<32>, prefill_smem<32>());
        });
        if (fs != BI_OK) return fs;
        prefill_kernel<32><<<grid, cthreads<32>(), prefill_smem<32>(),
                             stream>>>(
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
                                Hkv > 0 ? unbounded_pages(Hkv) : 1, Hq, Hkv, D,
                                scale, out, nullptr, 0, bi_stream(stream),
                                false);
}

extern "C" size_t bi_prefill_attn_workspace_size(int T, int R, int Hq,
                                                 int Hkv) {
    return bi_prefill_attn_ws_bytes(T, R, Hq, Hkv);
}

extern "C" size_t bi_prefill_attn_split_workspace_size(int T, int R, int Hq,
                                                       int Hkv,
                                                       int max_kv_len) {
    return bi_prefill_attn_split_ws_bytes(T, R, Hq, Hkv, max_kv_len);
}

extern "C" bi_status bi_prefill_attn_ws(
    const bi_bf16 *q, const int32_t *cu_q, const int32_t *seg_req, int R,
    int T, const int32_t *pos, int max_q, int max_kv_len,
    const bi_bf16 *k_pool, const bi_bf16 *v_pool, const int32_t *page_table,
    int max_pages, int Hq, int Hkv, int D, float scale, bi_bf16 *out,
    void *ws, size_t ws_bytes, void *stream) {
    BI_REQUIRE(!ws || bi_aligned16(ws), "bi_prefill_attn_ws: ws alignment");
    return bi_prefill_attn_pool(q, cu_q, seg_req, R, T, pos, max_q, max_kv_len,
                                k_pool, v_pool, page_table, max_pages,
                                Hkv > 0 ? unbounded_pages(Hkv) : 1, Hq, Hkv, D,
                                scale, out, ws, ws_bytes, bi_stream(stream),
                                false);
}
