// bi_gemm: y = x W^T on the tcgen05 tensor cores, batch-invariant.
//
// ybb.press, "LLM 推理确定性工程深度实战", section 2.2: library GEMMs pick tile
// shape, stage count and split-K from (M, N, K), and split-K with atomicAdd
// is not even run-to-run deterministic.  Section 4 gives the remedy this
// kernel follows: one tile shape for every M, a split count fixed per weight
// shape, a fixed-order second stage, no float atomics.
//
// Reduction order of one output y[m][n] (independent of M, of the row's
// place in its tile, and of which CTA does the work):
//   - K is cut into S = bi_gemm_splits(N, K) slices of whole 64-column
//     blocks, slice s covering blocks [s*KB/S, (s+1)*KB/S).
//   - Inside a slice: one tcgen05.mma chain (M=128, N=128, K=16 per
//     instruction) in ascending k, accumulating in fp32 in tensor memory,
//     starting from zero.
//   - Slices are summed in fp32 in slice order: ((p0 + p1) + p2) + ...
//
// Two schedules give the same bits:
//   split: a work unit is one (m-tile, n-tile, slice); slices go to memory
//          as fp32 partials and a consumer (bi_rmsnorm, bi_rope, or the
//          reduce kernel here) sums them in order.  Fills the GPU at small M.
//   fused: a work unit is one (m-tile, n-tile) with all its slices run one
//          after another; the epilogue warps add each finished slice to a
//          register running sum in slice order.  No partial traffic; used
//          when there are enough tiles.
//
// Persistent CTAs (one per SM, 192 threads) loop over work units: warp 0
// lane 0 issues TMA loads into a ring of shared-memory stages; warp 1 owns
// the TMEM allocation and lane 0 issues the MMAs into a ring of four TMEM
// accumulators; warps 2-5 are the epilogue (warp w reads TMEM lanes
// 32*(w%4) .. 32*(w%4)+31, i.e. tile rows), staging each 32-row piece of the
// result in a 128-byte-swizzled shared buffer and writing it with a TMA
// store, which clips rows past M and columns past N.  Every wait is bounded.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t IDESC = make_idesc_bf16(BM, BN);
constexpr int STAGES = 5;                 // 160 KB of operand stages
constexpr int NACC = 4;                   // TMEM accumulators (4 x 128 cols)
constexpr int STORE_BYTES = 32 * 128;     // one staged store: 32 rows x 128 B
constexpr int EPI_BYTES = 4 * 2 * STORE_BYTES;  // 4 warps x double buffer

constexpr size_t smem_bytes() {
    return 1024 /* alignment slack */ + (size_t)STAGES * STAGE_BYTES +
           EPI_BYTES + 256;
}

struct GemmArgs {
    int M, N, K, KB, S;
    int MT;     // m-tiles
    int units;  // work units (see unit_coords)
    int out_kind;
    int32_t *status;
};

// silu(g) * u = (g / (1 + e^-g)) * u, each operation rounded separately.
__device__ __forceinline__ float swiglu1(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// Unit u of the schedule.  Units are numbered with the m-tile fastest, so
// CTAs that run at the same time on neighbouring units read the same weight
// tile (the second read hits L2).
template <bool FUSED>
__device__ __forceinline__ void unit_coords(const GemmArgs &p, int u, int &m0,
                                            int &n0, int &nt, int &s_lo,
                                            int &s_hi) {
    const int mt = u % p.MT;
    int rest = u / p.MT;
    if (FUSED) {
        nt = rest;
        s_lo = 0;
        s_hi = p.S;
    } else {
        s_lo = rest % p.S;
        s_hi = s_lo + 1;
        nt = rest / p.S;
    }
    m0 = mt * BM;
    n0 = nt * BN;
}

// Epilogue store of one 32-row x 128-byte piece: the calling warp's lane r
// holds row r as 32 words.  The piece goes into this warp's staging buffer
// in the layout of the 128-byte TMA swizzle (16-byte unit j of row r at
// unit j ^ (r % 8), conflict-free for st.shared.v4) and out with one TMA
// store at (x, y, z).  Two buffers alternate; before reusing one, lane 0
// waits until the store issued from it has finished reading it.
struct Stager {
    uint8_t *buf;   // this warp's two buffers
    int count;

    __device__ __forceinline__ void put(const CUtensorMap *map,
                                       const uint32_t *w, int x, int y, int z,
                                       bool issue) {
        const int lane = threadIdx.x & 31;
        uint8_t *b = buf + (count & 1) * STORE_BYTES;
        if (count >= 2) {
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t addr =
                smem_u32(b) + lane * 128 + ((j ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                         "r"(w[4 * j]), "r"(w[4 * j + 1]), "r"(w[4 * j + 2]),
                         "r"(w[4 * j + 3])
                         : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            // One bulk group per piece (empty when the piece lies wholly
            // outside the output), so the wait above always covers the
            // store that last read this buffer.
            if (issue) tma_store_3d(map, b, x, y, z);
            bulk_commit();
        }
        ++count;
    }
};

template <bool FUSED>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint8_t *sE = sB + STAGES * B_BYTES;  // epilogue staging, 1024-aligned
    uint64_t *full = reinterpret_cast<uint64_t *>(sE + EPI_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;     // [NACC]
    uint64_t *acc_empty = acc_full + NACC;   // [NACC]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(acc_empty + NACC);

    constexpr uint32_t TMEM_COLS = NACC * BN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- producer --
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int m0, n0, nt, s_lo, s_hi;
            unit_coords<FUSED>(p, u, m0, n0, nt, s_lo, s_hi);
            for (int s = s_lo; s < s_hi && ok; ++s) {
                const int kb0 = (int)((int64_t)s * p.KB / p.S);
                const int kb1 = (int)((int64_t)(s + 1) * p.KB / p.S);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int st = it % STAGES;
                    const uint32_t round = it / STAGES;
                    if (round > 0 && !mbar_wait(&empty[st], (round - 1) & 1,
                                                p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
                    tma_load_2d(sA + st * A_BYTES, &tmA, kb * BK, m0,
                                &full[st]);
                    tma_load_2d(sB + st * B_BYTES, &tmB, kb * BK, n0,
                                &full[st]);
                }
            }
        }
        if (!ok) {
            // Let the copies already issued land before the CTA exits.
            for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait(&full[j % STAGES], (j / STAGES) & 1, p.status);
        }
    } else if (warp == 1 && lane == 0) {
        // --------------------------------------------------------- MMA --
        int it = 0, acc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int m0, n0, nt, s_lo, s_hi;
            unit_coords<FUSED>(p, u, m0, n0, nt, s_lo, s_hi);
            for (int s = s_lo; s < s_hi && ok; ++s, ++acc) {
                const int buf = acc % NACC;
                if (acc >= NACC &&
                    !mbar_wait(&acc_empty[buf], ((acc / NACC) - 1) & 1,
                               p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * BN;
                const int kb0 = (int)((int64_t)s * p.KB / p.S);
                const int kb1 = (int)((int64_t)(s + 1) * p.KB / p.S);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int st = it % STAGES;
                    if (!mbar_wait(&full[st], (it / STAGES) & 1, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(sA + st * A_BYTES);
                    const uint32_t b = smem_u32(sB + st * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc_mma_bf16(d_tmem, make_sw128_desc(a + 32 * k),
                                    make_sw128_desc(b + 32 * k), IDESC,
                                    (kb > kb0 || k > 0) ? 1u : 0u);
                    tc_commit(&empty[st]);
                }
                tc_commit(&acc_full[buf]);
            }
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------- epilogue --
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        Stager stg{sE + (warp - 2) * 2 * STORE_BYTES, 0};
        float run[FUSED ? BN : 1];
        int acc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int m0, n0, nt, s_lo, s_hi;
            unit_coords<FUSED>(p, u, m0, n0, nt, s_lo, s_hi);
            const int row0 = m0 + q * 32;
            const bool rows_live = row0 < p.M;
            for (int s = s_lo, j = 0; s < s_hi; ++s, ++j, ++acc) {
                const int buf = acc % NACC;
                if (!mbar_wait(&acc_full[buf], (acc / NACC) & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t base = lane_addr + buf * BN;
                if (FUSED) {
#pragma unroll
                    for (int c = 0; c < BN; c += 32) {
                        float v[32];
                        tmem_ld_32cols(base + c, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            run[c + i] =
                                (j == 0) ? v[i] : __fadd_rn(run[c + i], v[i]);
                    }
                } else if (p.out_kind == BI_OUT_SWIGLU) {
                    uint32_t w[32];
#pragma unroll
                    for (int c = 0; c < BN / 2; c += 32) {
                        float g[32], uu[32];
                        tmem_ld_32cols(base + c, g);
                        tmem_ld_32cols(base + BN / 2 + c, uu);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[c / 2 + i] = pack_bf16x2(
                                swiglu1(g[2 * i], uu[2 * i]),
                                swiglu1(g[2 * i + 1], uu[2 * i + 1]));
                    }
                    stg.put(&tmO, w, nt * (BN / 2), row0, 0, rows_live);
                } else if (p.out_kind == BI_OUT_BF16) {
#pragma unroll
                    for (int c = 0; c < BN; c += 64) {
                        uint32_t w[32];
                        float v[32];
                        tmem_ld_32cols(base + c, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                        tmem_ld_32cols(base + c + 32, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[16 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                        stg.put(&tmO, w, n0 + c, row0, 0,
                                rows_live && n0 + c < p.N);
                    }
                } else {  // fp32: partial slice s (or the only slice)
#pragma unroll
                    for (int c = 0; c < BN; c += 32) {
                        float v[32];
                        tmem_ld_32cols(base + c, v);
                        stg.put(&tmO, reinterpret_cast<const uint32_t *>(v),
                                n0 + c, row0, p.out_kind == BI_OUT_PARTIALS ? s : 0,
                                rows_live && n0 + c < p.N);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
            if (FUSED && ok) {
                if (p.out_kind == BI_OUT_SWIGLU) {
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        w[i] = pack_bf16x2(
                            swiglu1(run[2 * i], run[BN / 2 + 2 * i]),
                            swiglu1(run[2 * i + 1], run[BN / 2 + 2 * i + 1]));
                    stg.put(&tmO, w, nt * (BN / 2), row0, 0, rows_live);
                } else if (p.out_kind == BI_OUT_BF16) {
#pragma unroll
                    for (int c = 0; c < BN; c += 64) {
                        uint32_t w[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            w[i] = pack_bf16x2(run[c + 2 * i], run[c + 2 * i + 1]);
                        stg.put(&tmO, w, n0 + c, row0, 0,
                                rows_live && n0 + c < p.N);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < BN; c += 32)
                        stg.put(&tmO,
                                reinterpret_cast<const uint32_t *>(run + c),
                                n0 + c, row0, 0, rows_live && n0 + c < p.N);
                }
            }
        }
        if (lane == 0) bulk_wait<0>();  // stores done before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Second stage of the split schedule: y = sum_s ws[s] in slice order.
__global__ void reduce_slices_kernel(const float *__restrict__ ws, int S,
                                     int64_t MN, int out_kind, void *out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= MN) return;
    float v = ws[i];
    for (int s = 1; s < S; ++s) v = __fadd_rn(v, ws[(int64_t)s * MN + i]);
    if (out_kind == BI_OUT_BF16)
        reinterpret_cast<uint16_t *>(out)[i] = f32_to_bf16(v);
    else
        reinterpret_cast<float *>(out)[i] = v;
}

__global__ void pack_gate_up_kernel(const uint4 *__restrict__ wg,
                                    const uint4 *__restrict__ wu, int F,
                                    int K8, uint4 *__restrict__ wgu) {
    // Output row r: block b = r / 128, within-block j = r % 128;
    // j < 64 -> gate row 64b + j, else up row 64b + j - 64.
    const int64_t total = (int64_t)2 * F * K8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / K8, c = i % K8;
        const int64_t b = r / 128, j = r % 128;
        const uint4 *src = j < 64 ? wg + (b * 64 + j) * K8
                                  : wu + (b * 64 + j - 64) * K8;
        wgu[i] = src[c];
    }
}

template <bool FUSED>
bi_status set_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_kernel<FUSED>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_bytes());
    });
    return bi_cuda_check(err, "gemm smem attribute");
}

}  // namespace

extern "C" int bi_gemm_splits(int N, int K) {
    // A pure function of the weight shape.  Aim for about one work unit per
    // SM of a 152-SM GB300 at small M (two m-tiles give two per SM at
    // M = 256), with at least 4 k-blocks per slice and at most 8 slices.
    const int KB = (K + BK - 1) / BK;
    const int tiles = (N + BN - 1) / BN;
    int s = 152 / std::max(tiles, 1);
    s = std::min(s, 8);
    s = std::min(s, KB / 4);
    return std::max(s, 1);
}

extern "C" size_t bi_gemm_workspace_size(int M, int N, int K) {
    const int S = bi_gemm_splits(N, K);
    if (S <= 1 || M <= 0 || N <= 0) return 0;
    return (size_t)S * M * N * sizeof(float);
}

// Default schedule.  Either schedule gives the same bits, so this is a pure
// cost choice: fused once the output tiles alone fill the GPU.  (Measured on
// the 8B decode shapes at M = 256: with 48-96 tiles the fused schedule loses
// more to idle SMs than it saves in partial traffic.)
bool bi_gemm_default_fused(int M, int N, int K) {
    const int S = bi_gemm_splits(N, K);
    if (S <= 1) return false;
    const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    return tiles >= 148;
}

bi_status bi_gemm_sched(const bi_bf16 *x, int M, int K, const bi_bf16 *W,
                        int N, void *out, int out_kind, void *ws,
                        size_t ws_bytes, int mode, cudaStream_t stream) {
    BI_REQUIRE(M >= 0 && N > 0 && K > 0, "bi_gemm: bad shape M=%d N=%d K=%d",
               M, N, K);
    BI_REQUIRE(K % 8 == 0 && N % 8 == 0,
               "bi_gemm: K=%d and N=%d must be multiples of 8", K, N);
    if (M == 0) return BI_OK;
    BI_REQUIRE(x && W && out, "bi_gemm: null pointer");
    BI_REQUIRE(bi_aligned16(x) && bi_aligned16(W) && bi_aligned16(out),
               "bi_gemm: pointers must be 16-byte aligned");
    BI_REQUIRE(out_kind >= BI_OUT_PARTIALS && out_kind <= BI_OUT_SWIGLU,
               "bi_gemm: bad out_kind %d", out_kind);
    const int S = bi_gemm_splits(N, K);
    const int KB = (K + BK - 1) / BK;
    const int mt = (M + BM - 1) / BM, nt = (N + BN - 1) / BN;
    if (out_kind == BI_OUT_SWIGLU)
        BI_REQUIRE(N % BN == 0, "bi_gemm: SwiGLU needs N %% 128 == 0 (N=%d)", N);
    bool fused;
    if (mode == 1)
        fused = false;
    else if (mode == 2)
        fused = true;
    else
        fused = bi_gemm_default_fused(M, N, K);
    if (out_kind == BI_OUT_PARTIALS && S > 1) fused = false;
    if (S == 1) fused = false;
    if (out_kind == BI_OUT_SWIGLU && S > 1) fused = true;

    CUtensorMap ta, tb, to;
    bi_status st = bi_make_tmap_2d_bf16(&ta, x, K, M, (uint64_t)K * 2, BK, BM,
                                        true);
    if (st != BI_OK) return st;
    st = bi_make_tmap_2d_bf16(&tb, W, K, N, (uint64_t)K * 2, BK, BN, true);
    if (st != BI_OK) return st;

    GemmArgs a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.KB = KB;
    a.S = S;
    a.out_kind = out_kind;
    a.status = bi_status_ptr();

    void *dst = out;
    const bool need_reduce =
        !fused && S > 1 && out_kind != BI_OUT_PARTIALS;
    if (need_reduce) {
        const size_t need = (size_t)S * M * N * sizeof(float);
        if (!ws || ws_bytes < need)
            return bi_fail(BI_ERR_WORKSPACE_TOO_SMALL,
                           "bi_gemm: workspace %zu < %zu bytes", ws_bytes,
                           need);
        BI_REQUIRE(bi_aligned16(ws), "bi_gemm: workspace alignment");
        dst = ws;
        a.out_kind = BI_OUT_PARTIALS;
    }
    // Output map: fp32 [planes][M][N] in 32 x 32 boxes, or bf16 [M][cols]
    // in 64 x 32 boxes (128-byte rows, swizzled like the staging buffer).
    if (a.out_kind == BI_OUT_PARTIALS)
        st = bi_make_tmap_3d(&to, dst, true, N, M, S, 32, 32);
    else if (a.out_kind == BI_OUT_F32)
        st = bi_make_tmap_3d(&to, dst, true, N, M, 1, 32, 32);
    else if (a.out_kind == BI_OUT_BF16)
        st = bi_make_tmap_3d(&to, dst, false, N, M, 1, 64, 32);
    else
        st = bi_make_tmap_3d(&to, dst, false, N / 2, M, 1, 64, 32);
    if (st != BI_OK) return st;

    a.MT = mt;
    a.units = fused ? mt * nt : mt * nt * S;
    const int grid = std::min(a.units, bi_sm_count());
    if (fused) {
        if ((st = set_smem_attr<true>()) != BI_OK) return st;
        gemm_kernel<true><<<grid, THREADS, smem_bytes(), stream>>>(ta, tb, to,
                                                                   a);
    } else {
        if ((st = set_smem_attr<false>()) != BI_OK) return st;
        gemm_kernel<false><<<grid, THREADS, smem_bytes(), stream>>>(ta, tb, to,
                                                                    a);
    }
    BI_LAUNCH_CHECK("gemm launch");
    if (need_reduce) {
        const int64_t MN = (int64_t)M * N;
        reduce_slices_kernel<<<(unsigned)((MN + 255) / 256), 256, 0, stream>>>(
            static_cast<const float *>(ws), S, MN, out_kind, out);
        BI_LAUNCH_CHECK("gemm reduce launch");
    }
    return BI_OK;
}

extern "C" bi_status bi_gemm(const bi_bf16 *x, int M, int K, const bi_bf16 *W,
                             int N, void *out, int out_kind, void *ws,
                             size_t ws_bytes, void *stream) {
    return bi_gemm_sched(x, M, K, W, N, out, out_kind, ws, ws_bytes, 0,
                         bi_stream(stream));
}

extern "C" bi_status bi_pack_gate_up(const bi_bf16 *wg, const bi_bf16 *wu,
                                     int F, int K, bi_bf16 *wgu,
                                     void *stream) {
    BI_REQUIRE(wg && wu && wgu, "bi_pack_gate_up: null pointer");
    BI_REQUIRE(F > 0 && F % 64 == 0 && K > 0 && K % 8 == 0,
               "bi_pack_gate_up: F=%d must be a multiple of 64, K=%d of 8", F,
               K);
    BI_REQUIRE(bi_aligned16(wg) && bi_aligned16(wu) && bi_aligned16(wgu),
               "bi_pack_gate_up: pointers must be 16-byte aligned");
    const int K8 = K / 8;
    const int64_t total = (int64_t)2 * F * K8;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    pack_gate_up_kernel<<<blocks, 256, 0, bi_stream(stream)>>>(
        reinterpret_cast<const uint4 *>(wg), reinterpret_cast<const uint4 *>(wu),
        F, K8, reinterpret_cast<uint4 *>(wgu));
    BI_LAUNCH_CHECK("pack_gate_up launch");
    return BI_OK;
}
