// bi_gemm: y = x W^T on the tcgen05 tensor cores, batch-invariant.
//
// ybb.press, "LLM 推理确定性工程深度实战", section 2.2: library GEMMs pick tile
// shape, stage count and split-K from (M, N, K), and split-K with atomicAdd
// is not even run-to-run deterministic.  Section 4 gives the remedy this
// kernel follows: one tile shape for every M, a split count fixed per weight
// shape, a fixed-order second stage, no float atomics.
//
// Tile plan.  A tile is 256 rows x BN columns, BN in {128, 192, 256}; K is
// cut into S slices of whole 64-column blocks, slice s covering blocks
// [s*KB/S, (s+1)*KB/S).  (BN, S) = gemm_plan(N, K) is a pure function of the
// weight shape, never of M.  Reduction order of one output y[m][n]:
//   - inside a slice: one tcgen05.mma chain (M=128, N=BN, K=16 per
//     instruction) in ascending k, accumulating in fp32 in tensor memory,
//     starting from zero;
//   - slices are summed in fp32 in slice order ((p0 + p1) + p2) + ... by
//     the consumer (bi_rmsnorm, bi_rope, or the reduce kernels here).
//
// Why 256-row tiles: a decode batch (M <= 256) is one m-tile, so every W
// tile is loaded once for all rows, and per k-block an SM loads (256 + BN)
// rows of 128 B for 256 x BN x 64 multiply-adds.  Measured on GB300 an SM
// ingests about 112 GB/s and multiplies at about 12.5 TFLOP/s, so BN = 128
// is load-bound and BN >= 192 tensor-bound in steady state; the rest of a
// decode GEMM is fixed cost per launch (prologue, pipeline fill, epilogue:
// eight epilogue warps instead of four measured no faster).  gemm_plan
// ranks (BN, S, CTA pairs) by a time model calibrated on a sweep of every
// plan for the 8B projection shapes.
//
// Persistent CTAs (one per SM, 192 threads) loop over work units (m-tile,
// n-tile, slice), the m-tile fastest: warp 0 lane 0 issues TMA loads into a
// ring of shared-memory stages (A: 256 x 64, B: BN x 64, 128-byte swizzle);
// warp 1 owns the tensor memory and lane 0 issues, per 16-column step, one
// MMA per 128-row half into the two halves of a TMEM accumulator; warps 2-5
// are the epilogue (warp w reads TMEM lanes 32*(w%4) .. +31 of both halves),
// staging 32-row pieces in shared memory and writing them with TMA stores,
// which clip rows past M and columns past N.  Every wait is bounded.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int BM = 256;                   // tile rows
constexpr int HALF = 128;                 // rows per MMA (one TMEM lane each)
constexpr int BK = 64;                    // k-block: 128 bytes of bf16
constexpr int A_BYTES = BM * BK * 2;      // 32 KB
constexpr int THREADS = 192;
constexpr int STORE_BYTES = 32 * 128;     // one staged store: 32 rows x 128 B
constexpr int EPI_BYTES = 4 * 2 * STORE_BYTES;  // 4 warps x double buffer
constexpr int SMEM_LIMIT = 232448;        // opt-in shared memory per block
constexpr int TMEM_COLS = 512;
constexpr int MAX_SPLITS = 8;
constexpr int PLAN_SMS = 152;             // SMs the plan fills (GB300)

// ONE: every CTA runs at most one work unit.  Its epilogue then starts only
// after every load of the CTA has landed and every MMA has read its stage,
// so the epilogue staging reuses the first stage of the ring and the ring
// gets the space (BN = 192: four stages instead of three).
template <int BN, bool ONE = false>
struct Tile {
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_OWN = ONE ? 0 : EPI_BYTES;  // staging of its own
    static constexpr int FIT = (SMEM_LIMIT - EPI_OWN - 1024 - 256) / STAGE_BYTES;
    static constexpr int STAGES = FIT < 4 ? FIT : 4;
    static constexpr int ACC_COLS = 2 * BN;           // both halves
    static constexpr int NACC = TMEM_COLS / ACC_COLS;  // accumulators in TMEM
    static constexpr uint32_t IDESC = make_idesc_bf16(HALF, BN);
    static constexpr size_t SMEM =
        1024 + (size_t)STAGES * STAGE_BYTES + EPI_OWN + 256;
    static_assert(STAGES >= 2 && NACC >= 1, "tile does not fit");
    static_assert(ONE ? A_BYTES >= EPI_BYTES : true, "staging in stage 0");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory");
};

struct GemmArgs {
    int M, N, K, KB, S;
    int MT;     // m-tiles
    int units;  // MT * n-tiles * S
    int out_kind;
    int F;      // SwiGLU: output features (N / 2)
    int abox;   // rows of the A box: 256, or M rounded up to 16 when M < 256
    int32_t *status;
};

// silu(g) * u = (g / (1 + e^-g)) * u, each operation rounded separately.
// The exponential and the division are the fast hardware forms (__expf,
// __fdividef: a few fp32 ulp), far below the bf16 resolution of the
// output; the correctly rounded forms made the SwiGLU epilogue of the
// 8B gate/up GEMM 8 us slower (58 -> 50 us at M = 256).  The same fp32
// steps for every M, so the result stays batch-invariant.
__device__ __forceinline__ float swiglu1(float g, float u) {
    return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
}

__device__ __forceinline__ int slice_lo(const GemmArgs &p, int s) {
    return (int)((int64_t)s * p.KB / p.S);
}

// Unit u = (m-tile fastest, then slice, then n-tile).  CTAs that run at the
// same time on neighbouring units read the same weight tile.
__device__ __forceinline__ void unit_coords(const GemmArgs &p, int u, int &m0,
                                            int &nt, int &s) {
    const int mt = u % p.MT;
    const int rest = u / p.MT;
    s = rest % p.S;
    nt = rest / p.S;
    m0 = mt * BM;
}

// Epilogue store of one 32-row piece whose row r (lane r) is ROW_BYTES / 4
// words.  128-byte rows go to the staging buffer in the layout of the
// 128-byte TMA swizzle (16-byte unit j of row r at unit j ^ (r % 8),
// conflict-free for st.shared.v4); 64-byte rows are stored plainly.  The
// piece leaves with one TMA store at (x, y, z).  Two buffers alternate;
// before reusing one, lane 0 waits until the store issued from it has
// finished reading it.
struct Stager {
    uint8_t *buf;   // this warp's two buffers
    int count;

    template <int ROW_BYTES>
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
        for (int j = 0; j < ROW_BYTES / 16; ++j) {
            const uint32_t addr =
                ROW_BYTES == 128
                    ? smem_u32(b) + lane * 128 + ((j ^ (lane & 7)) << 4)
                    : smem_u32(b) + lane * ROW_BYTES + (j << 4);
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

// Epilogue of one accumulator block: this warp's 32 TMEM lanes (rows row0
// .. row0 + 31) x BN fp32 columns from `base`, for output column tile nt
// (BN columns; BN / 2 features for SwiGLU) and slice s; `live`: row0 < M.
template <int BN>
__device__ __forceinline__ void store_block(const GemmArgs &p,
                                            const CUtensorMap *tmO,
                                            Stager &stg, uint32_t base,
                                            int row0, int nt, int s,
                                            bool live) {
    const int n0 = nt * BN;
    if (p.out_kind == BI_OUT_SWIGLU) {
        // gate columns [0, w), up columns [w, 2w) of this tile
        const int f0 = nt * (BN / 2);
        const int w = min(BN / 2, p.F - f0);
        for (int c = 0; c < w; c += 32) {
            float g[32], uu[32];
            uint32_t wd[16];
            tmem_ld_32cols(base + c, g);
            tmem_ld_32cols(base + w + c, uu);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                wd[i] = pack_bf16x2(swiglu1(g[2 * i], uu[2 * i]),
                                    swiglu1(g[2 * i + 1], uu[2 * i + 1]));
            stg.put<64>(tmO, wd, f0 + c, row0, 0, live);
        }
    } else if (p.out_kind == BI_OUT_BF16) {
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
            uint32_t wd[32];
            float v[32];
            tmem_ld_32cols(base + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                wd[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            tmem_ld_32cols(base + c + 32, v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                wd[16 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            stg.put<128>(tmO, wd, n0 + c, row0, 0, live && n0 + c < p.N);
        }
    } else {  // fp32: partial slice s (or the only slice)
#pragma unroll
        for (int c = 0; c < BN; c += 32) {
            float v[32];
            tmem_ld_32cols(base + c, v);
            stg.put<128>(tmO, reinterpret_cast<const uint32_t *>(v), n0 + c,
                         row0, p.out_kind == BI_OUT_PARTIALS ? s : 0,
                         live && n0 + c < p.N);
        }
    }
}

template <int BN, bool ONE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, GemmArgs p) {
    using T = Tile<BN, ONE>;
    constexpr int STAGES = T::STAGES, NACC = T::NACC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    // epilogue staging, 1024-aligned: its own region, or stage 0's A tile
    uint8_t *sE = ONE ? sA : sB + STAGES * T::B_BYTES;
    uint64_t *full =
        reinterpret_cast<uint64_t *>(sB + STAGES * T::B_BYTES + T::EPI_OWN);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;     // [NACC]
    uint64_t *acc_empty = acc_full + NACC;   // [NACC]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(acc_empty + NACC);

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
    __syncthreads();  // the barriers exist
    // The producer needs no tensor memory: its loads start while warp 1
    // allocates it; warps 1-5 meet on named barrier 1 once it is held.
    uint32_t tmem = 0;
    if (warp >= 1) {
        if (warp == 1) tmem_alloc(tslot, TMEM_COLS);
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(THREADS - 32) : "memory");
        tc_fence_after();
        tmem = *tslot;
    }

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- producer --
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        // With one m-tile every W tile is read once: evict it from L2
        // first, so that x and the partial planes stay.
        const uint64_t pol = l2_evict_first_policy();
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            int m0, nt, s;
            unit_coords(p, u, m0, nt, s);
            const int kb1 = slice_lo(p, s + 1);
            for (int kb = slice_lo(p, s); kb < kb1; ++kb, ++it) {
                const int st = it % STAGES;
                const uint32_t round = it / STAGES;
                if (round > 0 &&
                    !mbar_wait(&empty[st], (round - 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[st],
                                      p.abox * BK * 2 + T::B_BYTES);
                tma_load_2d(sA + st * A_BYTES, &tmA, kb * BK, m0, &full[st]);
                if (p.MT == 1)
                    tma_load_2d_hint(sB + st * T::B_BYTES, &tmB, kb * BK,
                                     nt * BN, &full[st], pol);
                else
                    tma_load_2d(sB + st * T::B_BYTES, &tmB, kb * BK, nt * BN,
                                &full[st]);
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
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++acc) {
            int m0, nt, s;
            unit_coords(p, u, m0, nt, s);
            const int buf = acc % NACC;
            if (acc >= NACC &&
                !mbar_wait(&acc_empty[buf], ((acc / NACC) - 1) & 1,
                           p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d0 = tmem + buf * T::ACC_COLS, d1 = d0 + BN;
            const int kb0 = slice_lo(p, s), kb1 = slice_lo(p, s + 1);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int st = it % STAGES;
                if (!mbar_wait(&full[st], (it / STAGES) & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_u32(sA + st * A_BYTES);
                const uint32_t b = smem_u32(sB + st * T::B_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t bd = make_sw128_desc(b + 32 * k);
                    const uint32_t accumulate = (kb > kb0 || k > 0) ? 1u : 0u;
                    tc_mma_bf16(d0, make_sw128_desc(a + 32 * k), bd, T::IDESC,
                                accumulate);
                    if (p.abox > HALF)
                        tc_mma_bf16(d1,
                                    make_sw128_desc(a + HALF * 128 + 32 * k),
                                    bd, T::IDESC, accumulate);
                }
                tc_commit(&empty[st]);
            }
            if (ok) tc_commit(&acc_full[buf]);
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------- epilogue --
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        Stager stg{sE + (warp - 2) * 2 * STORE_BYTES, 0};
        int acc = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++acc) {
            int m0, nt, s;
            unit_coords(p, u, m0, nt, s);
            const int buf = acc % NACC;
            if (!mbar_wait(&acc_full[buf], (acc / NACC) & 1, p.status)) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row0 = m0 + h * HALF + q * 32;
                store_block<BN>(p, &tmO, stg,
                                lane_addr + buf * T::ACC_COLS + h * BN, row0,
                                nt, s, row0 < p.M);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
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

// ------------------------------------------------------------ CTA pairs --
//
// The same tile plan on pairs of SMs (a cluster of two CTAs): a unit is
// (m-tile of 256 rows, pair n-tile of 2 BN columns, slice).  Per k-block
// each CTA loads its own 128 rows of A and BN / 2 rows of each of the two
// BN-column halves of the pair tile's W block; the even CTA issues, per
// 16-column step, two tcgen05.mma.cta_group::2 (M = 256, N = BN), one per
// half, and each CTA receives its 128 rows of D in its own tensor memory.
// Against one CTA per 256 x BN tile, each SM loads (128 + BN) instead of
// (256 + BN) rows per k-block for the same number of outputs.  The
// reduction order of an output is the same chain of 16-column steps in
// ascending k, so the result is a function of (N, K) and the inputs only.
//
// Barriers: the even CTA's full[st] counts both CTAs' bytes (the odd CTA's
// loads complete on it through its shared::cluster address); empty[st] and
// acc_full[] are signalled in both CTAs by the pair commit; acc_empty[] of
// the even CTA collects the 8 epilogue warps of the pair.
template <int BN, bool ONE>
struct PairTile {
    static constexpr int A_CTA = HALF * BK * 2;             // 16 KB
    static constexpr int B_CTA = BN * BK * 2;               // 2 x BN/2 rows
    static constexpr int B_HALF = (BN / 2) * BK * 2;
    static constexpr int STAGE_BYTES = A_CTA + B_CTA;
    static constexpr int EPI_OWN = ONE ? 0 : EPI_BYTES;
    static constexpr int FIT =
        (SMEM_LIMIT - EPI_OWN - 1024 - 256) / STAGE_BYTES;
    static constexpr int STAGES = FIT < 8 ? FIT : 8;
    static constexpr int ACC_COLS = 2 * BN;
    static constexpr int NACC = TMEM_COLS / ACC_COLS;
    static constexpr uint32_t IDESC = make_idesc_bf16(2 * HALF, BN);
    static constexpr size_t SMEM =
        1024 + (size_t)STAGES * STAGE_BYTES + EPI_OWN + 256;
    static_assert(STAGES >= 2 && NACC >= 1, "pair tile does not fit");
    static_assert(ONE ? STAGES * A_CTA >= EPI_BYTES : true,
                  "staging in the A stages");
};

template <int BN, bool ONE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, GemmArgs p) {
    using T = PairTile<BN, ONE>;
    constexpr int STAGES = T::STAGES, NACC = T::NACC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * T::A_CTA;
    uint8_t *sE = ONE ? sA : sB + STAGES * T::B_CTA;
    uint64_t *full =
        reinterpret_cast<uint64_t *>(sB + STAGES * T::B_CTA + T::EPI_OWN);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + NACC;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(acc_empty + NACC);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 8);
        }
        mbar_fence_init();
    }
    cluster_sync_all();  // both CTAs' barriers exist before either signals
    if (warp == 1) tmem_alloc_pair(tslot, TMEM_COLS);
    tc_fence_before();
    cluster_sync_all();  // both CTAs hold the tensor memory
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- producer --
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        const uint32_t lead_full = mapa_rank(full, 0);
        // with one m-tile every W tile is read once (see gemm_kernel)
        const uint64_t pol = l2_evict_first_policy();
        int it = 0;
        bool ok = true;
        for (int u = cid; u < p.units && ok; u += ncl) {
            int m0, np, s;
            unit_coords(p, u, m0, np, s);
            const int kb1 = slice_lo(p, s + 1);
            for (int kb = slice_lo(p, s); kb < kb1; ++kb, ++it) {
                const int st = it % STAGES;
                const uint32_t round = it / STAGES;
                if (round > 0 &&
                    !mbar_wait(&empty[st], (round - 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                if (rank == 0)
                    mbar_arrive_expect_tx(&full[st], 2 * T::STAGE_BYTES);
                const uint32_t bar = lead_full + st * 8;
                tma_load_2d_pair(sA + st * T::A_CTA, &tmA, kb * BK,
                                 m0 + (int)rank * HALF, bar);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int wy = np * 2 * BN + j * BN + (int)rank * (BN / 2);
                    if (p.MT == 1)
                        tma_load_2d_pair_hint(sB + st * T::B_CTA + j * T::B_HALF,
                                              &tmB, kb * BK, wy, bar, pol);
                    else
                        tma_load_2d_pair(sB + st * T::B_CTA + j * T::B_HALF,
                                         &tmB, kb * BK, wy, bar);
                }
            }
        }
        // The pair commits of the last stages have reached this CTA's
        // empty barriers before it may leave.
        for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
            mbar_wait(&empty[j % STAGES], (j / STAGES) & 1, p.status);
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------------------------------------------- pair MMA --
        int it = 0, acc = 0;
        bool ok = true;
        for (int u = cid; u < p.units && ok; u += ncl, ++acc) {
            int m0, np, s;
            unit_coords(p, u, m0, np, s);
            const int buf = acc % NACC;
            if (acc >= NACC &&
                !mbar_wait(&acc_empty[buf], ((acc / NACC) - 1) & 1,
                           p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + buf * T::ACC_COLS;
            const int kb0 = slice_lo(p, s), kb1 = slice_lo(p, s + 1);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int st = it % STAGES;
                if (!mbar_wait(&full[st], (it / STAGES) & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_u32(sA + st * T::A_CTA);
                const uint32_t b = smem_u32(sB + st * T::B_CTA);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t ad = make_sw128_desc(a + 32 * k);
                    const uint32_t accumulate = (kb > kb0 || k > 0) ? 1u : 0u;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        tc_mma_pair_bf16(
                            d + j * BN, ad,
                            make_sw128_desc(b + j * T::B_HALF + 32 * k),
                            T::IDESC, accumulate);
                }
                tc_commit_pair(&empty[st]);
            }
            if (ok) tc_commit_pair(&acc_full[buf]);
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------- epilogue --
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t lead_acc_empty = mapa_rank(acc_empty, 0);
        Stager stg{sE + (warp - 2) * 2 * STORE_BYTES, 0};
        int acc = 0;
        for (int u = cid; u < p.units; u += ncl, ++acc) {
            int m0, np, s;
            unit_coords(p, u, m0, np, s);
            const int buf = acc % NACC;
            if (!mbar_wait(&acc_full[buf], (acc / NACC) & 1, p.status)) break;
            tc_fence_after();
            const int row0 = m0 + (int)rank * HALF + q * 32;
#pragma unroll
            for (int j = 0; j < 2; ++j)
                store_block<BN>(p, &tmO, stg,
                                lane_addr + buf * T::ACC_COLS + j * BN, row0,
                                2 * np + j, s, row0 < p.M);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lead_acc_empty + buf * 8);
        }
        if (lane == 0) bulk_wait<0>();  // stores done before the CTA exits
    }

    tc_fence_before();
    __syncwarp();
    cluster_sync_all();  // epilogues of both CTAs are done with the TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// Second stage: y = sum_s ws[s] in slice order.
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

// Second stage of SwiGLU with S > 1: gate and up sums (slice order) of
// feature f, then silu(g) * u.  Columns follow the bi_pack_gate_up
// interleave with blocks of w0 features.
__global__ void reduce_swiglu_kernel(const float *__restrict__ ws, int S,
                                     int M, int N, int F, int w0,
                                     uint16_t *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)M * F) return;
    const int64_t m = i / F;
    const int f = (int)(i % F);
    const int b = f / w0, j = f % w0;
    const int w = min(w0, F - b * w0);
    const int64_t gc = m * N + (int64_t)b * 2 * w0 + j, uc = gc + w;
    const int64_t MN = (int64_t)M * N;
    float g = ws[gc], u = ws[uc];
    for (int s = 1; s < S; ++s) {
        g = __fadd_rn(g, ws[s * MN + gc]);
        u = __fadd_rn(u, ws[s * MN + uc]);
    }
    out[i] = f32_to_bf16(swiglu1(g, u));
}

// Row r of the interleaved weight: block b = r / (2 w0) holds features
// [b w0, b w0 + w), w = min(w0, F - b w0): its first w rows are the gate
// rows of those features, the next w the up rows.
__global__ void pack_gate_up_kernel(const uint4 *__restrict__ wg,
                                    const uint4 *__restrict__ wu, int F,
                                    int K8, int w0, uint4 *__restrict__ wgu) {
    const int64_t total = (int64_t)2 * F * K8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / K8, c = i % K8;
        const int b = (int)(r / (2 * w0)), j = (int)(r % (2 * w0));
        const int w = min(w0, F - b * w0);
        const uint4 *src = j < w ? wg + ((int64_t)b * w0 + j) * K8
                                 : wu + ((int64_t)b * w0 + j - w) * K8;
        wgu[i] = src[c];
    }
}

template <int BN, bool ONE>
bi_status set_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_kernel<BN, ONE>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)Tile<BN, ONE>::SMEM);
    });
    return bi_cuda_check(err, "gemm smem attribute");
}

template <int BN, bool ONE>
bi_status set_pair_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_pair_kernel<BN, ONE>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)PairTile<BN, ONE>::SMEM);
    });
    return bi_cuda_check(err, "gemm pair smem attribute");
}

struct Plan {
    int bn, s;
    bool pair;  // CTA pairs (2 BN columns per unit) instead of single CTAs
};

// (BN, S, pair) for a weight of shape [N][K], from a time model of a
// 256-row batch on 152 SMs calibrated on GB300 with a sweep of every plan
// for the 8B projection shapes.  Per 64-column k-block an SM spends the
// longer of its loads, R rows x 128 B at 112 GB/s (R = 256 + BN for a
// single CTA, 128 + BN for a CTA of a pair), and its MMAs, 256 x BN x 64
// multiply-adds at 12.5 TFLOP/s (so BN = 128 is load-bound alone and
// MMA-bound in a pair, BN >= 192 MMA-bound either way).  The busiest SM
// runs waves * ceil(KB / S) k-blocks (waves = ceil(CTAs / 152)); a pair
// launch costs 6 us more (cluster set-up and teardown), and S > 1 adds
// 0.44 us per MB of fp32 partial planes (written once, read once).
// BN in {128, 192, 256}, S in 1 .. min(8, KB / 4); ties go to the smaller
// S, the smaller BN, then single CTAs.  Any plan gives M-invariant
// results, and the plan depends on (N, K) alone.
Plan gemm_plan(int N, int K) {
    const int KB = (K + BK - 1) / BK;
    const int smax = std::max(1, std::min(MAX_SPLITS, KB / 4));
    Plan best{128, 1, false};
    double best_us = -1.0;
    for (int s = 1; s <= smax; ++s) {
        for (int bn : {128, 192, 256}) {
            for (int pair = 0; pair < 2; ++pair) {
                const int64_t cols = pair ? 2 * bn : bn;
                const int64_t units = (int64_t)((N + cols - 1) / cols) * s;
                const int64_t ctas = pair ? 2 * units : units;
                const int64_t waves = (ctas + PLAN_SMS - 1) / PLAN_SMS;
                const double rows = pair ? HALF + bn : BM + bn;
                const double t_kb = std::max(rows * 128.0 / 112e3,
                                             256.0 * bn * 64 * 2 / 12.5e6);
                const double us =
                    (double)waves * ((KB + s - 1) / s) * t_kb +
                    (pair ? 6.0 : 0.0) +
                    (s > 1 ? 0.44 * s * 256.0 * N * 4.0 / 1e6 : 0.0);
                if (best_us < 0 || us < best_us) {
                    best_us = us;
                    best = {bn, s, pair != 0};
                }
            }
        }
    }
    return best;
}

template <int BN>
bi_status launch(const CUtensorMap &ta, const CUtensorMap &tb,
                 const CUtensorMap &to, const GemmArgs &a,
                 cudaStream_t stream) {
    const int grid = std::min(a.units, bi_sm_count());
    if (a.units <= grid) {  // one unit per CTA
        bi_status st = set_smem_attr<BN, true>();
        if (st != BI_OK) return st;
        gemm_kernel<BN, true><<<grid, THREADS, Tile<BN, true>::SMEM, stream>>>(
            ta, tb, to, a);
    } else {
        bi_status st = set_smem_attr<BN, false>();
        if (st != BI_OK) return st;
        gemm_kernel<BN, false>
            <<<grid, THREADS, Tile<BN, false>::SMEM, stream>>>(ta, tb, to, a);
    }
    BI_LAUNCH_CHECK("gemm launch");
    return BI_OK;
}

template <int BN>
bi_status launch_pair(const CUtensorMap &ta, const CUtensorMap &tb,
                      const CUtensorMap &to, const GemmArgs &a,
                      cudaStream_t stream) {
    const int pairs = std::min(a.units, bi_sm_count() / 2);
    if (a.units <= pairs) {  // one unit per pair
        bi_status st = set_pair_smem_attr<BN, true>();
        if (st != BI_OK) return st;
        gemm_pair_kernel<BN, true>
            <<<2 * pairs, THREADS, PairTile<BN, true>::SMEM, stream>>>(
                ta, tb, to, a);
    } else {
        bi_status st = set_pair_smem_attr<BN, false>();
        if (st != BI_OK) return st;
        gemm_pair_kernel<BN, false>
            <<<2 * pairs, THREADS, PairTile<BN, false>::SMEM, stream>>>(
                ta, tb, to, a);
    }
    BI_LAUNCH_CHECK("gemm pair launch");
    return BI_OK;
}

}  // namespace

extern "C" int bi_gemm_splits(int N, int K) {
    if (N <= 0 || K <= 0) return 1;
    return gemm_plan(N, K).s;
}

extern "C" int bi_gemm_tile_n(int N, int K) {
    if (N <= 0 || K <= 0) return 128;
    return gemm_plan(N, K).bn;
}

extern "C" size_t bi_gemm_workspace_size(int M, int N, int K) {
    const int S = bi_gemm_splits(N, K);
    if (S <= 1 || M <= 0 || N <= 0) return 0;
    return (size_t)S * M * N * sizeof(float);
}

extern "C" bi_status bi_gemm(const bi_bf16 *x, int M, int K, const bi_bf16 *W,
                             int N, void *out, int out_kind, void *ws,
                             size_t ws_bytes, void *stream_) {
    BI_REQUIRE(M >= 0 && N > 0 && K > 0, "bi_gemm: bad shape M=%d N=%d K=%d",
               M, N, K);
    BI_REQUIRE(K % 8 == 0 && N % 8 == 0,
               "bi_gemm: K=%d and N=%d must be multiples of 8", K, N);
    BI_REQUIRE(out_kind >= BI_OUT_PARTIALS && out_kind <= BI_OUT_SWIGLU,
               "bi_gemm: bad out_kind %d", out_kind);
    if (out_kind == BI_OUT_SWIGLU)
        BI_REQUIRE(N % 64 == 0,
                   "bi_gemm: SwiGLU needs N %% 64 == 0 (N=%d, 2F with F a "
                   "multiple of 32)",
                   N);
    if (M == 0) return BI_OK;
    BI_REQUIRE(x && W && out, "bi_gemm: null pointer");
    BI_REQUIRE(bi_aligned16(x) && bi_aligned16(W) && bi_aligned16(out),
               "bi_gemm: pointers must be 16-byte aligned");
    cudaStream_t stream = bi_stream(stream_);
    const Plan plan = gemm_plan(N, K);
    const int S = plan.s, BN = plan.bn;
    const int KB = (K + BK - 1) / BK;
    // n-tiles: BN columns, or 2 BN per CTA pair
    const int cols = plan.pair ? 2 * BN : BN;
    const int mt = (M + BM - 1) / BM, nt = (N + cols - 1) / cols;

    // A boxes: 256 rows per CTA, or 128 per CTA of a pair; W boxes: BN
    // rows, or BN / 2 per CTA of a pair and half of the pair tile.  A batch
    // of fewer than 256 rows (single CTAs) loads a box of M rounded up to
    // 16 rows: the TMA then fills no long out-of-bounds tail (measured:
    // M <= 8 took 17-21 us at 4096 x 4096 against 13.3 us for M >= 16).
    // Shared-memory rows past the box hold stale data that reaches only
    // accumulator rows >= M, which are never stored, and the MMA chain of
    // rows < 128 is the same instruction sequence, so the bits of every
    // stored row are those of the full box.
    const int abox = plan.pair ? HALF : (M < BM ? (M + 15) / 16 * 16 : BM);
    CUtensorMap ta, tb, to;
    bi_status st = bi_make_tmap_2d_bf16(&ta, x, K, M, (uint64_t)K * 2, BK,
                                        abox, true);
    if (st != BI_OK) return st;
    st = bi_make_tmap_2d_bf16(&tb, W, K, N, (uint64_t)K * 2, BK,
                              plan.pair ? BN / 2 : BN, true);
    if (st != BI_OK) return st;

    GemmArgs a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.KB = KB;
    a.S = S;
    a.MT = mt;
    a.units = mt * nt * S;
    a.out_kind = out_kind;
    a.F = N / 2;
    a.abox = abox;
    a.status = bi_status_ptr();

    void *dst = out;
    const bool need_reduce = S > 1 && out_kind != BI_OUT_PARTIALS;
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
    // Output map: fp32 [planes][M][N] in 32 x 32 boxes, bf16 [M][N] in
    // 64 x 32 boxes (128-byte rows, swizzled like the staging buffer), or
    // the SwiGLU bf16 [M][N/2] in plain 32 x 32 boxes (64-byte rows: a
    // tile's output width is a multiple of 32, not of 64).
    if (a.out_kind == BI_OUT_PARTIALS)
        st = bi_make_tmap_3d(&to, dst, true, N, M, S, 32, 32, true);
    else if (a.out_kind == BI_OUT_F32)
        st = bi_make_tmap_3d(&to, dst, true, N, M, 1, 32, 32, true);
    else if (a.out_kind == BI_OUT_BF16)
        st = bi_make_tmap_3d(&to, dst, false, N, M, 1, 64, 32, true);
    else
        st = bi_make_tmap_3d(&to, dst, false, N / 2, M, 1, 32, 32, false);
    if (st != BI_OK) return st;

    if (plan.pair) {
        if (BN == 128)
            st = launch_pair<128>(ta, tb, to, a, stream);
        else if (BN == 192)
            st = launch_pair<192>(ta, tb, to, a, stream);
        else
            st = launch_pair<256>(ta, tb, to, a, stream);
    } else {
        if (BN == 128)
            st = launch<128>(ta, tb, to, a, stream);
        else if (BN == 192)
            st = launch<192>(ta, tb, to, a, stream);
        else
            st = launch<256>(ta, tb, to, a, stream);
    }
    if (st != BI_OK) return st;
    if (need_reduce) {
        if (out_kind == BI_OUT_SWIGLU) {
            const int64_t MF = (int64_t)M * (N / 2);
            reduce_swiglu_kernel<<<(unsigned)((MF + 255) / 256), 256, 0,
                                   stream>>>(
                static_cast<const float *>(ws), S, M, N, N / 2, BN / 2,
                static_cast<uint16_t *>(out));
        } else {
            const int64_t MN = (int64_t)M * N;
            reduce_slices_kernel<<<(unsigned)((MN + 255) / 256), 256, 0,
                                   stream>>>(static_cast<const float *>(ws), S,
                                             MN, out_kind, out);
        }
        BI_LAUNCH_CHECK("gemm reduce launch");
    }
    return BI_OK;
}

extern "C" bi_status bi_pack_gate_up(const bi_bf16 *wg, const bi_bf16 *wu,
                                     int F, int K, bi_bf16 *wgu,
                                     void *stream) {
    BI_REQUIRE(F > 0 && F % 32 == 0 && K > 0 && K % 8 == 0,
               "bi_pack_gate_up: F=%d must be a multiple of 32, K=%d of 8", F,
               K);
    BI_REQUIRE(wg && wu && wgu, "bi_pack_gate_up: null pointer");
    BI_REQUIRE(bi_aligned16(wg) && bi_aligned16(wu) && bi_aligned16(wgu),
               "bi_pack_gate_up: pointers must be 16-byte aligned");
    const int K8 = K / 8;
    const int w0 = bi_gemm_tile_n(2 * F, K) / 2;
    const int64_t total = (int64_t)2 * F * K8;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    pack_gate_up_kernel<<<blocks, 256, 0, bi_stream(stream)>>>(
        reinterpret_cast<const uint4 *>(wg), reinterpret_cast<const uint4 *>(wu),
        F, K8, w0, reinterpret_cast<uint4 *>(wgu));
    BI_LAUNCH_CHECK("pack_gate_up launch");
    return BI_OK;
}
