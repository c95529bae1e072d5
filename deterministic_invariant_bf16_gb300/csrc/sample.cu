// bi_argmax_logits and philox_sample: token selection from fp32 logits.
//
// argmax: ybb.press section 1 notes that batch-dependent rounding can flip
// the argmax of the logits.  The comparison here is a total order
// (NaN above everything with the lower index winning among NaNs, then the
// larger value, then the lower index; -0 == +0), so the result is unique
// whatever order and split the elements are visited in: a row is split over
// a cluster of eight CTAs, whose bests are combined by the first.
//
// philox_sample: ybb.press section 6 item 3, one counter-based generator per
// request derived from (request_id, step): seed = request_id * 1000003 + step
// (mod 2^64).  The generator is Philox4x64-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11) with key (seed, 0)
// and counter 0; u = (word0 >> 40) * 2^-24.  The token is found by inverse
// CDF over p_i = exp((logit_i - max) / temperature) with fixed-order blocked
// prefix sums: thread k sums its contiguous slice in index order, the
// slice totals are scanned by a fixed shuffle pattern, so the result depends
// on nothing but the row.  p_i is taken as 2^((logit_i - max) * c) with
// c = rn(log2(e) / temperature) and the PTX base-2 exponential (relative
// error about 2^-22, well inside the rounding of the running sums).
//
// philox_sample_top: the same draw restricted to the top_k highest-ranked
// tokens (larger logit first, ties to the lower index) and, within them, the
// nucleus of mass top_p, the LLM-42 page's fixed sampling hyperparameters.
// One block per row finds the K-th ranked key by an 8-bit radix select,
// collects the keys at or above it (as soon as they fit a 2048-entry
// buffer), sorts them into rank order, and one thread runs the fp32 running
// sums in rank order; the cut and the draw are block-wide index searches.
// Everything depends on the row, request_id and step only.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int SEL_THREADS = 1024;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    const bool vn = isnan(v), bn = isnan(bv);
    if (vn || bn) return vn && bn ? i < bi : vn;
    if (v != bv) return v > bv;
    return i < bi;
}

__device__ __forceinline__ void warp_best(float &v, int &i) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

// Best (value, index) of the block; valid in thread 0.
__device__ __forceinline__ void block_best(float &v, int &i) {
    __shared__ float sv[32];
    __shared__ int si[32];
    warp_best(v, i);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sv[w] = v;
        si[w] = i;
    }
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        v = lane < nw ? sv[lane] : -INFINITY;
        i = lane < nw ? si[lane] : 0x7fffffff;
        warp_best(v, i);
    }
    __syncthreads();
}

// Argmax of one row by a cluster of AM_CLUSTER CTAs: CTA r of the cluster
// takes the r-th contiguous part of the row, and rank 0 combines the
// parts' bests read from the other CTAs' shared memory.  `better` is a
// strict total order, so the result is the same for any split.
constexpr int AM_CLUSTER = 8;
constexpr int AM_THREADS = 256;

__device__ __forceinline__ uint32_t ld_cluster_u32(const void *p,
                                                   uint32_t rank) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(v)
                 : "r"(mapa_rank(p, rank))
                 : "memory");
    return v;
}

__global__ void __cluster_dims__(AM_CLUSTER, 1, 1)
    __launch_bounds__(AM_THREADS)
    argmax_kernel(const float *__restrict__ logits, int V,
                  int32_t *__restrict__ ids) {
    const int t = blockIdx.x / AM_CLUSTER;
    const uint32_t part = cluster_rank();
    const float *row = logits + (int64_t)t * V;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if ((V & 3) == 0) {
        // UNROLL float4 loads in flight per thread over this CTA's part
        constexpr int UNROLL = 4;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int n4 = V / 4;
        const int per = (n4 + AM_CLUSTER - 1) / AM_CLUSTER;
        const int lo = min(n4, (int)part * per), hi = min(n4, lo + per);
        for (int k0 = lo + threadIdx.x; k0 < hi; k0 += UNROLL * AM_THREADS) {
            float4 x[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int k = k0 + u * AM_THREADS;
                x[u] = k < hi ? __ldg(r4 + k)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY,
                                            -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int k = k0 + u * AM_THREADS;
                const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (k < hi && better(xs[e], 4 * k + e, bv, bi)) {
                        bv = xs[e];
                        bi = 4 * k + e;
                    }
            }
        }
    } else {
        const int per = (V + AM_CLUSTER - 1) / AM_CLUSTER;
        const int lo = min(V, (int)part * per), hi = min(V, lo + per);
        for (int k = lo + threadIdx.x; k < hi; k += AM_THREADS)
            if (better(row[k], k, bv, bi)) {
                bv = row[k];
                bi = k;
            }
    }
    block_best(bv, bi);
    __shared__ float s_v;
    __shared__ int s_i;
    if (threadIdx.x == 0) {
        s_v = bv;
        s_i = bi;
    }
    cluster_sync_all();  // every part's best is in its CTA's shared memory
    if (part == 0 && threadIdx.x == 0) {
        for (uint32_t r = 1; r < AM_CLUSTER; ++r) {
            const float v = __uint_as_float(ld_cluster_u32(&s_v, r));
            const int i = (int)ld_cluster_u32(&s_i, r);
            if (better(v, i, bv, bi)) {
                bv = v;
                bi = i;
            }
        }
        ids[t] = bi;
    }
    cluster_sync_all();  // rank 0 has read the others before they exit
}

// ---------------------------------------------------------------- Philox --

struct U4 {
    uint64_t x[4];
};

__device__ __forceinline__ U4 philox4x64_10(U4 c, uint64_t k0, uint64_t k1) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint64_t hi0 = __umul64hi(M0, c.x[0]), lo0 = M0 * c.x[0];
        const uint64_t hi1 = __umul64hi(M1, c.x[2]), lo1 = M1 * c.x[2];
        U4 n;
        n.x[0] = hi1 ^ c.x[1] ^ k0;
        n.x[1] = lo1;
        n.x[2] = hi0 ^ c.x[3] ^ k1;
        n.x[3] = lo0;
        c = n;
    }
    return c;
}

__device__ __forceinline__ float sample_uniform(uint64_t request_id,
                                                uint64_t step) {
    const uint64_t seed = request_id * 1000003ull + step;
    U4 c = {{0, 0, 0, 0}};
    const U4 o = philox4x64_10(c, seed, 0);
    return (float)(o.x[0] >> 40) * 0x1.0p-24f;
}

// Inclusive scan of one value per thread over the block, fixed pattern:
// Hillis-Steele inside each warp, then the warp totals scanned the same way
// by warp 0.  Returns the exclusive prefix; *total gets the block sum.
__device__ __forceinline__ float block_exclusive_scan(float v, float *total) {
    __shared__ float wsum[32];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc = __fadd_rn(n, inc);
    }
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    if (w == 0) {
        float x = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x = __fadd_rn(n, x);
        }
        wsum[lane] = x;  // inclusive warp prefix
    }
    __syncthreads();
    const float before_warp = w > 0 ? wsum[w - 1] : 0.f;
    *total = wsum[(blockDim.x >> 5) - 1];
    // Exclusive prefix of this thread: the warps before it plus the
    // inclusive scan of the previous lane.
    float prev = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) prev = 0.f;
    return lane == 0 ? before_warp : __fadd_rn(before_warp, prev);
}

// One p of the sampling distribution: 2^((x - mx) * c), c = log2(e) / tau
// rounded once.  x == mx gives exactly 1 (also when c overflows for a
// subnormal tau); x = -inf gives 0.  ex2.approx.f32 without .ftz keeps
// subnormal results, as the definition's exp does.
__device__ __forceinline__ float sample_p(float x, float mx, float c) {
    const float d = __fsub_rn(x, mx);
    const float y = d == 0.f ? 0.f : __fmul_rn(d, c);
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// Two blocks per SM (32 registers a thread), so that a batch of up to
// 2 x 152 rows is one wave.
__global__ void __launch_bounds__(SEL_THREADS, 2)
    sample_kernel(const float *__restrict__ logits, int V,
                  const uint64_t *__restrict__ request_id,
                  const uint64_t *__restrict__ step, float tau,
                  int32_t *__restrict__ ids) {
    const int t = blockIdx.x;
    const float *row = logits + (int64_t)t * V;
    // The request's uniform, drawn by one thread before the row is read.
    __shared__ float s_u;
    if (threadIdx.x == 0) s_u = sample_uniform(request_id[t], step[t]);
    // 1. maximum (exact and order-free; NaN ignored), several loads in
    // flight per thread
    float mx = -INFINITY;
    if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
        constexpr int UNROLL = 4;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int n4 = V / 4;
        for (int k0 = threadIdx.x; k0 < n4; k0 += UNROLL * SEL_THREADS) {
            float4 x[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int k = k0 + u * SEL_THREADS;
                x[u] = k < n4 ? __ldg(r4 + k)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY,
                                            -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                mx = fmaxf(fmaxf(mx, fmaxf(x[u].x, x[u].y)),
                           fmaxf(x[u].z, x[u].w));
        }
    } else {
        for (int k = threadIdx.x; k < V; k += SEL_THREADS)
            mx = fmaxf(mx, row[k]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __shared__ float smx[32];
    if ((threadIdx.x & 31) == 0) smx[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = smx[0];
    for (int i = 1; i < SEL_THREADS / 32; ++i) mx = fmaxf(mx, smx[i]);
    // 2. contiguous slice sums in index order.  A warp's 32 slices are one
    // contiguous range; it is read 8 columns of every slice at a time, with
    // lane -> (slice 4 i + lane / 8, column lane % 8) so that each load
    // covers four 32-byte runs, and each lane then sums its own slice's 8
    // values from shared memory in index order.
    const float l2t = __fdiv_rn(1.4426950408889634f, tau);  // log2(e) / tau
    const int per = (V + SEL_THREADS - 1) / SEL_THREADS;
    const int lo = min(V, threadIdx.x * per), hi = min(V, lo + per);
    __shared__ float cols[SEL_THREADS / 32][32][9];
    float(*cw)[9] = cols[threadIdx.x >> 5];
    const int lane = threadIdx.x & 31;
    const int wbase = (threadIdx.x & ~31) * per;
    float part = 0.f;
    // the next column block is loaded into registers while the current
    // one is summed
    float nxt[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + (lane >> 3), c = lane & 7;
        const int e = wbase + r * per + c;
        nxt[i] = c < per && e < V ? __ldg(row + e) : 0.f;
    }
    for (int c0 = 0; c0 < per; c0 += 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) cw[4 * i + (lane >> 3)][lane & 7] = nxt[i];
        __syncwarp();
        const int c = c0 + 8 + (lane & 7);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const int e = wbase + r * per + c;
            nxt[i] = c < per && e < V ? __ldg(row + e) : 0.f;
        }
        const int n = min(8, hi - lo - c0);
        for (int j = 0; j < n; ++j)
            part = __fadd_rn(part, sample_p(cw[lane][j], mx, l2t));
        __syncwarp();
    }
    float total;
    const float prefix = block_exclusive_scan(part, &total);
    // 3. first index whose running sum exceeds u * total.  A slice whose
    // running sum cannot pass the target is skipped: for its n terms and
    // u = 2^-24 the slice's last running sum is at most
    // (prefix + sum p) (1 + u)^n (each rounded add of non-negative terms
    // grows by at most 1 + u) and sum p <= part / (1 - u)^(n - 1); both
    // factors are below f = 1 + 2 (n + 1) u while n u < 1/2, so with the
    // bound in double the skip never changes the result of the full scan.
    const float target = __fmul_rn(s_u, total);
    int first = 0x7fffffff;
    const double f = 1.0 + 2.0 * (double)(hi - lo + 1) * 0x1p-24;
    const double bound = ((double)prefix + (double)part * f) * f;
    // The slice is read 8 values at a time, all loads in flight before the
    // running sums use them.
    if (bound > (double)target) {
        constexpr int CH = 8;
        float cdf = prefix;
        for (int k0 = lo; k0 < hi && first == 0x7fffffff; k0 += CH) {
            float x[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i)
                x[i] = k0 + i < hi ? __ldg(row + k0 + i) : 0.f;
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                if (k0 + i < hi && first == 0x7fffffff) {
                    cdf = __fadd_rn(cdf, sample_p(x[i], mx, l2t));
                    if (cdf > target) first = k0 + i;
                }
            }
        }
    }
    // Integer min/max over the block: order-free, so deterministic.
    __shared__ int s_first, s_last;
    if (threadIdx.x == 0) {
        s_first = 0x7fffffff;
        s_last = -1;
    }
    __syncthreads();
    if (first != 0x7fffffff) atomicMin(&s_first, first);
    __syncthreads();
    if (s_first != 0x7fffffff) {
        if (threadIdx.x == 0) ids[t] = s_first;
        return;
    }
    // No running sum passed the target (rounding): the last index with
    // p > 0.
    int lp = -1;
    for (int k = hi - 1; k >= lo; --k)
        if (sample_p(row[k], mx, l2t) > 0.f) {
            lp = k;
            break;
        }
    if (lp >= 0) atomicMax(&s_last, lp);
    __syncthreads();
    if (threadIdx.x == 0) ids[t] = max(s_last, 0);
}


// ------------------------------------------------------ top-k / top-p --
//
// Token order: larger logit first, equal logits by lower index; NaN ranks
// as -inf, -0 as +0.  rank_key maps a logit to a uint32 whose unsigned
// order is that order of values (ties are then broken by index).
constexpr int TOPK_MAX = 1024;
constexpr int TOPK_CAND = 2048;  // candidate buffer (>= TOPK_MAX)

__device__ __forceinline__ uint32_t rank_key(float v) {
    if (isnan(v)) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Calls f(i, x, live) for every logit of the row, 4 float4 loads in flight
// per thread when aligned.  Every lane of a warp makes the same calls (the
// ones past the row with live = false), so f may use warp collectives.
template <class F>
__device__ __forceinline__ void for_each_logit(const float *row, int V,
                                               bool vec, F f) {
    if (vec) {
        constexpr int UNROLL = 4;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int n4 = V / 4;
        const int span = UNROLL * SEL_THREADS;
        for (int k0 = threadIdx.x & ~31; k0 < n4; k0 += span) {
            const int base = k0 + (threadIdx.x & 31);
            float4 x[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int k = base + u * SEL_THREADS;
                x[u] = k < n4 ? __ldg(r4 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int k = base + u * SEL_THREADS;
                const bool live = k < n4;
                f(4 * k, x[u].x, live);
                f(4 * k + 1, x[u].y, live);
                f(4 * k + 2, x[u].z, live);
                f(4 * k + 3, x[u].w, live);
            }
        }
    } else {
        for (int k0 = threadIdx.x & ~31; k0 < V; k0 += SEL_THREADS) {
            const int k = k0 + (threadIdx.x & 31);
            const bool live = k < V;
            f(k, live ? row[k] : 0.f, live);
        }
    }
}

// Exclusive prefix of one int per thread over the block (warp shuffles,
// then the warp totals); *total gets the block sum.  Integer: exact.
__device__ __forceinline__ int block_excl_scan_i32(int v, int *total) {
    __shared__ int wt[SEL_THREADS / 32];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) wt[w] = inc;
    __syncthreads();
    if (w == 0) {
        int x = wt[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        wt[lane] = x;
    }
    __syncthreads();
    *total = wt[SEL_THREADS / 32 - 1];
    const int r = (w > 0 ? wt[w - 1] : 0) + inc - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(SEL_THREADS)
    sample_top_kernel(const float *__restrict__ logits, int V,
                      const uint64_t *__restrict__ request_id,
                      const uint64_t *__restrict__ step, float tau, int K,
                      float top_p, int32_t *__restrict__ ids) {
    __shared__ uint32_t hist[256];
    __shared__ unsigned long long cand[TOPK_CAND];
    __shared__ float pw[TOPK_MAX], cs[TOPK_MAX];
    __shared__ int s_bin, s_above, s_eq, n_cand, s_n, s_first, s_last;
    const int t = blockIdx.x;
    const float *row = logits + (int64_t)t * V;
    const bool vec =
        (V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // 1. radix select, 8 bits a pass from the top: after each pass the
    // K-th ranked key matches `prefix` under `mask`, `above` keys rank above
    // the prefix and `rank` counts within it.  As soon as the keys at or
    // above the prefix fit the candidate buffer, one more pass collects
    // them all (the top K are among them, ranked above every other key);
    // otherwise the select runs to the full key theta.
    uint32_t prefix = 0, mask = 0;
    int rank = K, above = 0, n_eq = 0;
    bool early = false;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (threadIdx.x < 256) hist[threadIdx.x] = 0;
        __syncthreads();
        for_each_logit(row, V, vec, [&](int, float x, bool live) {
            const uint32_t k = rank_key(x);
            if (live && (k & mask) == prefix)
                atomicAdd(&hist[(k >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 8l .. 8l+7; suffix sums over the lanes
            uint32_t sl = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) sl += hist[8 * lane + j];
            uint32_t suf = sl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t n = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += n;
            }
            const unsigned top =
                __ballot_sync(0xffffffffu, suf >= (uint32_t)rank);
            const int L = 31 - __clz((int)top);
            if (lane == L) {
                uint32_t acc = suf - sl;
                int b = 8 * L + 7;
                for (; b > 8 * L; --b) {
                    if (acc + hist[b] >= (uint32_t)rank) break;
                    acc += hist[b];
                }
                s_bin = b;
                s_above = (int)acc;
                s_eq = (int)hist[b];
            }
        }
        __syncthreads();
        prefix |= (uint32_t)s_bin << shift;
        mask |= 0xffu << shift;
        rank -= s_above;
        above += s_above;
        n_eq = s_eq;
        __syncthreads();
        if (shift > 0 && above + n_eq <= TOPK_CAND) {
            early = true;
            break;
        }
    }

    // 2. candidates as (key << 32 | ~index), at most TOPK_CAND of them
    if (threadIdx.x == 0) n_cand = 0;
    for (int j = threadIdx.x; j < TOPK_CAND; j += SEL_THREADS) cand[j] = 0ull;
    __syncthreads();
    auto put = [&](int i, uint32_t k) {
        const int at = atomicAdd(&n_cand, 1);
        if (at < TOPK_CAND)
            cand[at] = ((unsigned long long)k << 32) | (0xffffffffu - (uint32_t)i);
    };
    const int need = K - above;  // (full select) tokens of key theta kept
    if (early || need == n_eq) {
        // every key at or above the prefix (early), or every key >= theta
        for_each_logit(row, V, vec, [&](int i, float x, bool live) {
            const uint32_t k = rank_key(x);
            if (live && (k & mask) >= prefix) put(i, k);
        });
    } else {
        // full key theta with ties at the cut: keys above theta, and the
        // first `need` tokens of key theta in index order (thread-ordered
        // pieces of 4 tokens, ranked by a block scan)
        const uint32_t theta = prefix;
        int base = 0;
        for (int c0 = 0; c0 < V; c0 += 4 * SEL_THREADS) {
            const int i0 = c0 + 4 * threadIdx.x;
            uint32_t k4[4];
            int eq = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                k4[e] = i0 + e < V ? rank_key(row[i0 + e]) : 0u;
                eq += (i0 + e < V && k4[e] == theta) ? 1 : 0;
            }
            int tot;
            int r = base + block_excl_scan_i32(eq, &tot);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (i0 + e >= V) continue;
                if (k4[e] > theta) {
                    put(i0 + e, k4[e]);
                } else if (k4[e] == theta) {
                    if (r < need) put(i0 + e, k4[e]);
                    ++r;
                }
            }
            base += tot;
        }
    }
    __syncthreads();

    // 3. rank order: bitonic sort, descending (empty entries are 0 and sort
    // last); the first K entries are the kept tokens
    for (int size = 2; size <= TOPK_CAND; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < TOPK_CAND; i += SEL_THREADS) {
                const int j = i ^ stride;
                if (j > i) {
                    const unsigned long long a = cand[i], b = cand[j];
                    const bool desc = (i & size) == 0;
                    if (desc ? a < b : a > b) {
                        cand[i] = b;
                        cand[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }

    // 4. weights, sequential running sums (one thread: the order is part of
    // the result), then the nucleus cut and the draw as block-wide searches
    const float l0 = key_value((uint32_t)(cand[0] >> 32));
    for (int j = threadIdx.x; j < K; j += SEL_THREADS)
        pw[j] = expf(__fdiv_rn(
            __fsub_rn(key_value((uint32_t)(cand[j] >> 32)), l0), tau));
    if (threadIdx.x == 0) {
        s_n = K - 1;
        s_first = 0x7fffffff;
        s_last = 0;
    }
    __syncthreads();
    auto index_of = [&](int j) {
        return (int32_t)(0xffffffffu - (uint32_t)(cand[j] & 0xffffffffull));
    };
    if (n_cand < K || l0 == -INFINITY) {
        if (threadIdx.x == 0) ids[t] = index_of(0);
        return;
    }
    if (threadIdx.x == 0) {
        float c = 0.0f;
#pragma unroll 8
        for (int j = 0; j < K; ++j) {
            c = __fadd_rn(c, pw[j]);
            cs[j] = c;
        }
    }
    __syncthreads();
    // (K <= TOPK_MAX = SEL_THREADS: one j per thread; a warp reduction
    // before each shared atomic)
    static_assert(TOPK_MAX == SEL_THREADS, "one rank position per thread");
    const int j = threadIdx.x;
    if (top_p < 1.0f) {
        const float cut = __fmul_rn(top_p, cs[K - 1]);
        const int c = __reduce_min_sync(
            0xffffffffu, j < K && cs[j] >= cut ? j : 0x7fffffff);
        if (lane == 0) atomicMin(&s_n, c);
        __syncthreads();
    }
    const int n = s_n;
    const float target =
        __fmul_rn(sample_uniform(request_id[t], step[t]), cs[n]);
    const int f = __reduce_min_sync(
        0xffffffffu, j <= n && cs[j] > target ? j : 0x7fffffff);
    const int l = __reduce_max_sync(0xffffffffu,
                                    j <= n && pw[j] > 0.0f ? j : 0);
    if (lane == 0) {
        atomicMin(&s_first, f);
        atomicMax(&s_last, l);
    }
    __syncthreads();
    if (threadIdx.x == 0)
        ids[t] = index_of(s_first != 0x7fffffff ? s_first : s_last);
}

}  // namespace

extern "C" bi_status bi_argmax_logits(const float *logits, int T, int V,
                                      int32_t *ids, void *stream) {
    BI_REQUIRE(T >= 0 && V > 0, "bi_argmax_logits: T=%d V=%d", T, V);
    if (T == 0) return BI_OK;
    BI_REQUIRE(logits && ids, "bi_argmax_logits: null pointer");
    BI_REQUIRE(bi_aligned16(logits), "bi_argmax_logits: logits alignment");
    argmax_kernel<<<T * AM_CLUSTER, AM_THREADS, 0, bi_stream(stream)>>>(
        logits, V, ids);
    BI_LAUNCH_CHECK("argmax launch");
    return BI_OK;
}

extern "C" bi_status philox_sample_top(const float *logits, int T, int V,
                                       const uint64_t *request_id,
                                       const uint64_t *step,
                                       float temperature, int top_k,
                                       float top_p, int32_t *ids,
                                       void *stream) {
    BI_REQUIRE(T >= 0 && V > 0, "philox_sample_top: T=%d V=%d", T, V);
    BI_REQUIRE(temperature >= 0.f, "philox_sample_top: temperature < 0");
    BI_REQUIRE(top_k >= 1, "philox_sample_top: top_k=%d", top_k);
    BI_REQUIRE(top_p > 0.f && top_p <= 1.f, "philox_sample_top: top_p=%g",
               (double)top_p);
    if (top_k > TOPK_MAX)
        return bi_fail(BI_ERR_UNSUPPORTED, "philox_sample_top: top_k=%d > %d",
                       top_k, TOPK_MAX);
    if (T == 0) return BI_OK;
    BI_REQUIRE(logits && ids, "philox_sample_top: null pointer");
    if (temperature == 0.f) return bi_argmax_logits(logits, T, V, ids, stream);
    BI_REQUIRE(request_id && step, "philox_sample_top: null request_id/step");
    sample_top_kernel<<<T, SEL_THREADS, 0, bi_stream(stream)>>>(
        logits, V, request_id, step, temperature, std::min(top_k, V), top_p,
        ids);
    BI_LAUNCH_CHECK("sample top launch");
    return BI_OK;
}

extern "C" bi_status philox_sample(const float *logits, int T, int V,
                                   const uint64_t *request_id,
                                   const uint64_t *step, float temperature,
                                   int32_t *ids, void *stream) {
    // (V < 2^30 keeps the kernel's in-row element offsets in 32 bits)
    BI_REQUIRE(T >= 0 && V > 0 && V < (1 << 30), "philox_sample: T=%d V=%d",
               T, V);
    BI_REQUIRE(temperature >= 0.f, "philox_sample: temperature < 0");
    if (T == 0) return BI_OK;
    BI_REQUIRE(logits && ids, "philox_sample: null pointer");
    if (temperature == 0.f) return bi_argmax_logits(logits, T, V, ids, stream);
    BI_REQUIRE(request_id && step, "philox_sample: null request_id/step");
    sample_kernel<<<T, SEL_THREADS, 0, bi_stream(stream)>>>(
        logits, V, request_id, step, temperature, ids);
    BI_LAUNCH_CHECK("sample launch");
    return BI_OK;
}
