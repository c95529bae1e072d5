// Host-side plumbing shared by every entry point: thread-local error text,
// the device status word, and tensor-map encoding through the driver entry
// point (so the library loads on machines without a driver).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

__device__ int32_t g_bi_device_status = 0;

static thread_local char t_last_error[512] = "";

bi_status bi_fail(bi_status code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return code;
}

bi_status bi_cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return BI_OK;
    return bi_fail(BI_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

extern "C" const char *bi_last_error(void) { return t_last_error; }

int32_t *bi_status_ptr() {
    // One address per device; looked up once per device.
    static std::mutex mu;
    static int32_t *ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bi_device_status) != cudaSuccess)
            return nullptr;
        ptrs[dev] = static_cast<int32_t *>(p);
    }
    return ptrs[dev];
}

int bi_sm_count() {
    static std::mutex mu;
    static int counts[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (counts[dev] <= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        counts[dev] = n;
    }
    return counts[dev];
}

extern "C" bi_status bi_device_status(int32_t *h_status, void *stream) {
    BI_REQUIRE(h_status, "bi_device_status: null output");
    int32_t *d = bi_status_ptr();
    if (!d) return bi_fail(BI_ERR_CUDA, "bi_device_status: no status word");
    cudaStream_t s = bi_stream(stream);
    int32_t zero = 0;
    bi_status st = bi_cuda_check(
        cudaMemcpyAsync(h_status, d, sizeof(int32_t), cudaMemcpyDeviceToHost, s),
        "read status");
    if (st != BI_OK) return st;
    st = bi_cuda_check(cudaStreamSynchronize(s), "sync status");
    if (st != BI_OK) return st;
    return bi_cuda_check(
        cudaMemcpy(d, &zero, sizeof zero, cudaMemcpyHostToDevice),
        "clear status");
}

// ------------------------------------------------------------ tensor maps --

typedef CUresult (*encode_tiled_fn)(CUtensorMap *, CUtensorMapDataType,
                                    cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

static encode_tiled_fn get_encode() {
    static encode_tiled_fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p,
                                             12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<encode_tiled_fn>(p);
    });
    return fn;
}

bi_status bi_make_tmap_3d(CUtensorMap *map, const void *base, bool f32,
                          uint64_t d0, uint64_t d1, uint64_t d2,
                          uint32_t box0, uint32_t box1, bool swizzle128,
                          uint32_t box2) {
    encode_tiled_fn enc = get_encode();
    if (!enc)
        return bi_fail(BI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const uint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map,
                     f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                         : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return bi_fail(BI_ERR_INVALID_ARG,
                       "cuTensorMapEncodeTiled (3-D) failed (%d): dims %llu x "
                       "%llu x %llu",
                       (int)r, (unsigned long long)d0, (unsigned long long)d1,
                       (unsigned long long)d2);
    return BI_OK;
}

bi_status bi_make_tmap_2d_bf16(CUtensorMap *map, const void *base,
                               uint64_t inner, uint64_t outer,
                               uint64_t row_stride_bytes, uint32_t box_inner,
                               uint32_t box_outer, bool swizzle128) {
    encode_tiled_fn enc = get_encode();
    if (!enc)
        return bi_fail(BI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return bi_fail(BI_ERR_INVALID_ARG,
                       "cuTensorMapEncodeTiled failed (%d): base %p inner %llu "
                       "outer %llu stride %llu",
                       (int)r, base, (unsigned long long)inner,
                       (unsigned long long)outer,
                       (unsigned long long)row_stride_bytes);
    return BI_OK;
}

// Test aid for the bounded waits: one thread initialises an mbarrier that
// expects one arrival, which never comes, and waits for its phase with
// the library's bounded wait (mbar_wait_for, the loop mbar_wait runs with
// the 2 s limit) and the given limit.  Nothing else touches the barrier, so
// the wait runs out, BI_ERR_TIMEOUT goes to the status word and the kernel
// returns: no copy, MMA or tensor memory is involved.
__global__ void wait_probe_kernel(uint64_t limit_ns, int32_t *status,
                                  int32_t *done) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        const bool ok = mbar_wait_for(&bar, 0, status, limit_ns);
        *done = ok ? 1 : 2;
    }
}

extern "C" bi_status bi_test_wait_timeout(int64_t limit_ns, int32_t *done,
                                          void *stream) {
    BI_REQUIRE(limit_ns >= 1000 && limit_ns <= 100000000,
               "bi_test_wait_timeout: limit %lld ns outside [1 us, 100 ms]",
               (long long)limit_ns);
    BI_REQUIRE(done, "bi_test_wait_timeout: null pointer");
    int32_t *st = bi_status_ptr();
    if (!st) return bi_fail(BI_ERR_CUDA, "bi_test_wait_timeout: no status");
    wait_probe_kernel<<<1, 32, 0, bi_stream(stream)>>>((uint64_t)limit_ns, st,
                                                      done);
    BI_LAUNCH_CHECK("wait probe launch");
    return BI_OK;
}
