// local_hess_compute_noalloc: the 16x16 block Hessians of ONE batch,
// computed without allocating any device memory.
//
// Who needs this: callers whose device memory is all reserved up front by
// a pooling allocator, so that a cudaMalloc on their hot path would fail or
// fragment the pool, and callers whose runtime forbids allocating while they
// run (for example code paths that must not synchronise the device, which
// cudaMalloc/cudaFree can do).  local_hess_create allocates its accumulator
// with cudaMalloc; this entry point instead uses a fixed scratch array that
// lives in the library's device image.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds it (kScratchBytes) until the process exits, and every call
// on a device shares it.  Each call clears the part it uses before the
// kernels run, so no state carries over from the previous call; calls whose
// work overlaps on the GPU (different streams, no ordering between them)
// race on the array and give wrong results.
//
// Host code may not use the array's name as a device address (in host code
// it is only a stand-in); the address comes from cudaGetSymbolAddress, taken
// once per device with that device current, on the first call made on the
// device.  Make that first call before any stream capture.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "hess.h"
#include "device_ptr.h"
#include "kernels.cuh"

namespace {

// 1,024 blocks of 16x16 fp64 (d <= 16,384) plus a 256-byte status area.
constexpr int kMaxBlocks = 1024;
constexpr size_t kAccBytes = static_cast<size_t>(kMaxBlocks) * 256 * sizeof(double);
constexpr size_t kScratchBytes = kAccBytes + 256;

static __device__ __align__(256) unsigned char g_local_scratch[kScratchBytes];

// The message is reported by hess_last_error() like every other call's.
hess_status noalloc_fail(hess_status s, const char* fmt, ...) {
    char buf[384];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    hk::set_last_error(buf);
    return s;
}

// Per-device set-up: kernel attributes and the device address of the
// scratch array.  Runs once per device, with that device current.
struct DeviceScratch {
    bool ready = false;
    void* ptr = nullptr;
    int sm_count = 0;
};

hess_status scratch_for_device(int dev, DeviceScratch& out) {
    static std::mutex mu;
    static DeviceScratch table[128];
    if (dev < 0 || dev >= 128) return noalloc_fail(HESS_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(mu);
    DeviceScratch& e = table[dev];
    if (!e.ready) {
        void* p = nullptr;
        cudaError_t err = cudaGetSymbolAddress(&p, g_local_scratch);
        if (err != cudaSuccess)
            return noalloc_fail(HESS_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed: %s",
                                cudaGetErrorString(err));
        err = hk::local_prepare();
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&e.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess)
            return noalloc_fail(HESS_ERR_CUDA, "no-alloc set-up failed: %s", cudaGetErrorString(err));
        e.ptr = p;
        e.ready = true;
    }
    out = e;
    return HESS_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn noalloc_encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) hess_status local_hess_compute_noalloc(
    const void* X, int64_t n_tokens, int64_t d, int32_t block, int32_t dtype, float* out,
    hess_stream_t stream) {
    if (n_tokens < 0) return noalloc_fail(HESS_ERR_INVALID, "n_tokens < 0");
    if (d <= 0) return noalloc_fail(HESS_ERR_INVALID, "d must be positive");
    if (!out) return noalloc_fail(HESS_ERR_INVALID, "out is NULL");
    if (block != 16) return noalloc_fail(HESS_ERR_UNSUPPORTED, "block must be 16 (got %d)", block);
    if (d % block != 0) return noalloc_fail(HESS_ERR_UNSUPPORTED, "d %% block != 0");
    if (d / block > kMaxBlocks)
        return noalloc_fail(HESS_ERR_UNSUPPORTED,
                            "d = %lld exceeds the no-alloc scratch limit of %d features",
                            static_cast<long long>(d), kMaxBlocks * 16);
    if (dtype != HESS_BF16) {
        if (dtype == HESS_F32) return noalloc_fail(HESS_ERR_UNSUPPORTED, "bf16 input only");
        return noalloc_fail(HESS_ERR_INVALID, "unknown dtype %d", dtype);
    }
    if (n_tokens > 0 && !X) return noalloc_fail(HESS_ERR_INVALID, "X is NULL with n_tokens > 0");
    if (n_tokens > 0 && reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return noalloc_fail(HESS_ERR_INVALID, "X is not 16-byte aligned");
    if (n_tokens > (int64_t(1) << 31) - hk::kLocalKBlock)
        return noalloc_fail(HESS_ERR_UNSUPPORTED, "n_tokens too large");
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return noalloc_fail(HESS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
    char why[128];
    if (const char* w = hk::device_ptr_problem(out, dev, why)) return noalloc_fail(HESS_ERR_INVALID, "out %s", w);
    if (n_tokens > 0)
        if (const char* w = hk::device_ptr_problem(X, dev, why)) return noalloc_fail(HESS_ERR_INVALID, "X %s", w);
    DeviceScratch sc;
    hess_status st = scratch_for_device(dev, sc);
    if (st != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n_blocks = static_cast<int>(d / block);
    const size_t out_bytes = static_cast<size_t>(n_blocks) * 256 * sizeof(float);
    if (n_tokens == 0) {
        err = cudaMemsetAsync(out, 0, out_bytes, s);
        return err == cudaSuccess ? HESS_OK
                                  : noalloc_fail(HESS_ERR_CUDA, "memset: %s", cudaGetErrorString(err));
    }
    double* acc = static_cast<double*>(sc.ptr);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(sc.ptr) + kAccBytes);
    // The previous call's sums are still in the array: clear what this call uses.
    err = cudaMemsetAsync(acc, 0, static_cast<size_t>(n_blocks) * 256 * sizeof(double), s);
    if (err == cudaSuccess) err = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
    if (err != cudaSuccess) return noalloc_fail(HESS_ERR_CUDA, "memset: %s", cudaGetErrorString(err));

    EncodeTiledFn enc = noalloc_encode_fn();
    if (!enc) return noalloc_fail(HESS_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    err = hk::ensure_context();
    if (err != cudaSuccess) return noalloc_fail(HESS_ERR_CUDA, "context: %s", cudaGetErrorString(err));
    hk::LocalParams p;
    std::memset(&p, 0, sizeof(p));
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n_tokens)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(hk::kLocalKBlock)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&p.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return noalloc_fail(HESS_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    p.acc = acc;
    p.status = status;
    p.timeout_ns = 2000000000ull;
    p.d = static_cast<int32_t>(d);
    p.n_groups = static_cast<int32_t>((d + hk::kLocalGroup - 1) / hk::kLocalGroup);
    p.total_kb = static_cast<int32_t>((n_tokens + hk::kLocalKBlock - 1) / hk::kLocalKBlock);
    const int64_t want = (2 * static_cast<int64_t>(sc.sm_count) + p.n_groups - 1) / p.n_groups;
    p.n_ranges = static_cast<int32_t>(want < 1 ? 1 : (want > p.total_kb ? p.total_kb : want));
    p.chunk_steps = 8;
    err = hk::launch_local_gram(p, p.n_groups * p.n_ranges, s);
    if (err == cudaSuccess)
        err = hk::launch_local_read(acc, out, n_blocks, 2.0 / static_cast<double>(n_tokens), s);
    if (err != cudaSuccess) return noalloc_fail(HESS_ERR_CUDA, "launch: %s", cudaGetErrorString(err));
    return HESS_OK;
}
