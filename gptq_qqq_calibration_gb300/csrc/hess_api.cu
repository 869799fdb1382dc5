// Host side of the C ABI declared in include/hess.h: handles, argument
// validation, the ragged-batch queue, tensor-map encoding and launches.
//
// Queue: hess_add_batch only records (pointer, tokens, stream).  A flush
// turns every queued batch of one dtype into one tensor map, concatenates
// their tokens into one stream of 128-token k-blocks and runs a single
// split-K SYRK pass over it, so the accumulator is read and written once per
// flush instead of once per batch (GPTQModel PR #2981, Changes: no transient
// d x d product per batch; the accumulator is allocated once).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "device_ptr.h"
#include "hess.h"
#include "kernels.cuh"
#include "schedule.cuh"

#define HESS_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_last_error;

hess_status fail(hess_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

#define CUDA_TRY(call)                                                                         \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return fail(HESS_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));        \
    } while (0)

// Host-side fault injection for tests: HESS_FAULT=alloc makes the *_create
// calls fail as if out of memory; HESS_FAULT=encode makes every tensor-map
// encoding fail as if the driver refused the descriptor.
bool injected(const char* what) {
    const char* f = std::getenv("HESS_FAULT");
    return f && std::strcmp(f, what) == 0;
}
bool injected_alloc_failure() { return injected("alloc"); }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// 2-D row-major [rows, cols] tensor map with a 128-byte-swizzled box of
// box_cols x box_rows elements; reads past the edges return zeros.
hess_status encode_2d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, size_t elem,
                      int64_t cols, int64_t rows, uint32_t box_cols, uint32_t box_rows,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(HESS_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    if (injected("encode")) return fail(HESS_ERR_UNSUPPORTED, "injected tensor-map failure (HESS_FAULT=encode)");
    CUDA_TRY(hk::ensure_context());
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(HESS_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d) for [%lld, %lld]",
                    static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(cols));
    return HESS_OK;
}

// Per-device one-time kernel set-up (dynamic shared-memory limits, how many
// SM pairs the pair kernel can keep resident).
hess_status prepare_device(int dev, int* max_pairs) {
    static std::mutex mu;
    static bool done[128] = {};
    static int pairs[128] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 128) return fail(HESS_ERR_UNSUPPORTED, "device index %d", dev);
    if (!done[dev]) {
        CUDA_TRY(hk::syrk_bf16_prepare());
        CUDA_TRY(hk::syrk_bf16_2sm_prepare(&pairs[dev]));
        CUDA_TRY(hk::syrk_f32_prepare());
        CUDA_TRY(hk::local_prepare());
        done[dev] = true;
    }
    if (max_pairs) *max_pairs = pairs[dev];
    return HESS_OK;
}


int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The handle's device status block: word 0 the status bits the kernels OR
// in, words 8..11 the state-blob trailer staged for a copy.
constexpr size_t kStatusBytes = 64;

// Largest single batch whose X a flush prefetches into L2 (a small fraction
// of the 129 MB L2, so it displaces little of the accumulator).
constexpr uint64_t kL2PrefetchMaxBytes = 32ull << 20;

}  // namespace

struct hess_ctx {
    std::mutex mu;
    int device = 0;
    int64_t d = 0;
    int T = 0;
    int n_tiles = 0;
    int sm_count = 0;
    float* acc = nullptr;  // (hi, lo) planes per upper tile
    uint32_t* status = nullptr;
    double* damp64 = nullptr;  // the damping value, then materialize's scratch
    float* damp32 = nullptr;
    cudaEvent_t ev = nullptr;
    // Pinned, mapped host copy of the status word (word 0) and of the damping
    // value (word 1), written by the materialize kernel itself (or by a copy
    // when N == 0).  The next call on the handle reads it once ev_status has
    // completed, without waiting.
    uint32_t* status_host = nullptr;
    uint32_t* status_host_dev = nullptr;  // its device address
    cudaEvent_t ev_status = nullptr;
    bool status_copy_pending = false;
    uint32_t fault = 0;  // a recorded device status word seen on the host (until reset)
    // The accumulator's last user: work on another stream waits for it
    // (flushes may read-modify-write tiles without atomics).
    cudaEvent_t ev_acc = nullptr;
    cudaStream_t acc_stream = nullptr;
    bool acc_used = false;
    int64_t N = 0;
    int64_t kernels = 0;  // kernel launches made for this handle (hess_kernel_launches)
    struct Pending {
        const void* ptr;
        int64_t n;
        cudaStream_t stream;
    };
    std::vector<Pending> pending;
    int32_t pending_dtype = -1;
    int64_t pending_tokens = 0;
    // options
    int64_t flush_tokens = 65536;
    int max_pending = hk::kMaxBatches;
    int chunk_tokens = 384;
    unsigned long long timeout_ns = 2000000000ull;
    int split_k = 0;
    int grid = 0;
    int pair_kernel = 0;  // bf16: 1 = pairs of SMs (256 x 128 tiles), 0 = one SM per tile
    int fold_every = 8;   // single-slab flushes per kAccPair flush (the others are kAccLo)
    int overlap = 1;      // launch flushes with programmatic stream serialization
    int lo_flushes = 0;   // kAccLo flushes since lo was last folded into hi
    int max_pairs = 0;
    hk::SyrkParams* params = nullptr;  // host staging of the launch parameters
};

struct local_hess_ctx {
    std::mutex mu;
    int device = 0;
    int64_t d = 0;
    int block = 16;
    int n_blocks = 0;
    int sm_count = 0;
    double* acc = nullptr;
    uint32_t* status = nullptr;
    int64_t N = 0;
    unsigned long long timeout_ns = 2000000000ull;
};

namespace {

hess_status check_device(int dev) {
    int cur = -1;
    CUDA_TRY(cudaGetDevice(&cur));
    if (cur != dev)
        return fail(HESS_ERR_INVALID, "handle belongs to device %d but device %d is current", dev, cur);
    return HESS_OK;
}

// A caller's buffer must be device memory of the handle's device (or
// managed memory); anything else is refused before a kernel could touch it.
hess_status check_buffer(const void* p, int dev, const char* name) {
    char why[128];
    if (const char* w = hk::device_ptr_problem(p, dev, why)) return fail(HESS_ERR_INVALID, "%s %s", name, w);
    return HESS_OK;
}

// Split-K factor (token slabs) from a per-unit cost model in SM cycles:
// each unit costs max(MMA, epilogue), waves of units run back to back.  The
// MMA part is ~4.7 cycles per token of a 128 x 128 tile; the epilogue writes
// a 128 KB (hi, lo) tile back: a plain read-modify-write with one slab (one
// writer per tile), compensated atomics with several, which cost about three
// times as much.  Small flushes are epilogue-bound and take one slab; large
// ones split to fill the waves.  Ties go to fewer slabs.
int choose_slabs(int n_tiles, int total_kb, int kb_tokens, int grid) {
    const int smax = std::max(1, std::min(64, total_kb));
    int best = 1;
    double best_cost = 0.0;
    for (int S = 1; S <= smax; ++S) {
        const long long units = static_cast<long long>(n_tiles) * S;
        const long long waves = (units + grid - 1) / grid;
        const double mma = 4.7 * kb_tokens * std::ceil(static_cast<double>(total_kb) / S);
        const double epi = S == 1 ? 12000.0 : 36000.0;
        const double cost = static_cast<double>(waves) * std::max(mma, epi);
        if (S == 1 || cost < best_cost * 0.98) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

// Order work on `s` after the accumulator's last user on another stream,
// and record `s` as its user.
hess_status order_acc(hess_ctx* h, cudaStream_t s) {
    if (h->acc_used && h->acc_stream != s) CUDA_TRY(cudaStreamWaitEvent(s, h->ev_acc, 0));
    return HESS_OK;
}
hess_status mark_acc(hess_ctx* h, cudaStream_t s) {
    CUDA_TRY(cudaEventRecord(h->ev_acc, s));
    h->acc_stream = s;
    h->acc_used = true;
    return HESS_OK;
}

// Write-back mode of the next flush.  A single-slab flush usually adds to
// the lo plane alone (kAccLo: 8 bytes per accumulator element instead of
// 16); every fold_every-th one adds to both planes (kAccPair), which also
// folds lo back into hi.  lo then never holds more than fold_every - 1
// undigested flush sums, each added with one fp32 rounding of at most
// (fold_every - 1) flushes' magnitude: relative to H, unbiased errors of
// about 2^-24 (fold_every / flushes)^(1/2) per entry.  Split-K flushes add
// compensated atomics to both planes and leave the count as it is.
int32_t next_acc_mode(hess_ctx* h, int exclusive) {
    if (!exclusive) return hk::kAccPair;
    if (h->lo_flushes + 1 < h->fold_every) {
        ++h->lo_flushes;
        return hk::kAccLo;
    }
    h->lo_flushes = 0;
    return hk::kAccPair;
}

hess_status flush_locked(hess_ctx* h, cudaStream_t stream) {
    if (h->pending.empty()) return HESS_OK;
    // Order the flush after the work that produced every queued batch.
    for (size_t i = 0; i < h->pending.size(); ++i) {
        cudaStream_t s = h->pending[i].stream;
        if (s == stream) continue;
        bool seen = false;
        for (size_t k = 0; k < i; ++k) seen |= h->pending[k].stream == s;
        if (seen) continue;
        CUDA_TRY(cudaEventRecord(h->ev, s));
        CUDA_TRY(cudaStreamWaitEvent(stream, h->ev, 0));
    }
    hk::SyrkParams& p = *h->params;
    const bool f32 = h->pending_dtype == HESS_F32;
    const int nb = static_cast<int>(h->pending.size());
    p.kb_start[0] = 0;
    const int kblock = f32 ? hk::kKBlockF32 : hk::kKBlock;
    for (int b = 0; b < nb; ++b) {
        const auto& q = h->pending[b];
        hess_status st =
            f32 ? encode_2d(&p.maps[b], q.ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, h->d, q.n, 32,
                            hk::kKBlockF32, hk::kF32Swizzle)
                : encode_2d(&p.maps[b], q.ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h->d, q.n, 64,
                            hk::kKBlock);
        if (st != HESS_OK) return st;
        p.kb_start[b + 1] = p.kb_start[b] + static_cast<int32_t>(ceil_div(q.n, kblock));
    }
    p.n_batches = nb;
    p.total_kb = p.kb_start[nb];
    p.n_tiles = h->n_tiles;
    p.tiles_per_dim = h->T;
    // fp32 input has a 5x tighter bound and 2x more MMA steps per token, so
    // its chains are 6x shorter in tokens (64 at the default chunk: on the
    // log-uniform d=4096 stream, 2.9e-6 of the mean diagonal, against 1.7e-6
    // at 32 tokens for 13 % less speed).
    p.chunk_kb = f32 ? std::max(1, h->chunk_tokens / 6 / hk::kKBlockF32)
                     : std::max(1, h->chunk_tokens / hk::kKBlock);
    p.d = static_cast<int32_t>(h->d);
    p.acc = h->acc;
    {
        hess_status st = order_acc(h, stream);
        if (st != HESS_OK) return st;
    }
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    // A flush of one bf16 batch that fits L2 many times over (the flush-per-call
    // regime) has its X prefetched into L2 by the CTAs before the grid wait, so
    // the first wave's loads do not wait on DRAM.
    p.l2_ptr = nullptr;
    p.l2_bytes = 0;
    if (!f32 && nb == 1) {
        const uint64_t bytes = static_cast<uint64_t>(h->pending[0].n) * static_cast<uint64_t>(h->d) * 2u;
        if (bytes <= kL2PrefetchMaxBytes) {
            p.l2_ptr = h->pending[0].ptr;
            p.l2_bytes = bytes;
        }
    }
    const bool pairs = !f32 && h->pair_kernel && h->max_pairs > 0;
    int grid = 0;
    cudaError_t e;
    if (pairs) {
        p.n_tiles = hk::pair_tile_count(h->T);
        const int pairs_max = h->grid > 0 ? std::max(1, h->grid / 2) : h->max_pairs;
        p.n_slabs = h->split_k > 0 ? std::min(h->split_k, p.total_kb)
                                   : choose_slabs(p.n_tiles, p.total_kb, hk::kKBlock, pairs_max);
        p.n_units = p.n_tiles * p.n_slabs;
        p.exclusive = p.n_slabs == 1 ? 1 : 0;
        p.acc_mode = next_acc_mode(h, p.exclusive);
        p.tail_split = 0;
        grid = 2 * std::min(pairs_max, p.n_units);
        e = hk::launch_syrk_bf16_2sm(p, grid, stream, h->overlap != 0);
        ++h->kernels;
    } else {
        const int grid_max = h->grid > 0 ? h->grid : h->sm_count;
        p.n_slabs = h->split_k > 0 ? std::min(h->split_k, p.total_kb)
                                   : choose_slabs(h->n_tiles, p.total_kb, kblock, grid_max);
        if (!f32 && h->split_k == 0 && p.n_slabs > 1 && h->fold_every > 1) {
            // A large bf16 flush runs as one slab that adds to the low part
            // with L2 reductions, its last wave split in halves
            // (tail_split_for): the waves stay balanced without split-K's
            // compensated atomics on both parts.  A fold that is due goes
            // first, as its own pass over the accumulator.  (The fp32
            // kernel, bound by its converters, measured 2 % faster with
            // split-K, and keeps it.)
            if (h->lo_flushes + 1 >= h->fold_every) {
                CUDA_TRY(hk::launch_renorm_pairs(h->acc, static_cast<size_t>(h->n_tiles), h->sm_count, stream));
                ++h->kernels;
                h->lo_flushes = 0;
            }
            p.n_slabs = 1;
        }
        p.n_units = p.n_tiles * p.n_slabs;
        p.exclusive = p.n_slabs == 1 ? 1 : 0;
        p.acc_mode = next_acc_mode(h, p.exclusive);
        p.tail_split = hk::syrk::tail_split_for(p.n_tiles, grid_max, p.total_kb, p.exclusive != 0, p.acc_mode);
        p.n_units += p.tail_split;
        grid = std::min(grid_max, p.n_units);
        e = f32 ? hk::launch_syrk_f32(p, grid, stream, h->overlap != 0)
                : hk::launch_syrk_bf16(p, grid, stream, h->overlap != 0);
        ++h->kernels;
    }
    h->pending.clear();
    h->pending_tokens = 0;
    h->pending_dtype = -1;
    if (e != cudaSuccess) return fail(HESS_ERR_CUDA, "SYRK launch failed: %s", cudaGetErrorString(e));
    {
        hess_status st = mark_acc(h, stream);
        if (st != HESS_OK) return st;
    }
    if (std::getenv("HESS_TRACE"))
        std::fprintf(stderr, "[hess] flush d=%lld batches=%d kblocks=%d slabs=%d%s grid=%d %s (max pairs %d)\n",
                     static_cast<long long>(h->d), nb, p.total_kb, p.n_slabs,
                     p.exclusive ? (p.acc_mode == hk::kAccLo ? " (exclusive, lo)" : " (exclusive, pair)") : "", grid,
                     f32 ? "f32" : (pairs ? "bf16-pairs" : "bf16"), h->max_pairs);
    return HESS_OK;
}

// The error a nonzero device status word stands for: an index guard that
// failed (HESS_ERR_INTERNAL) before a wait that ran out (HESS_ERR_TIMEOUT).
hess_status status_error(uint32_t st, const char* when) {
    if (st & hk::kStatusBadIndex)
        return fail(HESS_ERR_INTERNAL, "a kernel index guard failed%s (status 0x%x); hess_reset clears it", when, st);
    return fail(HESS_ERR_TIMEOUT, "a device-side wait ran out%s (status 0x%x); hess_reset clears it", when, st);
}

// A device status recorded earlier and already visible on the host (from the
// status copy of an earlier hess_materialize) fails the call.
hess_status check_reported(hess_ctx* h) {
    if (h->status_copy_pending && cudaEventQuery(h->ev_status) == cudaSuccess) {
        h->status_copy_pending = false;
        h->fault |= *reinterpret_cast<volatile uint32_t*>(h->status_host);
    }
    if (h->fault) return status_error(h->fault, " in an earlier call");
    return HESS_OK;
}

hess_status read_status(uint32_t* dev_status, cudaStream_t stream, uint32_t* seen = nullptr) {
    uint32_t st = 0;
    CUDA_TRY(cudaMemcpyAsync(&st, dev_status, sizeof(st), cudaMemcpyDeviceToHost, stream));
    CUDA_TRY(cudaStreamSynchronize(stream));
    if (seen) *seen |= st;
    if (st != 0) return status_error(st, "");
    return HESS_OK;
}

}  // namespace

// ------------------------------------------------------------------ full H

HESS_EXPORT hess_status hess_create(int64_t d, hess_t* out) {
    if (!out) return fail(HESS_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d <= 0) return fail(HESS_ERR_INVALID, "d must be positive (got %lld)", (long long)d);
    if (d > 32768) return fail(HESS_ERR_UNSUPPORTED, "d = %lld exceeds 32768", (long long)d);
    if (d % 8 != 0) return fail(HESS_ERR_UNSUPPORTED, "d = %lld is not a multiple of 8", (long long)d);
    if (injected_alloc_failure()) return fail(HESS_ERR_OOM, "injected allocation failure (HESS_FAULT=alloc)");
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    int max_pairs = 0;
    hess_status st = prepare_device(dev, &max_pairs);
    if (st != HESS_OK) return st;
    hess_ctx* h = new (std::nothrow) hess_ctx();
    if (!h) return fail(HESS_ERR_OOM, "host allocation failed");
    h->params = new (std::nothrow) hk::SyrkParams();
    if (!h->params) {
        delete h;
        return fail(HESS_ERR_OOM, "host allocation failed");
    }
    h->device = dev;
    h->max_pairs = max_pairs;
    h->d = d;
    h->T = static_cast<int>(ceil_div(d, hk::kTile));
    h->n_tiles = h->T * (h->T + 1) / 2;
    cudaError_t e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
    // The status block sits right after the accumulator tiles, so that one
    // memset clears both in hess_reset.
    const size_t acc_bytes = static_cast<size_t>(h->n_tiles) * hk::kTileWords * sizeof(float);
    if (e == cudaSuccess) e = cudaMalloc(&h->acc, acc_bytes + kStatusBytes);
    if (e == cudaSuccess) h->status = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(h->acc) + acc_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&h->damp64, hk::materialize_scratch_bytes(h->T));
    if (e == cudaSuccess) e = cudaMalloc(&h->damp32, sizeof(float));
    if (e == cudaSuccess) e = cudaMemset(h->acc, 0, acc_bytes + kStatusBytes);
    if (e == cudaSuccess) e = cudaMemset(h->damp64, 0, hk::materialize_scratch_bytes(h->T));
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_acc, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_status, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaHostAlloc(&h->status_host, 64, cudaHostAllocMapped);
    if (e == cudaSuccess) std::memset(h->status_host, 0, 64);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->status_host_dev), h->status_host, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        hess_status s = e == cudaErrorMemoryAllocation ? HESS_ERR_OOM : HESS_ERR_CUDA;
        cudaFree(h->acc);
        cudaFree(h->damp64);
        cudaFree(h->damp32);
        if (h->status_host) cudaFreeHost(h->status_host);
        if (h->ev) cudaEventDestroy(h->ev);
        if (h->ev_acc) cudaEventDestroy(h->ev_acc);
        if (h->ev_status) cudaEventDestroy(h->ev_status);
        delete h->params;
        delete h;
        return fail(s, "hess_create: %s", cudaGetErrorString(e));
    }
    *out = h;
    return HESS_OK;
}

HESS_EXPORT hess_status hess_add_batch(hess_t h, const void* X, int64_t n_tokens, int32_t dtype,
                                       hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (n_tokens < 0) return fail(HESS_ERR_INVALID, "n_tokens < 0");
    if (dtype != HESS_BF16 && dtype != HESS_F32) return fail(HESS_ERR_INVALID, "unknown dtype %d", dtype);
    if (n_tokens == 0) return HESS_OK;  // empty batch: no-op, N unchanged
    if (!X) return fail(HESS_ERR_INVALID, "X is NULL with n_tokens > 0");
    if (reinterpret_cast<uintptr_t>(X) % 16 != 0) return fail(HESS_ERR_INVALID, "X is not 16-byte aligned");
    if (n_tokens > (int64_t(1) << 31) - hk::kKBlock)
        return fail(HESS_ERR_UNSUPPORTED, "n_tokens exceeds 2^31 - %d in one batch", hk::kKBlock);
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_reported(h)) != HESS_OK) return st;
    if ((st = check_buffer(X, h->device, "X")) != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!h->pending.empty()) {
        const int64_t kb_now = ceil_div(n_tokens, hk::kKBlock);
        int64_t kb_pending = 0;
        for (const auto& q : h->pending) kb_pending += ceil_div(q.n, hk::kKBlock);
        if (dtype != h->pending_dtype || kb_pending + kb_now > (int64_t(1) << 30)) {
            st = flush_locked(h, s);
            if (st != HESS_OK) return st;
        }
    }
    h->pending.push_back({X, n_tokens, s});
    h->pending_dtype = dtype;
    h->pending_tokens += n_tokens;
    h->N += n_tokens;
    if (static_cast<int>(h->pending.size()) >= h->max_pending || h->pending_tokens >= h->flush_tokens) {
        st = flush_locked(h, s);
        if (st != HESS_OK && !h->pending.empty()) {
            // The flush failed before launching: this call leaves no trace
            // (the batch is neither queued nor counted); earlier batches stay
            // queued for the next flush.
            h->pending.pop_back();
            h->pending_tokens -= n_tokens;
            h->N -= n_tokens;
            if (h->pending.empty()) h->pending_dtype = -1;
        }
        return st;
    }
    return HESS_OK;
}

HESS_EXPORT hess_status hess_flush(hess_t h, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_reported(h)) != HESS_OK) return st;
    return flush_locked(h, static_cast<cudaStream_t>(stream));
}

HESS_EXPORT hess_status hess_materialize(hess_t h, float* H_out, double damp_percent,
                                         hess_stream_t stream, float* damp_value_out) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (!H_out) return fail(HESS_ERR_INVALID, "H_out is NULL");
    if (reinterpret_cast<uintptr_t>(H_out) % 16 != 0) return fail(HESS_ERR_INVALID, "H_out is not 16-byte aligned");
    if (!(damp_percent >= 0.0 && damp_percent < 1.0))
        return fail(HESS_ERR_INVALID, "damp_percent must be in [0, 1)");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_reported(h)) != HESS_OK) return st;
    if ((st = check_buffer(H_out, h->device, "H_out")) != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = flush_locked(h, s);
    if (st != HESS_OK) return st;
    if (h->N == 0) {
        CUDA_TRY(cudaMemsetAsync(H_out, 0, static_cast<size_t>(h->d) * h->d * sizeof(float), s));
        if (damp_value_out) {
            *damp_value_out = 0.0f;
            return read_status(h->status, s, &h->fault);
        }
        // the status word travels to the pinned host copy behind this work
        CUDA_TRY(cudaMemcpyAsync(h->status_host, h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    } else {
        const double scale = 2.0 / static_cast<double>(h->N);
        if ((st = order_acc(h, s)) != HESS_OK) return st;
        CUDA_TRY(hk::launch_materialize(h->acc, H_out, static_cast<int>(h->d), h->T, scale, damp_percent,
                                        h->damp64, h->damp32, h->status, h->status_host_dev, s));
        ++h->kernels;
        if ((st = mark_acc(h, s)) != HESS_OK) return st;
    }
    CUDA_TRY(cudaEventRecord(h->ev_status, s));
    if (damp_value_out) {
        // the kernel wrote the status word and the damping value to the
        // pinned host copy: wait for it, then read both there
        CUDA_TRY(cudaEventSynchronize(h->ev_status));
        h->status_copy_pending = false;
        const volatile uint32_t* m = h->status_host;
        h->fault |= m[0];
        if (m[0] != 0) return status_error(m[0], "");
        uint32_t bits = m[1];
        float v;
        std::memcpy(&v, &bits, sizeof(v));
        *damp_value_out = v;
        return HESS_OK;
    }
    // No wait here: a later call reports a timeout the host copy shows.
    h->status_copy_pending = true;
    return HESS_OK;
}

HESS_EXPORT int64_t hess_token_count(hess_t h) {
    if (!h) return -1;
    std::lock_guard<std::mutex> lk(h->mu);
    return h->N;
}

HESS_EXPORT int64_t hess_kernel_launches(hess_t h) {
    if (!h) return -1;
    std::lock_guard<std::mutex> lk(h->mu);
    return h->kernels;
}

HESS_EXPORT int64_t hess_pending_batches(hess_t h) {
    if (!h) return -1;
    std::lock_guard<std::mutex> lk(h->mu);
    return static_cast<int64_t>(h->pending.size());
}

HESS_EXPORT int64_t hess_dim(hess_t h) { return h ? h->d : -1; }

HESS_EXPORT hess_status hess_sync(hess_t h, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    return read_status(h->status, static_cast<cudaStream_t>(stream), &h->fault);
}

HESS_EXPORT hess_status hess_reset(hess_t h, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->pending.clear();
    h->pending_tokens = 0;
    h->pending_dtype = -1;
    h->N = 0;
    h->lo_flushes = 0;
    h->fault = 0;
    h->status_copy_pending = false;
    if ((st = order_acc(h, s)) != HESS_OK) return st;
    // the tiles and the status block after them, in one memset
    CUDA_TRY(cudaMemsetAsync(h->acc, 0,
                             static_cast<size_t>(h->n_tiles) * hk::kTileWords * sizeof(float) + kStatusBytes, s));
    return mark_acc(h, s);
}

HESS_EXPORT hess_status hess_set_option(hess_t h, int32_t option, int64_t value) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    switch (option) {
        case HESS_OPT_FLUSH_TOKENS:
            if (value < 1) return fail(HESS_ERR_INVALID, "flush_tokens must be >= 1");
            h->flush_tokens = value;
            return HESS_OK;
        case HESS_OPT_MAX_PENDING:
            if (value < 1 || value > hk::kMaxBatches)
                return fail(HESS_ERR_INVALID, "max_pending must be in [1, %d]", hk::kMaxBatches);
            h->max_pending = static_cast<int>(value);
            return HESS_OK;
        case HESS_OPT_CHUNK_TOKENS:
            if (value < hk::kKBlock || value > 65536 || value % hk::kKBlock)
                return fail(HESS_ERR_INVALID, "chunk_tokens must be a multiple of %d in [%d, 65536]",
                            hk::kKBlock, hk::kKBlock);
            h->chunk_tokens = static_cast<int>(value);
            return HESS_OK;
        case HESS_OPT_WAIT_TIMEOUT_NS:
            if (value < 0) return fail(HESS_ERR_INVALID, "timeout must be >= 0");
            h->timeout_ns = static_cast<unsigned long long>(value);
            return HESS_OK;
        case HESS_OPT_SPLIT_K:
            if (value < 0 || value > 4096) return fail(HESS_ERR_INVALID, "split_k must be in [0, 4096]");
            h->split_k = static_cast<int>(value);
            return HESS_OK;
        case HESS_OPT_GRID:
            if (value < 0 || value > 65535) return fail(HESS_ERR_INVALID, "grid must be in [0, 65535]");
            h->grid = static_cast<int>(value);
            return HESS_OK;
        case HESS_OPT_PAIR_KERNEL:
            if (value != 0 && value != 1) return fail(HESS_ERR_INVALID, "pair_kernel must be 0 or 1");
            h->pair_kernel = static_cast<int>(value);
            return HESS_OK;
        case HESS_OPT_OVERLAP_LAUNCHES:
            if (value != 0 && value != 1) return fail(HESS_ERR_INVALID, "overlap_launches must be 0 or 1");
            h->overlap = static_cast<int>(value);
            return HESS_OK;
        case HESS_OPT_FOLD_EVERY:
            if (value < 1 || value > 64) return fail(HESS_ERR_INVALID, "fold_every must be in [1, 64]");
            h->fold_every = static_cast<int>(value);
            h->lo_flushes = std::min(h->lo_flushes, h->fold_every - 1);
            return HESS_OK;
        default:
            return fail(HESS_ERR_INVALID, "unknown option %d", option);
    }
}

HESS_EXPORT hess_status hess_destroy(hess_t h) {
    if (!h) return HESS_OK;
    {
        std::lock_guard<std::mutex> lk(h->mu);
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(h->device);
        cudaDeviceSynchronize();
        cudaFree(h->acc);
        cudaFree(h->damp64);
        cudaFree(h->damp32);
        cudaFreeHost(h->status_host);
        cudaEventDestroy(h->ev);
        cudaEventDestroy(h->ev_acc);
        cudaEventDestroy(h->ev_status);
        cudaSetDevice(cur);
    }
    delete h->params;
    delete h;
    return HESS_OK;
}

// ------------------------------------------------- merge and clone (f2, f4)

HESS_EXPORT hess_status hess_merge(hess_t dst, hess_t src, hess_stream_t stream) {
    if (!dst || !src) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (dst == src) return fail(HESS_ERR_INVALID, "cannot merge a handle into itself");
    if (dst->d != src->d) return fail(HESS_ERR_INVALID, "widths differ (%lld vs %lld)",
                                      (long long)dst->d, (long long)src->d);
    if (dst->device != src->device)
        return fail(HESS_ERR_UNSUPPORTED, "handles live on different devices");
    // Lock in address order so that two merges in opposite directions cannot deadlock.
    std::mutex& m1 = dst < src ? dst->mu : src->mu;
    std::mutex& m2 = dst < src ? src->mu : dst->mu;
    std::lock_guard<std::mutex> l1(m1);
    std::lock_guard<std::mutex> l2(m2);
    hess_status st = check_device(dst->device);
    if (st != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = flush_locked(src, s)) != HESS_OK) return st;
    if ((st = flush_locked(dst, s)) != HESS_OK) return st;
    if ((st = order_acc(src, s)) != HESS_OK || (st = order_acc(dst, s)) != HESS_OK) return st;
    CUDA_TRY(hk::launch_add_pairs(dst->acc, src->acc, static_cast<size_t>(dst->n_tiles), dst->sm_count, s));
    ++dst->kernels;
    if ((st = mark_acc(src, s)) != HESS_OK || (st = mark_acc(dst, s)) != HESS_OK) return st;
    dst->N += src->N;
    dst->lo_flushes = 0;  // the merge leaves dst's pairs renormalised
    return HESS_OK;
}

HESS_EXPORT hess_status hess_clone(hess_t src, hess_t* out, hess_stream_t stream) {
    if (!out) return fail(HESS_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (!src) return fail(HESS_ERR_INVALID, "handle is NULL");
    {
        std::lock_guard<std::mutex> lk(src->mu);
        hess_status st = check_device(src->device);
        if (st != HESS_OK) return st;
    }
    // The new handle is created before src is locked (create synchronises
    // the device); the flush, the copy and the token count are then taken
    // under one hold of src's mutex, so a batch another thread adds to src
    // meanwhile is either in both the copied sums and N or in neither.
    hess_t h = nullptr;
    hess_status st = hess_create(src->d, &h);
    if (st != HESS_OK) return st;
    std::lock_guard<std::mutex> lk(src->mu);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = static_cast<size_t>(src->n_tiles) * hk::kTileWords * sizeof(float);
    if ((st = flush_locked(src, s)) != HESS_OK || (st = order_acc(src, s)) != HESS_OK) {
        hess_destroy(h);
        return st;
    }
    cudaError_t e = cudaMemcpyAsync(h->acc, src->acc, bytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaEventRecord(src->ev_acc, s);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_acc, s);
    if (e != cudaSuccess) {
        hess_destroy(h);
        return fail(HESS_ERR_CUDA, "clone copy failed: %s", cudaGetErrorString(e));
    }
    src->acc_stream = h->acc_stream = s;
    src->acc_used = h->acc_used = true;
    h->N = src->N;
    h->flush_tokens = src->flush_tokens;
    h->max_pending = src->max_pending;
    h->chunk_tokens = src->chunk_tokens;
    h->timeout_ns = src->timeout_ns;
    h->split_k = src->split_k;
    h->grid = src->grid;
    h->pair_kernel = src->pair_kernel;
    h->fold_every = src->fold_every;
    h->overlap = src->overlap;
    h->lo_flushes = src->lo_flushes;
    *out = h;
    return HESS_OK;
}

// ------------------------------------------------------ checkpoint / resume

// A state blob is the accumulator tiles followed by a 16-byte trailer:
// {kStateMagic, HESS_ABI_VERSION, kAccLo flushes not yet folded, 0}.  The
// trailer is stored by a kernel into the handle's status block (words
// kTrailerWord..+3) and copied from there, in stream order.
constexpr uint32_t kStateMagic = 0x48535431u;  // "HST1"
constexpr int kTrailerWord = 8;

int64_t acc_bytes(const hess_ctx* h) {
    return static_cast<int64_t>(h->n_tiles) * hk::kTileWords * static_cast<int64_t>(sizeof(float));
}

HESS_EXPORT int64_t hess_state_bytes(hess_t h) {
    if (!h) return 0;
    return acc_bytes(h) + 16;
}

HESS_EXPORT hess_status hess_export_state(hess_t h, void* dst, int64_t bytes, hess_stream_t stream,
                                          int64_t* n_tokens_out) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (!dst || !n_tokens_out) return fail(HESS_ERR_INVALID, "dst or n_tokens_out is NULL");
    const int64_t need = hess_state_bytes(h);
    if (bytes < need)
        return fail(HESS_ERR_INVALID, "state needs %lld bytes, got %lld", static_cast<long long>(need),
                    static_cast<long long>(bytes));
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = flush_locked(h, s)) != HESS_OK) return st;
    if ((st = order_acc(h, s)) != HESS_OK) return st;
    const size_t ab = static_cast<size_t>(acc_bytes(h));
    CUDA_TRY(cudaMemcpyAsync(dst, h->acc, ab, cudaMemcpyDefault, s));
    uint32_t* trailer = h->status + kTrailerWord;
    CUDA_TRY(hk::launch_store_words(trailer, kStateMagic, HESS_ABI_VERSION,
                                    static_cast<uint32_t>(h->lo_flushes), 0u, s));
    CUDA_TRY(cudaMemcpyAsync(static_cast<char*>(dst) + ab, trailer, 16, cudaMemcpyDefault, s));
    if ((st = mark_acc(h, s)) != HESS_OK) return st;
    *n_tokens_out = h->N;
    return HESS_OK;
}

HESS_EXPORT hess_status hess_import_state(hess_t h, const void* src, int64_t bytes, int64_t n_tokens,
                                          hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (!src) return fail(HESS_ERR_INVALID, "src is NULL");
    if (n_tokens < 0) return fail(HESS_ERR_INVALID, "n_tokens < 0");
    const int64_t need = hess_state_bytes(h);
    if (bytes != need)
        return fail(HESS_ERR_INVALID, "state of %lld bytes for a handle that holds %lld",
                    static_cast<long long>(bytes), static_cast<long long>(need));
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the trailer first (the call waits for it): it must name this library
    const size_t ab = static_cast<size_t>(acc_bytes(h));
    CUDA_TRY(cudaMemcpyAsync(h->status_host + kTrailerWord, static_cast<const char*>(src) + ab, 16,
                             cudaMemcpyDefault, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    const volatile uint32_t* tr = h->status_host + kTrailerWord;
    if (tr[0] != kStateMagic || tr[1] != HESS_ABI_VERSION || tr[2] > 64u)
        return fail(HESS_ERR_INVALID, "src is not a state blob of this library version");
    h->pending.clear();
    h->pending_tokens = 0;
    h->pending_dtype = -1;
    h->fault = 0;
    h->status_copy_pending = false;
    h->lo_flushes = std::min(static_cast<int>(tr[2]), h->fold_every - 1);
    if ((st = order_acc(h, s)) != HESS_OK) return st;
    CUDA_TRY(cudaMemcpyAsync(h->acc, src, ab, cudaMemcpyDefault, s));
    CUDA_TRY(cudaMemsetAsync(h->status, 0, kStatusBytes, s));
    h->N = n_tokens;
    return mark_acc(h, s);
}

// ----------------------------------------------------------- imatrix (f3)

struct imatrix_ctx {
    std::mutex mu;
    int device = 0;
    int64_t d = 0;
    int sm_count = 0;
    double* acc = nullptr;
    int64_t N = 0;
};

HESS_EXPORT hess_status imatrix_create(int64_t d, imatrix_t* out) {
    if (!out) return fail(HESS_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d <= 0) return fail(HESS_ERR_INVALID, "d must be positive");
    if (d % 8 != 0) return fail(HESS_ERR_UNSUPPORTED, "d = %lld is not a multiple of 8", (long long)d);
    if (d > (int64_t(1) << 24)) return fail(HESS_ERR_UNSUPPORTED, "d too large");
    if (injected_alloc_failure()) return fail(HESS_ERR_OOM, "injected allocation failure (HESS_FAULT=alloc)");
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    imatrix_ctx* h = new (std::nothrow) imatrix_ctx();
    if (!h) return fail(HESS_ERR_OOM, "host allocation failed");
    h->device = dev;
    h->d = d;
    cudaError_t e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaMalloc(&h->acc, d * sizeof(double));
    if (e == cudaSuccess) e = cudaMemset(h->acc, 0, d * sizeof(double));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        hess_status s = e == cudaErrorMemoryAllocation ? HESS_ERR_OOM : HESS_ERR_CUDA;
        cudaFree(h->acc);
        delete h;
        return fail(s, "imatrix_create: %s", cudaGetErrorString(e));
    }
    *out = h;
    return HESS_OK;
}

HESS_EXPORT hess_status imatrix_add(imatrix_t h, const void* X, int64_t n_tokens, int32_t dtype,
                                    hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (n_tokens < 0) return fail(HESS_ERR_INVALID, "n_tokens < 0");
    if (dtype != HESS_BF16 && dtype != HESS_F32) return fail(HESS_ERR_INVALID, "unknown dtype %d", dtype);
    if (n_tokens == 0) return HESS_OK;
    if (!X) return fail(HESS_ERR_INVALID, "X is NULL with n_tokens > 0");
    if (reinterpret_cast<uintptr_t>(X) % 16 != 0) return fail(HESS_ERR_INVALID, "X is not 16-byte aligned");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_buffer(X, h->device, "X")) != HESS_OK) return st;
    CUDA_TRY(hk::launch_colsumsq(X, dtype == HESS_F32, n_tokens, static_cast<int>(h->d), h->acc,
                                 h->sm_count, static_cast<cudaStream_t>(stream)));
    h->N += n_tokens;
    return HESS_OK;
}

HESS_EXPORT hess_status imatrix_read(imatrix_t h, float* out, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (!out) return fail(HESS_ERR_INVALID, "out is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_buffer(out, h->device, "out")) != HESS_OK) return st;
    CUDA_TRY(hk::launch_colsumsq_read(h->acc, out, static_cast<int>(h->d),
                                      static_cast<cudaStream_t>(stream)));
    return HESS_OK;
}

HESS_EXPORT int64_t imatrix_token_count(imatrix_t h) {
    if (!h) return -1;
    std::lock_guard<std::mutex> lk(h->mu);
    return h->N;
}

HESS_EXPORT hess_status imatrix_reset(imatrix_t h, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    h->N = 0;
    CUDA_TRY(cudaMemsetAsync(h->acc, 0, h->d * sizeof(double), static_cast<cudaStream_t>(stream)));
    return HESS_OK;
}

HESS_EXPORT hess_status imatrix_destroy(imatrix_t h) {
    if (!h) return HESS_OK;
    {
        std::lock_guard<std::mutex> lk(h->mu);
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(h->device);
        cudaDeviceSynchronize();
        cudaFree(h->acc);
        cudaSetDevice(cur);
    }
    delete h;
    return HESS_OK;
}

// ---------------------------------------------------------------- local H

HESS_EXPORT hess_status local_hess_create(int64_t d, int32_t block, local_hess_t* out) {
    if (!out) return fail(HESS_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d <= 0) return fail(HESS_ERR_INVALID, "d must be positive");
    if (block != 16) return fail(HESS_ERR_UNSUPPORTED, "block must be 16 (got %d)", block);
    if (d % block != 0) return fail(HESS_ERR_UNSUPPORTED, "d %% block != 0");
    if (d > (int64_t(1) << 20)) return fail(HESS_ERR_UNSUPPORTED, "d too large");
    if (injected_alloc_failure()) return fail(HESS_ERR_OOM, "injected allocation failure (HESS_FAULT=alloc)");
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    hess_status st = prepare_device(dev, nullptr);
    if (st != HESS_OK) return st;
    local_hess_ctx* h = new (std::nothrow) local_hess_ctx();
    if (!h) return fail(HESS_ERR_OOM, "host allocation failed");
    h->device = dev;
    h->d = d;
    h->block = block;
    h->n_blocks = static_cast<int>(d / block);
    const size_t bytes = static_cast<size_t>(h->n_blocks) * 256 * sizeof(double);
    cudaError_t e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaMalloc(&h->acc, bytes);
    if (e == cudaSuccess) e = cudaMalloc(&h->status, 64);
    if (e == cudaSuccess) e = cudaMemset(h->acc, 0, bytes);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, 64);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        hess_status s = e == cudaErrorMemoryAllocation ? HESS_ERR_OOM : HESS_ERR_CUDA;
        cudaFree(h->acc);
        cudaFree(h->status);
        delete h;
        return fail(s, "local_hess_create: %s", cudaGetErrorString(e));
    }
    *out = h;
    return HESS_OK;
}

HESS_EXPORT hess_status local_hess_add(local_hess_t h, const void* X, int64_t n_tokens, int64_t d,
                                       int32_t block, int32_t dtype, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (n_tokens < 0) return fail(HESS_ERR_INVALID, "n_tokens < 0");
    if (d != h->d) return fail(HESS_ERR_INVALID, "d = %lld does not match the handle (%lld)", (long long)d, (long long)h->d);
    if (block != h->block) return fail(HESS_ERR_INVALID, "block does not match the handle");
    if (dtype != HESS_BF16) {
        if (dtype == HESS_F32) return fail(HESS_ERR_UNSUPPORTED, "local_hess_add takes bf16 input");
        return fail(HESS_ERR_INVALID, "unknown dtype %d", dtype);
    }
    if (n_tokens == 0) return HESS_OK;
    if (!X) return fail(HESS_ERR_INVALID, "X is NULL with n_tokens > 0");
    if (reinterpret_cast<uintptr_t>(X) % 16 != 0) return fail(HESS_ERR_INVALID, "X is not 16-byte aligned");
    if (n_tokens > (int64_t(1) << 31) - hk::kLocalKBlock) return fail(HESS_ERR_UNSUPPORTED, "n_tokens too large");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_buffer(X, h->device, "X")) != HESS_OK) return st;
    hk::LocalParams p;
    std::memset(&p, 0, sizeof(p));
    st = encode_2d(&p.map, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h->d, n_tokens, 64, hk::kLocalKBlock);
    if (st != HESS_OK) return st;
    p.acc = h->acc;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    p.d = static_cast<int32_t>(h->d);
    p.n_groups = static_cast<int32_t>(ceil_div(h->d, hk::kLocalGroup));
    p.total_kb = static_cast<int32_t>(ceil_div(n_tokens, hk::kLocalKBlock));
    const int64_t want = ceil_div(2 * static_cast<int64_t>(h->sm_count), p.n_groups);
    p.n_ranges = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(want, p.total_kb)));
    p.chunk_steps = 8;
    const int64_t grid = static_cast<int64_t>(p.n_groups) * p.n_ranges;
    if (grid > 0x7fffffff) return fail(HESS_ERR_UNSUPPORTED, "grid too large");
    cudaError_t e = hk::launch_local_gram(p, static_cast<int>(grid), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(HESS_ERR_CUDA, "local launch failed: %s", cudaGetErrorString(e));
    h->N += n_tokens;
    return HESS_OK;
}

HESS_EXPORT hess_status local_hess_read(local_hess_t h, float* out, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    if (!out) return fail(HESS_ERR_INVALID, "out is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    if ((st = check_buffer(out, h->device, "out")) != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->N == 0) {
        CUDA_TRY(cudaMemsetAsync(out, 0, static_cast<size_t>(h->n_blocks) * 256 * sizeof(float), s));
        return HESS_OK;
    }
    CUDA_TRY(hk::launch_local_read(h->acc, out, h->n_blocks, 2.0 / static_cast<double>(h->N), s));
    return HESS_OK;
}

HESS_EXPORT int64_t local_hess_token_count(local_hess_t h) {
    if (!h) return -1;
    std::lock_guard<std::mutex> lk(h->mu);
    return h->N;
}

HESS_EXPORT hess_status local_hess_sync(local_hess_t h, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    return read_status(h->status, static_cast<cudaStream_t>(stream));
}

HESS_EXPORT hess_status local_hess_reset(local_hess_t h, hess_stream_t stream) {
    if (!h) return fail(HESS_ERR_INVALID, "handle is NULL");
    std::lock_guard<std::mutex> lk(h->mu);
    hess_status st = check_device(h->device);
    if (st != HESS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->N = 0;
    CUDA_TRY(cudaMemsetAsync(h->acc, 0, static_cast<size_t>(h->n_blocks) * 256 * sizeof(double), s));
    CUDA_TRY(cudaMemsetAsync(h->status, 0, 64, s));
    return HESS_OK;
}

HESS_EXPORT hess_status local_hess_destroy(local_hess_t h) {
    if (!h) return HESS_OK;
    {
        std::lock_guard<std::mutex> lk(h->mu);
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(h->device);
        cudaDeviceSynchronize();
        cudaFree(h->acc);
        cudaFree(h->status);
        cudaSetDevice(cur);
    }
    delete h;
    return HESS_OK;
}

HESS_EXPORT const char* hess_last_error(void) { return g_last_error.c_str(); }

namespace hk {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace hk

HESS_EXPORT int32_t hess_abi_version(void) { return HESS_ABI_VERSION; }
