// Companion statistics of the calibration Hessian:
//   * merge of two accumulators (per-device partials summed before the 2/N
//     scale: GPTQModel PR #2979 Summary and PR #2981 Changes);
//   * the imatrix per-column sum of squares, which NVIDIA Model-Optimizer
//     PR #3002 ("What does this PR do?") keeps as a float32 statistic because
//     it is not a GEMM.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>

#include "kernels.cuh"

namespace hk {
namespace {

__device__ __forceinline__ float two_sum(float a, float b, float& err) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return s;
}

// dst += src over (hi, lo) accumulator tiles.  Per element, each stored pair
// is first renormalised with an exact TwoSum (its lo may hold undigested
// flush sums), then: TwoSum of the hi parts, the lo parts and the error
// added, and the pair renormalised with Fast2Sum.  Four elements per thread
// (float4 of each plane), grid-stride over the tiles' planes.
__global__ void __launch_bounds__(256) add_pairs_kernel(float* __restrict__ dst,
                                                        const float* __restrict__ src,
                                                        size_t n_tiles) {
    const size_t per_tile = kTileElems / 4;
    const size_t n4 = n_tiles * per_tile;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t q = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; q < n4; q += stride) {
        const size_t t = q / per_tile, k = (q - t * per_tile) * 4;
        float* dh = dst + t * kTileWords + k;
        const float* sh = src + t * kTileWords + k;
        float4 ah = *reinterpret_cast<const float4*>(dh);
        float4 al = *reinterpret_cast<const float4*>(dh + kTileElems);
        const float4 bh = *reinterpret_cast<const float4*>(sh);
        const float4 bl = *reinterpret_cast<const float4*>(sh + kTileElems);
        float* const a_h[4] = {&ah.x, &ah.y, &ah.z, &ah.w};
        float* const a_l[4] = {&al.x, &al.y, &al.z, &al.w};
        const float b_h[4] = {bh.x, bh.y, bh.z, bh.w};
        const float b_l[4] = {bl.x, bl.y, bl.z, bl.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float fa, fb, e;
            const float ha = two_sum(*a_h[i], *a_l[i], fa);
            const float hb = two_sum(b_h[i], b_l[i], fb);
            const float s = two_sum(ha, hb, e);
            const float l = __fadd_rn(__fadd_rn(fa, fb), e);
            const float hi = __fadd_rn(s, l);
            *a_h[i] = hi;
            *a_l[i] = __fsub_rn(l, __fsub_rn(hi, s));  // Fast2Sum error (|s| >= |l|)
        }
        *reinterpret_cast<float4*>(dh) = ah;
        *reinterpret_cast<float4*>(dh + kTileElems) = al;
    }
}


__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// CTA = up to 4,096 consecutive features (thread l takes features 8l..8l+7)
// x one token slab, so the CTA reads whole contiguous stretches of each token
// row: a read stream over rows measured ~8 % faster on GB300 than CTAs that
// each take a 512-byte segment of every row.  Each thread walks the slab's
// tokens kRowsInFlight rows at a time and sums squares in fp32 chains of
// kChain tokens (round to nearest: unbiased), each chain folded into a
// compensated (hi, lo) pair; at the end it adds one fp64 value per feature to
// acc, so no shared memory or barrier is needed.
constexpr int kChain = 64;
constexpr int kRowThreads = 512;                 // threads per CTA
constexpr int kRowFeatures = kRowThreads * 8;    // features per CTA
constexpr int kRowsInFlight = 8;

template <class T>
__global__ void __launch_bounds__(kRowThreads) colsumsq_kernel(const T* __restrict__ X, int64_t n, int d,
                                                               int64_t slab, double* __restrict__ acc) {
    const int f0 = blockIdx.x * kRowFeatures + threadIdx.x * 8;
    if (f0 >= d) return;  // d is a multiple of 8: a thread has all 8 features or none
    const int64_t t0 = static_cast<int64_t>(blockIdx.y) * slab;
    const int64_t t1 = min(n, t0 + slab);
    const T* const col = X + f0;
    float hi[8] = {}, lo[8] = {};
    for (int64_t c0 = t0; c0 < t1; c0 += kChain) {
        const int64_t c1 = min(t1, c0 + kChain);
        float s[8] = {};
        int64_t t = c0;
        for (; t + kRowsInFlight <= c1; t += kRowsInFlight) {
            float x[kRowsInFlight][8];
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r) load8(col + (t + r) * d, x[r]);
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r)
#pragma unroll
                for (int k = 0; k < 8; ++k) s[k] = __fmaf_rn(x[r][k], x[r][k], s[k]);
        }
        for (; t < c1; ++t) {
            float x[8];
            load8(col + t * d, x);
#pragma unroll
            for (int k = 0; k < 8; ++k) s[k] = __fmaf_rn(x[k], x[k], s[k]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float e;
            hi[k] = two_sum(hi[k], s[k], e);
            lo[k] = __fadd_rn(lo[k], e);
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const double v = static_cast<double>(hi[k]) + static_cast<double>(lo[k]);
        if (v != 0.0) atomicAdd(acc + f0 + k, v);
    }
}

__global__ void __launch_bounds__(256) colsumsq_read_kernel(const double* __restrict__ acc,
                                                            float* __restrict__ out, int d) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < d) out[i] = static_cast<float>(acc[i]);
}

}  // namespace

cudaError_t launch_add_pairs(float* dst, const float* src, size_t n_tiles, int sm_count,
                             cudaStream_t s) {
    const size_t want = (n_tiles * (kTileElems / 4) + 255) / 256;
    const int grid = static_cast<int>(want < static_cast<size_t>(4 * sm_count) ? want : 4 * sm_count);
    add_pairs_kernel<<<grid, 256, 0, s>>>(dst, src, n_tiles);
    return cudaGetLastError();
}

namespace {
__global__ void store_words_kernel(uint4* dst, uint4 v) { *dst = v; }

// (hi, lo) <- TwoSum(hi, lo) over accumulator tiles: folds the low part's
// undigested flush sums into the high part, exactly.  Four elements per
// thread, grid-stride over the tiles' planes.
__global__ void __launch_bounds__(256) renorm_pairs_kernel(float* __restrict__ acc, size_t n_tiles) {
    const size_t per_tile = kTileElems / 4;
    const size_t n4 = n_tiles * per_tile;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t q = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; q < n4; q += stride) {
        const size_t t = q / per_tile, k = (q - t * per_tile) * 4;
        float* h = acc + t * kTileWords + k;
        float4 a = *reinterpret_cast<const float4*>(h);
        float4 b = *reinterpret_cast<const float4*>(h + kTileElems);
        float e;
        a.x = two_sum(a.x, b.x, e); b.x = e;
        a.y = two_sum(a.y, b.y, e); b.y = e;
        a.z = two_sum(a.z, b.z, e); b.z = e;
        a.w = two_sum(a.w, b.w, e); b.w = e;
        *reinterpret_cast<float4*>(h) = a;
        *reinterpret_cast<float4*>(h + kTileElems) = b;
    }
}
}  // namespace

cudaError_t launch_renorm_pairs(float* acc, size_t n_tiles, int sm_count, cudaStream_t s) {
    const size_t want = (n_tiles * (kTileElems / 4) + 255) / 256;
    const int grid = static_cast<int>(want < static_cast<size_t>(4 * sm_count) ? want : 4 * sm_count);
    renorm_pairs_kernel<<<grid, 256, 0, s>>>(acc, n_tiles);
    return cudaGetLastError();
}

cudaError_t launch_store_words(uint32_t* dst, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                               cudaStream_t s) {
    store_words_kernel<<<1, 1, 0, s>>>(reinterpret_cast<uint4*>(dst), make_uint4(w0, w1, w2, w3));
    return cudaGetLastError();
}

cudaError_t launch_colsumsq(const void* X, bool f32, int64_t n, int d, double* acc, int sm_count,
                            cudaStream_t s) {
    const int gx = (d + kRowFeatures - 1) / kRowFeatures;
    const int threads = std::min(kRowThreads, ((d / 8 + 31) / 32) * 32);
    // One wave: as many token slabs as the SMs hold CTAs of this kernel,
    // split evenly (a grid of ~1.7 waves ran its second wave two-thirds full).
    static std::atomic<int> resident[2] = {{0}, {0}};
    int per_sm = resident[f32 ? 1 : 0].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        int b = 0;
        const cudaError_t e =
            f32 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, colsumsq_kernel<float>, kRowThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, colsumsq_kernel<__nv_bfloat16>, kRowThreads, 0);
        if (e != cudaSuccess) return e;
        per_sm = std::max(1, b);
        resident[f32 ? 1 : 0].store(per_sm, std::memory_order_relaxed);
    }
    // About 16 warps per SM: one CTA of 512 threads at d >= 4,096 (more CTAs
    // per SM made the per-feature fp64 atomics cost more than they hid:
    // 53.2 against 47.1 us at two per SM, measured), more for narrow rows.
    const int ctas_per_sm = std::min(per_sm, std::max(1, kRowThreads / threads));
    int64_t slabs = std::max<int64_t>(1, static_cast<int64_t>(ctas_per_sm) * sm_count / gx);
    int64_t slab = std::max<int64_t>(1, (n + slabs - 1) / slabs);
    slabs = (n + slab - 1) / slab;
    if (slabs > 65535) {
        slabs = 65535;
        slab = (n + slabs - 1) / slabs;
        slabs = (n + slab - 1) / slab;
    }
    const dim3 grid(gx, static_cast<unsigned>(slabs));
    if (f32)
        colsumsq_kernel<float><<<grid, threads, 0, s>>>(static_cast<const float*>(X), n, d, slab, acc);
    else
        colsumsq_kernel<__nv_bfloat16>
            <<<grid, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(X), n, d, slab, acc);
    return cudaGetLastError();
}
cudaError_t launch_colsumsq_read(const double* acc, float* out, int d, cudaStream_t s) {
    colsumsq_read_kernel<<<(d + 255) / 256, 256, 0, s>>>(acc, out, d);
    return cudaGetLastError();
}

}  // namespace hk
