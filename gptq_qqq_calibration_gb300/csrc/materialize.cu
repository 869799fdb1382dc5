// Materialize kernels: scale the (hi, lo) accumulator by 2/N, add the damping
// term to the diagonal and write the full symmetric fp32 Hessian; and the
// read-out of the local 16x16 block Hessians.
//
// GPTQModel wiki "QQQ", Concepts (Quadratic error compensation): the merged
// Gram is scaled by 2 / total_samples, and the quantization pass adds
// damp_percent * mean(diag(H)) to the diagonal (step 3); "Quantizer API and
// results": the damping value handed back is that absolute amount.
// GPTQModel PR #2979 Summary: N counts token vectors.
//
// Readings: the mean of the diagonal is taken of the scaled matrix, in
// fp64; diagonal elements are computed in fp64 and rounded once to fp32;
// off-diagonal elements (hi + lo) * scale are computed in fp32 (the pair
// renormalised with an exact TwoSum, then an exact product by FMA) and
// rounded to within an ulp of the correctly rounded value;
// H_out[j][i] is a copy of H_out[i][j] (i <= j) so the result is exactly
// symmetric.
#include "kernels.cuh"
#include "ptx.cuh"

namespace hk {
namespace {

// Scratch words of one materialization (device memory of the handle):
// [0] the damping value (fp64), [1, 1 + 2T) the fp64 sums of the diagonal
// quarters, then a 32-bit arrival count of those quarters, zero between
// launches.
__host__ __device__ constexpr size_t ticket_offset(int T) { return sizeof(double) * (1 + 2 * static_cast<size_t>(T)); }

// One CTA per 64x64 quarter of an upper tile, the diagonal tiles' quarters
// first (so that the diagonal tail below overlaps the rest); blockIdx.x =
// 4 * (tile in that order) + quarter.  Each thread loads all of its
// 16-byte words of both planes first (4 columns of one row per word),
// computes (hi + lo) * 2/N in fp32 and writes the mirrored strictly-upper
// rows of H_out; pass 2 writes the direct strictly-upper rows through the
// shared-memory transpose.  Diagonal elements are left to the tail: each
// diagonal quarter stores the fp64 sum of its 64 diagonal (hi + lo), and the
// last of them to arrive takes the mean of the scaled diagonal (its partial
// sums added in a fixed order), writes the damping value and every diagonal
// element, rounded once from fp64, while other quarters may still run.
__global__ void __launch_bounds__(256) materialize_kernel(const float* __restrict__ acc,
                                                          float* __restrict__ H, int d, int T,
                                                          double scale, float scale_hi,
                                                          float scale_lo, double damp_percent,
                                                          double* __restrict__ scratch,
                                                          float* __restrict__ damp_f32,
                                                          const uint32_t* __restrict__ status,
                                                          uint32_t* __restrict__ status_mirror) {
    __shared__ float tr[64][65];
    // Launched to overlap the end of the flush before it: the accumulator
    // is read only once that kernel has completed.
    griddep_wait();
    __shared__ double wpart[8];
    __shared__ int last;
    const int a = (blockIdx.x >> 1) & 1, b = blockIdx.x & 1;
    int I, J;
    if (static_cast<int>(blockIdx.x >> 2) < T) {
        I = J = static_cast<int>(blockIdx.x >> 2);
    } else {
        // strictly upper tiles, row by row
        int rem = static_cast<int>(blockIdx.x >> 2) - T;
        I = 0;
        while (rem >= T - 1 - I) {
            rem -= T - 1 - I;
            ++I;
        }
        J = I + 1 + rem;
    }
    if (I == J && a > b) return;  // lower quarter of a diagonal tile: covered by its mirror
    const int t = tile_index(I, J, T);
    const bool diag = I == J && a == b;
    const int r0 = I * kTile + a * 64, c0 = J * kTile + b * 64;
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
    const float* tile = acc + static_cast<size_t>(t) * kTileWords;
    const int r = r0 + tx;
    float4 h4[4], l4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = tile_offset(a * 64 + tx, b * 64 + 4 * (ty + 4 * i));
        h4[i] = *reinterpret_cast<const float4*>(tile + k);
        l4[i] = *reinterpret_cast<const float4*>(tile + kTileElems + k);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = ty + 4 * i;
        const float hs[4] = {h4[i].x, h4[i].y, h4[i].z, h4[i].w};
        const float ls[4] = {l4[i].x, l4[i].y, l4[i].z, l4[i].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int c = c0 + 4 * q + m;
            // The stored pair may be unnormalised (the low part can hold
            // recent flushes' sums that nearly cancel the high part), so it
            // is first renormalised exactly: h = RN(hi + lo), l the error.
            float l;
            const float h = two_sum_f32(hs[m], ls[m], l);
            // (h + l) * (scale_hi + scale_lo): the exact product h * scale_hi
            // as p + pe, plus the small cross terms, then one rounding
            const float p = __fmul_rn(h, scale_hi);
            const float pe = __fmaf_rn(h, scale_hi, -p);
            const float cross = __fmaf_rn(l, scale_hi, __fmaf_rn(h, scale_lo, pe));
            const float v = __fadd_rn(p, cross);
            tr[4 * q + m][tx] = v;
            if (r < c && c < d) H[static_cast<size_t>(c) * d + r] = v;
        }
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = ty; rr < 64; rr += 4) {
        const int r2 = r0 + rr, c = c0 + tx;
        if (c < d && r2 < c) H[static_cast<size_t>(r2) * d + c] = tr[tx][rr];
    }
    if (!diag) return;

    // ---- diagonal quarter: its fp64 partial sum, then the arrival count
    if (ty == 0) {
        double s = 0.0;
        if (r < d) {
            const int k = tile_offset(a * 64 + tx, a * 64 + tx);
            s = static_cast<double>(tile[k]) + static_cast<double>(tile[kTileElems + k]);
        }
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if ((tx & 31) == 0) wpart[tx >> 5] = s;
    }
    __syncthreads();
    unsigned* const ticket = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(scratch) + ticket_offset(T));
    if (threadIdx.x == 0) {
        scratch[1 + 2 * I + a] = wpart[0] + wpart[1];
        __threadfence();
        last = atomicAdd(ticket, 1u) == static_cast<unsigned>(2 * T - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    {
        // the partial sums, in a fixed order: thread k takes k, k + 256, ...
        double s = 0.0;
        for (int i = threadIdx.x; i < 2 * T; i += blockDim.x) s += __ldcg(scratch + 1 + i);
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if ((threadIdx.x & 31) == 0) wpart[threadIdx.x >> 5] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < 8; ++w) s += wpart[w];
        const double damp = damp_percent * ((s * scale) / static_cast<double>(d));
        scratch[0] = damp;
        *damp_f32 = static_cast<float>(damp);
        *ticket = 0u;  // ready for the next launch (every quarter has arrived)
        // the handle's status word and the damping value, written straight
        // to their pinned host copy (mapped memory): the host reads them
        // there once this kernel has completed, with no copy in the stream
        if (status_mirror != nullptr) {
            volatile uint32_t* m = status_mirror;
            m[0] = *status;
            m[1] = __float_as_uint(static_cast<float>(damp));
            __threadfence_system();
        }
        wpart[0] = damp;
    }
    __syncthreads();
    const double damp = wpart[0];
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const int ti = i / kTile, rr = i % kTile;
        const float* e = acc + static_cast<size_t>(tile_index(ti, ti, T)) * kTileWords + tile_offset(rr, rr);
        const double v = static_cast<double>(e[0]) + static_cast<double>(e[kTileElems]);
        H[static_cast<size_t>(i) * d + i] = static_cast<float>(v * scale + damp);
    }
}

__global__ void __launch_bounds__(256) local_read_kernel(const double* __restrict__ acc,
                                                         float* __restrict__ out, double scale) {
    const int b = blockIdx.x;
    const int i = threadIdx.x >> 4, j = threadIdx.x & 15;
    const int lo = i < j ? i : j, hi = i < j ? j : i;
    out[static_cast<size_t>(b) * 256 + threadIdx.x] =
        static_cast<float>(acc[static_cast<size_t>(b) * 256 + lo * 16 + hi] * scale);
}

}  // namespace

size_t materialize_scratch_bytes(int T) { return ticket_offset(T) + sizeof(unsigned); }

cudaError_t launch_materialize(const float* acc, float* H_out, int d, int T, double scale,
                               double damp_percent, double* scratch, float* damp_f32, const uint32_t* status,
                               uint32_t* status_mirror, cudaStream_t s) {
    const int n_tiles = T * (T + 1) / 2;
    const float scale_hi = static_cast<float>(scale);
    const float scale_lo = static_cast<float>(scale - static_cast<double>(scale_hi));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(4 * n_tiles), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, materialize_kernel, acc, H_out, d, T, scale, scale_hi, scale_lo, damp_percent,
                              scratch, damp_f32, status, status_mirror);
}

cudaError_t launch_local_read(const double* acc, float* out, int n_blocks, double scale,
                              cudaStream_t s) {
    local_read_kernel<<<n_blocks, 256, 0, s>>>(acc, out, scale);
    return cudaGetLastError();
}

}  // namespace hk
