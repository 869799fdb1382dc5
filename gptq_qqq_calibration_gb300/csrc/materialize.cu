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
// off-diagonal elements (hi + lo) * scale are computed in fp32 with an exact
// product (FMA) and rounded to within an ulp of the correctly rounded value;
// H_out[j][i] is a copy of H_out[i][j] (i <= j) so the result is exactly
// symmetric.
#include "kernels.cuh"

namespace hk {
namespace {

constexpr int kDiagThreads = 1024;

__global__ void __launch_bounds__(kDiagThreads) diag_damp_kernel(const float* __restrict__ acc, int d,
                                                                 int T, double scale,
                                                                 double damp_percent,
                                                                 double* damp_out,
                                                                 float* damp_out_f32) {
    __shared__ double part[kDiagThreads / 32];
    double s = 0.0;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const int ti = i / kTile, r = i % kTile;
        const float* e = acc + static_cast<size_t>(tile_index(ti, ti, T)) * kTileWords + tile_offset(r, r);
        s += static_cast<double>(e[0]) + static_cast<double>(e[kTileElems]);
    }
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        s = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.0;
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (threadIdx.x == 0) {
            const double mean = (s * scale) / static_cast<double>(d);
            const double damp = damp_percent * mean;
            *damp_out = damp;
            *damp_out_f32 = static_cast<float>(damp);
        }
    }
}

// One CTA per 64x64 quarter of an upper tile.  Pass 1 reads the quarter,
// 4 columns of one row per thread (16-byte loads of each plane), computes
// (hi + lo) * 2/N in fp32 and writes the mirrored strictly-upper rows of
// H_out; a diagonal quarter then recomputes its diagonal in fp64 with the
// damping (kept out of the main loop, where a per-element branch would put
// fp64 work on every element); pass 2 writes the direct rows, diagonal
// included, through the shared-memory transpose.
__global__ void __launch_bounds__(256) materialize_kernel(const float* __restrict__ acc,
                                                          float* __restrict__ H, int d, int T,
                                                          double scale, float scale_hi,
                                                          float scale_lo,
                                                          const double* __restrict__ damp_ptr) {
    __shared__ float tr[64][65];
    const int t = blockIdx.x;
    const int a = blockIdx.y >> 1, b = blockIdx.y & 1;
    int I = 0, rem = t;
    while (rem >= T - I) {
        rem -= T - I;
        ++I;
    }
    const int J = I + rem;
    if (I == J && a > b) return;  // lower quarter of a diagonal tile: covered by its mirror
    const int r0 = I * kTile + a * 64, c0 = J * kTile + b * 64;
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
    const float* tile = acc + static_cast<size_t>(t) * kTileWords;
    const int r = r0 + tx;
    for (int q = ty; q < 16; q += 4) {
        const int k = tile_offset(a * 64 + tx, b * 64 + 4 * q);
        const float4 h4 = *reinterpret_cast<const float4*>(tile + k);
        const float4 l4 = *reinterpret_cast<const float4*>(tile + kTileElems + k);
        const float hs[4] = {h4.x, h4.y, h4.z, h4.w};
        const float ls[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int c = c0 + 4 * q + m;
            // (h + l) * (scale_hi + scale_lo): the exact product h * scale_hi
            // as p + pe, plus the small cross terms, then one rounding
            const float p = __fmul_rn(hs[m], scale_hi);
            const float pe = __fmaf_rn(hs[m], scale_hi, -p);
            const float cross = __fmaf_rn(ls[m], scale_hi, __fmaf_rn(hs[m], scale_lo, pe));
            const float v = __fadd_rn(p, cross);
            tr[4 * q + m][tx] = v;
            if (r < c && c < d) H[static_cast<size_t>(c) * d + r] = v;
        }
    }
    __syncthreads();
    if (I == J && a == b) {
        if (ty == 0 && r < d) {
            const int k = tile_offset(a * 64 + tx, a * 64 + tx);
            const double s = static_cast<double>(tile[k]) + static_cast<double>(tile[kTileElems + k]);
            tr[tx][tx] = static_cast<float>(s * scale + *damp_ptr);
        }
        __syncthreads();
    }
    for (int rr = ty; rr < 64; rr += 4) {
        const int r2 = r0 + rr, c = c0 + tx;
        if (r2 < d && c < d && r2 <= c) H[static_cast<size_t>(r2) * d + c] = tr[tx][rr];
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

cudaError_t launch_diag_damp(const float* acc, int d, int T, double scale, double damp_percent,
                             double* damp_out, float* damp_out_f32, cudaStream_t s) {
    diag_damp_kernel<<<1, kDiagThreads, 0, s>>>(acc, d, T, scale, damp_percent, damp_out,
                                                damp_out_f32);
    return cudaGetLastError();
}

cudaError_t launch_materialize(const float* acc, float* H_out, int d, int T, double scale,
                               const double* damp, cudaStream_t s) {
    const int n_tiles = T * (T + 1) / 2;
    const float scale_hi = static_cast<float>(scale);
    const float scale_lo = static_cast<float>(scale - static_cast<double>(scale_hi));
    materialize_kernel<<<dim3(n_tiles, 4), 256, 0, s>>>(acc, H_out, d, T, scale, scale_hi, scale_lo,
                                                        damp);
    return cudaGetLastError();
}

cudaError_t launch_local_read(const double* acc, float* out, int n_blocks, double scale,
                              cudaStream_t s) {
    local_read_kernel<<<n_blocks, 256, 0, s>>>(acc, out, scale);
    return cudaGetLastError();
}

}  // namespace hk
