// The quantization pass that consumes the calibration Hessian: GPTQModel
// wiki "QQQ", Concepts (Quadratic error compensation, steps 1-5), "Whole-row
// and grouped weight quantization", and "Quantizer API and results".
//
// Factor (steps 2-4).  Step 4 asks for U, upper triangular with
// U^T U = inv(H_damped).  With J the order-reversing permutation and
// L = chol_lower(J H J), U = J inv(L) J (U^T U = J L^-T L^-1 J = inv(H)), so
// one Cholesky and one triangular inverse give U without forming inv(H).
// Reversing both indices of a d x d row-major matrix reverses its flat
// array, which is how J . J is applied on the way in and out.  Both the
// Cholesky and the inverse run in 128-column blocks: a one-CTA kernel
// factors and inverts each diagonal block in shared memory; the panel
// solve, the trailing update and the block-row steps of the inverse are
// fp32 tile GEMMs.
//
// Quantize (step 5), per 128-column block: eight lanes per weight row walk
// the block's columns in order with U's diagonal block in shared memory
// (quantize, scaled error, update of the block's remaining columns); GEMMs
// then propagate the block's errors into the later columns, lazily in two
// levels (the rest of a 512-column super-block after each block, every
// column after the super-block once per super-block).
//
// All arithmetic is fp32 (the working-matrix precision of step 1) except the
// damping mean and the loss sum, which are accumulated in fp64.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <cuda_bf16.h>

#include "gptq.h"
#include "hess.h"
#include "kernels.cuh"

namespace {

constexpr int kNB = 128;          // column block of the factorization and of step 5
constexpr int kLd = kNB + 1;      // padded row of the diagonal-block tiles
constexpr int kGemmLd = 132;      // padded row of the GEMM k-slices
constexpr int kGemmCLowerTiles = 1;
constexpr int kPotrfThreads = 512;
constexpr int kBlockThreads = 128;
constexpr int kSuper = 4;          // blocks per lazy super-block of step 5
constexpr size_t kPotrfSmem = 2 * kNB * kLd * sizeof(float);
constexpr size_t kBlockSmem = kNB * kNB * sizeof(float);
constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------- steps 2-3

// dead[i] = (H_ii == 0); damp = damp_percent * mean_i(dead ? 1 : H_ii).
__global__ void __launch_bounds__(1024) gq_damp_kernel(const float* __restrict__ H, int d,
                                                       double damp_percent,
                                                       unsigned char* __restrict__ dead,
                                                       double* __restrict__ damp64,
                                                       float* __restrict__ damp32) {
    __shared__ double part[32];
    double s = 0.0;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const float h = H[static_cast<size_t>(i) * (d + 1)];
        const bool z = (h == 0.0f);
        dead[i] = z;
        s += z ? 1.0 : static_cast<double>(h);
    }
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        s = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.0;
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        if (threadIdx.x == 0) {
            const double damp = damp_percent * (s / d);
            *damp64 = damp;
            *damp32 = static_cast<float>(damp);
        }
    }
}

// G = J H_damped J, lower triangle only (zeros above the diagonal).  A dead
// diagonal entry becomes 1 before damping.  Thread = 4 consecutive outputs.
__global__ void gq_rotate_in_kernel(const float* __restrict__ H, float* __restrict__ G, int d,
                                    const unsigned char* __restrict__ dead,
                                    const double* __restrict__ damp64) {
    const size_t n4 = static_cast<size_t>(d) * d / 4;
    const double damp = *damp64;
    for (size_t q = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; q < n4;
         q += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(H)[n4 - 1 - q];
        const float src[4] = {v.w, v.z, v.y, v.x};
        const size_t e = 4 * q;
        const int i = static_cast<int>(e / d);
        const int j0 = static_cast<int>(e % d);
        float out[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int j = j0 + t;
            float x = j > i ? 0.0f : src[t];
            if (j == i) {
                const int r = d - 1 - i;
                x = static_cast<float>(static_cast<double>(dead[r] ? 1.0f : x) + damp);
            }
            out[t] = x;
        }
        reinterpret_cast<float4*>(G)[q] = make_float4(out[0], out[1], out[2], out[3]);
    }
}

// ------------------------------------------------------------- step 4

// Factor the diagonal block k of F in place (F = L L^T, lower) and write
// inv(L_kk) to Dinv.  A pivot that is not a positive finite number sets
// status bit 1 and is replaced by 1 so the kernel still ends normally.
__global__ void __launch_bounds__(kPotrfThreads) gq_potrf_kernel(float* __restrict__ F, int d, int k,
                                                                 float* __restrict__ Dinv,
                                                                 int* __restrict__ status) {
    extern __shared__ float sm[];
    float* S = sm;               // [kNB][kLd]: the block, then L
    float* X = sm + kNB * kLd;   // [kNB][kLd]: inv(L)
    const int tid = threadIdx.x;
    float* blk = F + static_cast<size_t>(k) * kNB * d + static_cast<size_t>(k) * kNB;
    for (int e = tid; e < kNB * kNB; e += kPotrfThreads) {
        const int i = e >> 7, j = e & (kNB - 1);
        S[i * kLd + j] = j <= i ? blk[static_cast<size_t>(i) * d + j] : 0.0f;
        X[i * kLd + j] = 0.0f;
    }
    __syncthreads();

    // Right-looking, one column per step.  Thread (row = tid % 128,
    // part = tid / 128) updates columns c = j+1+part, j+5+part, ... of its row.
    const int row = tid & (kNB - 1), part = tid >> 7;
    bool bad = false;
    for (int j = 0; j < kNB; ++j) {
        float p = S[j * kLd + j];
        if (!(p > 0.0f) || !(p < INFINITY)) {
            bad = true;
            p = 1.0f;
        }
        const float l = sqrtf(p);
        if (part == 0 && row > j) S[row * kLd + j] = __fdiv_rn(S[row * kLd + j], l);
        __syncthreads();  // column j scaled; every thread has read the pivot
        if (part == 0 && row == j) S[j * kLd + j] = l;
        if (row > j) {
            // Four elements per round, all loads before the stores (the
            // compiler cannot prove the stores miss the next loads).
            const float lr = S[row * kLd + j];
            int c = j + 1 + part;
            for (; c + 12 <= row; c += 16) {
                const float a0 = S[row * kLd + c], a1 = S[row * kLd + c + 4];
                const float a2 = S[row * kLd + c + 8], a3 = S[row * kLd + c + 12];
                const float b0 = S[c * kLd + j], b1 = S[(c + 4) * kLd + j];
                const float b2 = S[(c + 8) * kLd + j], b3 = S[(c + 12) * kLd + j];
                S[row * kLd + c] = fmaf(-lr, b0, a0);
                S[row * kLd + c + 4] = fmaf(-lr, b1, a1);
                S[row * kLd + c + 8] = fmaf(-lr, b2, a2);
                S[row * kLd + c + 12] = fmaf(-lr, b3, a3);
            }
            for (; c <= row; c += 4) S[row * kLd + c] = fmaf(-lr, S[c * kLd + j], S[row * kLd + c]);
        }
        __syncthreads();
    }
    if (bad && tid == 0) atomicOr(status, 1);
    __shared__ float rdiag[kNB];
    if (tid < kNB) rdiag[tid] = __frcp_rn(S[tid * kLd + tid]);
    __syncthreads();

    // inv(L) by forward substitution: column j = tid / 4 is solved by four
    // threads (consecutive lanes) that split each dot product.
    {
        const int col = tid >> 2, q = tid & 3;
        const int first = (tid >> 5) * 8;  // smallest column of this warp
        for (int i = first; i < kNB; ++i) {
            float a0 = 0.0f, a1 = 0.0f;
            if (i > col) {
                int m = col + q;
                for (; m + 4 < i; m += 8) {
                    a0 = fmaf(S[i * kLd + m], X[m * kLd + col], a0);
                    a1 = fmaf(S[i * kLd + m + 4], X[(m + 4) * kLd + col], a1);
                }
                if (m < i) a0 = fmaf(S[i * kLd + m], X[m * kLd + col], a0);
            }
            float acc = a0 + a1;
            acc += __shfl_xor_sync(kFull, acc, 1);
            acc += __shfl_xor_sync(kFull, acc, 2);
            if (i >= col && q == 0) X[i * kLd + col] = ((i == col ? 1.0f : 0.0f) - acc) * rdiag[i];
            __syncwarp();
        }
    }
    __syncthreads();
    float* inv = Dinv + static_cast<size_t>(k) * kNB * kNB;
    for (int e = tid; e < kNB * kNB; e += kPotrfThreads) {
        const int i = e >> 7, j = e & (kNB - 1);
        blk[static_cast<size_t>(i) * d + j] = S[i * kLd + j];
        inv[e] = X[i * kLd + j];
    }
}

struct GemmArgs {
    const float* A;  // M x K, row-major, lda
    const float* B;  // K x N row-major (ldb), or N x K when transposed
    float* C;        // M x N row-major, ldc
    int M, N, K, lda, ldb, ldc;
    float alpha;
    int beta;  // 0: C = alpha AB; 1: C = C + alpha AB
    int flags;
};

// C = beta C + alpha A op(B) in fp32 (FMA chains along k, one rounding per
// step).  128 x 128 output tile per CTA, k-slices of 8 double-buffered in
// shared memory, 8 x 8 outputs per thread.  N % 128 == 0 and K % 8 == 0;
// rows of A and C beyond M are skipped.  A CTA reads only the rows of A and
// the columns of op(B) of its own tile, and writes C after all its reads,
// so C may alias A when N == 128, or alias B when K == 128 and op(B) is not
// transposed.
template <bool kTransB>
__global__ void __launch_bounds__(256) gq_gemm_kernel(const GemmArgs g) {
    const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
    if ((g.flags & kGemmCLowerTiles) && n0 > m0) return;
    __shared__ __align__(16) float As[2][8][kGemmLd];
    __shared__ __align__(16) float Bs[2][8][kGemmLd];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int r_row = tid >> 1, r_col = (tid & 1) * 4;      // row-of-8 loader (A, transposed B)
    const int b_k = tid >> 5, b_n = (tid & 31) * 4;         // plain B loader
    const bool a_ok = m0 + r_row < g.M;
    const float* a_src = g.A + static_cast<size_t>(a_ok ? m0 + r_row : 0) * g.lda + r_col;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    float4 ra, rb;
    auto load = [&](int k0) {
        // Plain loads: C may alias A or B, so the read-only path is not used.
        ra = a_ok ? *reinterpret_cast<const float4*>(a_src + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (kTransB)
            rb = *reinterpret_cast<const float4*>(g.B + static_cast<size_t>(n0 + r_row) * g.ldb + k0 + r_col);
        else
            rb = *reinterpret_cast<const float4*>(g.B + static_cast<size_t>(k0 + b_k) * g.ldb + n0 + b_n);
    };
    auto store = [&](int buf) {
        As[buf][r_col + 0][r_row] = ra.x;
        As[buf][r_col + 1][r_row] = ra.y;
        As[buf][r_col + 2][r_row] = ra.z;
        As[buf][r_col + 3][r_row] = ra.w;
        if (kTransB) {
            Bs[buf][r_col + 0][r_row] = rb.x;
            Bs[buf][r_col + 1][r_row] = rb.y;
            Bs[buf][r_col + 2][r_row] = rb.z;
            Bs[buf][r_col + 3][r_row] = rb.w;
        } else {
            *reinterpret_cast<float4*>(&Bs[buf][b_k][b_n]) = rb;
        }
    };

    load(0);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < g.K; k0 += 8) {
        const bool more = k0 + 8 < g.K;
        if (more) load(k0 + 8);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) store(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (m >= g.M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float4* cp = reinterpret_cast<float4*>(g.C + static_cast<size_t>(m) * g.ldc + n0 + h * 64 + tx * 4);
            float4 o = make_float4(g.alpha * acc[i][h * 4 + 0], g.alpha * acc[i][h * 4 + 1],
                                   g.alpha * acc[i][h * 4 + 2], g.alpha * acc[i][h * 4 + 3]);
            if (g.beta) {
                const float4 c = *cp;
                o.x += c.x;
                o.y += c.y;
                o.z += c.z;
                o.w += c.w;
            }
            *cp = o;
        }
    }
}

__global__ void gq_identity_kernel(float* __restrict__ X, int d) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < d) X[static_cast<size_t>(i) * (d + 1)] = 1.0f;
}

// dst = src reversed as a flat array of 4 * n4 floats: J src J for a square
// row-major matrix.
__global__ void gq_reverse_copy_kernel(const float* __restrict__ src, float* __restrict__ dst, size_t n4) {
    for (size_t q = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; q < n4;
         q += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(src)[n4 - 1 - q];
        reinterpret_cast<float4*>(dst)[q] = make_float4(a.w, a.z, a.y, a.x);
    }
}

// ------------------------------------------------------------- step 5

// Working copy of W in fp32 with dead input columns zeroed (steps 1-2).
template <class T>
__global__ void gq_load_w_kernel(const T* __restrict__ W, float* __restrict__ Wc, size_t n4, int d,
                                 const unsigned char* __restrict__ dead) {
    for (size_t q = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; q < n4;
         q += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>((4 * q) % d);
        float x[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) x[t] = dead[c + t] ? 0.0f : static_cast<float>(W[4 * q + t]);
        reinterpret_cast<float4*>(Wc)[q] = make_float4(x[0], x[1], x[2], x[3]);
    }
}

// Whole-row scale s = max|w_row| / 7 (1 / 7 for an all-zero row), one warp per row.
__global__ void gq_rowscale_kernel(const float* __restrict__ Wc, int64_t rows, int d,
                                   float* __restrict__ rowscale, float* __restrict__ scales_out) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    const float* w = Wc + r * d;
    float m = 0.0f;
    for (int c = lane * 4; c < d; c += 128) {
        const float4 v = *reinterpret_cast<const float4*>(w + c);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (lane == 0) {
        const float s = __fdiv_rn(m > 0.0f ? m : 1.0f, 7.0f);
        rowscale[r] = s;
        scales_out[r] = s;
    }
}

struct BlockArgs {
    float* Wc;              // rows x d working matrix
    const float* U;         // d x d upper factor
    float* Wq;              // rows x d dequantized output
    signed char* codes;     // rows x d codes or NULL
    float* scales;          // rows x n_groups
    float* Err;             // scaled errors of this block: rows x 128 at stride ld_err
    const float* rowscale;  // whole-row scales (grouped == 0)
    double* loss;
    int64_t rows;
    int d, b, n_groups, grouped, ld_err;
};

constexpr int kRowLanes = 8;   // lanes per weight row
constexpr int kLaneCols = 16;  // consecutive block columns per lane
constexpr int kBlockRows = kBlockThreads / kRowLanes;

// One 128-column block of step 5.  Eight lanes hold one weight row, 16
// consecutive block columns each (four rows per warp).  Column i is
// quantized by the lane that holds it, its scaled error
// err = (w - q) / U_ii is broadcast to the row's lanes, and every lane
// applies w_j -= err * U_ij to its columns (U_ij = 0 for j < i, so columns
// already quantized keep their value; the lane then parks err in the slot of
// column i).  The code is rint(w / s) with w / s rounded to nearest as an
// fp32 division: w * (1/s) is used unless it lies within 1e-4 of a half
// integer, where the correctly rounded quotient decides.  Grouped blocks
// take their scale from the block's values as they stand when the block
// starts.
__global__ void __launch_bounds__(kBlockThreads) gq_block_kernel(const BlockArgs a) {
    extern __shared__ float4 us4[];  // U[b0:b0+128, b0:b0+128], row-major
    __shared__ float inv_u[kNB];
    __shared__ double red[kBlockThreads / 32];
    const float* Us = reinterpret_cast<const float*>(us4);
    const int b0 = a.b * kNB;
    for (int e = threadIdx.x; e < kNB * 32; e += kBlockThreads) {
        const int i = e >> 5, q = e & 31;
        us4[e] = __ldg(reinterpret_cast<const float4*>(a.U + static_cast<size_t>(b0 + i) * a.d + b0 + q * 4));
    }
    for (int i = threadIdx.x; i < kNB; i += kBlockThreads)
        inv_u[i] = __frcp_rn(__ldg(a.U + static_cast<size_t>(b0 + i) * (a.d + 1)));
    __syncthreads();
    const int lane = threadIdx.x & 31, sl = lane & (kRowLanes - 1), grp = lane & ~(kRowLanes - 1);
    double lsum = 0.0;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kBlockRows; base < a.rows;
         base += static_cast<int64_t>(gridDim.x) * kBlockRows) {
        const int64_t r = base + threadIdx.x / kRowLanes;
        const bool ok = r < a.rows;
        float w[kLaneCols];
        if (ok) {
            const float4* src = reinterpret_cast<const float4*>(a.Wc + r * a.d + b0 + kLaneCols * sl);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 v = src[t];
                w[4 * t] = v.x;
                w[4 * t + 1] = v.y;
                w[4 * t + 2] = v.z;
                w[4 * t + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int t = 0; t < kLaneCols; ++t) w[t] = 0.0f;
        }
        float s;
        if (a.grouped) {
            float m = 0.0f;
#pragma unroll
            for (int t = 0; t < kLaneCols; ++t) m = fmaxf(m, fabsf(w[t]));
            for (int o = kRowLanes / 2; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
            s = __fdiv_rn(m > 0.0f ? m : 1.0f, 7.5f);
        } else {
            s = ok ? a.rowscale[r] : 1.0f;
        }
        const float inv_s = __frcp_rn(s);
        uint32_t cw[kLaneCols / 4] = {0u, 0u, 0u, 0u};
        float lf = 0.0f;
        for (int so = 0; so < kRowLanes; ++so) {
#pragma unroll
            for (int k = 0; k < kLaneCols; ++k) {
                const int i = so * kLaneCols + k;
                float err = 0.0f;
                if (sl == so) {
                    const float x = w[k];
                    const float y = __fmul_rn(x, inv_s);
                    float q = rintf(y);
                    if (fabsf(fabsf(__fsub_rn(y, q)) - 0.5f) < 1e-4f) q = rintf(__fdiv_rn(x, s));
                    q = fminf(fmaxf(q, -8.0f), 7.0f);
                    err = __fmul_rn(__fsub_rn(x, __fmul_rn(s, q)), inv_u[i]);
                    lf = fmaf(err, err, lf);
                    cw[k >> 2] |= (static_cast<uint32_t>(static_cast<int>(q)) & 0xffu) << (8 * (k & 3));
                }
                err = __shfl_sync(kFull, err, grp | so);
                const float4* up = reinterpret_cast<const float4*>(Us + i * kNB + kLaneCols * sl);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float4 u = up[t];
                    w[4 * t] = __fsub_rn(w[4 * t], __fmul_rn(err, u.x));
                    w[4 * t + 1] = __fsub_rn(w[4 * t + 1], __fmul_rn(err, u.y));
                    w[4 * t + 2] = __fsub_rn(w[4 * t + 2], __fmul_rn(err, u.z));
                    w[4 * t + 3] = __fsub_rn(w[4 * t + 3], __fmul_rn(err, u.w));
                }
                if (sl == so) w[k] = err;
            }
        }
        if (ok) {
            float4* ep = reinterpret_cast<float4*>(a.Err + r * a.ld_err + kLaneCols * sl);
            float4* qp = reinterpret_cast<float4*>(a.Wq + r * a.d + b0 + kLaneCols * sl);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                ep[t] = make_float4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
                float qf[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    qf[u] = __fmul_rn(s, static_cast<float>(static_cast<signed char>((cw[t] >> (8 * u)) & 0xffu)));
                qp[t] = make_float4(qf[0], qf[1], qf[2], qf[3]);
            }
            if (a.codes)
                *reinterpret_cast<uint4*>(a.codes + r * a.d + b0 + kLaneCols * sl) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            if (a.grouped && sl == 0) a.scales[r * a.n_groups + a.b] = s;
            lsum += static_cast<double>(lf);
        }
    }
    for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
    if (lane == 0) red[threadIdx.x >> 5] = lsum;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int i = 0; i < kBlockThreads / 32; ++i) t += red[i];
        if (t != 0.0) atomicAdd(a.loss, 0.5 * t);
    }
}

// ------------------------------------------------------------- host side

hess_status gq_fail(hess_status s, const char* fmt, ...) {
    char buf[384];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    hk::set_last_error(buf);
    return s;
}

#define GQ_TRY(call)                                                                           \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return gq_fail(HESS_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));     \
    } while (0)

template <bool kTransB>
cudaError_t gemm(const float* A, int lda, const float* B, int ldb, float* C, int ldc, int M, int N, int K,
                 float alpha, int beta, int flags, cudaStream_t s) {
    if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
    GemmArgs g{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, flags};
    const dim3 grid(N / 128, (M + 127) / 128);
    gq_gemm_kernel<kTransB><<<grid, 256, 0, s>>>(g);
    return cudaGetLastError();
}

int stride_grid(size_t items, int sm_count) {
    const size_t want = (items + 255) / 256;
    const size_t cap = static_cast<size_t>(sm_count) * 8;
    return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

struct gptq_ctx {
    std::mutex mu;
    int device = 0;
    int sm_count = 0;
    int64_t d = 0, max_rows = 0;
    int n_blocks = 0;
    float* F = nullptr;         // d x d: J H J, then L, then (after prepare) U
    float* X = nullptr;         // d x d: inv(L) workspace
    float* Dinv = nullptr;      // n_blocks x 128 x 128 inverses of the diagonal blocks
    float* Wc = nullptr;        // max_rows x d working matrix
    float* Err = nullptr;       // max_rows x (kSuper * 128) errors of one super-block
    float* rowscale = nullptr;  // max_rows
    unsigned char* dead = nullptr;
    double* damp64 = nullptr;
    float* damp32 = nullptr;
    double* loss = nullptr;
    int* status = nullptr;
    bool prepared = false;
    int64_t n_tokens = 0;
};

namespace {

hess_status gq_check_device(int dev) {
    int cur = -1;
    GQ_TRY(cudaGetDevice(&cur));
    if (cur != dev)
        return gq_fail(HESS_ERR_INVALID, "handle belongs to device %d but device %d is current", dev, cur);
    return HESS_OK;
}

void gq_free(gptq_ctx* g) {
    cudaFree(g->F);
    cudaFree(g->X);
    cudaFree(g->Dinv);
    cudaFree(g->Wc);
    cudaFree(g->Err);
    cudaFree(g->rowscale);
    cudaFree(g->dead);
    cudaFree(g->damp64);
    cudaFree(g->damp32);
    cudaFree(g->loss);
    cudaFree(g->status);
}

bool misaligned(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 != 0; }

// Steps 2-4 on a device H (d x d fp32, symmetric), leaving U in g->F.
hess_status prepare_locked(gptq_ctx* g, const float* H, double damp_percent, cudaStream_t s,
                           float* damp_out) {
    const int d = static_cast<int>(g->d), n = g->n_blocks;
    const size_t dd = static_cast<size_t>(d) * d;
    g->prepared = false;
    GQ_TRY(cudaMemsetAsync(g->status, 0, sizeof(int), s));
    gq_damp_kernel<<<1, 1024, 0, s>>>(H, d, damp_percent, g->dead, g->damp64, g->damp32);
    GQ_TRY(cudaGetLastError());
    gq_rotate_in_kernel<<<stride_grid(dd / 4, g->sm_count), 256, 0, s>>>(H, g->F, d, g->dead, g->damp64);
    GQ_TRY(cudaGetLastError());
    // Blocked right-looking Cholesky of F = J H J.
    for (int k = 0; k < n; ++k) {
        gq_potrf_kernel<<<1, kPotrfThreads, kPotrfSmem, s>>>(g->F, d, k, g->Dinv, g->status);
        GQ_TRY(cudaGetLastError());
        const int rem = d - (k + 1) * kNB;
        if (rem == 0) break;
        float* A21 = g->F + static_cast<size_t>(k + 1) * kNB * d + static_cast<size_t>(k) * kNB;
        float* A22 = g->F + static_cast<size_t>(k + 1) * kNB * (d + 1);
        // L21 = A21 inv(L11)^T, in place (one 128-wide column tile).
        GQ_TRY(gemm<true>(A21, d, g->Dinv + static_cast<size_t>(k) * kNB * kNB, kNB, A21, d, rem, kNB, kNB,
                          1.0f, 0, 0, s));
        // A22 -= L21 L21^T on the tiles at or below the diagonal.
        GQ_TRY(gemm<true>(A21, d, A21, d, A22, d, rem, rem, kNB, -1.0f, 1, kGemmCLowerTiles, s));
    }
    // X = inv(L), block row by block row: X_k = inv(L_kk) (I_k - sum_{j<k} L_kj X_j),
    // with the sum accumulated into X by rank-128 updates after each row.
    GQ_TRY(cudaMemsetAsync(g->X, 0, dd * sizeof(float), s));
    gq_identity_kernel<<<(d + 255) / 256, 256, 0, s>>>(g->X, d);
    GQ_TRY(cudaGetLastError());
    for (int k = 0; k < n; ++k) {
        float* Xk = g->X + static_cast<size_t>(k) * kNB * d;
        const int cols = (k + 1) * kNB;
        GQ_TRY(gemm<false>(g->Dinv + static_cast<size_t>(k) * kNB * kNB, kNB, Xk, d, Xk, d, kNB, cols, kNB,
                           1.0f, 0, 0, s));
        const int rem = d - (k + 1) * kNB;
        if (rem == 0) break;
        const float* Lk = g->F + static_cast<size_t>(k + 1) * kNB * d + static_cast<size_t>(k) * kNB;
        GQ_TRY(gemm<false>(Lk, d, Xk, d, Xk + static_cast<size_t>(kNB) * d, d, rem, cols, kNB, -1.0f, 1, 0, s));
    }
    // U = J X J into F.
    gq_reverse_copy_kernel<<<stride_grid(dd / 4, g->sm_count), 256, 0, s>>>(g->X, g->F, dd / 4);
    GQ_TRY(cudaGetLastError());
    int status = 0;
    float damp = 0.0f;
    GQ_TRY(cudaMemcpyAsync(&status, g->status, sizeof(int), cudaMemcpyDeviceToHost, s));
    GQ_TRY(cudaMemcpyAsync(&damp, g->damp32, sizeof(float), cudaMemcpyDeviceToHost, s));
    GQ_TRY(cudaStreamSynchronize(s));
    if (damp_out) *damp_out = damp;
    if (status & 1)
        return gq_fail(HESS_ERR_NOT_PD, "the damped Hessian is not positive definite in fp32 "
                                        "(a Cholesky pivot was <= 0 or not finite)");
    g->prepared = true;
    return HESS_OK;
}

}  // namespace

#define GQ_EXPORT extern "C" __attribute__((visibility("default")))

GQ_EXPORT hess_status gptq_create(int64_t d, int64_t max_rows, gptq_t* out) {
    if (!out) return gq_fail(HESS_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d <= 0 || max_rows < 0) return gq_fail(HESS_ERR_INVALID, "d must be positive and max_rows >= 0");
    if (d % kNB != 0) return gq_fail(HESS_ERR_UNSUPPORTED, "d must be a multiple of 128 (got %lld)",
                                     static_cast<long long>(d));
    if (d > 32768) return gq_fail(HESS_ERR_UNSUPPORTED, "d > 32768");
    if (max_rows > (int64_t(1) << 26)) return gq_fail(HESS_ERR_UNSUPPORTED, "max_rows > 2^26");
    int dev = 0;
    GQ_TRY(cudaGetDevice(&dev));
    gptq_ctx* g = new (std::nothrow) gptq_ctx();
    if (!g) return gq_fail(HESS_ERR_OOM, "host allocation failed");
    g->device = dev;
    g->d = d;
    g->max_rows = max_rows;
    g->n_blocks = static_cast<int>(d / kNB);
    const size_t dd = static_cast<size_t>(d) * d;
    const size_t rows = static_cast<size_t>(max_rows > 0 ? max_rows : 1);
    cudaError_t e = cudaDeviceGetAttribute(&g->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gq_potrf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kPotrfSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gq_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kBlockSmem));
    if (e == cudaSuccess) e = cudaMalloc(&g->F, dd * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->X, dd * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->Dinv, static_cast<size_t>(d) * kNB * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->Wc, rows * d * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->Err, rows * kSuper * kNB * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->rowscale, rows * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->dead, static_cast<size_t>(d));
    if (e == cudaSuccess) e = cudaMalloc(&g->damp64, sizeof(double));
    if (e == cudaSuccess) e = cudaMalloc(&g->damp32, sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->loss, sizeof(double));
    if (e == cudaSuccess) e = cudaMalloc(&g->status, sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        const hess_status s = e == cudaErrorMemoryAllocation ? HESS_ERR_OOM : HESS_ERR_CUDA;
        gq_free(g);
        delete g;
        return gq_fail(s, "gptq_create: %s", cudaGetErrorString(e));
    }
    *out = g;
    return HESS_OK;
}

GQ_EXPORT hess_status gptq_prepare(gptq_t g, const float* H, int64_t n_tokens, double damp_percent,
                                   hess_stream_t stream, float* damp_value_out) {
    if (!g) return gq_fail(HESS_ERR_INVALID, "handle is NULL");
    if (!H) return gq_fail(HESS_ERR_INVALID, "H is NULL");
    if (misaligned(H)) return gq_fail(HESS_ERR_INVALID, "H is not 16-byte aligned");
    if (n_tokens < 0) return gq_fail(HESS_ERR_INVALID, "n_tokens < 0");
    if (!(damp_percent >= 0.0 && damp_percent < 1.0))
        return gq_fail(HESS_ERR_INVALID, "damp_percent must be in [0, 1)");
    std::lock_guard<std::mutex> lk(g->mu);
    hess_status st = gq_check_device(g->device);
    if (st != HESS_OK) return st;
    st = prepare_locked(g, H, damp_percent, static_cast<cudaStream_t>(stream), damp_value_out);
    if (st == HESS_OK) g->n_tokens = n_tokens;
    return st;
}

GQ_EXPORT hess_status gptq_prepare_hess(gptq_t g, hess_t h, double damp_percent, hess_stream_t stream,
                                        float* damp_value_out) {
    if (!g || !h) return gq_fail(HESS_ERR_INVALID, "handle is NULL");
    if (hess_dim(h) != g->d)
        return gq_fail(HESS_ERR_INVALID, "Hessian width %lld != quantizer width %lld",
                       static_cast<long long>(hess_dim(h)), static_cast<long long>(g->d));
    if (!(damp_percent >= 0.0 && damp_percent < 1.0))
        return gq_fail(HESS_ERR_INVALID, "damp_percent must be in [0, 1)");
    std::lock_guard<std::mutex> lk(g->mu);
    hess_status st = gq_check_device(g->device);
    if (st != HESS_OK) return st;
    // The undamped H lands in the inverse workspace, which prepare reads
    // (into F) before it reuses it.
    st = hess_materialize(h, g->X, 0.0, stream, nullptr);
    if (st != HESS_OK) return st;
    st = prepare_locked(g, g->X, damp_percent, static_cast<cudaStream_t>(stream), damp_value_out);
    if (st == HESS_OK) g->n_tokens = hess_token_count(h);
    return st;
}

GQ_EXPORT hess_status gptq_read_factor(gptq_t g, float* U_out, hess_stream_t stream) {
    if (!g) return gq_fail(HESS_ERR_INVALID, "handle is NULL");
    if (!U_out) return gq_fail(HESS_ERR_INVALID, "U_out is NULL");
    std::lock_guard<std::mutex> lk(g->mu);
    hess_status st = gq_check_device(g->device);
    if (st != HESS_OK) return st;
    if (!g->prepared) return gq_fail(HESS_ERR_INVALID, "no factor: gptq_prepare has not succeeded");
    GQ_TRY(cudaMemcpyAsync(U_out, g->F, static_cast<size_t>(g->d) * g->d * sizeof(float),
                           cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
    return HESS_OK;
}

GQ_EXPORT hess_status gptq_quantize(gptq_t g, const void* W, int32_t w_dtype, int64_t rows,
                                    int32_t group_size, float* Wq_out, float* scales_out,
                                    int8_t* codes_out, hess_stream_t stream, double* avg_loss_out) {
    if (!g) return gq_fail(HESS_ERR_INVALID, "handle is NULL");
    if (rows < 0) return gq_fail(HESS_ERR_INVALID, "rows < 0");
    if (rows > g->max_rows)
        return gq_fail(HESS_ERR_INVALID, "rows %lld > max_rows %lld", static_cast<long long>(rows),
                       static_cast<long long>(g->max_rows));
    if (w_dtype != HESS_BF16 && w_dtype != HESS_F32) return gq_fail(HESS_ERR_INVALID, "unknown dtype %d", w_dtype);
    if (group_size != -1 && group_size != kNB)
        return gq_fail(HESS_ERR_UNSUPPORTED, "group_size must be -1 or 128 (got %d)", group_size);
    if (rows > 0) {
        if (!W || !Wq_out || !scales_out) return gq_fail(HESS_ERR_INVALID, "W, Wq_out or scales_out is NULL");
        if (misaligned(W) || misaligned(Wq_out) || misaligned(codes_out))
            return gq_fail(HESS_ERR_INVALID, "W, Wq_out and codes_out must be 16-byte aligned");
    }
    std::lock_guard<std::mutex> lk(g->mu);
    hess_status st = gq_check_device(g->device);
    if (st != HESS_OK) return st;
    if (!g->prepared) return gq_fail(HESS_ERR_INVALID, "no factor: gptq_prepare has not succeeded");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int d = static_cast<int>(g->d), n = g->n_blocks;
    const bool grouped = group_size == kNB;
    GQ_TRY(cudaMemsetAsync(g->loss, 0, sizeof(double), s));
    if (rows > 0) {
        const size_t n4 = static_cast<size_t>(rows) * d / 4;
        if (w_dtype == HESS_F32)
            gq_load_w_kernel<float><<<stride_grid(n4, g->sm_count), 256, 0, s>>>(
                static_cast<const float*>(W), g->Wc, n4, d, g->dead);
        else
            gq_load_w_kernel<__nv_bfloat16><<<stride_grid(n4, g->sm_count), 256, 0, s>>>(
                static_cast<const __nv_bfloat16*>(W), g->Wc, n4, d, g->dead);
        GQ_TRY(cudaGetLastError());
        if (!grouped) {
            gq_rowscale_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, s>>>(
                g->Wc, rows, d, g->rowscale, scales_out);
            GQ_TRY(cudaGetLastError());
        }
        const int wanted = static_cast<int>((rows + kBlockRows - 1) / kBlockRows);
        const int grid = std::min(wanted, 3 * g->sm_count);
        const int ld_err = kSuper * kNB;
        // Two-level lazy update: after each block only the rest of its
        // super-block (kSuper blocks) is updated; the columns after the
        // super-block get one K = kSuper * 128 update.
        for (int sb0 = 0; sb0 < n; sb0 += kSuper) {
            const int sb1 = std::min(n, sb0 + kSuper);
            for (int b = sb0; b < sb1; ++b) {
                float* err_b = g->Err + (b - sb0) * kNB;
                BlockArgs a{g->Wc, g->F, Wq_out, reinterpret_cast<signed char*>(codes_out), scales_out, err_b,
                            g->rowscale, g->loss, rows, d, b, grouped ? n : 1, grouped ? 1 : 0, ld_err};
                gq_block_kernel<<<grid, kBlockThreads, kBlockSmem, s>>>(a);
                GQ_TRY(cudaGetLastError());
                const int in_super = (sb1 - b - 1) * kNB;  // columns left in this super-block
                if (in_super > 0)
                    GQ_TRY(gemm<false>(err_b, ld_err, g->F + static_cast<size_t>(b) * kNB * d + (b + 1) * kNB, d,
                                       g->Wc + (b + 1) * kNB, d, static_cast<int>(rows), in_super, kNB, -1.0f, 1, 0,
                                       s));
            }
            const int rest = d - sb1 * kNB;
            if (rest > 0)
                GQ_TRY(gemm<false>(g->Err, ld_err, g->F + static_cast<size_t>(sb0) * kNB * d + sb1 * kNB, d,
                                   g->Wc + sb1 * kNB, d, static_cast<int>(rows), rest, (sb1 - sb0) * kNB, -1.0f, 1,
                                   0, s));
        }
    }
    if (avg_loss_out) {
        double loss = 0.0;
        GQ_TRY(cudaMemcpyAsync(&loss, g->loss, sizeof(double), cudaMemcpyDeviceToHost, s));
        GQ_TRY(cudaStreamSynchronize(s));
        *avg_loss_out = g->n_tokens > 0 ? loss / static_cast<double>(g->n_tokens) : loss;
    }
    return HESS_OK;
}

GQ_EXPORT hess_status gptq_destroy(gptq_t g) {
    if (!g) return HESS_OK;
    {
        std::lock_guard<std::mutex> lk(g->mu);
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(g->device);
        cudaDeviceSynchronize();
        gq_free(g);
        cudaSetDevice(cur);
    }
    delete g;
    return HESS_OK;
}
