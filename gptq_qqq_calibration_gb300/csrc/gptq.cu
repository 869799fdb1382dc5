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

#include "device_ptr.h"
#include "gptq.h"
#include "hess.h"
#include "kernels.cuh"

namespace {

constexpr int kNB = 128;          // column block of the factorization and of step 5
constexpr int kLd = kNB + 1;      // padded row of the diagonal-block tiles
constexpr int kGemmLd = 132;      // padded row of the GEMM k-slices
constexpr int kGemmCLowerTiles = 1;
constexpr int kPotrfThreads = 256;
constexpr int kBlockThreads = 128;
constexpr int kSuper = 4;          // blocks per lazy super-block of step 5
constexpr size_t kBlockSmem = kNB * kNB * sizeof(float);
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kGemmTimeoutNs = 2000000000ull;  // bound of every wait in the tensor GEMM

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
// inv(L_kk) to Dinv.  The 128 columns go in sub-panels of kSub:
//   1. one warp factors the kSub x kSub diagonal sub-block in registers
//      (lane i holds row i; pivots and column entries travel by shuffle) and
//      inverts it by forward substitution (lane j holds column j of the
//      inverse).  The unrolled code of this step is kept small enough to stay
//      in the instruction cache: with 32 columns it was fetch-bound;
//   2. all warps solve the rows below the sub-panel, L21 = A21 inv(L11)^T,
//      in 4 x 4 register tiles;
//   3. all warps apply the rank-kSub update to the rows and columns after it.
// The 128 x 128 inverse is built alongside, right-looking by block columns:
// with B = I, block row p becomes X_p = Y_p B_p (Y_p the sub-block inverse)
// once its sub-panel is factored, and every later block row then takes
// B_i -= L_ip X_p; these steps share the sub-panel loop's barriers.
// A pivot that is not a positive finite number sets status bit 1 and is
// replaced by 1 so the kernel still ends normally.
constexpr int kSub = 16;             // sub-panel width (one warp's register factor)
constexpr int kSubT = kSub / 4;       // 4-wide tiles across a sub-panel
constexpr int kLtLd = kNB + 4;        // transposed panel rows (float4-aligned)
constexpr int kYtLd = kSub + 4;       // transposed sub-block inverse rows
constexpr size_t kPotrfFloats =
    2 * kNB * kLd + kSub * kLtLd + kSub * kYtLd + kNB;
constexpr size_t kPotrfSmem = kPotrfFloats * sizeof(float);

// Step 1 of the diagonal-block kernel for the sub-panel at column P, run by
// one warp: register factor of the kSub x kSub diagonal sub-block and its
// inverse (into S, Xs's diagonal sub-block, Yt and rl).  Returns true if a
// pivot was replaced.  Inlined at both call sites: as a call it cost the
// critical warp more than the duplicated code costs the instruction cache.
__device__ __forceinline__ bool potrf_sub_block(float* S, float* Xs, float* Yt, float* rl, int P, int lane) {
    bool bad = false;
    // Lanes kSub..31 take part in the shuffles only.
    const bool in = lane < kSub;
    float dv[kSub];
#pragma unroll
    for (int c = 0; c < kSub; ++c) dv[c] = in ? S[(P + lane) * kLd + P + c] : 0.0f;
#pragma unroll
    for (int j = 0; j < kSub; ++j) {
        float piv = __shfl_sync(kFull, dv[j], j);
        if (!(piv > 0.0f) || !(piv < INFINITY)) {
            bad = true;
            piv = 1.0f;
        }
        // 1/sqrt by the hardware estimate and one Newton step,
        // y <- y (1.5 - 0.5 x y^2): the pivot chain is the
        // sequential path of the whole factorization.
        float il = rsqrtf(piv);
        il = __fmul_rn(il, fmaf(-0.5f * piv * il, il, 1.5f));
        const float l = __fmul_rn(piv, il);
        if (lane == j) dv[j] = l;
        else if (lane > j) dv[j] = __fmul_rn(dv[j], il);
        if (lane == 0) rl[P + j] = il;
#pragma unroll
        for (int c = 0; c < kSub; ++c) {
            if (c > j) {  // resolved at compile time
                const float lc = __shfl_sync(kFull, dv[j], c);
                if (lane >= c) dv[c] = fmaf(-dv[j], lc, dv[c]);
            }
        }
    }
    if (in) {
#pragma unroll
        for (int c = 0; c < kSub; ++c) S[(P + lane) * kLd + P + c] = c <= lane ? dv[c] : 0.0f;
    }
    __syncwarp();
    // Column `lane` of the sub-block inverse: solve L y = e_lane.
    float acc[kSub];
#pragma unroll
    for (int i = 0; i < kSub; ++i) acc[i] = i == lane ? 1.0f : 0.0f;
#pragma unroll
    for (int m = 0; m < kSub; ++m) {
        acc[m] = __fmul_rn(acc[m], rl[P + m]);
#pragma unroll
        for (int i = 0; i < kSub; ++i)
            if (i > m) acc[i] = fmaf(-S[(P + i) * kLd + P + m], acc[m], acc[i]);
    }
    if (in) {
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            Xs[(P + i) * kLd + P + lane] = acc[i];  // Y[i][lane] (0 for i < lane)
            Yt[lane * kYtLd + i] = acc[i];           // Yt[m][c] = Y[c][m]
        }
    }
    return bad;
}

__global__ void __launch_bounds__(kPotrfThreads, 1) gq_potrf_kernel(float* __restrict__ F, int d, int k,
                                                                 float* __restrict__ Dinv,
                                                                 float* __restrict__ DinvT,
                                                                 int* __restrict__ status) {
    extern __shared__ __align__(16) float sm[];
    float* S = sm;                  // [kNB][kLd]: the block, then L
    float* Xs = S + kNB * kLd;      // [kNB][kLd]: inv(L)
    float* Lt = Xs + kNB * kLd;     // [kSub][kLtLd]: L21 of the current sub-panel, transposed
    float* Yt = Lt + kSub * kLtLd;  // [kSub][kYtLd]: inverse of the current sub-block, transposed
    float* rl = Yt + kSub * kYtLd;  // [kNB]: 1 / L_ii
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float* blk = F + static_cast<size_t>(k) * kNB * d + static_cast<size_t>(k) * kNB;
    constexpr int kVecPerThread = kNB * kNB / 4 / kPotrfThreads;
    {
        float4 v[kVecPerThread];  // every load in flight before the first store
#pragma unroll
        for (int it = 0; it < kVecPerThread; ++it) {
            const int e4 = tid + it * kPotrfThreads, i = e4 >> 5, j = (e4 & 31) * 4;
            v[it] = *reinterpret_cast<const float4*>(blk + static_cast<size_t>(i) * d + j);
        }
#pragma unroll
        for (int it = 0; it < kVecPerThread; ++it) {
            const int e4 = tid + it * kPotrfThreads, i = e4 >> 5, j = (e4 & 31) * 4;
            const float x[4] = {v[it].x, v[it].y, v[it].z, v[it].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                S[i * kLd + j + u] = j + u <= i ? x[u] : 0.0f;
                Xs[i * kLd + j + u] = 0.0f;
            }
        }
    }
    __syncthreads();
    bool bad = false;
    for (int p = 0; p < kNB / kSub; ++p) {
        const int P = p * kSub;
        if (p == 0) {  // later sub-panels are factored inside step 3 of the previous one
            if (warp == 0) bad |= potrf_sub_block(S, Xs, Yt, rl, P, lane);
        }
        __syncthreads();
        const int R0 = P + kSub;  // first row after the sub-panel
        const int nb = kNB - R0;
        // 2. In registers: tiles of L21 = A21 Y^T (threads [0, n2)) and tiles of
        //    block row p of the inverse, X_p,j = Y B_p,j for the columns before
        //    the sub-panel (threads [n2, n2 + P)); B_p,j holds I - sum L X there.
        const int n2 = (nb / 4) * kSubT;
        int mode = 0, r0 = 0, c0 = 0;
        float a2[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int u = 0; u < 4; ++u) a2[t][u] = 0.0f;
        if (tid < n2) {
            mode = 1;
            r0 = R0 + 4 * (tid / kSubT);
            c0 = 4 * (tid % kSubT);
            for (int m = 0; m < c0 + 4; ++m) {  // Y[c][m] = 0 for m > c
                const float4 y = *reinterpret_cast<const float4*>(&Yt[m * kYtLd + c0]);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float av = S[(r0 + t) * kLd + P + m];
                    a2[t][0] = fmaf(av, y.x, a2[t][0]);
                    a2[t][1] = fmaf(av, y.y, a2[t][1]);
                    a2[t][2] = fmaf(av, y.z, a2[t][2]);
                    a2[t][3] = fmaf(av, y.w, a2[t][3]);
                }
            }
        } else if (tid < n2 + P) {
            mode = 2;
            const int q = tid - n2;
            r0 = 4 * (q % kSubT);  // row within block row p
            c0 = 4 * (q / kSubT);  // column < P
            for (int m = 0; m < r0 + 4; ++m) {  // Y[t][m] = 0 for m > t
                const float4 y = *reinterpret_cast<const float4*>(&Yt[m * kYtLd + r0]);
                const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float bv = Xs[(P + m) * kLd + c0 + u];
#pragma unroll
                    for (int t = 0; t < 4; ++t) a2[t][u] = fmaf(yv[t], bv, a2[t][u]);
                }
            }
        }
        __syncthreads();  // every read of A21 and B_p is done
        if (mode == 1) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u) S[(r0 + t) * kLd + P + c0 + u] = a2[t][u];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<float4*>(&Lt[(c0 + u) * kLtLd + (r0 - R0)]) =
                    make_float4(a2[0][u], a2[1][u], a2[2][u], a2[3][u]);
        } else if (mode == 2) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u) Xs[(P + r0 + t) * kLd + c0 + u] = a2[t][u];
        }
        __syncthreads();
        if (nb == 0) break;
        // 3. On 4 x 4 tiles: A22 -= L21 L21^T at or below the diagonal
        //    (triangular index idx < n3), and B_i,j -= L_ip X_p,j for the rows
        //    after the sub-panel and the columns up to its end (the rest).
        //    Look-ahead: warp 0 updates the next diagonal sub-block (the
        //    first kSubT (kSubT + 1) / 2 tiles) and factors it at once, while
        //    the other warps apply the rest of the update; the next
        //    sub-panel's factor touches none of their tiles.
        const int nt = nb / 4;
        const int n3 = nt * (nt + 1) / 2;
        const int ct = (P + kSub) / 4;
        constexpr int kDiagTiles = kSubT * (kSubT + 1) / 2;
        auto tile = [&](int idx) {
            float a3[4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u) a3[t][u] = 0.0f;
            if (idx < n3) {
                int ta = static_cast<int>((sqrtf(8.0f * idx + 1.0f) - 1.0f) * 0.5f);
                while (ta * (ta + 1) / 2 > idx) --ta;
                while ((ta + 1) * (ta + 2) / 2 <= idx) ++ta;
                const int tb = idx - ta * (ta + 1) / 2;  // 0 <= tb <= ta < nt
#pragma unroll 4
                for (int m = 0; m < kSub; ++m) {
                    const float4 x = *reinterpret_cast<const float4*>(&Lt[m * kLtLd + 4 * ta]);
                    const float4 y = *reinterpret_cast<const float4*>(&Lt[m * kLtLd + 4 * tb]);
                    const float xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t)
#pragma unroll
                        for (int u = 0; u < 4; ++u) a3[t][u] = fmaf(xv[t], yv[u], a3[t][u]);
                }
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int u = 0; u < 4; ++u) S[(R0 + 4 * ta + t) * kLd + R0 + 4 * tb + u] -= a3[t][u];
            } else {
                const int q = idx - n3;
                const int ta = q / ct, tb = q % ct;  // row tile after R0, column tile
#pragma unroll 4
                for (int m = 0; m < kSub; ++m) {
                    const float4 x = *reinterpret_cast<const float4*>(&Lt[m * kLtLd + 4 * ta]);
                    const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float bv = Xs[(P + m) * kLd + 4 * tb + u];
#pragma unroll
                        for (int t = 0; t < 4; ++t) a3[t][u] = fmaf(xv[t], bv, a3[t][u]);
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int u = 0; u < 4; ++u) Xs[(R0 + 4 * ta + t) * kLd + 4 * tb + u] -= a3[t][u];
            }
        };
        if (warp == 0) {
            if (lane < kDiagTiles) tile(lane);
            __syncwarp();
            bad |= potrf_sub_block(S, Xs, Yt, rl, R0, lane);
        } else {
            for (int idx = kDiagTiles + tid - 32; idx < n3 + nt * ct; idx += kPotrfThreads - 32) tile(idx);
        }
        __syncthreads();
    }
    if (bad && tid == 0) atomicOr(status, 1);

    float* inv = Dinv + static_cast<size_t>(k) * kNB * kNB;
#pragma unroll 4
    for (int it = 0; it < kVecPerThread; ++it) {
        const int e4 = tid + it * kPotrfThreads, i = e4 >> 5, j = (e4 & 31) * 4;
        float l[4], x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            l[u] = j + u <= i ? S[i * kLd + j + u] : 0.0f;
            x[u] = j + u <= i ? Xs[i * kLd + j + u] : 0.0f;
        }
        *reinterpret_cast<float4*>(blk + static_cast<size_t>(i) * d + j) = make_float4(l[0], l[1], l[2], l[3]);
        *reinterpret_cast<float4*>(inv + i * kNB + j) = make_float4(x[0], x[1], x[2], x[3]);
    }
    // inv(L_kk)^T: row i holds column i of the inverse (nonzero from row i down).
    float* invT = DinvT + static_cast<size_t>(k) * kNB * kNB;
#pragma unroll 4
    for (int it = 0; it < kVecPerThread; ++it) {
        const int e4 = tid + it * kPotrfThreads, i = e4 >> 5, j = (e4 & 31) * 4;
        float y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) y[u] = i <= j + u ? Xs[(j + u) * kLd + i] : 0.0f;
        *reinterpret_cast<float4*>(invT + i * kNB + j) = make_float4(y[0], y[1], y[2], y[3]);
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
    long long sA, sB, sC;  // element strides between the problems of a batch (grid z)
    int diag_step;         // lower-tile test of problem z: skip tiles with n0 > m0 + z * diag_step
};

// C = beta C + alpha A op(B) in fp32 (FMA chains along k, one rounding per
// step).  BM x 128 output tile per CTA (BM = 128, or 32 for narrow problems
// whose 128-row grid would not fill the SMs), k-slices of 8 double-buffered
// in shared memory, BM/16 x 8 outputs per thread.  N % 128 == 0 and
// K % 8 == 0; rows of A and C beyond M are skipped.  A CTA reads only the
// rows of A and the columns of op(B) of its own tile, and writes C after all
// its reads, so C may alias A when N == 128, or alias B when K == 128, op(B)
// is not transposed and one row tile covers M (BM = 128 >= M).
template <bool kTransB, int BM>
__global__ void __launch_bounds__(256) gq_gemm_kernel(const GemmArgs g) {
    static_assert(BM == 128 || BM == 32, "tile height");
    constexpr int RM = BM / 16;  // rows per thread
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * 128;
    if ((g.flags & kGemmCLowerTiles) && n0 >= m0 + BM + static_cast<int>(blockIdx.z) * g.diag_step) return;
    const float* Ab = g.A + blockIdx.z * g.sA;
    const float* Bb = g.B + blockIdx.z * g.sB;
    float* Cb = g.C + blockIdx.z * g.sC;
    __shared__ __align__(16) float As[2][8][BM + 4];
    __shared__ __align__(16) float Bs[2][8][kGemmLd];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int r_row = tid >> 1, r_col = (tid & 1) * 4;  // row-of-8 loader (A, transposed B)
    const int b_k = tid >> 5, b_n = (tid & 31) * 4;     // plain B loader
    const bool a_loader = r_row < BM;
    const bool a_ok = a_loader && m0 + r_row < g.M;
    const float* a_src = Ab + static_cast<size_t>(a_ok ? m0 + r_row : 0) * g.lda + r_col;
    float acc[RM][8];
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    float4 ra, rb;
    auto load = [&](int k0) {
        // Plain loads: C may alias A or B, so the read-only path is not used.
        ra = a_ok ? *reinterpret_cast<const float4*>(a_src + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (kTransB)
            rb = *reinterpret_cast<const float4*>(Bb + static_cast<size_t>(n0 + r_row) * g.ldb + k0 + r_col);
        else
            rb = *reinterpret_cast<const float4*>(Bb + static_cast<size_t>(k0 + b_k) * g.ldb + n0 + b_n);
    };
    auto store = [&](int buf) {
        if (a_loader) {
            As[buf][r_col + 0][r_row] = ra.x;
            As[buf][r_col + 1][r_row] = ra.y;
            As[buf][r_col + 2][r_row] = ra.z;
            As[buf][r_col + 3][r_row] = ra.w;
        }
        if (kTransB) {
            Bs[buf][r_col + 0][r_row] = rb.x;
            Bs[buf][r_col + 1][r_row] = rb.y;
            Bs[buf][r_col + 2][r_row] = rb.z;
            Bs[buf][r_col + 3][r_row] = rb.w;
        } else {
            *reinterpret_cast<float4*>(&Bs[buf][b_k][b_n]) = rb;
        }
    };
    // the row of thread row i within the tile
    auto row_of = [&](int i) { return BM == 128 ? (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4) : ty * RM + i; };

    load(0);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < g.K; k0 += 8) {
        const bool more = k0 + 8 < g.K;
        if (more) load(k0 + 8);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            float a[RM];
            if constexpr (BM == 128) {
                const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
                const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
                a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
                a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            } else {
                const float2 a0 = *reinterpret_cast<const float2*>(&As[buf][kk][ty * RM]);
                a[0] = a0.x; a[1] = a0.y;
            }
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < RM; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) store(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }

#pragma unroll
    for (int i = 0; i < RM; ++i) {
        const int m = m0 + row_of(i);
        if (m >= g.M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float4* cp = reinterpret_cast<float4*>(Cb + static_cast<size_t>(m) * g.ldc + n0 + h * 64 + tx * 4);
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
    float* ErrT;            // scaled errors of this block, transposed: 128 x rows at stride ld_errt
    const float* rowscale;  // whole-row scales (grouped == 0)
    double* loss;
    int64_t rows;
    int d, b, n_groups, grouped, ld_errt;
};

constexpr int kRowLanes = 8;   // lanes per weight row
constexpr int kLaneCols = 16;  // consecutive block columns per lane
constexpr int kBlockRows = kBlockThreads / kRowLanes;

// One 128-column block of step 5.  Eight lanes hold one weight row (four
// rows per warp); lane l holds block columns 32t + 4l + u (t, u = 0..3), so
// every row-of-U load and every global access of the eight lanes covers 128
// contiguous bytes.  Column i is quantized by the lane that holds it, its
// scaled error err = (w - q) / U_ii is broadcast to the row's lanes, and
// every lane applies w_j -= err * U_ij to its columns (U_ij = 0 for j < i, so
// columns already quantized keep their value; the owner then parks err in
// the slot of column i).  Every lane evaluates the quantizer on its own slot
// and only the owner's result is used, so the common path has no divergent
// branch.  The code is rint(w / s) with w / s rounded to nearest as an fp32
// division: w * (1/s) is used unless it lies within 1e-4 of a half integer,
// where the correctly rounded quotient decides (a warp-uniform, rarely taken
// branch).  Grouped blocks take their scale from the block's values as they
// stand when the block starts.
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
        float w[kLaneCols];  // slot 4t + u <-> block column 32t + 4 sl + u
        if (ok) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 v = *reinterpret_cast<const float4*>(a.Wc + r * a.d + b0 + 32 * t + 4 * sl);
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
        uint32_t cw[4] = {0u, 0u, 0u, 0u};
        float lf = 0.0f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            for (int so = 0; so < kRowLanes; ++so) {
                const bool own = sl == so;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = 4 * t + u;
                    const int i = 32 * t + 4 * so + u;
                    // every lane evaluates its slot k; the owner's result counts
                    const float x = w[k];
                    const float y = __fmul_rn(x, inv_s);
                    float q = rintf(y);
                    const bool tie = fabsf(fabsf(__fsub_rn(y, q)) - 0.5f) < 1e-4f;
                    if (__any_sync(kFull, tie && own)) {
                        if (tie && own) q = rintf(__fdiv_rn(x, s));
                    }
                    q = fminf(fmaxf(q, -8.0f), 7.0f);
                    const float e = __fmul_rn(__fsub_rn(x, __fmul_rn(s, q)), inv_u[i]);
                    lf = own ? fmaf(e, e, lf) : lf;
                    cw[t] |= own ? (static_cast<uint32_t>(static_cast<int>(q)) & 0xffu) << (8 * u) : 0u;
                    const float err = __shfl_sync(kFull, e, grp | so);
#pragma unroll
                    for (int tt = 0; tt < 4; ++tt) {
                        const float4 uv = *reinterpret_cast<const float4*>(Us + i * kNB + 32 * tt + 4 * sl);
                        w[4 * tt] = __fsub_rn(w[4 * tt], __fmul_rn(err, uv.x));
                        w[4 * tt + 1] = __fsub_rn(w[4 * tt + 1], __fmul_rn(err, uv.y));
                        w[4 * tt + 2] = __fsub_rn(w[4 * tt + 2], __fmul_rn(err, uv.z));
                        w[4 * tt + 3] = __fsub_rn(w[4 * tt + 3], __fmul_rn(err, uv.w));
                    }
                    w[k] = own ? err : w[k];
                }
            }
        }
        if (ok) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int c = 32 * t + 4 * sl;
#pragma unroll
                for (int u = 0; u < 4; ++u) a.ErrT[static_cast<size_t>(c + u) * a.ld_errt + r] = w[4 * t + u];
                float qf[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    qf[u] = __fmul_rn(s, static_cast<float>(static_cast<signed char>((cw[t] >> (8 * u)) & 0xffu)));
                *reinterpret_cast<float4*>(a.Wq + r * a.d + b0 + c) = make_float4(qf[0], qf[1], qf[2], qf[3]);
                if (a.codes) *reinterpret_cast<uint32_t*>(a.codes + r * a.d + b0 + c) = cw[t];
            }
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

// `narrow_ok`: 32-row tiles may be used (not when C aliases B, whose
// column tile would then be shared by several CTAs).
template <bool kTransB>
cudaError_t gemm(int sm_count, const float* A, int lda, const float* B, int ldb, float* C, int ldc, int M,
                 int N, int K, float alpha, int beta, int flags, cudaStream_t s, int batch = 1,
                 long long sA = 0, long long sB = 0, long long sC = 0, int diag_step = 0,
                 bool narrow_ok = true) {
    if (M <= 0 || N <= 0 || K <= 0 || batch <= 0) return cudaSuccess;
    GemmArgs g{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, flags, sA, sB, sC, diag_step};
    // 128-row tiles unless they leave SMs idle; then 32-row tiles (4x the CTAs).
    const long long tiles128 = static_cast<long long>(N / 128) * ((M + 127) / 128) * batch;
    if (tiles128 >= sm_count || !narrow_ok) {
        gq_gemm_kernel<kTransB, 128><<<dim3(N / 128, (M + 127) / 128, batch), 256, 0, s>>>(g);
    } else {
        gq_gemm_kernel<kTransB, 32><<<dim3(N / 128, (M + 31) / 32, batch), 256, 0, s>>>(g);
    }
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
    float* ErrT = nullptr;      // (kSuper * 128) x ld_errt: errors of one super-block, transposed
    int ld_errt = 0;            // max_rows rounded up to a multiple of 4 (16-byte rows)
    float* rowscale = nullptr;  // max_rows
    unsigned char* dead = nullptr;
    double* damp64 = nullptr;
    float* damp32 = nullptr;
    double* loss = nullptr;
    int* status = nullptr;
    float* DinvT = nullptr;          // the inverses of the diagonal blocks, transposed
    float* L21T[2] = {nullptr, nullptr};  // 128 x (d - 128): a step's panel, transposed (two steps in flight)
    float* MkT = nullptr;            // 128 x (d - 128): (L_ik inv(L_kk))^T of one step
    cudaStream_t side = nullptr;     // inverse block rows, alongside the Cholesky
    cudaEvent_t ev_fork = nullptr, ev_panel = nullptr, ev_side = nullptr;
    cudaEvent_t ev_l21t[2] = {nullptr, nullptr};  // the side stream has read panel buffer 0 / 1
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

// A caller's buffer must be device memory of the handle's device (or
// managed memory); anything else is refused before a kernel could touch it.
hess_status gq_check_buffer(const void* p, int dev, const char* name) {
    char why[128];
    if (const char* w = hk::device_ptr_problem(p, dev, why)) return gq_fail(HESS_ERR_INVALID, "%s %s", name, w);
    return HESS_OK;
}

void gq_free(gptq_ctx* g) {
    cudaFree(g->F);
    cudaFree(g->X);
    cudaFree(g->Dinv);
    cudaFree(g->Wc);
    cudaFree(g->ErrT);
    cudaFree(g->rowscale);
    cudaFree(g->dead);
    cudaFree(g->damp64);
    cudaFree(g->damp32);
    cudaFree(g->loss);
    cudaFree(g->status);
    cudaFree(g->DinvT);
    cudaFree(g->L21T[0]);
    cudaFree(g->L21T[1]);
    cudaFree(g->MkT);
    for (int i = 0; i < 2; ++i)
        if (g->ev_l21t[i]) cudaEventDestroy(g->ev_l21t[i]);
    if (g->side) cudaStreamDestroy(g->side);
    if (g->ev_fork) cudaEventDestroy(g->ev_fork);
    if (g->ev_panel) cudaEventDestroy(g->ev_panel);
    if (g->ev_side) cudaEventDestroy(g->ev_side);
}

bool misaligned(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 != 0; }

// Steps 2-4 on a device H (d x d fp32, symmetric), leaving U in g->F.
hess_status prepare_locked(gptq_ctx* g, const float* H, double damp_percent, cudaStream_t s,
                           float* damp_out) {
    const int d = static_cast<int>(g->d), n = g->n_blocks;
    const size_t dd = static_cast<size_t>(d) * d;
    g->prepared = false;
    GQ_TRY(cudaMemsetAsync(g->status, 0, 2 * sizeof(int), s));
    gq_damp_kernel<<<1, 1024, 0, s>>>(H, d, damp_percent, g->dead, g->damp64, g->damp32);
    GQ_TRY(cudaGetLastError());
    gq_rotate_in_kernel<<<stride_grid(dd / 4, g->sm_count), 256, 0, s>>>(H, g->F, d, g->dead, g->damp64);
    GQ_TRY(cudaGetLastError());
    // Blocked right-looking Cholesky of F = J H J on `s`, and alongside it on
    // the side stream the block rows of inv(L): with B = I - (strictly lower
    // sums), X_k = inv(L_kk) B_k, and after step k every later block row
    // takes B_i -= (L_ik inv(L_kk)) B_k.  The factors M_k = L_ik inv(L_kk)
    // are formed from the finished panel, so only the Cholesky itself is on
    // the critical path; the products X_k = inv(L_kk) B_k run at the end in
    // one batched launch.  The side stream reads only finished panels and
    // inv(L_kk) and writes only X and M_k (reused in its own order).
    GQ_TRY(cudaMemsetAsync(g->X, 0, dd * sizeof(float), s));
    gq_identity_kernel<<<(d + 255) / 256, 256, 0, s>>>(g->X, d);
    GQ_TRY(cudaGetLastError());
    GQ_TRY(cudaEventRecord(g->ev_fork, s));
    GQ_TRY(cudaStreamWaitEvent(g->side, g->ev_fork, 0));
    uint32_t* gemm_status = reinterpret_cast<uint32_t*>(g->status) + 1;
    for (int k = 0; k < n; ++k) {
        gq_potrf_kernel<<<1, kPotrfThreads, kPotrfSmem, s>>>(g->F, d, k, g->Dinv, g->DinvT, g->status);
        GQ_TRY(cudaGetLastError());
        const int rem = d - (k + 1) * kNB;
        if (rem == 0) break;
        const float* A21 = g->F + static_cast<size_t>(k + 1) * kNB * d + static_cast<size_t>(k) * kNB;
        float* A22 = g->F + static_cast<size_t>(k + 1) * kNB * (d + 1);
        const float* Dk = g->Dinv + static_cast<size_t>(k) * kNB * kNB;
        const float* DkT = g->DinvT + static_cast<size_t>(k) * kNB * kNB;
        float* L21T = g->L21T[k & 1];  // 128 x rem, leading dimension rem
        // The side stream reads a panel two steps before its buffer is reused.
        if (k >= 2) GQ_TRY(cudaStreamWaitEvent(s, g->ev_l21t[k & 1], 0));
        // L21^T = inv(L11) A21^T (CUDA cores; 128 rows).
        GQ_TRY(gemm<true>(g->sm_count, Dk, kNB, A21, d, L21T, rem, kNB, rem, kNB, 1.0f, 0, 0, s));
        GQ_TRY(cudaEventRecord(g->ev_panel, s));
        // A22 -= L21 L21^T on the tensor cores, tiles at or below the diagonal.
        GQ_TRY(hk::launch_gemm_tf32(L21T, rem, L21T, rem, A22, d, rem, rem, kNB, -1.0f, gemm_status,
                                    kGemmTimeoutNs, g->sm_count, s, /*lower=*/true));
        // Side stream: M_k^T = inv(L11)^T L21^T, then B[k+1:, :k+1] -= M_k B_k.
        GQ_TRY(cudaStreamWaitEvent(g->side, g->ev_panel, 0));
        GQ_TRY(gemm<false>(g->sm_count, DkT, kNB, L21T, rem, g->MkT, rem, kNB, rem, kNB, 1.0f, 0, 0, g->side));
        GQ_TRY(cudaEventRecord(g->ev_l21t[k & 1], g->side));
        float* Bk = g->X + static_cast<size_t>(k) * kNB * d;
        GQ_TRY(hk::launch_gemm_tf32(g->MkT, rem, Bk, d, Bk + static_cast<size_t>(kNB) * d, d, rem, (k + 1) * kNB,
                                    kNB, -1.0f, gemm_status, kGemmTimeoutNs, g->sm_count, g->side));
    }
    GQ_TRY(cudaEventRecord(g->ev_side, g->side));
    GQ_TRY(cudaStreamWaitEvent(s, g->ev_side, 0));
    // X_k = inv(L_kk) B_k for every block row k, in place; tiles right of
    // the diagonal block hold zeros and are skipped.
    GQ_TRY(gemm<false>(g->sm_count, g->Dinv, kNB, g->X, d, g->X, d, kNB, d, kNB, 1.0f, 0, kGemmCLowerTiles, s, n,
                       static_cast<long long>(kNB) * kNB, static_cast<long long>(kNB) * d,
                       static_cast<long long>(kNB) * d, kNB, /*narrow_ok=*/false));
    // U = J X J into F.
    gq_reverse_copy_kernel<<<stride_grid(dd / 4, g->sm_count), 256, 0, s>>>(g->X, g->F, dd / 4);
    GQ_TRY(cudaGetLastError());
    int status[2] = {0, 0};
    float damp = 0.0f;
    GQ_TRY(cudaMemcpyAsync(status, g->status, 2 * sizeof(int), cudaMemcpyDeviceToHost, s));
    GQ_TRY(cudaMemcpyAsync(&damp, g->damp32, sizeof(float), cudaMemcpyDeviceToHost, s));
    GQ_TRY(cudaStreamSynchronize(s));
    if (damp_out) *damp_out = damp;
    if (status[1] != 0)
        return gq_fail(HESS_ERR_TIMEOUT, "a device-side wait of the tensor-core GEMM ran out (status 0x%x)",
                       status[1]);
    if (status[0] & 1)
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
    g->ld_errt = static_cast<int>((rows + 3) / 4 * 4);
    if (e == cudaSuccess) e = cudaMalloc(&g->ErrT, static_cast<size_t>(kSuper) * kNB * g->ld_errt * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->rowscale, rows * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->dead, static_cast<size_t>(d));
    if (e == cudaSuccess) e = cudaMalloc(&g->damp64, sizeof(double));
    if (e == cudaSuccess) e = cudaMalloc(&g->damp32, sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->loss, sizeof(double));
    // status[0]: Cholesky pivot flag; status[1]: device-side wait limits of the tensor GEMM
    if (e == cudaSuccess) e = cudaMalloc(&g->status, 4 * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(g->status, 0, 4 * sizeof(int));
    if (e == cudaSuccess) e = hk::gemm_tf32_prepare();
    if (e == cudaSuccess) e = cudaMalloc(&g->DinvT, static_cast<size_t>(d) * kNB * sizeof(float));
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
        e = cudaMalloc(&g->L21T[i], static_cast<size_t>(d) * kNB * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&g->MkT, static_cast<size_t>(d) * kNB * sizeof(float));
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&g->ev_l21t[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&g->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->ev_panel, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->ev_side, cudaEventDisableTiming);
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
    if ((st = gq_check_buffer(H, g->device, "H")) != HESS_OK) return st;
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
    if ((st = gq_check_buffer(U_out, g->device, "U_out")) != HESS_OK) return st;
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
    if (rows > 0) {
        if ((st = gq_check_buffer(W, g->device, "W")) != HESS_OK) return st;
        if ((st = gq_check_buffer(Wq_out, g->device, "Wq_out")) != HESS_OK) return st;
        if ((st = gq_check_buffer(scales_out, g->device, "scales_out")) != HESS_OK) return st;
        if (codes_out && (st = gq_check_buffer(codes_out, g->device, "codes_out")) != HESS_OK) return st;
    }
    if (!g->prepared) return gq_fail(HESS_ERR_INVALID, "no factor: gptq_prepare has not succeeded");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int d = static_cast<int>(g->d), n = g->n_blocks;
    const bool grouped = group_size == kNB;
    GQ_TRY(cudaMemsetAsync(g->loss, 0, sizeof(double), s));
    GQ_TRY(cudaMemsetAsync(g->status + 1, 0, sizeof(int), s));
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
        const int ldt = g->ld_errt;
        uint32_t* gemm_status = reinterpret_cast<uint32_t*>(g->status) + 1;
        // Two-level lazy update on the tensor cores (C -= P^T Q with P the
        // transposed errors and Q a panel of U): after each block only the
        // rest of its super-block (kSuper blocks) is updated; the columns
        // after the super-block get one K = kSuper * 128 update.
        for (int sb0 = 0; sb0 < n; sb0 += kSuper) {
            const int sb1 = std::min(n, sb0 + kSuper);
            for (int b = sb0; b < sb1; ++b) {
                float* errt_b = g->ErrT + static_cast<size_t>(b - sb0) * kNB * ldt;
                BlockArgs a{g->Wc, g->F, Wq_out, reinterpret_cast<signed char*>(codes_out), scales_out, errt_b,
                            g->rowscale, g->loss, rows, d, b, grouped ? n : 1, grouped ? 1 : 0, ldt};
                gq_block_kernel<<<grid, kBlockThreads, kBlockSmem, s>>>(a);
                GQ_TRY(cudaGetLastError());
                const int in_super = (sb1 - b - 1) * kNB;  // columns left in this super-block
                if (in_super > 0)
                    GQ_TRY(hk::launch_gemm_tf32(errt_b, ldt, g->F + static_cast<size_t>(b) * kNB * d + (b + 1) * kNB,
                                                d, g->Wc + (b + 1) * kNB, d, static_cast<int>(rows), in_super, kNB,
                                                -1.0f, gemm_status, kGemmTimeoutNs, g->sm_count, s));
            }
            const int rest = d - sb1 * kNB;
            if (rest > 0)
                GQ_TRY(hk::launch_gemm_tf32(g->ErrT, ldt, g->F + static_cast<size_t>(sb0) * kNB * d + sb1 * kNB, d,
                                            g->Wc + sb1 * kNB, d, static_cast<int>(rows), rest, (sb1 - sb0) * kNB,
                                            -1.0f, gemm_status, kGemmTimeoutNs, g->sm_count, s));
        }
    }
    if (avg_loss_out) {
        double loss = 0.0;
        int gst = 0;
        GQ_TRY(cudaMemcpyAsync(&loss, g->loss, sizeof(double), cudaMemcpyDeviceToHost, s));
        GQ_TRY(cudaMemcpyAsync(&gst, g->status + 1, sizeof(int), cudaMemcpyDeviceToHost, s));
        GQ_TRY(cudaStreamSynchronize(s));
        if (gst != 0)
            return gq_fail(HESS_ERR_TIMEOUT, "a device-side wait of the tensor-core GEMM ran out (status 0x%x)", gst);
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
