// C[M x N] += alpha * P^T Q on the tensor cores, for the fp32 contractions of
// the quantization pass (GPTQModel wiki "QQQ", Concepts, step 5: the
// propagation of a block's scaled errors into the later columns).
//
//   P: K x M fp32, row-major (M contiguous), leading dimension ldp
//   Q: K x N fp32, row-major (N contiguous), leading dimension ldq
//   C: M x N fp32, row-major, leading dimension ldc (read-modify-write)
//
// fp32 accuracy from tf32 MMAs: every value is split x = hi + lo with hi = x
// rounded to nearest tf32 and lo = x - hi (exact), and
//     p q = hi_p hi_q + (hi_p lo_q + lo_p hi_q) + lo_p lo_q,
// of which the last term (relative 2^-22, zero mean) is dropped.  hi*hi
// accumulates in one tensor-memory bank and the two cross terms in the other,
// so the small terms never ride on the large running sum.
//
// Tile: 128 columns of C (the MMA's M, one tensor-memory lane each) x 128 rows
// of C (the MMA's N), the whole K per tile; tensor memory holds two tiles
// (2 x 2 banks x 128 columns) so one tile's write-back overlaps the next
// tile's MMAs.  Warp roles follow the fp32 SYRK kernel:
//   * warp 0 lane 0 stages 32 x 32 fp32 boxes of P and Q (128-byte swizzle,
//     32-byte granules: the MN-major tf32 layout) into a 3-deep landing ring;
//   * six converter warps (2-3 and 12-15) split each landed stage into hi /
//     lo planes of a 2-deep ring at the same offsets, each taking every
//     sixth 2 KB round;
//   * warp 1 lane 0 issues tcgen05.mma kind::tf32 (M = N = 128, K = 8);
//   * warps 4-11 add bank 0 + bank 1 and write C[r][c] += alpha * sum, a
//     warp's 32 lanes covering 32 consecutive columns of one row.
//     Warpgroups 0 and 3 give registers to them with setmaxnreg.
// Tensor-memory accumulation rounds toward zero; with K <= 512 (64 steps
// per bank) the drift is ~1e-6 of each update.  Every wait is bounded.
#include <cuda.h>

#include "device_ptr.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace hk {
namespace {

constexpr int kKB = 32;                               // k per stage
constexpr int kLand = 3;                              // landing stages
constexpr int kCvt = 2;                               // converted stages
constexpr uint32_t kBoxBytes = kKB * 128;             // 32 k x 32 fp32
constexpr uint32_t kOpBytes = 4 * kBoxBytes;          // 128 columns
constexpr uint32_t kLandBytes = 2 * kOpBytes;         // Q | P raw
constexpr uint32_t kCvtBytes = 4 * kOpBytes;          // Q hi | Q lo | P hi | P lo
constexpr int kEpiWarps = 8;
// Warpgroup 0: warp 0 (producer), warp 1 (MMA issuer), warps 2-3
// (converters 0-1); warpgroups 1-2: the write-back; warpgroup 3:
// converters 2-5.  Converter ci takes rounds ci, ci + kCvtWarps, ... of
// kRoundWords 16-byte words.
constexpr int kCvtWarps = 6;
constexpr int kFirstEpiWarp = 4;
constexpr int kFirstHighCvt = kFirstEpiWarp + kEpiWarps;  // warps 12-15
constexpr int kThreads = (kFirstHighCvt + 4) * 32;
constexpr int kRoundWords = 128;
constexpr uint32_t kRegsLaunch = 128;  // 65536 / 512
constexpr uint32_t kRegsLow = 64;
constexpr uint32_t kRegsHigh = 192;
static_assert(2 * 128 * kRegsLow + kEpiWarps * 32 * kRegsHigh <= kThreads * kRegsLaunch,
              "register re-split exceeds the launch's registers");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = instr_desc_mn_major(2u /*tf32*/, 128, 128);
// land_full, land_empty (kLand each); cvt_full, cvt_empty (kCvt each);
// accf, acce (2 each); drain
constexpr int kNumBarriers = 2 * kLand + 2 * kCvt + 5;
constexpr uint32_t kCvtBase = kLand * kLandBytes;
constexpr size_t kSmemBytes = 1024 + kLand * kLandBytes + kCvt * kCvtBytes + 8 * kNumBarriers + 16;
constexpr unsigned long long kDrainNs = 1000000000ull;

// Walks the (tile, k-block) sequence of this CTA: tiles u = blockIdx.x,
// blockIdx.x + gridDim.x, ...; tile u covers C columns 128 (u % tiles_n)
// and C rows 128 (u / tiles_n).
struct Cursor {
    int u;
    int kb;
    bool valid;
};

__device__ __forceinline__ void cur_start(const GemmTf32Params& p, Cursor& c) {
    c.u = blockIdx.x;
    c.kb = 0;
    c.valid = c.u < p.n_units;
}

__device__ __forceinline__ void cur_next(const GemmTf32Params& p, Cursor& c) {
    if (++c.kb < p.n_kb) return;
    c.kb = 0;
    c.u += gridDim.x;
    c.valid = c.u < p.n_units;
}

// First C column (n0) and row (m0) of tile u.
__device__ __forceinline__ void unit_tile(const GemmTf32Params& p, int u, int& n0, int& m0) {
    if (p.lower) {  // u = a (a + 1) / 2 + b, b <= a: row tile a, column tile b
        int a = static_cast<int>((sqrtf(8.0f * u + 1.0f) - 1.0f) * 0.5f);
        while (a * (a + 1) / 2 > u) --a;
        while ((a + 1) * (a + 2) / 2 <= u) ++a;
        n0 = (u - a * (a + 1) / 2) * 128;
        m0 = a * 128;
    } else {
        n0 = (u % p.tiles_n) * 128;
        m0 = (u / p.tiles_n) * 128;
    }
}

// hi = x rounded to nearest tf32 (low 13 bits cleared), lo = x - hi exactly.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    const uint32_t u = __float_as_uint(x);
    hi = __uint_as_float((u + 0x1000u) & 0xFFFFE000u);
    lo = __fsub_rn(x, hi);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_tf32_kernel(const __grid_constant__ GemmTf32Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kLand * kLandBytes + kCvt * kCvtBytes;
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(
        gbase + kLand * kLandBytes + kCvt * kCvtBytes + 8 * kNumBarriers);
    auto land_full = [&](int s) { return bar0 + 8u * s; };
    auto land_empty = [&](int s) { return bar0 + 8u * (kLand + s); };
    auto cvt_full = [&](int s) { return bar0 + 8u * (2 * kLand + s); };
    auto cvt_empty = [&](int s) { return bar0 + 8u * (2 * kLand + kCvt + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kLand + 2 * kCvt + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kLand + 2 * kCvt + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kLand + 2 * kCvt + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLand; ++s) {
            mbar_init(land_full(s), 1);
            mbar_init(land_empty(s), kCvtWarps);
        }
        for (int s = 0; s < kCvt; ++s) {
            mbar_init(cvt_full(s), kCvtWarps);
            mbar_init(cvt_empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const unsigned long long limit = p.timeout_ns;

    // Converter `ci` splits its rounds of landed stage number `converted`
    // into hi / lo planes, then signals the MMA issuer and the producer.
    auto convert_stage = [&](int ci, uint32_t converted) -> bool {
        const int s = converted % kLand;
        const int c = converted % kCvt;
        if (!mbar_wait(land_full(s), (converted / kLand) & 1u, limit) ||
            !mbar_wait(cvt_empty(c), ((converted / kCvt) & 1u) ^ 1u, limit))
            return false;
        constexpr int kRoundsPerOp = static_cast<int>(kOpBytes / 16 / kRoundWords);
        constexpr int kLd = kRoundWords / 32;  // 16-byte loads per lane per round
        constexpr int n_rounds = 2 * kRoundsPerOp;
        const uint32_t src = base + s * kLandBytes;
        const uint32_t dst = base + kCvtBase + c * kCvtBytes;
        // the word of load k of round rr, for this lane, within its operand
        auto word = [&](int rr, int k) { return ((rr % kRoundsPerOp) * kLd + k) * 32 + lane; };
#pragma unroll 1
        for (int rr = ci; rr < n_rounds; rr += 2 * kCvtWarps) {
            // two rounds' loads in flight when this warp has a second one
            const int rr2 = rr + kCvtWarps;
            const bool two = rr2 < n_rounds;
            uint4 x[2 * kLd];
#pragma unroll
            for (int k = 0; k < kLd; ++k) x[k] = lds128(src + (rr / kRoundsPerOp) * kOpBytes + word(rr, k) * 16);
            if (two) {
#pragma unroll
                for (int k = 0; k < kLd; ++k)
                    x[kLd + k] = lds128(src + (rr2 / kRoundsPerOp) * kOpBytes + word(rr2, k) * 16);
            }
#pragma unroll
            for (int k = 0; k < 2 * kLd; ++k) {
                if (k >= kLd && !two) break;
                const int q = k < kLd ? rr : rr2;
                const uint32_t hp = dst + (q / kRoundsPerOp) * 2 * kOpBytes;
                const uint32_t lp = hp + kOpBytes;
                const uint32_t off = word(q, k % kLd) * 16;
                float h0, h1, h2, h3, l0, l1, l2, l3;
                split_tf32(__uint_as_float(x[k].x), h0, l0);
                split_tf32(__uint_as_float(x[k].y), h1, l1);
                split_tf32(__uint_as_float(x[k].z), h2, l2);
                split_tf32(__uint_as_float(x[k].w), h3, l3);
                sts128(hp + off, make_uint4(__float_as_uint(h0), __float_as_uint(h1),
                                            __float_as_uint(h2), __float_as_uint(h3)));
                sts128(lp + off, make_uint4(__float_as_uint(l0), __float_as_uint(l1),
                                            __float_as_uint(l2), __float_as_uint(l3)));
            }
        }
        // generic-proxy writes (and reads of the landing slot) must be
        // ordered before the async proxy (MMA, next TMA)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(cvt_full(c));
            mbar_arrive(land_empty(s));
        }
        return true;
    };

    // Converter ci walks every (tile, k-block) of this CTA in order.
    auto run_converter = [&](int ci) {
        Cursor C;
        cur_start(p, C);
        uint32_t converted = 0;
        bool ok = true;
        while (ok && C.valid) {
            if (!convert_stage(ci, converted)) {
                ok = false;
                break;
            }
            ++converted;
            cur_next(p, C);
        }
        if (!ok && lane == 0) atomicOr(p.status, kStatusTimeoutLoad);
    };

    if (warp < kFirstEpiWarp || warp >= kFirstHighCvt) {
      setmaxnreg_dec<kRegsLow>();
      if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            Cursor L;
            cur_start(p, L);
            uint32_t issued = 0;
            while (L.valid) {
                const int s = issued % kLand;
                // a reused landing slot must have been read by every converter
                if (issued >= static_cast<uint32_t>(kLand) &&
                    !mbar_wait(land_empty(s), ((issued / kLand) + 1u) & 1u, limit)) {
                    ok = false;
                    break;
                }
                int n0, m0;  // first C column (Q) and row (P)
                unit_tile(p, L.u, n0, m0);
                const int k0 = L.kb * kKB;
                const uint32_t dst = base + s * kLandBytes;
                mbar_arrive_expect_tx(land_full(s), kLandBytes);
                for (int bx = 0; bx < 4; ++bx)
                    tma_load_2d(dst + bx * kBoxBytes, &p.q_map, land_full(s), n0 + 32 * bx, k0);
                for (int bx = 0; bx < 4; ++bx)
                    tma_load_2d(dst + kOpBytes + bx * kBoxBytes, &p.p_map, land_full(s), m0 + 32 * bx, k0);
                ++issued;
                cur_next(p, L);
            }
            if (!ok) atomicOr(p.status, kStatusTimeoutLoad);
            // Every issued copy must land before the CTA may exit: the last
            // copy of each slot (earlier ones landed before their slot was reused).
            const uint32_t first = issued > static_cast<uint32_t>(kLand) ? issued - kLand : 0u;
            for (uint32_t k = first; k < issued; ++k) {
                if (!mbar_wait(land_full(k % kLand), (k / kLand) & 1u, kDrainNs)) {
                    atomicOr(p.status, kStatusTimeoutDrain);
                    break;
                }
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            uint32_t consumed = 0;
            int ab = 0;
            uint32_t aphase = 0;
            for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                if (!mbar_wait(acce_bar(ab), aphase ^ 1u, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + static_cast<uint32_t>(ab) * 256u;
                const uint32_t d1 = d0 + 128u;
                for (int kb = 0; kb < p.n_kb; ++kb) {
                    const int cs = consumed % kCvt;
                    if (!mbar_wait(cvt_full(cs), (consumed / kCvt) & 1u, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sQ = base + kCvtBase + cs * kCvtBytes;  // Q hi | Q lo
                    const uint32_t sP = sQ + 2 * kOpBytes;                 // P hi | P lo
#pragma unroll
                    for (int j = 0; j < kKB / 8; ++j) {
                        const uint32_t off = j * 1024u;
                        const uint64_t qhi = smem_desc_sw128(sQ + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                        const uint64_t qlo = smem_desc_sw128(sQ + kOpBytes + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                        const uint64_t phi = smem_desc_sw128(sP + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                        const uint64_t plo = smem_desc_sw128(sP + kOpBytes + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                        const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
                        umma_tf32(d0, qhi, phi, kIdesc, acc);
                        umma_tf32(d1, qhi, plo, kIdesc, acc);
                        umma_tf32(d1, qlo, phi, kIdesc, 1u);
                    }
                    tc_commit(cvt_empty(cs));
                    ++consumed;
                }
                if (!ok) break;
                tc_commit(accf_bar(ab));
                if (++ab == 2) {
                    ab = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) atomicOr(p.status, kStatusTimeoutMma);
            // Wait for every MMA this thread issued before tensor memory is freed.
            tc_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, kDrainNs)) atomicOr(p.status, kStatusTimeoutDrain);
        }
      } else {
        // ------------------------------------------------ converters
        run_converter(warp < kFirstEpiWarp ? warp - 2 : warp - kFirstHighCvt + 2);
      }
    } else {
        // ------------------------------------------------ write-back (warps 4-11)
        // Warp w reads tensor-memory lanes 32 (w % 4) .. +31 (C columns) and
        // 64 of the tile's 128 C rows.
        setmaxnreg_inc<kRegsHigh>();
        const int q = warp & 3;
        const int part = (warp - kFirstEpiWarp) >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        int ab = 0;
        uint32_t aphase = 0;
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            if (!mbar_wait(accf_bar(ab), aphase, limit)) {
                ok = false;
                break;
            }
            tc_fence_after();
            int n0, m0;
            unit_tile(p, u, n0, m0);
            const int col = n0 + q * 32 + lane;
            const uint32_t tb = tmem + lane_off + static_cast<uint32_t>(ab) * 256u + part * 64u;
            // 32 rows per step: their 32 loads of C are in flight together
            // while the tensor-memory columns are read.
#pragma unroll 1
            for (int it = 0; it < 8; it += 4) {
                const int r0 = m0 + part * 64 + it * 8;
                float cv[32];
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    cv[t] = r0 + t < p.M ? p.C[static_cast<size_t>(r0 + t) * p.ldc + col] : 0.0f;
                uint32_t b0[4][8], b1[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld8x2_sync(tb + (it + j) * 8, tb + 128 + (it + j) * 8, b0[j], b1[j]);
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    if (r0 + t < p.M)
                        p.C[static_cast<size_t>(r0 + t) * p.ldc + col] =
                            cv[t] + p.alpha * (__uint_as_float(b0[t / 8][t % 8]) + __uint_as_float(b1[t / 8][t % 8]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(ab));
            if (++ab == 2) {
                ab = 0;
                aphase ^= 1u;
            }
        }
        if (!ok && lane == 0) atomicOr(p.status, kStatusTimeoutEpilogue);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn gemm_encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// fp32 [outer][inner] row-major with leading dimension ld, 32 x 32 boxes
// (zeros beyond the edges), 128-byte swizzle with 32-byte atoms.
cudaError_t encode_fp32(CUtensorMap* map, const float* ptr, int inner, int outer, int ld) {
    EncodeTiledFn fn = gemm_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cudaError_t ce = ensure_context();
    if (ce != cudaSuccess) return ce;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * sizeof(float)};
    const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(kKB)};
    const cuuint32_t es[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, kF32Swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t gemm_tf32_prepare() {
    cudaError_t e = cudaFuncSetAttribute(gemm_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gemm_tf32_kernel, kThreads, kSmemBytes);
    if (e == cudaSuccess && blocks < 1) e = cudaErrorLaunchOutOfResources;
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits until the CTA's pool has the registers: the pool
    // must be what the re-split was sized for, or the write-back would never start.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, gemm_tf32_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kRegsLaunch)) return cudaErrorLaunchOutOfResources;
    return cudaSuccess;
}

cudaError_t launch_gemm_tf32(const float* P, int ldp, const float* Q, int ldq, float* C, int ldc, int M, int N,
                             int K, float alpha, uint32_t* status, unsigned long long timeout_ns, int grid_max,
                             cudaStream_t s, bool lower) {
    if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
    if (N % 128 != 0 || K % kKB != 0 || ldp % 4 || ldq % 4 || ldc % 4) return cudaErrorInvalidValue;
    if (lower && M != N) return cudaErrorInvalidValue;
    GemmTf32Params p{};
    cudaError_t e = encode_fp32(&p.p_map, P, M, K, ldp);
    if (e == cudaSuccess) e = encode_fp32(&p.q_map, Q, N, K, ldq);
    if (e != cudaSuccess) return e;
    p.C = C;
    p.ldc = ldc;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.tiles_n = N / 128;
    p.n_kb = K / kKB;
    p.lower = lower ? 1 : 0;
    p.n_units = lower ? p.tiles_n * (p.tiles_n + 1) / 2 : p.tiles_n * ((M + 127) / 128);
    p.status = status;
    p.timeout_ns = timeout_ns;
    const int grid = p.n_units < grid_max ? p.n_units : grid_max;
    gemm_tf32_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hk
