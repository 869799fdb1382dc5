// Symmetric rank-k update S += X^T X for fp32 activations on sm_103a.
//
// The pages' fp32 option copies each batch to float32 and runs a float32
// GEMM on CUDA cores (NVIDIA Model-Optimizer PR #3002, "What does this PR
// do?").  Here the same sums run on the tensor cores with a split that keeps
// fp32 accuracy: every value is written x = hi + lo, hi = x rounded to
// nearest tf32 (11 significant bits) and lo = x - hi (exact), and
//     x_i x_j ~ hi_i hi_j + (hi_i lo_j + lo_i hi_j)
// The tf32 rounding of lo (relative 2^-22 of x, zero mean because hi is
// rounded to nearest) is lost, and so is lo_i lo_j: below 2^-24 of x_i x_j,
// the size of one fp32 rounding of the product, and never negative on the
// diagonal (a bias of about -2e-8 of each diagonal entry).
//
// How (same skeleton as the bf16 kernel, 128x128 tiles, 32-token k-blocks):
//   * warp 0 lane 0 stages raw fp32 boxes (32 tokens x 32 features,
//     128-byte swizzle with 32-byte granules, the layout MN-major tf32
//     operands need) into a 3-deep landing ring, and refills a landing slot
//     once every converter has read it;
//   * six converter warps (2-3 and 12-15) turn each landed stage into hi /
//     lo planes of a 2-deep MMA ring, at the same byte offsets (so the
//     swizzle carries over), each taking every sixth round of 2 KB;
//   * warp 1 issues tcgen05.mma kind::tf32 (M=N=128, K=8): hi*hi into bank 0
//     and the two cross terms into bank 1, so they never ride on the large
//     running sum;
//   * warps 4-11 run the shared compensated epilogue (bank 0 + bank 1 folded
//     into registers by TwoSum, added to the (hi, lo) accumulator at the
//     end of a unit).  Warpgroups 0 and 3 give registers to them with
//     setmaxnreg.
// Tensor-core accumulation rounds toward zero, so chunks are short (64
// tokens by default: 8 hi*hi steps).  Every wait is bounded.
#include "syrk_common.cuh"

namespace hk {
namespace {

using syrk::kDrainLimitNs;
using syrk::kEpiWarps;
using syrk::Unit;
using syrk::unit_at;

constexpr int kKB = kKBlockF32;                     // tokens per k-block
constexpr int kLand = 3;                            // landing stages
constexpr int kCvt = 2;                             // converted stages
constexpr uint32_t kBoxBytes = kKB * 128;           // 32 tokens x 32 fp32
constexpr uint32_t kOpBytes = 4 * kBoxBytes;        // 128 features
constexpr uint32_t kLandBytes = 2 * kOpBytes;       // A | B raw
constexpr uint32_t kCvtBytes = 4 * kOpBytes;        // A hi | A lo | B hi | B lo
// Warpgroup 0: warp 0 (producer), warp 1 (MMA issuer), warps 2-3
// (converters 0-1); warpgroups 1-2: the epilogue; warpgroup 3: converters
// 2-5.  Converter ci takes rounds ci, ci + kCvtWarps, ... of kRoundWords
// 16-byte words.  The launch gives every thread kRegsLaunch registers;
// warpgroups 0 and 3 hand most of theirs to the epilogue's (hi, lo) state.
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
constexpr int kNumBarriers = 2 * kLand + 2 * kCvt + 5;
constexpr uint32_t kCvtBase = kLand * kLandBytes;
constexpr size_t kSmemBytes =
    1024 + kLand * kLandBytes + kCvt * kCvtBytes + 8 * kNumBarriers + 16;

// Walks the (unit, k-block) sequence of this CTA.
struct Cursor {
    int u;
    Unit un;
    int kb;
    int b;  // batch holding kb
    bool valid;
};

__device__ __forceinline__ void cursor_seek(const SyrkParams& p, Cursor& c) {
    while (c.u < p.n_units) {
        if (syrk::unit_checked(p, c.u, c.un)) {
            c.kb = c.un.k0;
            c.b = 0;
            while (c.b + 1 < p.n_batches && p.kb_start[c.b + 1] <= c.kb) ++c.b;
            c.valid = true;
            return;
        }
        c.u += gridDim.x;
    }
    c.valid = false;
}

__device__ __forceinline__ void cursor_start(const SyrkParams& p, Cursor& c) {
    c.u = blockIdx.x;
    cursor_seek(p, c);
}

__device__ __forceinline__ void cursor_next(const SyrkParams& p, Cursor& c) {
    if (++c.kb < c.un.k1) {
        while (c.b + 1 < p.n_batches && p.kb_start[c.b + 1] <= c.kb) ++c.b;
        return;
    }
    c.u += gridDim.x;
    cursor_seek(p, c);
}

// hi = x rounded to nearest tf32 (low 13 bits cleared), lo = x - hi exactly.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    const uint32_t u = __float_as_uint(x);
    hi = __uint_as_float((u + 0x1000u) & 0xFFFFE000u);
    lo = __fsub_rn(x, hi);
}

template <bool kExcl>
__global__ void __launch_bounds__(kThreads, 1) syrk_f32_kernel(const __grid_constant__ SyrkParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kLand * kLandBytes + kCvt * kCvtBytes;
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(
        gbase + kLand * kLandBytes + kCvt * kCvtBytes + 8 * kNumBarriers);
    auto land_full = [&](int s) { return bar0 + 8u * s; };
    auto cvt_full = [&](int s) { return bar0 + 8u * (kLand + s); };
    auto cvt_empty = [&](int s) { return bar0 + 8u * (kLand + kCvt + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (kLand + 2 * kCvt + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (kLand + 2 * kCvt + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (kLand + 2 * kCvt + 4);
    auto land_empty = [&](int s) { return bar0 + 8u * (kLand + 2 * kCvt + 5 + s); };

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
    // Set-up above may overlap the end of the previous kernel of the stream
    // (programmatic dependent launch); X and the accumulator are read only
    // after it has completed, and before any bounded wait starts.  The next
    // flush of the stream may then start on the SMs this grid leaves.
    if (threadIdx.x == 0) syrk::prefetch_first_map(p);
    griddep_wait();
    griddep_launch_dependents();
    const unsigned long long limit = p.timeout_ns;

    // Converter `ci` (0..kCvtWarps-1) splits its rounds of landed stage
    // number `converted` (unit C) into hi / lo planes, then signals the MMA
    // issuer (cvt_full) and the producer (land_empty).
    auto convert_stage = [&](int ci, const Cursor& C, uint32_t converted) -> bool {
        const int s = converted % kLand;
        const int c = converted % kCvt;
        if (!mbar_wait(land_full(s), (converted / kLand) & 1u, limit) ||
            !mbar_wait(cvt_empty(c), ((converted / kCvt) & 1u) ^ 1u, limit))
            return false;
        const bool diag = C.un.I == C.un.J;
        constexpr int kRoundsPerOp = static_cast<int>(kOpBytes / 16 / kRoundWords);
        constexpr int kLd = kRoundWords / 32;  // 16-byte loads per lane per round
        const int n_rounds = (diag ? 1 : 2) * kRoundsPerOp;
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
        // visible to / ordered before the async proxy (MMA, next TMA)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(cvt_full(c));
            mbar_arrive(land_empty(s));
        }
        return true;
    };

    // Converter ci walks every (unit, k-block) of this CTA in order.
    auto run_converter = [&](int ci) {
        Cursor C;
        cursor_start(p, C);
        uint32_t converted = 0;
        bool ok = true;
        while (ok && C.valid) {
            if (!convert_stage(ci, C, converted)) {
                ok = false;
                break;
            }
            ++converted;
            cursor_next(p, C);
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
            cursor_start(p, L);
            uint32_t issued = 0;
            int pref = -1;  // batch whose successor's tensor map was prefetched
            while (L.valid) {
                if (L.b != pref) {
                    if (L.b + 1 < p.n_batches) prefetch_tensormap(&p.maps[L.b + 1]);
                    pref = L.b;
                }
                const int s = issued % kLand;
                // a reused landing slot must have been read by every converter
                if (issued >= static_cast<uint32_t>(kLand) &&
                    !mbar_wait(land_empty(s), ((issued / kLand) + 1u) & 1u, limit)) {
                    ok = false;
                    break;
                }
                const bool diag = L.un.I == L.un.J;
                const CUtensorMap* m = &p.maps[L.b];
                const int tok = (L.kb - p.kb_start[L.b]) * kKB;
                const uint32_t dst = base + s * kLandBytes;
                mbar_arrive_expect_tx(land_full(s), diag ? kOpBytes : kLandBytes);
                for (int bx = 0; bx < 4; ++bx)
                    tma_load_2d(dst + bx * kBoxBytes, m, land_full(s), L.un.I * kTile + 32 * bx, tok);
                if (!diag)
                    for (int bx = 0; bx < 4; ++bx)
                        tma_load_2d(dst + kOpBytes + bx * kBoxBytes, m, land_full(s),
                                    L.un.J * kTile + 32 * bx, tok);
                ++issued;
                cursor_next(p, L);
            }
            if (!ok) atomicOr(p.status, kStatusTimeoutLoad);
            // Every issued copy must land before the CTA may exit: the last
            // copy of each slot (earlier ones landed before their slot was reused).
            const uint32_t first = issued > static_cast<uint32_t>(kLand) ? issued - kLand : 0u;
            for (uint32_t k = first; k < issued; ++k) {
                if (!mbar_wait(land_full(k % kLand), (k / kLand) & 1u, kDrainLimitNs)) {
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
                Unit un;
                if (!syrk::unit_checked(p, u, un)) continue;
                const bool diag = un.I == un.J;
                for (int c0 = un.k0; c0 < un.k1; c0 += p.chunk_kb) {
                    const int c1 = min(c0 + p.chunk_kb, un.k1);
                    if (!mbar_wait(acce_bar(ab), aphase ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d0 = tmem + static_cast<uint32_t>(ab) * 256u;
                    const uint32_t d1 = d0 + 128u;
                    for (int kb = c0; kb < c1; ++kb) {
                        const int cs = consumed % kCvt;
                        if (!mbar_wait(cvt_full(cs), (consumed / kCvt) & 1u, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = base + kCvtBase + cs * kCvtBytes;
                        const uint32_t sB = diag ? sA : sA + 2 * kOpBytes;
#pragma unroll
                        for (int j = 0; j < kKB / 8; ++j) {
                            const uint32_t off = j * 1024u;
                            const uint64_t ahi = smem_desc_sw128(sA + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                            const uint64_t alo =
                                smem_desc_sw128(sA + kOpBytes + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                            const uint64_t bhi = smem_desc_sw128(sB + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                            const uint64_t blo =
                                smem_desc_sw128(sB + kOpBytes + off, kBoxBytes, kF32Sbo, kF32DescLayout);
                            const uint32_t acc = (kb > c0 || j > 0) ? 1u : 0u;
                            umma_tf32(d0, ahi, bhi, kIdesc, acc);
                            umma_tf32(d1, ahi, blo, kIdesc, acc);
                            umma_tf32(d1, alo, bhi, kIdesc, 1u);
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
            }
            if (!ok) atomicOr(p.status, kStatusTimeoutMma);
            tc_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, kDrainLimitNs)) atomicOr(p.status, kStatusTimeoutDrain);
        }
      } else {
        // ------------------------------------------------ converters
        run_converter(warp < kFirstEpiWarp ? warp - 2 : warp - kFirstHighCvt + 2);
      }
    } else {
        // ------------------------------------------------ epilogue (warps 4-11)
        setmaxnreg_inc<kRegsHigh>();
        syrk::epilogue<kExcl, 0>(p, tmem, warp, lane, kFirstEpiWarp, accf_bar(0), acce_bar(0), limit);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t syrk_f32_prepare() {
    cudaError_t e = cudaFuncSetAttribute(syrk_f32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(syrk_f32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    // One CTA of kThreads must fit an SM with this register and shared-memory use.
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, syrk_f32_kernel<false>, kThreads, kSmemBytes);
    if (e == cudaSuccess && blocks < 1) e = cudaErrorLaunchOutOfResources;
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits until the CTA's pool has the registers: the pool
    // must be what the re-split was sized for, or the epilogue would never start.
    for (auto fn : {syrk_f32_kernel<false>, syrk_f32_kernel<true>}) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kRegsLaunch)) return cudaErrorLaunchOutOfResources;
    }
    return cudaSuccess;
}

cudaError_t launch_syrk_f32(const SyrkParams& p, int grid, cudaStream_t s, bool overlap) {
    return syrk::launch_syrk(p.exclusive ? syrk_f32_kernel<true> : syrk_f32_kernel<false>, p, grid, kThreads,
                             kSmemBytes, s, overlap);
}

}  // namespace hk
