// Symmetric rank-k update S += X^T X for bf16 activations on sm_103a.
//
// What it computes: for every upper-triangle tile (I, J), I <= J, of the
// d x d Gram, acc_IJ += sum_t X[t, I-block]^T X[t, J-block] over the tokens
// of every queued batch (GPTQModel PR #2979 Summary: H = (2/n) sum x x^T;
// NVIDIA Model-Optimizer PR #3002, "What does this PR do?": bf16 inputs,
// products exact in fp32, fp32 accumulation).  The 2/N scale is applied at
// materialize time.
//
// How:
//   * one persistent CTA per SM walks a static list of units
//     (tile, token slab); the token stream is the concatenation of the
//     queued batches, so many small ragged batches form one split-K pass;
//   * warp 0 stages X boxes of 64 tokens x 64 features with TMA
//     (128-byte swizzle) into a 6-deep shared-memory ring; on diagonal
//     tiles A and B are the same slab and are loaded once;
//   * warp 1 issues tcgen05.mma (M=128, N=128, K=16, both operands
//     MN-major straight from the row-major X boxes) into one of two fp32
//     tensor-memory accumulators; after `chunk_kb` k-blocks it hands the
//     chain to the epilogue and continues in the other accumulator;
//   * warps 2-5 fold each chain into an on-chip compensated sum (hi, lo) in
//     tensor memory (TwoSum), so no fp32 chain runs longer than one chunk,
//     and at the end of a unit add hi + lo in fp64 to the accumulator in
//     global memory (red.add.f64; several slabs may add to one tile).
// Every mbarrier wait is bounded; on timeout a status bit is set, in-flight
// copies and MMAs are drained, tensor memory is freed and the kernel returns.
#include "kernels.cuh"
#include "ptx.cuh"

namespace hk {
namespace {

constexpr int kStages = 6;
constexpr uint32_t kBoxBytes = 64 * 128;            // 64 tokens x 128 bytes
constexpr uint32_t kOperandBytes = 2 * kBoxBytes;   // 128 features
constexpr uint32_t kStageBytes = 2 * kOperandBytes; // A and B
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;  // acc0 | acc1 | hi | lo, 128 columns each
constexpr uint32_t kColHi = 256, kColLo = 384;
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
constexpr uint32_t kIdesc = instr_desc_mn_major(1u /*bf16*/, 128, 128);
constexpr size_t kBarrierBytes = 8 * (2 * kStages + 5) + 16;
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + kBarrierBytes;

struct Unit {
    int t, I, J, k0, k1;
};

__device__ __forceinline__ bool unit_at(const SyrkParams& p, int u, Unit& un) {
    const int slab = u / p.n_tiles;
    const int t = u - slab * p.n_tiles;
    int i = 0, rem = t;
    while (rem >= p.tiles_per_dim - i) {
        rem -= p.tiles_per_dim - i;
        ++i;
    }
    un.t = t;
    un.I = i;
    un.J = i + rem;
    un.k0 = static_cast<int>(static_cast<long long>(slab) * p.total_kb / p.n_slabs);
    un.k1 = static_cast<int>(static_cast<long long>(slab + 1) * p.total_kb / p.n_slabs);
    return un.k1 > un.k0;
}

__device__ __forceinline__ float two_sum(float a, float b, float& err) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return s;
}

__global__ void __launch_bounds__(kThreads, 1) syrk_bf16_kernel(const __grid_constant__ SyrkParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kStages * kStageBytes;
    uint32_t* const tmem_slot =
        reinterpret_cast<uint32_t*>(gbase + kStages * kStageBytes + 8 * (2 * kStages + 5));
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);
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

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;       // stages with a load issued
            uint32_t issued_par = 0;   // parity of the last load per stage
            for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                Unit un;
                if (!unit_at(p, u, un)) continue;
                const bool diag = un.I == un.J;
                const uint32_t bytes = diag ? kOperandBytes : kStageBytes;
                int b = 0;
                while (p.kb_start[b + 1] <= un.k0) ++b;
                for (int kb = un.k0; kb < un.k1; ++kb) {
                    while (p.kb_start[b + 1] <= kb) ++b;
                    const int tok = (kb - p.kb_start[b]) * kKBlock;
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    const CUtensorMap* m = &p.maps[b];
                    const uint32_t sA = base + stage * kStageBytes;
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    tma_load_2d(sA, m, full_bar(stage), un.I * kTile, tok);
                    tma_load_2d(sA + kBoxBytes, m, full_bar(stage), un.I * kTile + 64, tok);
                    if (!diag) {
                        tma_load_2d(sA + kOperandBytes, m, full_bar(stage), un.J * kTile, tok);
                        tma_load_2d(sA + kOperandBytes + kBoxBytes, m, full_bar(stage),
                                    un.J * kTile + 64, tok);
                    }
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) atomicOr(p.status, kStatusTimeoutLoad);
            // Every issued copy must land before the CTA may exit.
            for (int s = 0; s < kStages; ++s) {
                if ((issued >> s) & 1u) {
                    if (!mbar_wait(full_bar(s), (issued_par >> s) & 1u, kDrainLimitNs))
                        atomicOr(p.status, kStatusTimeoutDrain);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            int ab = 0;
            uint32_t aphase = 0;
            for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                Unit un;
                if (!unit_at(p, u, un)) continue;
                const bool diag = un.I == un.J;
                for (int c0 = un.k0; c0 < un.k1; c0 += p.chunk_kb) {
                    const int c1 = min(c0 + p.chunk_kb, un.k1);
                    if (!mbar_wait(acce_bar(ab), aphase ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + static_cast<uint32_t>(ab) * 128u;
                    for (int kb = c0; kb < c1; ++kb) {
                        if (!mbar_wait(full_bar(stage), phase, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = base + stage * kStageBytes;
                        const uint32_t sB = diag ? sA : sA + kOperandBytes;
#pragma unroll
                        for (int j = 0; j < kKBlock / 16; ++j) {
                            const uint64_t ad = smem_desc_sw128(sA + j * 2048u, kBoxBytes, 1024u);
                            const uint64_t bd = smem_desc_sw128(sB + j * 2048u, kBoxBytes, 1024u);
                            umma_f16(dt, ad, bd, kIdesc, (kb > c0 || j > 0) ? 1u : 0u);
                        }
                        tc_commit(empty_bar(stage));
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
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
            // Wait for every MMA this thread issued before tensor memory is freed.
            tc_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, kDrainLimitNs)) atomicOr(p.status, kStatusTimeoutDrain);
        }
    } else {
        // ------------------------------------------------ epilogue (4 warps)
        const int q = warp & 3;  // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        int ab = 0;
        uint32_t aphase = 0;
        for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
            Unit un;
            if (!unit_at(p, u, un)) continue;
            const int nch = (un.k1 - un.k0 + p.chunk_kb - 1) / p.chunk_kb;
            double* const out = p.acc + static_cast<size_t>(un.t) * kTileElems + row;
            for (int c = 0; c < nch; ++c) {
                if (!mbar_wait(accf_bar(ab), aphase, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[4][32];
                const uint32_t ta = tmem + lane_off + static_cast<uint32_t>(ab) * 128u;
#pragma unroll
                for (int pc = 0; pc < 4; ++pc) tmem_ld32_sync(ta + pc * 32, v[pc]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce_bar(ab));
                if (++ab == 2) {
                    ab = 0;
                    aphase ^= 1u;
                }
                const bool first = c == 0, last = c == nch - 1;
#pragma unroll
                for (int pc = 0; pc < 4; ++pc) {
                    const uint32_t th = tmem + lane_off + kColHi + pc * 32;
                    const uint32_t tl = tmem + lane_off + kColLo + pc * 32;
                    if (first && last) {
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            red_add_f64(out + (pc * 32 + k) * kTile,
                                        static_cast<double>(__uint_as_float(v[pc][k])));
                    } else if (first) {
                        uint32_t z[32];
#pragma unroll
                        for (int k = 0; k < 32; ++k) z[k] = 0u;
                        tmem_st32_sync(th, v[pc]);
                        tmem_st32_sync(tl, z);
                    } else {
                        uint32_t hi[32], lo[32];
                        tmem_ld32_sync(th, hi);
                        tmem_ld32_sync(tl, lo);
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            float e;
                            const float s =
                                two_sum(__uint_as_float(hi[k]), __uint_as_float(v[pc][k]), e);
                            hi[k] = __float_as_uint(s);
                            lo[k] = __float_as_uint(__fadd_rn(__uint_as_float(lo[k]), e));
                        }
                        if (last) {
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                red_add_f64(out + (pc * 32 + k) * kTile,
                                            static_cast<double>(__uint_as_float(hi[k])) +
                                                static_cast<double>(__uint_as_float(lo[k])));
                        } else {
                            tmem_st32_sync(th, hi);
                            tmem_st32_sync(tl, lo);
                        }
                    }
                }
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

}  // namespace

size_t syrk_bf16_smem_bytes() { return kSmemBytes; }

cudaError_t syrk_bf16_prepare() {
    return cudaFuncSetAttribute(syrk_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemBytes));
}

cudaError_t launch_syrk_bf16(const SyrkParams& p, int grid, cudaStream_t s) {
    syrk_bf16_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hk
