// Symmetric rank-k update S += X^T X for bf16 activations, run by pairs of
// SMs (tcgen05 cta_group::2) on 256 x 128 tiles.
//
// Same sums as syrk_bf16.cu (GPTQModel PR #2979 Summary; NVIDIA
// Model-Optimizer PR #3002, "What does this PR do?"), laid out for the
// per-SM operand feed that bounds the single-SM kernel: a pair computes a
// 256-row x 128-column tile, each SM receiving its 128 rows of A and 64 of the
// 128 columns of B, i.e. 48 KB per 128 tokens instead of 64 KB for the same
// tensor work.
//
// Tiles: rows in blocks of 256 (I2), columns in blocks of 128 (J), J >= 2*I2
// so that the upper triangle is covered.  CTA r of the pair owns rows
// 256*I2 + 128*r .. +127 of the tile, i.e. 128x128 accumulator tile
// (2*I2 + r, J); blocks strictly below the diagonal are computed (the MMA
// spans 256 rows) but not stored.
//
// Roles (both CTAs run all of them, except where noted):
//   * warp 0: TMA producer for this CTA's A (2 boxes) and B (1 box) of 128
//     tokens, into a 4-deep ring; the copies of both CTAs count their bytes
//     on the even CTA's barrier (pair-mode TMA), which expects both;
//   * warp 1 of the even CTA: issues tcgen05.mma.cta_group::2 (M=256, N=128,
//     K=16), alternating 16-token steps between two accumulator banks, and
//     multicasts every commit to both CTAs;
//   * warps 4-11: the shared compensated epilogue (chunk sums into `mid`,
//     folded into (hi, lo) every 8 chunks) on this CTA's 128 rows; they
//     release accumulator buffers on the even CTA's barrier (relaxed arrive:
//     their tensor-memory loads have completed, and a release would wait for
//     the unrelated accumulator atomics still in flight).
// Every wait is bounded; both CTAs meet at a cluster barrier before tensor
// memory is freed, so neither exits while the other still reads its memory.
// After a timeout a CTA cannot watch its own copies land (they count on the
// even CTA's barrier), so it pauses 2 ms before that barrier.
#include "syrk_common.cuh"

namespace hk {
namespace {

using syrk::kDrainLimitNs;
using syrk::kEpiWarps;
using syrk::PairUnit;

constexpr int kStages = 4;
constexpr uint32_t kBoxBytes = kKBlock * 128;       // kKBlock tokens x 64 bf16
constexpr uint32_t kABytes = 2 * kBoxBytes;         // this CTA's 128 rows
constexpr uint32_t kBBytes = kBoxBytes;             // this CTA's 64 columns
constexpr uint32_t kStageBytes = kABytes + kBBytes;  // 48 KB
// Warpgroup 0: warp 0 (producer), warp 1 (MMA issuer on the even CTA),
// warps 2-3 idle; warpgroups 1-2: the epilogue, which takes most of
// warpgroup 0's registers for its (mid, hi, lo) fold state.
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;
constexpr uint32_t kRegsLaunch = 168;  // 65536 / 384, rounded down to 8
constexpr uint32_t kRegsLow = 56;
constexpr uint32_t kRegsHigh = 224;
static_assert(128 * kRegsLow + kEpiWarps * 32 * kRegsHigh <= kThreads * kRegsLaunch,
              "register re-split exceeds the launch's registers");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = instr_desc_mn_major(1u /*bf16*/, 256, 128);
constexpr int kNumBarriers = 2 * kStages + 5;
constexpr unsigned long long kAbortSettleNs = 2000000ull;
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 8 * kNumBarriers + 16;

template <bool kExcl>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    syrk_bf16_2sm_kernel(const __grid_constant__ SyrkParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kStages * kStageBytes;
    uint32_t* const tmem_slot =
        reinterpret_cast<uint32_t*>(gbase + kStages * kStageBytes + 8 * kNumBarriers);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    __shared__ int aborted;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int n_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        aborted = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // Set-up above may overlap the end of the previous kernel of the stream
    // (programmatic dependent launch); X and the accumulator are read only
    // after it has completed, and before any bounded wait starts.  The next
    // flush of the stream may then start on the SMs this grid leaves.
    griddep_wait();
    griddep_launch_dependents();
    const unsigned long long limit = p.timeout_ns;

    if (warp < kFirstEpiWarp) {
      setmaxnreg_dec<kRegsLow>();
      if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            for (int u = pair; ok && u < p.n_units; u += n_pairs) {
                PairUnit un;
                if (!syrk::pair_unit_checked(p, u, un)) continue;
                const int xa = un.I2 * 256 + static_cast<int>(rank) * 128;
                const int xb = un.J * kTile + static_cast<int>(rank) * 64;
                int b = 0;
                while (b + 1 < p.n_batches && p.kb_start[b + 1] <= un.k0) ++b;
                int pref = -1;  // batch whose successor's tensor map was prefetched
                for (int kb = un.k0; kb < un.k1; ++kb) {
                    while (b + 1 < p.n_batches && p.kb_start[b + 1] <= kb) ++b;
                    if (b != pref) {
                        // the next batch's map reaches the descriptor cache
                        // while this batch's stages load
                        if (b + 1 < p.n_batches) prefetch_tensormap(&p.maps[b + 1]);
                        pref = b;
                    }
                    const int tok = (kb - p.kb_start[b]) * kKBlock;
                    if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    const CUtensorMap* m = &p.maps[b];
                    const uint32_t sA = base + stage * kStageBytes;
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytes);
                    tma_load_2d_pair(sA, m, fb, xa, tok);
                    tma_load_2d_pair(sA + kBoxBytes, m, fb, xa + 64, tok);
                    tma_load_2d_pair(sA + kABytes, m, fb, xb, tok);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicOr(p.status, kStatusTimeoutLoad);
                aborted = 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------- MMA issuer (even CTA)
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            int ab = 0;
            uint32_t aphase = 0;
            for (int u = pair; ok && u < p.n_units; u += n_pairs) {
                PairUnit un;
                if (!syrk::pair_unit_checked(p, u, un)) continue;
                for (int c0 = un.k0; c0 < un.k1; c0 += p.chunk_kb) {
                    const int c1 = min(c0 + p.chunk_kb, un.k1);
                    if (!mbar_wait_cluster(acce_bar(ab), aphase ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + static_cast<uint32_t>(ab) * 256u;
                    for (int kb = c0; kb < c1; ++kb) {
                        if (!mbar_wait_cluster(full_bar(stage), phase, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sA = base + stage * kStageBytes;
                        const uint32_t sB = sA + kABytes;
#pragma unroll
                        for (int j = 0; j < kKSteps; ++j) {
                            const uint64_t ad = smem_desc_sw128(sA + j * 2048u, kBoxBytes, 1024u);
                            // B is one 64-column slice per CTA: no second slice to
                            // stride to (a zero stride keeps any read inside it)
                            const uint64_t bd = smem_desc_sw128(sB + j * 2048u, 0u, 1024u);
                            umma_f16_pair(dt + (j & 1) * 128u, ad, bd, kIdesc,
                                          (kb > c0 || j > 1) ? 1u : 0u);
                        }
                        tc_commit_pair_mc(empty_bar(stage), 0x3);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc_commit_pair_mc(accf_bar(ab), 0x3);
                    if (++ab == 2) {
                        ab = 0;
                        aphase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicOr(p.status, kStatusTimeoutMma);
                aborted = 1;
            }
            // Wait for every MMA issued before the pair's memories are released.
            tc_commit_pair_mc(drain_bar, 0x1);
            if (!mbar_wait(drain_bar, 0, kDrainLimitNs)) atomicOr(p.status, kStatusTimeoutDrain);
        }
      }
    } else {
        // ------------------------------------------------ epilogue (8 warps)
        setmaxnreg_inc<kRegsHigh>();
        const int T = p.tiles_per_dim;
        const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
        syrk::epilogue_t<kExcl, syrk::kMidGroup>(
            p, tmem, warp, lane, kFirstEpiWarp, accf_bar(0), pair, n_pairs,
            [&](int u, int& k0, int& k1, int& out_tile) {
                PairUnit un;
                if (!syrk::pair_unit_checked(p, u, un)) return false;
                k0 = un.k0;
                k1 = un.k1;
                out_tile = syrk::pair_out_tile(un, static_cast<int>(rank), T);
                return true;
            },
            [&](uint32_t bar, uint32_t parity) { return mbar_wait_cluster(bar, parity, limit); },
            [&](int b) { mbar_arrive_cluster_relaxed(acce_leader0 + 8u * b); });
        if (p.status != nullptr && lane == 0 && *reinterpret_cast<volatile uint32_t*>(p.status) != 0)
            aborted = 1;
    }

    // After a timeout, give copies that count on the peer's barrier time to land.
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(&aborted) != 0) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kAbortSettleNs) __nanosleep(1000);
    }

    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t syrk_bf16_2sm_prepare(int* max_pairs) {
    cudaError_t e = cudaFuncSetAttribute(syrk_bf16_2sm_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(syrk_bf16_2sm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits until the CTA's pool has the registers: the pool
    // must be what the re-split was sized for, or the epilogue would never start.
    for (auto fn : {syrk_bf16_2sm_kernel<false>, syrk_bf16_2sm_kernel<true>}) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kRegsLaunch)) return cudaErrorLaunchOutOfResources;
    }
    cudaLaunchConfig_t cfg = {};
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, syrk_bf16_2sm_kernel<false>, &cfg);
    if (e != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        clusters = sms / 2;
    }
    *max_pairs = clusters;
    return cudaSuccess;
}

cudaError_t launch_syrk_bf16_2sm(const SyrkParams& p, int grid, cudaStream_t s, bool overlap) {
    return syrk::launch_syrk(p.exclusive ? syrk_bf16_2sm_kernel<true> : syrk_bf16_2sm_kernel<false>, p, grid, kThreads,
                             kSmemBytes, s, overlap);
}

}  // namespace hk
