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
//   * warp 0 stages X boxes of 128 tokens x 64 features with TMA
//     (128-byte swizzle) into a 3-deep shared-memory ring; on diagonal
//     tiles A and B are the same slab and are loaded once;
//   * warp 1 issues tcgen05.mma (M=128, N=128, K=16, both operands
//     MN-major straight from the row-major X boxes).  Consecutive 16-token
//     steps alternate between two fp32 accumulator banks in tensor memory,
//     and after `chunk_kb` k-blocks the pair is handed to the epilogue while
//     the MMAs continue in a second pair (2 buffers x 2 banks x 128 columns);
//   * warps 4-11 add the two banks, sum the chunks into a `mid` pair of
//     registers with round-to-nearest adds, and every 8 chunks fold mid
//     into a compensated (hi, lo) pair with an exact TwoSum, on packed fp32
//     pairs; at the end of a unit they add (hi, lo) to the (hi, lo)
//     accumulator tile in global memory with fp32 arithmetic (compensated
//     atomics when several slabs add to one tile).  Warpgroup 0 (warps 0-3)
//     gives registers to the epilogue warpgroups with setmaxnreg.
// Why the short chains: tcgen05 accumulation into tensor memory rounds
// toward zero, so each MMA step of a chain loses about half an ulp of its
// running sum (measured on GB300: relative bias -1.8e-6 at 1,024 tokens, -2.6e-4 at
// 65,536).  The default 384-token chunk, two 192-token chains, keeps it
// near 3e-7 of each entry.
// Every mbarrier wait is bounded; on timeout a status bit is set, in-flight
// copies and MMAs are drained, tensor memory is freed and the kernel returns.
#include "syrk_common.cuh"

namespace hk {
namespace {

using syrk::Unit;
using syrk::unit_at;
using syrk::kEpiWarps;
using syrk::kDrainLimitNs;

constexpr int kStages = 3;
constexpr uint32_t kBoxBytes = kKBlock * 128;       // kKBlock tokens x 128 bytes
constexpr uint32_t kOperandBytes = 2 * kBoxBytes;   // 128 features
constexpr uint32_t kStageBytes = 2 * kOperandBytes; // A and B
// Warpgroup 0: warp 0 (producer), warp 1 (MMA issuer), warps 2-3 idle;
// warpgroups 1-2: the epilogue.  The launch gives every thread kRegsLaunch
// registers; warpgroup 0 hands most of its share to the epilogue's
// (mid, hi, lo) fold state.
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;
constexpr uint32_t kRegsLaunch = 168;  // 65536 / 384, rounded down to 8
constexpr uint32_t kRegsLow = 56;
constexpr uint32_t kRegsHigh = 224;
static_assert(128 * kRegsLow + kEpiWarps * 32 * kRegsHigh <= kThreads * kRegsLaunch,
              "register re-split exceeds the launch's registers");
constexpr uint32_t kTmemCols = 512;  // [buffer][bank] x 128 columns
constexpr uint32_t kIdesc = instr_desc_mn_major(1u /*bf16*/, 128, 128);
constexpr int kNumBarriers = 2 * kStages + 5;
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + 8 * kNumBarriers + 16;

template <bool kExcl>
__global__ void __launch_bounds__(kThreads, 1) syrk_bf16_kernel(const __grid_constant__ SyrkParams p) {
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

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
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
    if (threadIdx.x == 0) {
        syrk::prefetch_first_map(p);
        // A small one-batch flush: each CTA sends its share of X toward L2.
        if (p.l2_bytes > 0) {
            const uint64_t share = ((p.l2_bytes + gridDim.x - 1) / gridDim.x + 15) & ~15ull;
            const uint64_t off = share * blockIdx.x;
            if (off < p.l2_bytes) {
                const uint64_t len = min(share, p.l2_bytes - off);
                prefetch_l2_bulk(static_cast<const uint8_t*>(p.l2_ptr) + off, static_cast<uint32_t>(len));
            }
        }
        // The X boxes of the first unit's first ring fill (kStages stages)
        // start toward L2 too.  Only L2 is touched, and it stays coherent
        // with any write of the previous kernel still in flight: the loads
        // after the grid wait read the finished data.  (Prefetching the next
        // units' first stages as well made flushes slower: the prefetches
        // queue ahead of the loads.)
        Unit un;
        if (static_cast<int>(blockIdx.x) < p.n_units && syrk::unit_at(p, blockIdx.x, un) &&
            syrk::unit_in_range(p, un)) {
            int b = 0;
            for (int kb = un.k0; kb < un.k1 && kb < un.k0 + kStages; ++kb) {
                while (b + 1 < p.n_batches && p.kb_start[b + 1] <= kb) ++b;
                const int tok = (kb - p.kb_start[b]) * kKBlock;
                tma_prefetch_2d(&p.maps[b], un.I * kTile, tok);
                tma_prefetch_2d(&p.maps[b], un.I * kTile + 64, tok);
                if (un.I != un.J) {
                    tma_prefetch_2d(&p.maps[b], un.J * kTile, tok);
                    tma_prefetch_2d(&p.maps[b], un.J * kTile + 64, tok);
                }
            }
        }
    }
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
            uint32_t issued = 0;       // stages with a load issued
            uint32_t issued_par = 0;   // parity of the last load per stage
            for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                Unit un;
                if (!syrk::unit_checked(p, u, un)) continue;
                const bool diag = un.I == un.J;
                const uint32_t bytes = diag ? kOperandBytes : kStageBytes;
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
            // Descriptor of stage 0's first step.  Shared-memory addresses stay
            // below 2^18, so the 14-bit address field (address / 16) takes the
            // stage and step offsets without a carry into the next field; the
            // additions take fewer instructions on the issuer's path than
            // building each descriptor (measured: 1 % on the ragged stream).
            const uint64_t desc0 = smem_desc_sw128(base, kBoxBytes, 1024u);
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
                    const uint32_t dt = tmem + static_cast<uint32_t>(ab) * 256u;
                    for (int kb = c0; kb < c1; ++kb) {
                        if (!mbar_wait(full_bar(stage), phase, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // this stage's A and B descriptors: offsets added to
                        // the address field of stage 0's (2,048 bytes per step)
                        const uint64_t ad_s = desc0 + ((static_cast<uint32_t>(stage) * kStageBytes) >> 4);
                        const uint64_t bd_s = diag ? ad_s : ad_s + (kOperandBytes >> 4);
#pragma unroll
                        for (int j = 0; j < kKSteps; ++j) {
                            const uint64_t ad = ad_s + j * (2048u >> 4);
                            const uint64_t bd = bd_s + j * (2048u >> 4);
                            // even steps -> bank 0, odd steps -> bank 1; each bank
                            // starts afresh at the first step of the chunk.  Rows
                            // past a batch's end hold TMA's zeros and add nothing:
                            // issuing them costs less than a per-stage test on
                            // this thread's critical path (measured)
                            umma_f16(dt + (j & 1) * 128u, ad, bd, kIdesc,
                                     (kb > c0 || j > 1) ? 1u : 0u);
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
      }
    } else {
        // ------------------------------------------------ epilogue (8 warps)
        setmaxnreg_inc<kRegsHigh>();
        syrk::epilogue<kExcl, syrk::kMidGroup>(p, tmem, warp, lane, kFirstEpiWarp, accf_bar(0),
                                               acce_bar(0), limit);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t syrk_bf16_prepare() {
    cudaError_t e = cudaFuncSetAttribute(syrk_bf16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(syrk_bf16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    // One CTA of kThreads must fit an SM with this register and shared-memory use.
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, syrk_bf16_kernel<false>, kThreads, kSmemBytes);
    if (e == cudaSuccess && blocks < 1) e = cudaErrorLaunchOutOfResources;
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits until the CTA's pool has the registers: the pool
    // must be what the re-split was sized for, or the epilogue would never start.
    for (auto fn : {syrk_bf16_kernel<false>, syrk_bf16_kernel<true>}) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kRegsLaunch)) return cudaErrorLaunchOutOfResources;
    }
    return cudaSuccess;
}

cudaError_t launch_syrk_bf16(const SyrkParams& p, int grid, cudaStream_t s, bool overlap) {
    return syrk::launch_syrk(p.exclusive ? syrk_bf16_kernel<true> : syrk_bf16_kernel<false>, p, grid, kThreads,
                             kSmemBytes, s, overlap);
}

}  // namespace hk
