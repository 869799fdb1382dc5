// Batched 16x16 block Grams for local_hessian: for every block b of 16
// consecutive features, L_b += X_b^T X_b over the tokens of one batch.
//
// NVIDIA Model-Optimizer PR #3002, "What does this PR do?": local_hessian
// builds 16x16 per-block Hessians with a bf16-in, fp32-out batched GEMM; the
// result only weights a scale search and is never inverted.
//
// The work is a stream over X with 16 flops per byte, so it is HBM-bound:
//   * CTA (g, r) owns feature group g (256 features = 16 blocks) and one
//     contiguous range of token k-blocks (64 tokens each); the grid covers
//     every SM twice so all of them stream;
//   * warp 8 stages [64 tokens x 256 features] with four 128-byte-swizzled
//     TMA boxes per stage (full 128-byte lines of every token row) into a
//     3-deep ring;
//   * each of warps 0-7 owns two 16-feature blocks: per 16 tokens one
//     ldmatrix.x4.trans gives the A fragment of X_b^T (16 features x 16
//     tokens) whose halves are also the two B fragments of X_b, so two
//     mma.sync m16n8k16 make the 16x16 block;
//   * the register accumulators are folded into a compensated (hi, lo) pair
//     every `chunk_steps` steps and added in fp64 to the accumulator at the
//     end (red.add.f64), so no fp32 chain is longer than one chunk.
#include "kernels.cuh"
#include "ptx.cuh"

namespace hk {
namespace {

constexpr int kStages = 3;
constexpr uint32_t kBoxBytes = kLocalKBlock * 128;  // 64 tokens x 64 bf16
constexpr uint32_t kStageBytes = 4 * kBoxBytes;      // 256 features
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 8 * 2 * kStages;

__device__ __forceinline__ float two_sum(float a, float b, float& err) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return s;
}

__global__ void __launch_bounds__(kThreads) local_gram_kernel(const __grid_constant__ LocalParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar0 = base + kStages * kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x % p.n_groups;
    const int r = blockIdx.x / p.n_groups;
    const int kb0 = static_cast<int>(static_cast<long long>(r) * p.total_kb / p.n_ranges);
    const int kb1 = static_cast<int>(static_cast<long long>(r + 1) * p.total_kb / p.n_ranges);
    const int feat0 = g * kLocalGroup;
    const int n_boxes = min(4, (p.d - feat0 + 63) / 64);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = base + stage * kStageBytes;
                mbar_arrive_expect_tx(full_bar(stage), n_boxes * kBoxBytes);
                for (int bx = 0; bx < n_boxes; ++bx)
                    tma_load_2d(dst + bx * kBoxBytes, &p.map, full_bar(stage), feat0 + bx * 64,
                                kb * kLocalKBlock);
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) atomicOr(p.status, kStatusTimeoutLoad);
            for (int s = 0; s < kStages; ++s)
                if ((issued >> s) & 1u)
                    if (!mbar_wait(full_bar(s), (issued_par >> s) & 1u, kDrainLimitNs))
                        atomicOr(p.status, kStatusTimeoutDrain);
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int box = warp >> 1;                // 64-feature box of this warp
    const int fw = (warp & 1) * 32;           // first feature of the warp in the box
    const int blk_feat = feat0 + box * 64 + fw;  // global first feature of block 0
    const bool active0 = blk_feat < p.d;
    const bool active1 = blk_feat + 16 < p.d;
    // ldmatrix row this lane addresses: matrices (tok 0-7|f 0-7), (tok 0-7|f 8-15),
    // (tok 8-15|f 0-7), (tok 8-15|f 8-15).
    const int mq = lane >> 3;
    const int tok_l = (mq >> 1) * 8 + (lane & 7);
    const int fch = (fw >> 3) + (mq & 1);  // 16-byte chunk of block 0 for this lane

    float acc[2][2][4], hi[2][2][4], lo[2][2][4];
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 2; ++y)
#pragma unroll
            for (int z = 0; z < 4; ++z) acc[x][y][z] = hi[x][y][z] = lo[x][y][z] = 0.f;

    bool ok = true;
    int stage = 0, steps = 0;
    uint32_t phase = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, p.timeout_ns)) {
            ok = false;
            break;
        }
        if (active0) {
            const uint32_t sbox = base + stage * kStageBytes + box * kBoxBytes;
#pragma unroll
            for (int j = 0; j < kLocalKBlock / 16; ++j) {
                const int t = j * 16 + tok_l;
                const uint32_t rowa = sbox + t * 128;
#pragma unroll
                for (int bl = 0; bl < 2; ++bl) {
                    if (bl == 1 && !active1) break;
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4_trans(rowa + (((fch + 2 * bl) ^ (t & 7)) << 4), a0, a1, a2, a3);
                    mma_bf16_16816(acc[bl][0], a0, a1, a2, a3, a0, a2);
                    mma_bf16_16816(acc[bl][1], a0, a1, a2, a3, a1, a3);
                }
                if (++steps == p.chunk_steps) {
                    steps = 0;
#pragma unroll
                    for (int x = 0; x < 2; ++x)
#pragma unroll
                        for (int y = 0; y < 2; ++y)
#pragma unroll
                            for (int z = 0; z < 4; ++z) {
                                float e;
                                hi[x][y][z] = two_sum(hi[x][y][z], acc[x][y][z], e);
                                lo[x][y][z] = __fadd_rn(lo[x][y][z], e);
                                acc[x][y][z] = 0.f;
                            }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(p.status, kStatusTimeoutEpilogue);
        return;
    }
    // Fragment (row gi, col gj) of n-tile nt: c0 (gi, 2c), c1 (gi, 2c+1),
    // c2 (gi+8, 2c), c3 (gi+8, 2c+1), columns offset by 8*nt.
    const int gi = lane >> 2, gc = (lane & 3) * 2;
#pragma unroll
    for (int bl = 0; bl < 2; ++bl) {
        if (!(bl == 0 ? active0 : active1)) continue;
        const int block = (blk_feat + 16 * bl) / 16;
        double* out = p.acc + static_cast<size_t>(block) * 256;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                float e;
                const float h = two_sum(hi[bl][nt][z], acc[bl][nt][z], e);
                const double v = static_cast<double>(h) +
                                 static_cast<double>(__fadd_rn(lo[bl][nt][z], e));
                const int i = gi + ((z >> 1) << 3);
                const int j = nt * 8 + gc + (z & 1);
                red_add_f64(out + i * 16 + j, v);
            }
    }
}

}  // namespace

cudaError_t local_prepare() {
    return cudaFuncSetAttribute(local_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemBytes));
}

cudaError_t launch_local_gram(const LocalParams& p, int grid, cudaStream_t s) {
    local_gram_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hk
