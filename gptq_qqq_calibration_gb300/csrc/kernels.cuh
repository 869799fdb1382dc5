// Parameter blocks and launchers shared by the host library and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace hk {

// Edge of a tile of H (features).  The accumulator holds the upper-triangle
// tiles (I <= J), tile-major.  Each element is an unevaluated sum hi + lo of
// two fp32 values (about 48 significant bits), so that every update is fp32
// arithmetic (GB300's fp64 pipe runs at ~1/64 of its fp32 rate).  A tile is a
// plane of hi then a plane of lo.  A plane holds 4-column blocks: element
// (r, c) sits at tile_offset(r, c), so that one thread moves 4 columns of its
// row with a 16-byte access and a warp's 32 rows are 512 contiguous bytes.
// The lo plane is kTileElems further.
constexpr int kTile = 128;
constexpr int kTileElems = kTile * kTile;
constexpr int kTileWords = 2 * kTileElems;
__host__ __device__ constexpr int tile_offset(int r, int c) { return ((c >> 2) * kTile + r) * 4 + (c & 3); }
// Tokens per pipeline stage ("k-block") of the bf16 SYRK kernels.  Larger
// stages mean fewer barrier round trips per token between the TMA producer
// and the MMA issuer; on GB300, 128-token stages (3 in flight) run 1.14x
// faster than 64-token stages (6 in flight) with the same bytes in flight.
constexpr int kKBlock = 128;
// 16-token MMA steps per bf16 k-block.
constexpr int kKSteps = kKBlock / 16;
// Tokens per k-block of the fp32-input SYRK kernel.
constexpr int kKBlockF32 = 32;
// Shared-memory layout of the fp32 operand boxes.  MN-major tf32 operands of
// tcgen05.mma need the 128-byte swizzle with 32-byte granules (TMA
// SWIZZLE_128B_ATOM_32B, descriptor mode 1), whose K groups are 4 rows of
// 128 bytes (stride 512 bytes).  Measured on GB300: the 16-byte-granule
// swizzle gives zeros, and a 1,024-byte K-group stride gives wrong sums.
constexpr CUtensorMapSwizzle kF32Swizzle = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
constexpr uint32_t kF32DescLayout = 1u;
constexpr uint32_t kF32Sbo = 512u;
// Batches one fused flush can hold; their tensor maps travel in the kernel
// parameter block (up to 32 KB on sm_70 and later).
constexpr int kMaxBatches = 192;

// Device status word bits (OR-ed by kernels; read by hess_sync).
constexpr uint32_t kStatusTimeoutLoad = 1u;
constexpr uint32_t kStatusTimeoutMma = 2u;
constexpr uint32_t kStatusTimeoutEpilogue = 4u;
constexpr uint32_t kStatusTimeoutDrain = 8u;
// A kernel's index guard failed (a unit outside the upper triangle or the
// flush, a batch or accumulator tile out of range): the access was skipped.
constexpr uint32_t kStatusBadIndex = 16u;

// How an exclusive (single-slab) launch adds a unit's compensated sum
// (hi', lo') to its accumulator tile.  kAccPair renormalises the stored pair
// and adds exactly: (hi, lo) <- TwoSum(hi, lo) + (hi', lo').  kAccLo touches
// only the lo plane, lo <- lo + (hi' + lo') rounded to nearest, which halves
// the accumulator bytes a launch moves; lo then holds the last few launches'
// sums undigested (hi + lo stays the value) until the next kAccPair launch
// folds it back.  Every reader of the accumulator takes hi + lo, so both
// states are valid inputs everywhere.
constexpr int32_t kAccPair = 0;
constexpr int32_t kAccLo = 1;

// One fused split-K pass over the queued batches of one dtype.
struct SyrkParams {
    CUtensorMap maps[kMaxBatches];      // batch b: dims {d, n_b}, 128B swizzle
    int32_t kb_start[kMaxBatches + 1];  // prefix sum of ceil(n_b / kKBlock)
    int32_t n_batches;
    int32_t total_kb;       // k-blocks over all batches
    int32_t n_slabs;        // token slabs (split-K factor)
    int32_t n_tiles;        // upper-triangle tiles
    int32_t tiles_per_dim;  // ceil(d / kTile)
    int32_t chunk_kb;       // k-blocks per tensor-memory accumulation chunk
    int32_t d;
    int32_t n_units;        // n_tiles * n_slabs
    int32_t exclusive;      // 1: one token slab, so each accumulator tile has one writer and the
                            // epilogue reads, adds and stores it (else compensated atomics)
    int32_t acc_mode;       // exclusive launches: kAccPair or kAccLo
    int32_t tail_split;     // single-slab kAccLo launches: the last tail_split tiles of the tile
                            // order run as two units of half the k-blocks each (their lo sums
                            // meet in L2), so that the last wave of units is as short as the rest
                            // allow; n_units = n_tiles + tail_split
    float* acc;             // (hi, lo) accumulator (tile layout above)
    uint32_t* status;
    unsigned long long timeout_ns;
    const void* l2_ptr;     // bf16 flushes of one small batch: its X (l2_bytes, a multiple of 16),
    uint64_t l2_bytes;      // which the CTAs prefetch into L2 before the grid wait; else 0
};

// Upper-triangle tile index of tile (I, J), I <= J < T (row-major over I).
__host__ __device__ inline int tile_index(int I, int J, int T) {
    return I * T - (I * (I - 1)) / 2 + (J - I);
}

cudaError_t syrk_bf16_prepare();  // sets the dynamic shared-memory limit (per device)
// `overlap`: launch with programmatic stream serialization, so that the
// kernel's set-up may run while the previous kernel of the stream ends (every
// SYRK kernel waits for the previous grid before it reads X or the
// accumulator).
cudaError_t launch_syrk_bf16(const SyrkParams& p, int grid, cudaStream_t s, bool overlap);

// Pair-of-SMs bf16 kernel (256 x 128 tiles): n_tiles counts pair tiles,
// sum over I2 < ceil(T/2) of (T - 2*I2); the grid is 2 CTAs per pair.
cudaError_t syrk_bf16_2sm_prepare(int* max_pairs);
cudaError_t launch_syrk_bf16_2sm(const SyrkParams& p, int grid, cudaStream_t s, bool overlap);
__host__ __device__ inline int pair_tile_count(int T) {
    int n = 0;
    for (int i = 0; 2 * i < T; ++i) n += T - 2 * i;
    return n;
}

// Tensor-core fp32 GEMM C[M x N] += alpha P^T Q (gemm_tf32.cu); P is K x M and
// Q is K x N, both row-major with the minor dimension contiguous.
struct GemmTf32Params {
    CUtensorMap p_map;  // P: dims {M, K}, 32 x 32 boxes, fp32, 128B swizzle with 32B atoms
    CUtensorMap q_map;  // Q: dims {N, K}
    float* C;
    int32_t ldc, M, N, K;
    float alpha;
    int32_t tiles_n;  // N / 128
    int32_t n_kb;     // K / 32
    int32_t n_units;  // tiles_n * ceil(M / 128), or T (T + 1) / 2 tiles when lower
    int32_t lower;    // 1: square C, only the 128 x 128 tiles at or below the diagonal
    uint32_t* status;
    unsigned long long timeout_ns;
};
cudaError_t gemm_tf32_prepare();
// Encodes the tensor maps and launches.  P, Q, C 16-byte aligned; ldp, ldq,
// ldc multiples of 4; N % 128 == 0; K % 32 == 0; M >= 1.
// `lower`: M == N and only the tiles at or below the diagonal are computed
// (the diagonal tiles in full).
cudaError_t launch_gemm_tf32(const float* P, int ldp, const float* Q, int ldq, float* C, int ldc, int M, int N,
                             int K, float alpha, uint32_t* status, unsigned long long timeout_ns, int grid_max,
                             cudaStream_t s, bool lower = false);

cudaError_t syrk_f32_prepare();
cudaError_t launch_syrk_f32(const SyrkParams& p, int grid, cudaStream_t s, bool overlap);

// Materialize: damp = damp_percent * mean_i(acc_ii * scale) into damp_out
// (fp64) and damp_out_f32; then H_out (row-major d x d fp32).
// Scratch of one materialization: the fp64 damping value, per-quarter sums
// of the diagonal and an arrival count (zeroed once, left zero by each launch).
size_t materialize_scratch_bytes(int T);
// The kernel waits for the previous kernel of the stream (it is launched to
// overlap that kernel's end).  With status_mirror non-null (a device pointer
// to mapped pinned host memory) it also writes there *status (word 0) and
// the fp32 damping value (word 1).
cudaError_t launch_materialize(const float* acc, float* H_out, int d, int T, double scale,
                               double damp_percent, double* scratch, float* damp_f32, const uint32_t* status,
                               uint32_t* status_mirror, cudaStream_t s);

// Local 16x16 block Grams.
constexpr int kLocalKBlock = 64;   // tokens per stage
constexpr int kLocalGroup = 256;   // features per CTA (16 blocks)
struct LocalParams {
    CUtensorMap map;        // X: dims {d, n}, box {64, kLocalKBlock}, 128B swizzle
    double* acc;            // [d/16][16][16] fp64, full blocks
    uint32_t* status;
    unsigned long long timeout_ns;
    int32_t d;
    int32_t n_groups;       // ceil(d / kLocalGroup)
    int32_t n_ranges;       // token ranges per group
    int32_t total_kb;       // ceil(n / kLocalKBlock)
    int32_t chunk_steps;    // 16-token MMA steps per register chain
};
cudaError_t local_prepare();
cudaError_t launch_local_gram(const LocalParams& p, int grid, cudaStream_t s);
cudaError_t launch_local_read(const double* acc, float* out, int n_blocks, double scale,
                              cudaStream_t s);

// Four 32-bit words stored to 16-byte-aligned device memory, in stream order.
cudaError_t launch_store_words(uint32_t* dst, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                               cudaStream_t s);

// (hi, lo) <- TwoSum(hi, lo) over n_tiles accumulator tiles (folds lo into hi).
cudaError_t launch_renorm_pairs(float* acc, size_t n_tiles, int sm_count, cudaStream_t s);

// dst += src over n_tiles (hi, lo) accumulator tiles (accumulator merge).
cudaError_t launch_add_pairs(float* dst, const float* src, size_t n_tiles, int sm_count,
                             cudaStream_t s);
// acc[i] += sum_t X[t][i]^2 (fp64 accumulator), X row-major [n, d], d % 8 == 0.
cudaError_t launch_colsumsq(const void* X, bool f32, int64_t n, int d, double* acc, int sm_count,
                            cudaStream_t s);
cudaError_t launch_colsumsq_read(const double* acc, float* out, int d, cudaStream_t s);

// Sets the thread-local message returned by hess_last_error().
void set_last_error(const char* msg);

}  // namespace hk
