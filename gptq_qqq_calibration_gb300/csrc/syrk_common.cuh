// Pieces shared by the bf16 and fp32 SYRK kernels: the unit schedule and
// the compensated epilogue that folds tensor-memory chunks into registers.
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

namespace hk {
namespace syrk {

// Before the wait for the previous grid (which reads nothing of the
// previous kernel's output): the first unit's tensor map is fetched into
// the descriptor cache and the parameters into the constant cache.
__device__ __forceinline__ void prefetch_first_map(const SyrkParams& p) {
    Unit un;
    if (static_cast<int>(blockIdx.x) < p.n_units && unit_at(p, blockIdx.x, un) && unit_in_range(p, un)) {
        int b = 0;
        while (b + 1 < p.n_batches && p.kb_start[b + 1] <= un.k0) ++b;
        prefetch_tensormap(&p.maps[b]);
    }
}

constexpr int kEpiWarps = 8;                   // 2 per tensor-memory lane quarter
constexpr int kMidGroup = 8;                   // chunks summed in `mid` between folds
constexpr int kEpiCols = 4 * 128 / kEpiWarps;  // accumulator columns per warp
constexpr unsigned long long kDrainLimitNs = 1000000000ull;

// Epilogue of one CTA (kEpiWarps warps starting at first_warp).
// Tensor memory holds 2 buffers x 2 banks x 128 columns; chunk c of a unit
// sits in buffer (chunk counter & 1).  Each warp reads its lane quarter
// (warp % 4) and kEpiCols of the 128 columns and adds the two banks, on
// packed fp32 pairs.  The chunk sums reach a compensated (hi, lo) pair in
// one of two ways:
//   * kGroup == 0: every chunk sum is folded in with Fast2Sum;
//   * kGroup > 0: chunk sums are added into `mid` with plain round-to-nearest
//     adds (unbiased; over kGroup chunks their error is ~sqrt(kGroup) half-
//     ulps of mid, i.e. ~1e-8 of the entry at the end of a long unit), and
//     mid is folded in with an exact TwoSum every kGroup chunks and at the
//     end of the unit.  This needs 3 x kEpiCols registers of state per
//     thread (a re-split register budget) for about half the arithmetic.
// At the end of a unit, (hi, lo) is added to the (hi, lo) accumulator tile
// `out_tile` (skipped when it is negative): by a plain read-modify-write when
// the launch has one token slab (kExcl, the kernel instance chosen when
// p.exclusive is set) -- of both planes (kAccPair) or of the lo plane alone
// (kAccLo) -- else by compensated fp32 atomics.
//   unit_fn(u, k0, k1, out_tile) -> false if unit u is empty;
//   wait_full(bar, parity) waits for a filled accumulator buffer;
//   arrive_empty(b) releases buffer b to the MMA issuer.
template <bool kExcl, int kGroup, class UnitFn, class WaitFn, class ArriveFn>
__device__ __forceinline__ void epilogue_t(const SyrkParams& p, uint32_t tmem, int warp, int lane,
                                           int first_warp, uint32_t accf_bar0, int u0, int ustride,
                                           UnitFn unit_fn, WaitFn wait_full, ArriveFn arrive_empty) {
    const int q = warp & 3;
    const int part = (warp - first_warp) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(part) * kEpiCols;
    uint64_t hi[kEpiCols / 2], lo[kEpiCols / 2];  // this thread's columns, as pairs
    uint64_t mid[kGroup > 0 ? kEpiCols / 2 : 1];
    bool ok = true;
    int ab = 0;
    uint32_t aphase = 0;
    for (int u = u0; ok && u < p.n_units; u += ustride) {
        int k0, k1, out_tile;
        if (!unit_fn(u, k0, k1, out_tile)) continue;
        if constexpr (kExcl) {
            // the tile's old values travel to L2 while the unit's MMAs run
            if (out_tile >= 0 && warp == first_warp && lane == 0) {
                if (p.acc_mode == kAccLo)
                    prefetch_l2_bulk(p.acc + static_cast<size_t>(out_tile) * kTileWords + kTileElems,
                                     kTileElems * sizeof(float));
                else
                    prefetch_l2_bulk(p.acc + static_cast<size_t>(out_tile) * kTileWords,
                                     kTileWords * sizeof(float));
            }
        }
        const int nch = (k1 - k0 + p.chunk_kb - 1) / p.chunk_kb;
        if constexpr (kGroup > 0) {
#pragma unroll
            for (int i = 0; i < kEpiCols / 2; ++i) hi[i] = lo[i] = mid[i] = 0ull;
        }
        int g = 0;  // chunks in mid
        for (int c = 0; c < nch; ++c) {
            if (!wait_full(accf_bar0 + 8u * ab, aphase)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tb = tmem + lane_off + static_cast<uint32_t>(ab) * 256u + col0;
#pragma unroll
            for (int it = 0; it < kEpiCols / 8; ++it) {
                uint32_t b0[8], b1[8];
                tmem_ld8x2_sync(tb + it * 8, tb + 128 + it * 8, b0, b1);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t v = add2(pack2(b0[2 * k], b0[2 * k + 1]),
                                            pack2(b1[2 * k], b1[2 * k + 1]));
                    const int i = it * 4 + k;
                    if constexpr (kGroup > 0) {
                        mid[i] = add2(mid[i], v);
                    } else if (c == 0) {
                        hi[i] = v;
                        lo[i] = 0ull;
                    } else {
                        // The running sum dominates the chunk for the large
                        // (diagonal-like) entries that set the error, where
                        // Fast2Sum is exact; elsewhere it errs like one add.
                        uint64_t e;
                        hi[i] = fast_two_sum2(hi[i], v, e);
                        lo[i] = add2(lo[i], e);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_empty(ab);
            if (++ab == 2) {
                ab = 0;
                aphase ^= 1u;
            }
            if constexpr (kGroup > 0) {
                // fold mid while the MMAs fill the other buffer
                if (++g == kGroup || c + 1 == nch) {
#pragma unroll
                    for (int i = 0; i < kEpiCols / 2; ++i) {
                        uint64_t e;
                        hi[i] = two_sum2(hi[i], mid[i], e);
                        lo[i] = add2(lo[i], e);
                        mid[i] = 0ull;
                    }
                    g = 0;
                }
            }
        }
        if (!ok) break;
        if (out_tile < 0) continue;
        if (out_tile >= p.tiles_per_dim * (p.tiles_per_dim + 1) / 2) {  // guard: not a tile of H
            atomicOr(p.status, kStatusBadIndex);
            continue;
        }
        // this thread's row of the hi plane, from column col0 on (4-column
        // blocks of 4 words); the lo plane is kTileElems further
        float* const out = p.acc + static_cast<size_t>(out_tile) * kTileWords + tile_offset(row, col0);
        if constexpr (kExcl) {
          if (p.acc_mode == kAccLo) {
            // Sole writer, lo plane only: lo += hi' + lo', with the add done
            // in L2 by vector reductions (round to nearest, like an fp32
            // add): nothing comes back to the SM, so the epilogue moves on
            // to the next unit at once.
#pragma unroll
            for (int q = 0; q < kEpiCols / 4; ++q) {
                float4 v;
                unpack2(add2(hi[2 * q], lo[2 * q]), v.x, v.y);
                unpack2(add2(hi[2 * q + 1], lo[2 * q + 1]), v.z, v.w);
                red_add_v4_f32(out + kTileElems + q * 4 * kTile, v);
            }
          } else {
            // Sole writer of this tile in this launch: a plain read-modify-
            // write of (hi, lo) += (hi', lo'), 16-byte accesses, kRmw
            // columns' loads in flight at a time (with kGroup > 0 the dead
            // `mid` registers hold them).  The stored pair is renormalised
            // first with an exact TwoSum (lo may hold undigested kAccLo
            // sums), then the hi parts are added with an exact TwoSum.
            constexpr int kRmw = kGroup > 0 ? 32 : 8;
#pragma unroll
            for (int g = 0; g < kEpiCols / kRmw; ++g) {
                float4 oh[kRmw / 4], ol[kRmw / 4];
#pragma unroll
                for (int i = 0; i < kRmw / 4; ++i) {
                    const int q = (kRmw * g) / 4 + i;  // 4-column block of this thread
                    oh[i] = *reinterpret_cast<const float4*>(out + q * 4 * kTile);
                    ol[i] = *reinterpret_cast<const float4*>(out + kTileElems + q * 4 * kTile);
                }
#pragma unroll
                for (int i = 0; i < kRmw / 4; ++i) {
                    const int q = (kRmw * g) / 4 + i;
                    uint64_t f0, f1, e0, e1;
                    const uint64_t h0 = two_sum2(pack2(__float_as_uint(oh[i].x), __float_as_uint(oh[i].y)),
                                                 pack2(__float_as_uint(ol[i].x), __float_as_uint(ol[i].y)), f0);
                    const uint64_t h1 = two_sum2(pack2(__float_as_uint(oh[i].z), __float_as_uint(oh[i].w)),
                                                 pack2(__float_as_uint(ol[i].z), __float_as_uint(ol[i].w)), f1);
                    const uint64_t s0 = two_sum2(h0, hi[2 * q], e0);
                    const uint64_t s1 = two_sum2(h1, hi[2 * q + 1], e1);
                    const uint64_t t0 = add2(add2(f0, lo[2 * q]), e0);
                    const uint64_t t1 = add2(add2(f1, lo[2 * q + 1]), e1);
                    float4 nh, nl;
                    unpack2(s0, nh.x, nh.y);
                    unpack2(s1, nh.z, nh.w);
                    unpack2(t0, nl.x, nl.y);
                    unpack2(t1, nl.z, nl.w);
                    *reinterpret_cast<float4*>(out + q * 4 * kTile) = nh;
                    *reinterpret_cast<float4*>(out + kTileElems + q * 4 * kTile) = nl;
                }
            }
          }
        } else {
            // Several slabs add to this tile: an atomic add of hi' to hi
            // returns the old value, from which the exact rounding error of
            // that add is recovered (the stored sum is old + hi' rounded to
            // nearest) and added, with lo', to lo.  Atomics go out in groups
            // so that their round trips overlap.
            constexpr int kAtomQ = 4;  // 4-column blocks per group
#pragma unroll
            for (int g = 0; g < kEpiCols / (4 * kAtomQ); ++g) {
                float4 hv[kAtomQ], lv[kAtomQ], old[kAtomQ];
#pragma unroll
                for (int i = 0; i < kAtomQ; ++i) {
                    const int q = kAtomQ * g + i;
                    unpack2(hi[2 * q], hv[i].x, hv[i].y);
                    unpack2(hi[2 * q + 1], hv[i].z, hv[i].w);
                    unpack2(lo[2 * q], lv[i].x, lv[i].y);
                    unpack2(lo[2 * q + 1], lv[i].z, lv[i].w);
                }
#pragma unroll
                for (int i = 0; i < kAtomQ; ++i)
                    old[i] = atom_add_v4_f32(out + (kAtomQ * g + i) * 4 * kTile, hv[i]);
#pragma unroll
                for (int i = 0; i < kAtomQ; ++i) {
                    float e;
                    float4 l = lv[i];
                    two_sum_f32(old[i].x, hv[i].x, e);
                    l.x = __fadd_rn(l.x, e);
                    two_sum_f32(old[i].y, hv[i].y, e);
                    l.y = __fadd_rn(l.y, e);
                    two_sum_f32(old[i].z, hv[i].z, e);
                    l.z = __fadd_rn(l.z, e);
                    two_sum_f32(old[i].w, hv[i].w, e);
                    l.w = __fadd_rn(l.w, e);
                    red_add_v4_f32(out + kTileElems + (kAtomQ * g + i) * 4 * kTile, l);
                }
            }
        }
    }
    if (!ok && lane == 0) atomicOr(p.status, kStatusTimeoutEpilogue);
}

// Launches a SYRK kernel.  With `overlap`, the launch allows programmatic
// dependent launch: its CTAs may start on SMs that the previous kernel of the
// stream has released, before that kernel ends.  Every SYRK kernel does its
// set-up (barriers, tensor memory), then waits for the previous grid
// (griddep_wait) before anything else, and lets its own dependents start
// (griddep_launch_dependents).
template <class Kernel>
inline cudaError_t launch_syrk(Kernel kernel, const SyrkParams& p, int grid, int threads, size_t smem,
                               cudaStream_t s, bool overlap) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// The single-CTA form: units in blockIdx.x + k * gridDim.x order, local barriers.
template <bool kExcl, int kGroup>
__device__ __forceinline__ void epilogue(const SyrkParams& p, uint32_t tmem, int warp, int lane,
                                         int first_warp, uint32_t accf_bar0, uint32_t acce_bar0,
                                         unsigned long long limit) {
    epilogue_t<kExcl, kGroup>(
        p, tmem, warp, lane, first_warp, accf_bar0, blockIdx.x, gridDim.x,
        [&](int u, int& k0, int& k1, int& out_tile) {
            Unit un;
            if (!unit_checked(p, u, un)) return false;
            k0 = un.k0;
            k1 = un.k1;
            out_tile = un.t;
            return true;
        },
        [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, limit); },
        [&](int b) { mbar_arrive(acce_bar0 + 8u * b); });
}

}  // namespace syrk
}  // namespace hk
