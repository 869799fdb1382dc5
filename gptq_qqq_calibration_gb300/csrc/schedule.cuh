// The unit schedule of a fused SYRK pass: which (tile, token slab) each
// persistent CTA takes, for the single-SM and pair-of-SMs kernels, and the
// host rule that splits the last wave.  Host and device functions, so that
// the kernels, the host library and a CPU test of the schedule
// (tests/schedule_check.cu) run the same code.
#pragma once

#include "kernels.cuh"

namespace hk {
namespace syrk {

// A unit is one 128x128 upper tile (I, J) over one slab [k0, k1) of the
// flush's k-blocks.  Units are numbered slab-major so that the CTAs running
// at the same time stream the same tokens.  With p.tail_split > 0 (one
// slab): units below n_tiles - tail_split are whole tiles; the rest are the
// last tail_split tiles, each as its first and second half of the k-blocks.
struct Unit {
    int t, I, J, k0, k1;
};

__host__ __device__ inline bool unit_at(const SyrkParams& p, int u, Unit& un) {
    int t;
    if (p.tail_split > 0) {
        const int whole = p.n_tiles - p.tail_split;
        if (u < whole) {
            t = u;
            un.k0 = 0;
            un.k1 = p.total_kb;
        } else {
            const int v = u - whole;
            t = whole + (v >> 1);
            const int mid = p.total_kb >> 1;
            un.k0 = (v & 1) ? mid : 0;
            un.k1 = (v & 1) ? p.total_kb : mid;
        }
    } else {
        const int slab = u / p.n_tiles;
        t = u - slab * p.n_tiles;
        un.k0 = static_cast<int>(static_cast<long long>(slab) * p.total_kb / p.n_slabs);
        un.k1 = static_cast<int>(static_cast<long long>(slab + 1) * p.total_kb / p.n_slabs);
    }
    int i = 0, rem = t;
    while (rem >= p.tiles_per_dim - i) {
        rem -= p.tiles_per_dim - i;
        ++i;
    }
    un.t = t;
    un.I = i;
    un.J = i + rem;
    return un.k1 > un.k0;
}

// The kernels' guard before a unit's addresses are formed: a tile inside the
// upper triangle and a slab inside the flush.
__host__ __device__ inline bool unit_in_range(const SyrkParams& p, const Unit& un) {
    return un.t >= 0 && un.t < p.n_tiles && un.I >= 0 && un.I <= un.J && un.J < p.tiles_per_dim &&
           un.k0 >= 0 && un.k0 < un.k1 && un.k1 <= p.total_kb;
}

// Pair-of-SMs units: tiles of 256 rows (I2) x 128 columns (J), J >= 2 I2,
// n_tiles = pair_tile_count(T) per slab.  CTA `rank` of the pair stores
// accumulator tile (2 I2 + rank, J) unless it lies below the diagonal or
// past the last row block (out tile -1).
struct PairUnit {
    int I2, J, k0, k1;
};

__host__ __device__ inline bool pair_unit_at(const SyrkParams& p, int u, PairUnit& un) {
    const int slab = u / p.n_tiles;
    const int t = u - slab * p.n_tiles;
    const int T = p.tiles_per_dim;
    int i = 0, rem = t;
    while (rem >= T - 2 * i) {
        rem -= T - 2 * i;
        ++i;
    }
    un.I2 = i;
    un.J = 2 * i + rem;
    un.k0 = static_cast<int>(static_cast<long long>(slab) * p.total_kb / p.n_slabs);
    un.k1 = static_cast<int>(static_cast<long long>(slab + 1) * p.total_kb / p.n_slabs);
    return un.k1 > un.k0;
}

__host__ __device__ inline int pair_out_tile(const PairUnit& un, int rank, int T) {
    const int rb = 2 * un.I2 + rank;
    return (rb < T && rb <= un.J) ? tile_index(rb, un.J, T) : -1;
}

__host__ __device__ inline bool pair_unit_in_range(const SyrkParams& p, const PairUnit& un) {
    return un.I2 >= 0 && 2 * un.I2 <= un.J && un.J < p.tiles_per_dim && un.k0 >= 0 && un.k0 < un.k1 &&
           un.k1 <= p.total_kb;
}

#ifdef __CUDACC__
// Device forms: false for an empty unit, and for one that fails its range
// guard, which also records kStatusBadIndex.  Every role of a kernel walks
// the units through these, so a bad unit is skipped by all of them alike.
__device__ __forceinline__ bool unit_checked(const SyrkParams& p, int u, Unit& un) {
    if (!unit_at(p, u, un)) return false;
    if (unit_in_range(p, un)) return true;
    atomicOr(p.status, kStatusBadIndex);
    return false;
}
__device__ __forceinline__ bool pair_unit_checked(const SyrkParams& p, int u, PairUnit& un) {
    if (!pair_unit_at(p, u, un)) return false;
    if (pair_unit_in_range(p, un)) return true;
    atomicOr(p.status, kStatusBadIndex);
    return false;
}
#endif

// Host rule: a single-slab flush that adds to the lo plane with reductions
// (two writers per tile are fine) and whose last wave would fill at most
// half the grid runs that wave's tiles as two half units each.
__host__ __device__ inline int tail_split_for(int n_tiles, int grid_max, int total_kb, bool exclusive,
                                              int32_t acc_mode) {
    const int rem = n_tiles % grid_max;
    return (exclusive && acc_mode == kAccLo && n_tiles > grid_max && rem > 0 && 2 * rem <= grid_max &&
            total_kb >= 2)
               ? rem
               : 0;
}

}  // namespace syrk
}  // namespace hk
