// Host-only check of the SYRK unit schedule (compiled by
// tests/test_schedule_cpu.py with nvcc; it runs on the CPU, no GPU needed).
//
// The kernels walk their work through hk::syrk::unit_at (single-SM tiles,
// split-K slabs, the tail split) and hk::syrk::pair_unit_at /
// pair_out_tile (pairs of SMs).  This program calls those same functions
// for many flush shapes and checks that:
//   * every unit lies in the upper triangle and inside the flush's k-blocks
//     (the guard the kernels apply, unit_in_range / pair_unit_in_range);
//   * for every upper tile the k-ranges of its units cover [0, total_kb)
//     exactly once (no k-block summed twice or missed);
//   * for the pair kernel, every upper tile is stored by exactly one CTA of
//     one pair unit per slab, and tiles below the diagonal are never stored;
//   * tile_offset maps a tile's 128 x 128 elements one to one onto its plane.
// Prints "schedule ok <configurations>" and exits 0, or prints the first
// failure and exits 1.
#include <cstdio>
#include <vector>

#include "schedule.cuh"

using hk::SyrkParams;
namespace sy = hk::syrk;

static int fail(const char* what, int T, int kb, int slabs, int tail, int u) {
    std::printf("FAIL %s: tiles_per_dim=%d total_kb=%d slabs=%d tail_split=%d unit=%d\n", what, T, kb, slabs,
                tail, u);
    return 1;
}

static int check_single(int T, int total_kb, int slabs, int tail) {
    SyrkParams p{};
    p.tiles_per_dim = T;
    p.n_tiles = T * (T + 1) / 2;
    p.total_kb = total_kb;
    p.n_slabs = slabs;
    p.tail_split = tail;
    p.n_units = p.n_tiles * slabs + tail;
    // cover[t][kb]: how many units sum k-block kb of tile t
    std::vector<int> cover(static_cast<size_t>(p.n_tiles) * total_kb, 0);
    for (int u = 0; u < p.n_units; ++u) {
        sy::Unit un;
        if (!sy::unit_at(p, u, un)) continue;  // empty slab
        if (!sy::unit_in_range(p, un)) return fail("unit out of range", T, total_kb, slabs, tail, u);
        if (hk::tile_index(un.I, un.J, T) != un.t) return fail("tile index", T, total_kb, slabs, tail, u);
        for (int k = un.k0; k < un.k1; ++k) ++cover[static_cast<size_t>(un.t) * total_kb + k];
    }
    for (size_t i = 0; i < cover.size(); ++i)
        if (cover[i] != 1) return fail("k-block not covered exactly once", T, total_kb, slabs, tail, static_cast<int>(i));
    return 0;
}

static int check_pair(int T, int total_kb, int slabs) {
    SyrkParams p{};
    p.tiles_per_dim = T;
    p.n_tiles = hk::pair_tile_count(T);
    p.total_kb = total_kb;
    p.n_slabs = slabs;
    p.tail_split = 0;
    p.n_units = p.n_tiles * slabs;
    const int n_acc = T * (T + 1) / 2;
    std::vector<int> cover(static_cast<size_t>(n_acc) * total_kb, 0);
    for (int u = 0; u < p.n_units; ++u) {
        sy::PairUnit un;
        if (!sy::pair_unit_at(p, u, un)) continue;
        if (!sy::pair_unit_in_range(p, un)) return fail("pair unit out of range", T, total_kb, slabs, 0, u);
        for (int rank = 0; rank < 2; ++rank) {
            const int t = sy::pair_out_tile(un, rank, T);
            const int rb = 2 * un.I2 + rank;
            if (t < 0) {
                if (rb < T && rb <= un.J) return fail("upper tile not stored", T, total_kb, slabs, 0, u);
                continue;
            }
            if (t >= n_acc || rb > un.J) return fail("stored tile out of range", T, total_kb, slabs, 0, u);
            if (hk::tile_index(rb, un.J, T) != t) return fail("pair tile index", T, total_kb, slabs, 0, u);
            for (int k = un.k0; k < un.k1; ++k) ++cover[static_cast<size_t>(t) * total_kb + k];
        }
    }
    for (size_t i = 0; i < cover.size(); ++i)
        if (cover[i] != 1) return fail("pair: k-block not covered exactly once", T, total_kb, slabs, 0, static_cast<int>(i));
    return 0;
}

static int check_tile_offset() {
    std::vector<int> seen(hk::kTileElems, 0);
    for (int r = 0; r < hk::kTile; ++r)
        for (int c = 0; c < hk::kTile; ++c) {
            const int o = hk::tile_offset(r, c);
            if (o < 0 || o >= hk::kTileElems || seen[o]++) return fail("tile_offset", r, c, 0, 0, 0);
        }
    return 0;
}

int main() {
    int n = 0;
    if (check_tile_offset()) return 1;
    const int kbs[] = {1, 2, 3, 7, 64, 513};
    const int grids[] = {1, 2, 3, 4, 7, 152};
    for (int T = 1; T <= 36; ++T) {
        const int n_tiles = T * (T + 1) / 2;
        for (int kb : kbs) {
            for (int slabs : {1, 2, 3, 7, 40}) {
                if (slabs > kb) continue;
                if (check_single(T, kb, slabs, 0)) return 1;
                if (check_pair(T, kb, slabs)) return 1;
                n += 2;
            }
            // the tail split as the host chooses it, for every grid size
            for (int g : grids) {
                const int tail = sy::tail_split_for(n_tiles, g, kb, true, hk::kAccLo);
                if (tail < 0 || tail > n_tiles) return fail("tail split size", T, kb, 1, tail, g);
                if (tail > 0) {
                    // the last wave: at most half the grid before the split, full after
                    if (2 * tail > g) return fail("tail split larger than half the grid", T, kb, 1, tail, g);
                    if (sy::tail_split_for(n_tiles, g, kb, true, hk::kAccPair) != 0 ||
                        sy::tail_split_for(n_tiles, g, kb, false, hk::kAccLo) != 0)
                        return fail("tail split outside single-slab lo flushes", T, kb, 1, tail, g);
                }
                if (check_single(T, kb, 1, tail)) return 1;
                ++n;
            }
            // every tail size the schedule can take
            for (int tail = 1; tail <= n_tiles && kb >= 2; tail += (n_tiles > 40 ? 7 : 1)) {
                if (check_single(T, kb, 1, tail)) return 1;
                ++n;
            }
        }
    }
    std::printf("schedule ok %d\n", n);
    return 0;
}
