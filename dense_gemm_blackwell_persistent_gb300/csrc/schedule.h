// schedule.h -- static work schedule of the persistent GEMM: which output
// tiles and which K ranges each resident CTA pair ("unit") processes.
//
// Whole tiles in data-parallel waves, then a stream-K part for a partial
// last wave.  With T tiles on P units and R = T mod P > 0, plain waves would
// leave P - R units idle for a whole tile time.  Instead the first W - 1
// waves (W = T / P) run whole tiles and the remaining S = P + R tiles -- the
// last full wave plus the partial one -- have their S*KB k-blocks cut into P
// contiguous ranges of near-equal length, one per unit.  Every range is
// longer than a tile (S > P), so a tile is split between at most two units:
//
//   * contributor 0 holds the tile's first k-blocks; that piece ends its
//     unit's range, so it is the unit's last work item;
//   * contributor 1 holds the rest; that piece starts its unit's range, so
//     it is the unit's first stream-K item and is finished long before.
//
// Contributor 1 publishes its fp32 partial in a workspace slot (one slot per
// unit: a unit starts at most one range) and raises a flag; contributor 0
// waits for the flag, adds the partial to its own accumulator and writes C.
// With two addends the fp32 sum does not depend on which one is "own", so
// results are deterministic.
//
// With fewer tiles than units (W = 0) and T <= P/2, each tile is instead
// split into two K halves on 2T units (same protocol, same roles).
//
// Stream-K is used only when it is predicted to pay: the time saved, in
// k-blocks of one unit, must exceed kFixupKBlocks, an estimate of the
// publish/wait/add cost of a split tile.
//
// Prior art: the persistent grid of "Collective matrix multiplication"
// (grid = number of SMs, static tile loop); the split of the reduction
// dimension with an fp32 accumulator cast once at the end follows the
// K-accumulating matmul of "Chapter 7: Writing Custom Kernels with Pallas",
// §4.1'/§4.4 (there one program runs all K steps of a block; here two units
// share them and one of them adds the two partial sums).
//
// Plain C++ with host/device qualifiers so the host code and the CPU tests
// can run exactly the logic the kernel runs.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define GB300_HD __host__ __device__ __forceinline__
#else
#define GB300_HD inline
#endif

namespace gb300 {

// Division by a divisor fixed for the whole launch, as a multiply and a
// shift (T. Granlund and P. L. Montgomery, "Division by Invariant Integers
// using Multiplication", PLDI 1994): for 1 <= d < 2^31 and 0 <= x < 2^31,
// with l = ceil(log2 d) and p = 31 + l, m = ceil(2^p / d) < 2^32 and
// x / d = floor(x * m / 2^p).  Why it is exact: m * d = 2^p + e with
// 0 <= e < d, so x * m / 2^p = x / d + x * e / (d * 2^p), and the second term
// is below 2^31 / 2^p = 2^-l <= 1 / d, too little to reach the next integer
// from x / d, whose fraction is at most (d - 1) / d.  The host builds it once
// per launch; the kernel's tile decode then needs no division instructions.
// d == 1 is a plain copy (p - 32 would be negative).
struct FastDiv {
    uint32_t d;     // the divisor
    uint32_t mul;   // m (unused when d == 1)
    uint32_t shr;   // p - 32
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.mul = 0;
    f.shr = 0;
    if (d > 1) {
        uint32_t l = 0;
        while ((uint64_t(1) << l) < d) ++l;   // ceil(log2 d)
        const uint32_t p = 31 + l;
        f.mul = (uint32_t)(((uint64_t(1) << p) + d - 1) / d);
        f.shr = p - 32;
    }
    return f;
}

#if defined(__CUDACC__)
__host__ __device__ __forceinline__ uint32_t mul_hi_u32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
    return __umulhi(a, b);
#else
    return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}
#else
inline uint32_t mul_hi_u32(uint32_t a, uint32_t b) { return (uint32_t)(((uint64_t)a * b) >> 32); }
#endif

// x / f.d for 0 <= x < 2^31.
GB300_HD uint32_t fast_div(const FastDiv& f, uint32_t x) { return f.d == 1 ? x : mul_hi_u32(x, f.mul) >> f.shr; }

// Estimated cost of a split tile's fix-up, in k-blocks of MMA time: on
// GB300 the finishing unit's tail (bulk copy of the other partial, add,
// store) measured ~3-4.5 µs against ~2 µs for a plain last epilogue, and the
// units' end times spread by a few µs more; 12 k-blocks of a 256-wide tile
// are ~3.5 µs.
constexpr int kFixupKBlocks = 12;

struct Schedule {
    int tiles;        // T: output tiles
    int units;        // P: units that run (the grid)
    int kb;           // KB: k-blocks per tile
    int dp_waves;     // whole tiles per unit before the stream-K part (all of T when sk_tiles == 0)
    int sk_tiles;     // S: tiles whose k-blocks are spread over all units (0 = none)
};

// One unit of work for every role of a unit: tile `tile`, k-blocks
// [kb_begin, kb_end).  For a split tile (`ncontrib` == 2), `contrib` is 0
// for the piece holding the tile's first k-blocks (it finishes the tile)
// and 1 for the other, `slot` is the workspace slot of contributor 1's
// partial (the index of its unit) and `sk_index` the tile's index in the
// stream-K part (its flag).
struct Work {
    int tile;
    int kb_begin, kb_end;
    int contrib, ncontrib;
    int slot;
    int sk_index;
};

GB300_HD Schedule make_schedule(int tiles, int units, int kb, bool allow_stream_k) {
    Schedule s;
    s.tiles = tiles;
    s.kb = kb;
    const int waves = tiles / units, rem = tiles % units;
    if (allow_stream_k && rem != 0 && kb >= 2) {
        if (waves >= 1 && (int64_t)(units - rem) * kb > (int64_t)kFixupKBlocks * units) {
            s.units = units;
            s.dp_waves = waves - 1;
            s.sk_tiles = units + rem;
            return s;
        }
        if (waves == 0 && 2 * tiles <= units && kb > 2 * kFixupKBlocks) {
            s.units = 2 * tiles;
            s.dp_waves = 0;
            s.sk_tiles = tiles;
            return s;
        }
    }
    // whole tiles only, never more units than tiles
    s.units = units < tiles ? units : tiles;
    if (s.units < 1) s.units = 1;
    s.dp_waves = (tiles + s.units - 1) / s.units;
    s.sk_tiles = 0;
    return s;
}

// First stream-K k-block (in the concatenated stream-K k-block space) of unit u.
GB300_HD int64_t sk_begin(const Schedule& s, int u) {
    return (int64_t)u * ((int64_t)s.sk_tiles * s.kb) / s.units;
}

// The unit whose stream-K range contains k-block x (0 <= x < S*KB).
GB300_HD int sk_owner(const Schedule& s, int64_t x) {
    const int64_t total = (int64_t)s.sk_tiles * s.kb;
    // largest u with floor(u*total/P) <= x  <=>  u < (x+1)*P/total
    int64_t u = ((x + 1) * s.units + total - 1) / total - 1;
    if (u >= s.units) u = s.units - 1;
    if (u < 0) u = 0;
    return (int)u;
}

// Number of work items of unit u: its whole tiles plus its stream-K pieces.
GB300_HD int work_count(const Schedule& s, int u) {
    if (s.sk_tiles == 0) return u < s.tiles ? (s.tiles - 1 - u) / s.units + 1 : 0;
    const int64_t b0 = sk_begin(s, u), b1 = sk_begin(s, u + 1);
    if (b1 <= b0) return s.dp_waves;
    const int q0 = (int)(b0 / s.kb), q1 = (int)((b1 - 1) / s.kb);
    return s.dp_waves + (q1 - q0 + 1);
}

// All `kb` k-blocks of tile `tile`, by one unit.
GB300_HD Work whole_tile(int tile, int kb) {
    Work w;
    w.tile = tile;
    w.kb_begin = 0;
    w.kb_end = kb;
    w.contrib = 0;
    w.ncontrib = 1;
    w.slot = -1;
    w.sk_index = -1;
    return w;
}

// The j-th work item of unit u (0 <= j < work_count(s, u)).
GB300_HD Work work_item(const Schedule& s, int u, int j) {
    if (j < s.dp_waves || s.sk_tiles == 0) return whole_tile(u + j * s.units, s.kb);
    Work w;
    const int64_t b0 = sk_begin(s, u), b1 = sk_begin(s, u + 1);
    const int q = (int)(b0 / s.kb) + (j - s.dp_waves);
    const int64_t tile_lo = (int64_t)q * s.kb, tile_hi = tile_lo + s.kb;
    const int64_t lo = b0 > tile_lo ? b0 : tile_lo;
    const int64_t hi = b1 < tile_hi ? b1 : tile_hi;
    const int first = sk_owner(s, tile_lo);
    const int last = sk_owner(s, tile_hi - 1);
    w.tile = s.dp_waves * s.units + q;
    w.kb_begin = (int)(lo - tile_lo);
    w.kb_end = (int)(hi - tile_lo);
    w.contrib = u - first;
    w.ncontrib = last - first + 1;
    w.slot = w.ncontrib > 1 ? last : -1;
    w.sk_index = q;
    return w;
}

// Dynamic work list (cluster launch control): the grid has one cluster per
// list of tiles.  Cluster c < units owns the whole tiles c, c + units, ...,
// c + (waves - 1)·units of the persistent waves; cluster c >= units owns
// the single tile units·waves + (c - units).  A running unit does its own
// list, then the lists of clusters the hardware cancels for it, so every
// tile runs exactly once whichever clusters start.  units = tiles, waves = 1
// makes every tile a list of its own.
GB300_HD int dyn_list_count(int tiles, int units, int waves) { return units + (tiles - units * waves); }
GB300_HD int dyn_list_len(int c, int units, int waves) { return c < units ? waves : 1; }
GB300_HD int dyn_list_tile(int c, int k, int units, int waves) {
    return c < units ? c + k * units : units * waves + (c - units);
}

}  // namespace gb300
