// schedule.h -- static work schedule of the persistent GEMM: which output
// tiles and which K ranges each resident CTA pair ("unit") processes.
//
// Data-parallel waves, then a stream-K tail.  With T tiles on P units,
// W = T / P full waves run whole tiles (unit u takes tiles u, u+P, ...).
// The R = T - W*P tiles left over would leave P - R units idle for a whole
// tile time, so instead their R*KB k-blocks (KB per tile) are cut into P
// contiguous ranges of near-equal length, one per unit.  A range may start
// or end inside a tile; each piece of a tile ("segment") accumulates a
// partial sum over its k-blocks.  Every contributor of a split tile stores
// its fp32 partial in a workspace slot and bumps the tile's counter; the
// last to arrive adds all partials in contributor order (a fixed order, so
// results do not depend on timing) and writes C.
//
// Prior art: the persistent grid of "Collective matrix multiplication"
// (grid = number of SMs, static tile loop); the split of the reduction
// dimension across programs with an fp32 accumulator written once at the
// end follows the K-accumulating matmul of "Chapter 7: Writing Custom
// Kernels with Pallas", §4.1'/§4.4 (there the K steps of one block run in
// one program; here the last contributor does the final accumulation).
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

struct Schedule {
    int tiles;        // T: output tiles
    int units;        // P: resident CTA pairs (or single CTAs)
    int kb;           // KB: k-blocks per tile
    int dp_waves;     // W: whole tiles per unit in the data-parallel part
    int sk_tiles;     // R: tiles whose k-blocks are spread over all units (0 = none)
};

// One unit of work for every role of a unit: tile `tile`, k-blocks
// [kb_begin, kb_end).  For a split tile, `ncontrib` > 1, `contrib` is this
// segment's position among the tile's contributors, `slot` is this unit's
// workspace slot for the partial, `sk_index` the tile's index in the tail.
struct Work {
    int tile;
    int kb_begin, kb_end;
    int contrib, ncontrib;
    int slot;
    int sk_index;
};

// Decide the split.  Stream-K is used only when the last wave is at most
// 7/8 full and every unit gets at least two k-blocks of the tail.
GB300_HD Schedule make_schedule(int tiles, int units, int kb, bool allow_stream_k) {
    Schedule s;
    s.tiles = tiles;
    s.units = units;
    s.kb = kb;
    const int rem = tiles % units;
    const int64_t tail_work = (int64_t)rem * kb;
    const bool split = allow_stream_k && rem != 0 && (int64_t)rem * 8 <= (int64_t)units * 7 &&
                       tail_work >= 2 * (int64_t)units;
    if (split) {
        s.dp_waves = tiles / units;
        s.sk_tiles = rem;
    } else {
        s.dp_waves = (tiles + units - 1) / units;
        s.sk_tiles = 0;
    }
    return s;
}

// First tail k-block (in the concatenated tail k-block space) of unit u.
GB300_HD int64_t sk_begin(const Schedule& s, int u) {
    return (int64_t)u * ((int64_t)s.sk_tiles * s.kb) / s.units;
}

// The unit whose tail range contains tail k-block x (0 <= x < R*KB).
GB300_HD int sk_owner(const Schedule& s, int64_t x) {
    const int64_t total = (int64_t)s.sk_tiles * s.kb;
    // largest u with floor(u*total/P) <= x  <=>  u < (x+1)*P/total
    int64_t u = ((x + 1) * s.units + total - 1) / total - 1;
    if (u >= s.units) u = s.units - 1;
    if (u < 0) u = 0;
    return (int)u;
}

// Local index (0 or 1) of tail tile q within unit u's segments: a tail
// range is shorter than one tile, so it touches at most two tiles.
GB300_HD int sk_local_index(const Schedule& s, int u, int q) {
    const int first_tile = (int)(sk_begin(s, u) / s.kb);
    return q > first_tile ? 1 : 0;
}

GB300_HD int sk_slot(int u, int local) { return 2 * u + local; }

// Number of work items of unit u: its data-parallel tiles plus its tail
// segments.
GB300_HD int work_count(const Schedule& s, int u) {
    int dp = 0;
    if (s.sk_tiles == 0) {
        dp = u < s.tiles ? (s.tiles - 1 - u) / s.units + 1 : 0;
        return dp;
    }
    dp = s.dp_waves;
    const int64_t b0 = sk_begin(s, u), b1 = sk_begin(s, u + 1);
    if (b1 <= b0) return dp;
    const int q0 = (int)(b0 / s.kb), q1 = (int)((b1 - 1) / s.kb);
    return dp + (q1 - q0 + 1);
}

// The j-th work item of unit u (0 <= j < work_count(s, u)).
GB300_HD Work work_item(const Schedule& s, int u, int j) {
    Work w;
    if (j < s.dp_waves || s.sk_tiles == 0) {
        w.tile = u + j * s.units;
        w.kb_begin = 0;
        w.kb_end = s.kb;
        w.contrib = 0;
        w.ncontrib = 1;
        w.slot = -1;
        w.sk_index = -1;
        return w;
    }
    const int seg = j - s.dp_waves;                 // 0 or 1
    const int64_t b0 = sk_begin(s, u), b1 = sk_begin(s, u + 1);
    const int q = (int)(b0 / s.kb) + seg;
    const int64_t tile_lo = (int64_t)q * s.kb, tile_hi = tile_lo + s.kb;
    const int64_t lo = b0 > tile_lo ? b0 : tile_lo;
    const int64_t hi = b1 < tile_hi ? b1 : tile_hi;
    w.tile = s.dp_waves * s.units + q;
    w.kb_begin = (int)(lo - tile_lo);
    w.kb_end = (int)(hi - tile_lo);
    const int first = sk_owner(s, tile_lo);
    const int last = sk_owner(s, tile_hi - 1);
    w.contrib = u - first;
    w.ncontrib = last - first + 1;
    w.slot = sk_slot(u, seg);
    w.sk_index = q;
    return w;
}

// Workspace slot holding contributor c's partial of tail tile q.
GB300_HD int contributor_slot(const Schedule& s, int q, int c) {
    const int first = sk_owner(s, (int64_t)q * s.kb);
    const int u = first + c;
    return sk_slot(u, sk_local_index(s, u, q));
}

}  // namespace gb300
