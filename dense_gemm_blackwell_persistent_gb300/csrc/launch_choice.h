// launch_choice.h -- how the host shapes a launch: CTAs per work unit, tile
// width and the kind of work list.  Plain C++ (no CUDA calls), so that the
// host code and the CPU tests run exactly the same decisions; gemm_api.cu
// feeds them the plan's options and the resident-unit counts it queried on
// the device.
//
// The measurements behind each rule are given with the rule.  The sources
// for the rules themselves: whole waves of persistent units ("Collective
// matrix multiplication": grid = number of SMs), 2-CTA pairs and clusters
// sharing an operand by multicast ("Writing Mosaic GPU kernels with Pallas",
// "Collective MMA", clusters and collective copies), and tiles handed out at
// run time ("Writing Mosaic GPU kernels with Pallas", "Cluster launch
// control").
#pragma once
#include <stdint.h>

#include "gemm.h"

namespace gb300 {

constexpr int kLaunchTileWidths = 5;
constexpr int kLaunchWidths[kLaunchTileWidths] = {256, 224, 192, 160, 128};   // widest first
constexpr int kLaunchRowsPerCta = 128;   // rows of A per CTA (TMEM lanes)
constexpr int kLaunchMnBox = 64;         // elements of M or N per MN-major TMA box

// Raster group height (tile rows walked column by column together) when the
// caller leaves it to the library: all the tile rows when one batch
// element's A is at most kWholeGroupABytes, so that the waves walk the
// columns once with A resident in L2; else 8.  Measured on GB300: 4096³
// (A 32 MB) sustained for 4 s +1.0–1.5% with the whole height (16) over 8
// in three runs, bursts level; 8192³ (A 128 MB) level from 8 to 16.
constexpr int64_t kWholeGroupABytes = int64_t(48) << 20;

inline int launch_group_m(int forced, int64_t tiles_m, int64_t a_bytes) {
    int g = forced > 0 ? forced : (a_bytes <= kWholeGroupABytes ? (int)(tiles_m < (1 << 20) ? tiles_m : 1 << 20) : 8);
    if (g > tiles_m) g = (int)tiles_m;
    return g < 1 ? 1 : g;
}

// CTAs per MMA when the caller leaves it to the library (option 0): single
// CTAs for problems too small to fill half a wave of CTA pairs, as long as
// their 128×128 tiles still fit in one wave of single CTAs; pairs
// otherwise.  A pair's launch and cluster set-up cost more than it saves
// there: measured on GB300 (flushed, single vs pair, µs): 256³ 8.2 vs 10.3,
// 768³ 10.6 vs 12.3, 1024³ 12.3 vs 12.7, 256×4096×1024 12.1 vs 14.0,
// 128×4096×4096 23.5 vs 24.7, 2048×256×4096 22.2 vs 23.9; from a full wave
// of pair tiles on the pairs win clearly (1024×4096×4096: 76 pair tiles).
// `pair_units` and `single_units`: resident units of each size.
inline int launch_auto_pair(int64_t M, int64_t N, int64_t batch, int64_t pair_units, int64_t single_units) {
    const int64_t pair_tiles = batch * ((M + 2 * kLaunchRowsPerCta - 1) / (2 * kLaunchRowsPerCta)) * ((N + 255) / 256);
    const int64_t single_tiles = batch * ((M + kLaunchRowsPerCta - 1) / kLaunchRowsPerCta) * ((N + 127) / 128);
    return (2 * pair_tiles <= pair_units && single_tiles <= single_units) ? 1 : 2;
}

// CTAs per work unit: 1 (pair = 1), 2 (a CTA pair) or 4 (two pairs sharing B
// through TMA multicast).  Multicast is used only while the process sees
// a single GPU, so no code of a process that may drive several GPUs
// multicasts.  Automatic choice (multicast = -1): when the rows of K are not
// a multiple of 128 bytes every 128-byte box row straddles an extra 32-byte
// sector, the load path becomes the bound, and halving the B reads wins
// (measured +29% at 4000×3000×5000); with aligned rows the pairs' use of all
// SMs wins (4-CTA clusters fit on 144 of the 152 SMs).  An explicit request
// for multicast that cannot be honoured is refused by the caller, not here.
inline int launch_unit_ctas(int pair, int multicast, int visible_devices, int64_t K, int in_elem_bytes,
                            int layout) {
    if (pair != 2) return 1;
    const bool mc = visible_devices == 1 &&
                    (multicast == 1 || (multicast < 0 && layout == 0 && (K * in_elem_bytes) % 128 != 0));
    return mc ? 4 : 2;
}

// With an MN-major B, whether every CTA's share of the tile's B rows (as
// held for the MMA and as loaded) is whole 64-element TMA boxes.  If not, a
// 1- or 2-CTA unit uses the padded kernel form (shares rounded up to whole
// boxes); a 4-CTA unit cannot.
inline bool launch_b_boxes_exact(int bn, int cluster) {
    const int pair = cluster >= 2 ? 2 : 1;
    return (bn / pair) % kLaunchMnBox == 0 && (bn / cluster) % kLaunchMnBox == 0;
}
inline bool launch_width_fits_layout(int bn, int cluster, int layout) {
    return !(layout & GEMM_B_MN_MAJOR) || cluster <= 2 || launch_b_boxes_exact(bn, cluster);
}

// Tile width: the candidate that minimises (waves of resident units) × (SM
// cycles per k-block of that width), preferring the wider tile when two are
// within 1%.  Cycles per k-block measured on GB300 at 8192³ (GEMM_TRACE
// cycle stamps, steady state): CTA pairs (also the 4-CTA multicast unit)
// 520 / 453 / 432 / 429 / 485 for widths 256 / 224 / 192 / 160 / 128 —
// only 256 and 224 run at (within ~3% of) the MMA's own rate, narrower tiles
// wait on a ~460-cycle floor — and single CTAs 673 / 652 / 528 / 506 / 482.
// So 224 is picked at 4096³ (304 tiles = 4 whole waves on 76 pairs) and at
// 1024×4096×4096, 256 at 8192³.  `forced` > 0 is a width the caller asked
// for.  `units`: resident units of this size.  Returns 0 when no width fits
// (a forced width the layout cannot use).
inline int launch_tile_n(int forced, int64_t M, int64_t N, int cluster, int layout, int64_t batch, int64_t units) {
    if (forced > 0) return launch_width_fits_layout(forced, cluster, layout) ? forced : 0;
    static constexpr int64_t kCyclesPair[kLaunchTileWidths] = {520, 453, 432, 429, 485};
    static constexpr int64_t kCyclesSingle[kLaunchTileWidths] = {673, 652, 528, 506, 482};
    const int64_t* cycles = cluster >= 2 ? kCyclesPair : kCyclesSingle;
    if (units < 1) units = 1;
    const int64_t tiles_m = batch * ((M + kLaunchRowsPerCta * cluster - 1) / (kLaunchRowsPerCta * cluster));
    int best = 0;
    int64_t best_cost = INT64_MAX;
    for (int i = 0; i < kLaunchTileWidths; ++i) {   // widest first
        const int bn = kLaunchWidths[i];
        if (!launch_width_fits_layout(bn, cluster, layout)) continue;
        const int64_t tiles = tiles_m * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + units - 1) / units) * cycles[i];
        if (cost * 100 < best_cost * 99) {   // a narrower tile must be > 1% cheaper
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

// Dynamic work list of a launch (cluster launch control): `units`
// persistent clusters with `waves` whole tiles each, then one single-tile
// cluster per remaining tile.  Mode 1 hands out only the partial last
// wave (the whole waves keep the static placement of tiles on SMs); mode 2
// every tile.  Returns false for the static schedule: mode 0, or mode 1
// when the tiles fill whole waves or fit in one.
//
// Automatic choice (mode -1): mode 1 from kDynamicMinWaves whole waves on.
// On GB300 some SMs run a 256-wide tile up to 4% slower than others (the
// same SMs in every launch), so over many waves the static units drift
// apart and the slowest one sets the end; handing out the partial last wave
// lets the fast units take it.  Measured against the static schedule:
// 8192³ 588 → 570 µs, 7168³ 389 → 384, 8192×8192×4096 291 → 286,
// 8192×4096×8192 294 → 289, 5120³ 158 → 155 (6 to 13 waves); level at 3 to
// 5 waves; slower by 1.5-4 µs at 1 or 2 waves (3072³, 3328×4096×4096,
// 4000×3000×5000), where the drift is small and the handed-out tiles lose
// the static placement (~5% slower per tile when every tile is handed out).
// Mode 2 measured slower than mode 1 almost everywhere.  Plans with a CTA
// cap or stream-K keep the static schedule unless mode 1 or 2 is set
// explicitly.
constexpr int64_t kDynamicMinWaves = 6;

inline bool launch_dynamic_lists(int mode, bool capped, bool stream_k, int64_t tiles, int64_t resident, int* units,
                                 int* waves) {
    if (mode < 0) mode = (!capped && !stream_k && tiles / resident >= kDynamicMinWaves) ? 1 : 0;
    if (mode == 2) {
        *units = (int)tiles;
        *waves = 1;
        return true;
    }
    if (mode == 1 && tiles > resident && tiles % resident != 0) {
        *units = (int)resident;
        *waves = (int)(tiles / resident);
        return true;
    }
    return false;
}

// Split-K for problems with few tiles and a long K: the product becomes S
// products over K slices (k-blocks [s·KB/S, (s+1)·KB/S)), one fp32 partial
// each, then a reduction sums the S partials in order and writes C.  S is a
// power of two up to kSplitMax that divides the k-blocks, keeps at least
// kSplitMinKBlocks per slice, keeps every slice's tiles in one wave
// (tiles·S <= resident units) and fits the workspace; it is the S that
// minimises k-blocks per slice + kSplitCostKBlocks (the reduction and its
// launch, ~3 µs ≈ 12 k-blocks of a 256-wide tile), and must beat the
// unsplit K loop by a quarter.  `forced` > 1 asks for that S (still subject
// to the divisibility, wave and workspace limits); 0 turns it off.
// Returns 1 for no split.
constexpr int kSplitMax = 32;
constexpr int64_t kSplitMinKBlocks = 4;
constexpr int64_t kSplitCostKBlocks = 12;

inline int launch_split_k(int forced, int64_t tiles, int64_t units, int64_t k_blocks, int64_t slice_floats,
                          int64_t workspace_floats) {
    if (forced == 0 || tiles <= 0 || k_blocks <= 0) return 1;
    int best = 1;
    int64_t best_cost = k_blocks;
    for (int s = 2; s <= kSplitMax; s *= 2) {
        if (k_blocks % s != 0 || k_blocks / s < kSplitMinKBlocks) continue;
        if (tiles * s > units || slice_floats * s > workspace_floats) continue;
        if (forced > 1) {
            if (s == forced) return s;
            continue;
        }
        const int64_t cost = k_blocks / s + kSplitCostKBlocks;
        if (cost * 4 <= k_blocks * 3 && cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

}  // namespace gb300
