// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// C[M×N] = A[M×K] · B[N×K]ᵀ, bf16/f16 (or 8-bit float) in, fp32 accumulate
// in TMEM, C out as fp32/bf16/f16.  One CTA (or one CTA pair) stays resident
// per SM (pair of SMs) and walks a list of output tiles: a static list, or
// one that grows at run time through cluster launch control (the tiles of
// clusters that have not started).
//
// Roles inside a CTA (192 threads):
//   warp 0      TMA producer: fills a kStages-deep shared-memory ring with
//               64-wide K slices of A and B (128-byte swizzle, zero fill
//               outside the tensor).  Ring slots are guarded by full/empty
//               mbarriers.
//   warp 1      allocates TMEM; in the leader CTA one thread issues
//               tcgen05.mma into one of two TMEM accumulators (columns
//               0.. and 256.., kBN wide each) and commits completions to
//               the mbarriers.
//   warps 2..5  epilogue: TMEM -> registers -> swizzled shared staging ->
//               TMA store in 32-column boxes, while the MMA thread already
//               fills the other accumulator with the next tile (the stores
//               paced over that tile's K loop).
//
// The tile width kBN (256, 224, 192, 160 or 128) is chosen per problem on
// the host so that the tile count fills whole waves of resident CTA pairs.
//
// With a CTA pair (kCluster >= 2) two CTAs form one 256×kBN tile: each holds
// its own 128 rows of A and kBN/2 rows (half) of B, the leader issues
// tcgen05.mma.cta_group::2 with M = 256, and each CTA's TMEM receives its own
// 128 rows of the result.  This is the collective MMA of "Writing Mosaic GPU
// kernels with Pallas", "Collective MMA" (A and D per CTA, B split between
// the pair) with the B halves loaded as partitioned, leader-tracked copies.
// With kCluster == 4 two such pairs stacked along M share their B tile: the
// same-rank CTAs of the two pairs each fetch half of their common B rows and
// multicast it to both ("Writing Mosaic GPU kernels with Pallas", clusters
// and collective copies: every CTA on the cluster axis issues the identical
// copy and receives the data), which cuts L2-to-SM traffic by a quarter.
//
// Design sources on the pages (prior art, restated for this hardware):
//   * tiles of A (BM×BK) and B (BN×BK) staged in shared memory, loaded by
//     TMA under an mbarrier with expected bytes, consumed by tcgen05.mma in
//     K = 16 steps, accumulators in TMEM: "Optimizing Blackwell Matrix
//     Multiplication in Mojo (Part 2)", "Kernel 2: TMA and Tensor Core".
//   * 128-byte swizzle, Swizzle<3,4,3>, one box of 64 K elements per row:
//     same page, "Kernel 3: Swizzling" and "Swizzling math".
//   * epilogue through swizzled shared memory and TMA stores with commit
//     groups: same page, "Kernel 4".
//   * first MMA of a tile overwrites (accumulate flag 0): same page, Kernel 2
//     code (c_scale 0 on the first MMA).
//   * multi-slot ring with full/empty barriers and slot refill once the
//     consumer released it: "Writing Mosaic GPU kernels with Pallas",
//     "Barrier" and the pipelined Hopper matmul.
//   * grouped rasterisation for L2 reuse: same reference, "Utilizing L2
//     cache" (grid reordered as (m // mt, n, mt)).
//   * persistent grid of one CTA per SM: "Collective matrix multiplication"
//     (grid = number of SMs).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "schedule.h"

namespace gb300 {

// Optional timeline tracing (build with -DGEMM_TRACE): per-CTA
// %globaltimer stamps, wait totals and SM cycle counts in a device buffer of
// kTraceSlots 64-bit words per CTA.  Without GEMM_TRACE the macros compile
// to nothing.
constexpr int kTraceSlots = 136;
enum TraceSlot {
    kTrEntry = 0,         // %globaltimer at entry (thread 0; written at teardown)
    kTrClcWaitProducerNs = 1, kTrClcWaitEpiNs = 2,   // dynamic work list: time waiting for responses
    kTrFirstFull = 3,     // MMA warp: first full ring slot
    kTrTeardown = 4, kTrExit = 5,
    kTrFullWaitNs = 6, kTrEmptyWaitNs = 7, kTrAccEmptyWaitNs = 8,   // per-role wait totals
    kTrWorkItems = 9,     // MMA warp: all work items issued
    kTrClcWaitMmaNs = 10,
    kTrEpiDone = 11,      // epilogue warp 2: the CTA's stores have read shared memory
    kTrClusterArrived = 12, kTrClusterDone = 13, kTrDealloc = 14,
    kTrClkFirstFull = 15, // SM cycles (clock64) at first_full ...
    kTrMmaEnd = 16,       // + item (8 items): last MMA of the item issued
    kTrEpiStart = 24,     // + item
    kTrEpiEnd = 32,       // + item
    kTrPartialDone = 40,  // + item: stream-K partial published
    kTrReduceDone = 48,   // + item: stream-K tile finished (the piece holding its first k-blocks)
    kTrClkMmaEnd = 56,    // ... and at mma_end + item: cycles per k-block
    kTrClkPro = 64,       // + 0..8: SM cycles at the prologue steps (see timeline.PROLOGUE)
    kTrDynTile = 72,      // + 1 + r (r < 7): the list (cluster) that response r handed to this unit
    kTrSmid = 80,         // %smid of the CTA, + 1
    kTrProducerDone = 84, // producer warp: every slot's last use released
    kTrMmaDone = 85,      // MMA warp: every accumulator release awaited
    kTrEpiLoopDone = 86,  // epilogue warp 2: left its loop
    kTrLastEpi = 88,      // + 12 * epilogue warp + step: SM cycles in the unit's last tile (see LastEpiStep)
};
// Steps of the last tile's epilogue, stamped by each epilogue warp's lane 0.
enum LastEpiStep { kLeStart = 0, kLeFirstData = 1, kLeChunk = 2 /* + chunk c: its store issued */,
                   kLeCommitted = 10, kLeStoresRead = 11 };
#ifdef GEMM_TRACE
#define GEMM_TR_ON() (p.trace && blockIdx.x < (unsigned)p.trace_ctas)
#define GEMM_TR(slot) do { if (GEMM_TR_ON()) p.trace[blockIdx.x * kTraceSlots + (slot)] = global_timer_ns(); } while (0)
#define GEMM_TR_ITEM(base, item) do { if ((item) < 8) GEMM_TR((base) + (item)); } while (0)
#define GEMM_TR_SET(slot, v) do { if (GEMM_TR_ON()) p.trace[blockIdx.x * kTraceSlots + (slot)] = (v); } while (0)
#define GEMM_TR_NOW() global_timer_ns()
// Prologue cycle stamps stay in registers (constant indices) until the
// teardown writes them, so that taking them costs a few cycles and no
// memory traffic; the %globaltimer points above are too heavy for steps of
// a few hundred cycles.
#define GEMM_TR_CLK(step) (tr_clk[(step)] = (unsigned long long)clock64())
#define GEMM_TR_CLK_FLUSH()                                                            \
    do {                                                                               \
        if (GEMM_TR_ON())                                                              \
            for (int s_ = 0; s_ < 9; ++s_)                                             \
                if (tr_clk[s_]) p.trace[blockIdx.x * kTraceSlots + kTrClkPro + s_] = tr_clk[s_]; \
        if (GEMM_TR_ON() && tr_entry_ns) p.trace[blockIdx.x * kTraceSlots + kTrEntry] = tr_entry_ns; \
    } while (0)
#else
#define GEMM_TR_CLK_FLUSH() do { } while (0)
#define GEMM_TR_CLK(step) do { } while (0)
#define GEMM_TR(slot) do { } while (0)
#define GEMM_TR_ITEM(base, item) do { } while (0)
#define GEMM_TR_SET(slot, v) do { } while (0)
#define GEMM_TR_NOW() 0ull
#endif

constexpr int kNumThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kBlockKBytes = 128;        // K bytes per k-block: one 128-byte swizzle row
constexpr int kMmaKBytes = 32;           // K bytes of one MMA (16 bf16/f16 or 32 fp8 elements)
// MN-major operands (A stored K×M, B stored K×N) arrive in boxes of 64
// elements along M or N (one 128-byte row) × 64 K rows: 8 KB per box.
constexpr int kMnBoxElems = 64;
constexpr int kMnBoxBytes = kMnBoxElems * 128;
constexpr int kRowsPerCta = 128;         // TMEM lanes = rows of A per CTA
constexpr int kAccStride = 256;          // TMEM columns between the two accumulators
constexpr int kTmemCols = 2 * kAccStride;
constexpr int kStageBytesA = kRowsPerCta * kBlockKBytes;
constexpr int kChunkCols = 32;           // accumulator columns per epilogue store box
// Dynamic scheduling: responses of cluster launch control in flight or not
// yet read by every role of the cluster (a ring, so that the issuer never
// overwrites a response a lagging epilogue warp has still to read).
constexpr int kClcSlots = 4;
constexpr uint32_t kClcResponseBytes = 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // default bound on any single wait
constexpr int kRoleStallTest = 8;  // status[1] of the timeout a test provokes on purpose

constexpr int kOutBF16 = 0, kOutF16 = 1, kOutF32 = 2;
constexpr int kIn16 = 0, kInF8 = 1;      // operand width: bf16/f16 (kind::f16) or E4M3/E5M2 (kind::f8f6f4)
constexpr int kErrCuda = -4;      // device side: the launch's shared memory is not 1 KB aligned
constexpr int kErrTimeout = -7;
constexpr int kRoleSmemBase = 9;  // status[1] for kErrCuda; status[3] = the base address
constexpr int kRoleLayout = 10;   // status[1] for kErrCuda: an MN-major operand this tile cannot hold
constexpr int kRoleClc = 11;      // status[1] of a timeout on the dynamic work list's ring (detail: item)
constexpr int kErrInternal = -9;  // GEMM_DEBUG builds: a consistency check failed
constexpr int kRoleDebug = 12;    // status[1] for kErrInternal; status[3] = which check (DebugCheck)

// Consistency checks of GEMM_DEBUG builds (status[3] of a kErrInternal record).
enum DebugCheck {
    kChkWorkItem = 1,     // a work item's tile or k-block range outside the problem
    kChkTileCoords = 2,   // tile coordinates (batch element, tile row, tile column) outside the tile grid
    kChkOperandRows = 3,  // first A or B row of a load beyond the tile grid's rows
    kChkRing = 4,         // ring stage or phase out of range
    kChkKBlock = 5,       // k-block outside [0, k_blocks)
    kChkAccumulator = 6,  // accumulator buffer or phase out of range
    kChkStoreBox = 7,     // epilogue store box outside the tile grid
};

struct Params {
    // What decoding a work item reads comes first, so that it shares one
    // constant-cache line.
    Schedule sched;    // whole-tile waves + stream-K part
    // Divisors of the tile decode as multiply-shift dividers: tiles per
    // batch element, tiles per raster group (group_m * tiles_n), the group
    // height, and the height of the last group (tiles_m mod group_m, or
    // group_m when that is 0).
    FastDiv fd_batch, fd_group, fd_gm, fd_gm_last;
    // Dynamic work list (cluster launch control): 1 = on.  Cluster c < dyn_units
    // owns tiles c, c + dyn_units, ... (dyn_waves of them); cluster c >=
    // dyn_units owns tile dyn_units * dyn_waves + (c - dyn_units).
    int dynamic, dyn_units, dyn_waves;
    int tiles_m, tiles_n, group_m, k_blocks;
    int tiles_per_batch;        // tiles_m * tiles_n; tile t is in batch element t / tiles_per_batch
    int a_batched, b_batched;   // 0: every batch element reads the same A / B (batch coordinate 0)
    int M, N, K, num_tiles;
    uint32_t idesc;
    int* status;       // [0] first error code, [1] role, [2] block, [3] detail
    float* partials;   // stream-K: one partial-tile slot per unit, or null
    int* flags;        // stream-K: "partial published" per (split tile, CTA, epilogue warp)
    unsigned long long wait_limit_ns;   // bound on any single wait
    int stall_test;    // 1: the MMA warp waits on a barrier nothing completes (tests of the timeout path)
    int a_mn, b_mn;    // 1: A stored K×M / B stored K×N (MN-major in shared memory)
    unsigned long long* trace;  // GEMM_TRACE builds only: kTraceSlots words per CTA
    int trace_ctas;             // CTAs the trace buffer holds (CTAs with a higher index record nothing)
    // Per-launch clock record, or null: CTA 0 writes the SM cycles and the
    // %globaltimer nanoseconds between its entry and its exit (their ratio
    // is the SM clock the launch ran at).
    unsigned long long* clock_rec;
};

// fp32 partial of one epilogue warp: 32 rows × 256 columns, stored as
// float4 groups [column/4][row] so that a warp's accesses are contiguous.
constexpr int kPartialFloats = 32 * 256;
constexpr int kFixupBytes = kPartialFloats * 4;   // shared memory per epilogue warp for a fix-up

// kCluster: CTAs per work unit -- 1 (one CTA, tcgen05 cta_group::1), 2 (a
// CTA pair issuing cta_group::2 MMAs) or 4 (two pairs stacked along M that
// share the B tile: each CTA loads a quarter of it and multicasts it to
// the same-rank CTA of the other pair).  kBN: tile width (accumulator
// columns, a multiple of 32 up to 256).  kOut: C element type.  kIn:
// operand width; a k-block is one 128-byte swizzle row of K either way
// (64 bf16/f16 or 128 fp8 elements), so shared-memory layout, descriptors
// and the ring are the same for both.  kBMnPad: B is MN-major and a CTA's
// share of it is rounded up to whole 64-element boxes in shared memory (the
// extra rows are loaded but never read by the MMA), for tile widths whose
// share is not a multiple of 64 (e.g. 112 rows of a 256×224 pair tile).
template <int kCluster, int kBN, int kOut, int kIn, bool kBMnPad = false>
struct Cfg {
    static_assert(kCluster == 1 || kCluster == 2 || kCluster == 4, "1, 2 or 4 CTAs per unit");
    static_assert(kBN % 32 == 0 && kBN >= 64 && kBN <= 256, "tile width");
    static constexpr int kPair = kCluster >= 2 ? 2 : 1;           // CTAs per MMA
    static constexpr int kPairs = kCluster / kPair;                // MMA groups per unit
    static constexpr int kTileM = kRowsPerCta * kCluster;         // rows per unit tile
    static constexpr int kRowsB = kBN / kPair;                    // B rows held per CTA
    static constexpr int kRowsBLoad = kBN / kCluster;             // B rows each CTA loads
    static_assert(kRowsBLoad % 8 == 0, "B boxes must fill 1 KB swizzle atoms");
    static constexpr int kBlockKElems = kIn == kInF8 ? kBlockKBytes : kBlockKBytes / 2;   // TMA K coordinate step
    static_assert(!kBMnPad || (kCluster <= 2 && kIn == kIn16), "padded MN-major B: 1- or 2-CTA units, 16-bit");
    static constexpr int kBoxesB = (kRowsBLoad + kMnBoxElems - 1) / kMnBoxElems;   // MN-major B boxes per load
    static constexpr int kStageBytesB = kBMnPad ? kBoxesB * kMnBoxBytes : kRowsB * kBlockKBytes;
    static constexpr int kLoadBytesB = kBMnPad ? kBoxesB * kMnBoxBytes : kRowsBLoad * kBlockKBytes;
    static constexpr int kStageBytes = kStageBytesA + kStageBytesB;
    static constexpr int kOutBytes = kOut == kOutF32 ? 4 : 2;
    static constexpr int kRowBytes = kChunkCols * kOutBytes;    // 128 (fp32) or 64 (16-bit)
    static constexpr int kSlotBytes = 32 * kRowBytes;           // one 32-row store box
    static constexpr int kStagingBytes = kEpiWarps * 2 * kSlotBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kMiscBytes = 16 + kClcSlots * (int)kClcResponseBytes;   // TMEM address, abort flag; responses
    static constexpr int kFixed = kStagingBytes + kBarBytes + kMiscBytes;
    static constexpr int kStagesFit = (232448 - kFixed) / kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static_assert(kStages >= 3, "ring too shallow");
    static constexpr int kOffB = kStages * kStageBytesA;
    static constexpr int kOffStaging = kOffB + kStages * kStageBytesB;
    static constexpr int kOffBars = kOffStaging + kStagingBytes;
    static constexpr int kOffMisc = kOffBars + kBarBytes;
    static constexpr int kOffClc = kOffMisc + 16;   // the responses (kOffMisc is 1 KB + kBarBytes aligned)
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert((2 * kStages + 4 + kEpiWarps + 2 * kClcSlots) * 8 <= kBarBytes, "barrier area");
    static_assert(kOffClc % 16 == 0, "cluster launch control responses are 16-byte aligned");
    static constexpr uint32_t kPartialBytes = kBN * 32 * 4;   // one epilogue warp's fp32 partial
    static_assert(kEpiWarps * kFixupBytes <= kOffStaging, "fix-up buffers must fit in the operand ring");
    static_assert(kEpiWarps * (kBN / kChunkCols) * kSlotBytes <= kOffStaging,
                  "the last tile's store boxes must fit in the operand ring");
    static_assert(kStageBytesA % 1024 == 0 && kStageBytesB % 1024 == 0, "1 KB aligned tiles");
    static constexpr uint32_t kTxBytes = kStageBytes * kPair;   // bytes landing in a pair, tracked by its leader
};

// tcgen05 shared-memory matrix descriptor for an MN-major tile written by TMA
// with 128-byte swizzle in kMnBoxBytes boxes: each box holds 64 elements of
// M (or N) per 128-byte row and 64 rows of K.  Swizzle atoms are 64
// elements × 8 K rows (1 KB); the leading byte offset steps to the next 64
// elements along M/N (the next box), the stride byte offset to the next 8
// rows of K.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address / 16
    d |= (uint64_t)(kMnBoxBytes >> 4) << 16;         // leading byte offset: next 64 elements of M/N
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: next 8 rows of K
    d |= (uint64_t)1 << 46;                          // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle
    return d;
}

// tcgen05 shared-memory matrix descriptor for a K-major tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address / 16
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused when swizzled)
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: 8 rows × 128 B
    d |= (uint64_t)1 << 46;                     // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                     // layout: 128-byte swizzle
    return d;
}

// Output tile of linear tile index t: batch element bt = t / tiles_per_batch;
// within it, groups of `group_m` tile rows are walked column by column, so
// the tiles in flight at once share rows of A and columns of Bᵀ in L2.
// Every other group walks its columns right to left: the B panels a group
// ends on are the first the next one needs, while they are still in L2
// (8192³: DRAM reads 1108 → 1020 MB per launch, 567 → 561 µs).
__device__ __forceinline__ void tile_coords(const Params& p, int t, int& bt, int& mt, int& nt) {
    bt = (int)fast_div(p.fd_batch, (uint32_t)t);
    t -= bt * p.tiles_per_batch;
    const int g = (int)fast_div(p.fd_group, (uint32_t)t);
    const int first_m = g * p.group_m;
    const int r = t - g * (int)p.fd_group.d;
    // the group's height: group_m, or fewer in the last group
    const FastDiv& gs = first_m + p.group_m > p.tiles_m ? p.fd_gm_last : p.fd_gm;
    const int q = (int)fast_div(gs, (uint32_t)r);
    mt = first_m + (r - q * (int)gs.d);
    nt = (g & 1) ? p.tiles_n - 1 - q : q;
}

__device__ __forceinline__ void record_error(const Params& p, int role, int detail, int code = kErrTimeout) {
    if (atomicCAS(p.status, 0, code) == 0) {
        p.status[1] = role;
        p.status[2] = (int)blockIdx.x;
        p.status[3] = detail;
    }
}

// GEMM_DEBUG builds: `cond` must hold; if not, record kErrInternal (role
// kRoleDebug, detail `what`) and raise the CTA's abort flag, so that every
// role leaves its loop without the access and the CTA tears down as after a
// timeout.  Other builds: no code, always true.
#ifdef GEMM_DEBUG
__device__ __forceinline__ bool debug_check(bool cond, volatile uint32_t* abort_flag, const Params& p, int what) {
    if (!cond) {
        record_error(p, kRoleDebug, what, kErrInternal);
        *abort_flag = 1;
    }
    return cond;
}
// A check taken by a whole warp: true only if it holds for every lane.
#define GEMM_WARP_CHECK(cond, what) __all_sync(0xffffffffu, debug_check((cond), abort_flag, p, (what)))
#else
#define GEMM_WARP_CHECK(cond, what) true
#endif

// Suspend-time hints of the waits (ns; 0 = the hardware's own limit): the
// epilogue warps wait for an accumulator for a whole tile's K loop, the
// producer and MMA warps for ring slots a few hundred cycles at a time.
#ifndef GEMM_EPI_WAIT_HINT_NS
#define GEMM_EPI_WAIT_HINT_NS 20000
#endif
#ifndef GEMM_RING_WAIT_HINT_NS
#define GEMM_RING_WAIT_HINT_NS 0
#endif
constexpr uint32_t kEpiWaitHintNs = GEMM_EPI_WAIT_HINT_NS;
constexpr uint32_t kRingWaitHintNs = GEMM_RING_WAIT_HINT_NS;

template <bool kClusterScope, uint32_t kHintNs>
__device__ __forceinline__ bool try_wait_once(uint32_t bar, uint32_t parity) {
    if constexpr (kHintNs == 0)
        return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    else
        return kClusterScope ? mbar_try_wait_cluster_hint(bar, parity, kHintNs)
                             : mbar_try_wait_hint(bar, parity, kHintNs);
}

// Wait for the phase of parity `parity` of `bar`, for at most p.wait_limit_ns.
// Returns false (and raises the CTA's abort flag) if the bound expires or
// another role of this CTA has already aborted.
template <bool kClusterScope, uint32_t kHintNs = 0>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             const Params& p, int role, int detail) {
    if (try_wait_once<kClusterScope, kHintNs>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (try_wait_once<kClusterScope, kHintNs>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > p.wait_limit_ns) {
            record_error(p, role, detail);
            *abort_flag = 1;
            return false;
        }
    }
}

// Wait until *flag == 1 (another CTA's release), for at most p.wait_limit_ns:
// lane 0 polls, the warp gets the outcome.  On expiry records a timeout and
// raises the CTA's abort flag; gives up early if another role aborted.
__device__ __forceinline__ bool wait_flag_bounded(const int* flag, volatile uint32_t* abort_flag, const Params& p,
                                                  int role, int detail) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0 && ld_acquire_gpu(flag) != 1) {
        const uint64_t t0 = global_timer_ns();
        while (true) {
            __nanosleep(100);
            if (ld_acquire_gpu(flag) == 1) break;
            if (*abort_flag) {
                ok = 0;
                break;
            }
            if (global_timer_ns() - t0 > p.wait_limit_ns) {
                record_error(p, role, detail);
                *abort_flag = 1;
                ok = 0;
                break;
            }
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int out) {
    if (out == kOutBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

template <int kCluster, int kBN, int kOut, int kIn, bool kBMnPad>
__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_tn_persistent(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const Params p) {
    using C = Cfg<kCluster, kBN, kOut, kIn, kBMnPad>;
    constexpr int kPair = C::kPair;
    constexpr int kStages = C::kStages;
    constexpr int kChunks = kBN / kChunkCols;

    // The 128-byte-swizzled operand tiles need 1 KB alignment.  The dynamic
    // shared window is declared 1 KB aligned rather than padded by 1 KB:
    // that padding is what a 7th ring slot of a 256x224 tile needs.  Every
    // CTA of the launch has the same layout, so if the window were ever
    // misaligned all of them would record the error and return here,
    // before touching any barrier, TMEM or cluster peer.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
#ifdef GEMM_TRACE
    unsigned long long tr_clk[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    unsigned long long tr_entry_ns = 0;
    if (threadIdx.x == 0) {
        GEMM_TR_CLK(0);
        tr_entry_ns = global_timer_ns();
        GEMM_TR_SET(kTrSmid, (unsigned long long)sm_id() + 1);
    }
#endif
    // Clock record: CTA 0's first thread stamps entry here and exit at the end.
    const bool clock_owner = p.clock_rec != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
    unsigned long long clk_entry = 0, ns_entry = 0;
    if (clock_owner) {
        clk_entry = (unsigned long long)clock64();
        ns_entry = global_timer_ns();
    }
    const uint32_t base = smem_addr(smem_raw);
    uint8_t* smem = smem_raw;
    if (base & 1023u) {
        if (threadIdx.x == 0) record_error(p, kRoleSmemBase, (int)base, kErrCuda);
        return;
    }
    // An MN-major operand needs whole 64-element boxes per CTA and 16-bit
    // elements (a box holds the 64 K rows of a 16-bit k-block); the host only
    // launches such tiles, and a launch that did not would otherwise wait for
    // bytes that never come.  Uniform over the launch, before any barrier.
    if (((p.a_mn || p.b_mn) && kIn == kInF8) || (p.a_mn && kRowsPerCta % kMnBoxElems != 0) ||
        (kBMnPad && !p.b_mn) ||
        (p.b_mn && !kBMnPad && (C::kRowsB % kMnBoxElems != 0 || C::kRowsBLoad % kMnBoxElems != 0))) {
        if (threadIdx.x == 0) record_error(p, kRoleLayout, kBN, kErrCuda);
        return;
    }

    const uint32_t bars = base + C::kOffBars;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * kStages + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * kStages + 2 + b); };
    auto fix_bar = [&](int e) { return bars + 8u * (2 * kStages + 4 + e); };   // per epilogue warp
    auto clc_full = [&](int s) { return bars + 8u * (2 * kStages + 4 + kEpiWarps + s); };
    auto clc_empty = [&](int s) { return bars + 8u * (2 * kStages + 4 + kEpiWarps + kClcSlots + s); };
    auto clc_resp = [&](int s) { return base + (uint32_t)C::kOffClc + kClcResponseBytes * (uint32_t)s; };
    // Readers of each response: every CTA's producer and epilogue warps and
    // each pair's MMA warp.
    constexpr int kClcReaders = kCluster * (1 + kEpiWarps) + C::kPairs;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = kCluster > 1 ? cluster_cta_rank() : 0u;   // rank in the unit's cluster
    const uint32_t rank = crank & (uint32_t)(kPair - 1);             // rank in the MMA pair (0 = leader)
    const uint32_t pidx = crank / kPair;                             // which pair of the unit
    const uint32_t leader = crank & ~(uint32_t)(kPair - 1);          // cluster rank of this pair's leader
    const int pair_id = kCluster > 1 ? (int)cluster_id_x() : (int)blockIdx.x;   // work unit

    // Operand rows of this CTA for output tile `tile` (A: its 128 rows; B: the
    // rows of the pair's B tile that this CTA loads).
    auto operand_rows = [&](int tile, int& a_row, int& b_row, int& bt) {
        int mt, nt;
        tile_coords(p, tile, bt, mt, nt);
        a_row = mt * C::kTileM + (int)crank * kRowsPerCta;
        b_row = nt * kBN + (int)rank * C::kRowsB + (int)pidx * C::kRowsBLoad;
    };

    // ---- the work list
    // Static: the schedule's items for this unit.  Dynamic ("Writing Mosaic
    // GPU kernels with Pallas", "Cluster launch control"): the grid has one
    // cluster per list of tiles -- the persistent units' lists of whole waves
    // and one single-tile list per tile of the partial last wave (or one per
    // tile of the problem).  A cluster does its own list, then the lists of
    // clusters that have not started, which the hardware cancels on its
    // request, until a request finds none left; so units that run fast
    // take the tail.  The producer of the cluster's first CTA sends request r
    // when it starts the last item of a list; the response lands in ring
    // slot r % kClcSlots of every CTA of the cluster, and each reading warp
    // releases the slot on the first CTA's empty barrier.  Nothing is
    // requested after a request that failed.
    const bool dyn = p.dynamic != 0;
    const int nwork = dyn ? 0 : work_count(p.sched, pair_id);
    auto list_len = [&](int c) { return dyn_list_len(c, p.dyn_units, p.dyn_waves); };
    auto list_tile = [&](int c, int k) { return dyn_list_tile(c, k, p.dyn_units, p.dyn_waves); };
    // Position in this unit's work: whose list, the next item in it, its
    // length, the next response to read.
    struct Cursor {
        int owner, pos, len, resp;
    };
    const Cursor cursor0 = {pair_id, 0, dyn ? list_len(pair_id) : nwork, 0};
    uint64_t clc_wait_ns = 0;   // trace builds only
    // The next item of cursor `cur` into w: 1 = there is one, 0 = the work
    // has ended, -1 = a wait gave up.  Called by whole warps.
    auto get_work = [&](Cursor& cur, Work& w) -> int {
        if (!dyn) {
            if (cur.pos >= cur.len) return 0;
            w = work_item(p.sched, pair_id, cur.pos++);
            return 1;
        }
        while (cur.pos >= cur.len) {
            const int r = cur.resp++, s = r % kClcSlots;
            const uint64_t tw = GEMM_TR_NOW();
            if (!__all_sync(0xffffffffu, wait_bounded<(kCluster > 1)>(clc_full(s), (uint32_t)(r / kClcSlots) & 1u,
                                                                       abort_flag, p, kRoleClc, r)))
                return -1;
            clc_wait_ns += GEMM_TR_NOW() - tw;
            const int x = clc_response(clc_resp(s));
            __syncwarp();
            if (lane == 0) {
                if constexpr (kCluster > 1) mbar_arrive_cluster(map_shared_rank(clc_empty(s), 0));
                else mbar_arrive_local(clc_empty(s));
            }
            if (x < 0) return 0;
            cur.owner = x / kCluster;
            cur.pos = 0;
            cur.len = list_len(cur.owner);
            if (warp == 0 && lane == 0 && r < 7) GEMM_TR_SET(kTrDynTile + 1 + r, (unsigned long long)cur.owner + 1);
        }
        w = whole_tile(list_tile(cur.owner, cur.pos++), p.k_blocks);
        return 1;
    };
#ifdef GEMM_DEBUG
    auto item_ok = [&](const Work& w) {
        return w.tile >= 0 && w.tile < p.num_tiles && w.kb_begin >= 0 && w.kb_begin < w.kb_end &&
               w.kb_end <= p.k_blocks;
    };
    auto rows_ok = [&](int a_row, int b_row, int bt) {
        return bt >= 0 && bt * p.tiles_per_batch < p.num_tiles && a_row >= 0 && a_row < p.tiles_m * C::kTileM &&
               b_row >= 0 && b_row < p.tiles_n * kBN;
    };
#endif

    // The unit's first work item, without waiting: a static list's first
    // item, or the first tile of the unit's own dynamic list (every list
    // has one).  The same item get_work() returns first.
    auto first_item = [&](Work& w) -> bool {
        if (!dyn) {
            if (nwork <= 0) return false;
            w = work_item(p.sched, pair_id, 0);
        } else {
            w = whole_tile(list_tile(pair_id, 0), p.k_blocks);
        }
        return true;
    };
    // The first k-blocks of the first item are loaded by epilogue warp 2 at
    // start-up (see below): as many as the ring holds.
    auto preissued = [&](const Work& w) { return min(kStages, w.kb_end - w.kb_begin); };
    // A unit's odd work items load their k-blocks last to first: the wave
    // after a wave then starts on the k-blocks its predecessor read last,
    // still in L2 (8192³: DRAM reads 965 → 826 MB per launch, 560 → 556 µs).
    // Only the order of the fp32 sum changes, the same every run.
    constexpr bool kReverseOddItems = true;

    // Loads of k-block kb of a work item into ring slot `stage`, by one lane:
    // the pair leader announces the pair's bytes on its full barrier; then
    // this CTA's A rows and its share of the tile's B rows (in a 4-CTA unit a
    // quarter, written to this CTA and to the same-rank CTA of the other
    // pair).  In a pair the copies complete on the leader's barrier.
    auto issue_loads = [&](int kb, uint32_t stage, int a_row, int b_row, int za, int zb) {
        const uint32_t fb = full_bar(stage);
        const uint32_t a_dst = base + stage * kStageBytesA;
        const uint32_t b_dst = base + C::kOffB + stage * C::kStageBytesB;
        if (rank == 0) mbar_arrive_expect_tx(fb, C::kTxBytes);
        const uint32_t fb_leader = kCluster > 1 ? map_shared_rank(fb, leader) : fb;
        const uint16_t mask = (uint16_t)((1u << rank) | (1u << (rank + 2)));
        auto copy_a = [&](uint32_t dst, int x, int y) {
            if constexpr (kCluster > 1) tma_load_3d_pair(dst, &tmA, fb_leader, x, y, za);
            else tma_load_3d(dst, &tmA, fb, x, y, za);
        };
        auto copy_b = [&](uint32_t dst, int x, int y) {
            if constexpr (kCluster == 4)
                tma_load_3d_pair_multicast(dst, &tmB, fb_leader, mask, x, y, zb);
            else if constexpr (kCluster == 2) tma_load_3d_pair(dst, &tmB, fb_leader, x, y, zb);
            else tma_load_3d(dst, &tmB, fb, x, y, zb);
        };
        const int kx = kb * C::kBlockKElems;
        const uint32_t b_q = b_dst + pidx * C::kLoadBytesB;
        // K-major: one box {one 128-byte row of K, rows} at (k, row).
        // MN-major: boxes {64 elements, 64 K rows} at (row, k).
        if (p.a_mn) {
            for (int h = 0; h < kRowsPerCta / kMnBoxElems; ++h)
                copy_a(a_dst + h * kMnBoxBytes, a_row + h * kMnBoxElems, kx);
        } else {
            copy_a(a_dst, kx, a_row);
        }
        if (p.b_mn) {
            for (int h = 0; h < C::kBoxesB; ++h) copy_b(b_q + h * kMnBoxBytes, b_row + h * kMnBoxElems, kx);
        } else {
            copy_b(b_q, kx, b_row);
        }
    };

    // ---- set-up: barriers, TMEM, tensor-map prefetch
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), C::kPairs);   // one MMA commit per pair that reads this slot
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiWarps * kPair);
        }
        for (int e = 0; e < kEpiWarps; ++e) mbar_init(fix_bar(e), 1);
        for (int s = 0; s < kClcSlots; ++s) {
            mbar_init(clc_full(s), 1);              // the requester's expect-tx arrival + 16 bytes
            mbar_init(clc_empty(s), kClcReaders);   // used in the cluster's first CTA
        }
        *abort_flag = 0;
        fence_mbar_init_cluster();
        GEMM_TR_CLK(1);
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
        GEMM_TR_CLK(2);
    }
    // The barrier inits are published CTA-wide and to the peer CTAs by the
    // cluster barrier (a CTA barrier without a cluster).  The MMA warp
    // arrives on it before allocating TMEM and waits after, so the producer's
    // first loads do not wait for the allocation; the TMEM address reaches
    // the epilogue warps through a named barrier of warps 1-5.
    // Epilogue warp 2, idle until the first accumulator is full, decodes the
    // first work item while the barriers are set up and, once they are
    // visible, issues that item's first ring-full of loads (the producer
    // warp starts after them).  Each warp fetches its instructions on its
    // own, so after an L2 flush the cold code of the decode and of the
    // first issue is fetched while warp 0 initialises the barriers instead
    // of after it.
    Work w_first;
    int pre_rows[3] = {0, 0, 0};   // a_row, b_row, batch element of the first item
    bool pre_ok = false;
    if constexpr (kCluster > 1) cluster_arrive();
    if (warp == 2) {
        pre_ok = first_item(w_first);
        if (pre_ok) operand_rows(w_first.tile, pre_rows[0], pre_rows[1], pre_rows[2]);
        if (lane == 0) GEMM_TR_SET(kTrClkPro + 5, (unsigned long long)clock64());
    }
    if constexpr (kCluster == 1) __syncthreads();
    if (threadIdx.x == 0) GEMM_TR_CLK(3);
    if (warp == 1) {
        tmem_alloc<kPair>(smem_addr(tmem_holder), kTmemCols);
        tmem_relinquish<kPair>();
    }
    if constexpr (kCluster > 1) cluster_wait();
    if (threadIdx.x == 0) GEMM_TR_CLK(4);
    // Launched as a programmatic dependent of the previous kernel on the
    // stream, this grid may have started while that kernel still runs: the
    // set-up above touches only this CTA's shared memory, TMEM and the kernel
    // parameters.  Every thread waits here for the previous grids' completion
    // before any load of A or B, any store of C and any use of the plan's
    // device memory.
    griddep_wait();
    if (warp == 2 && pre_ok) {
#ifdef GEMM_DEBUG
        pre_ok = GEMM_WARP_CHECK(item_ok(w_first) && rows_ok(pre_rows[0], pre_rows[1], pre_rows[2]), kChkOperandRows);
#endif
        if (lane == 0) GEMM_TR_SET(kTrClkPro + 6, (unsigned long long)clock64());
        if (pre_ok && elect_one_sync()) {
            const int za = p.a_batched ? pre_rows[2] : 0, zb = p.b_batched ? pre_rows[2] : 0;
            const int n = preissued(w_first);
            for (int i = 0; i < n; ++i) issue_loads(w_first.kb_begin + i, (uint32_t)i, pre_rows[0], pre_rows[1], za, zb);
            GEMM_TR_SET(kTrClkPro + 7, (unsigned long long)clock64());
        }
        __syncwarp();
    }
    uint32_t tmem_base = 0;
    if (warp >= 1) {
        tc_fence_before_sync();
        named_bar_sync(1, kNumThreads - 32);
        tc_fence_after_sync();
        tmem_base = *tmem_holder;
        if (warp == 1 && lane == 0) GEMM_TR_CLK(8);
    }

    // The producer and MMA loops run on the whole warp, so that stage, phase
    // and the descriptors stay warp-uniform (the TMA and tcgen05.mma operands
    // live in uniform registers); one elected lane issues the instructions.
    // A single-lane loop in a divergent branch measured ~25% slower per K
    // block on GB300.
    if (warp == 0) {
        // ================= TMA producer
        {
            const bool issuer = elect_one_sync();
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            uint64_t empty_wait_ns = 0;   // trace builds only
            // Request r of the dynamic list: once every reader has released
            // slot r % kClcSlots, announce its 16 bytes on each CTA's full
            // barrier and send the request.
            auto request = [&](int r) -> bool {
                const int s = r % kClcSlots;
                if (!__all_sync(0xffffffffu,
                                wait_bounded<(kCluster > 1)>(clc_empty(s), ((uint32_t)(r / kClcSlots) & 1u) ^ 1u,
                                                             abort_flag, p, kRoleClc, -1 - r)))
                    return false;
                if (issuer) {
                    if constexpr (kCluster > 1) {
                        for (uint32_t c = 0; c < (uint32_t)kCluster; ++c)
                            mbar_arrive_expect_tx_cluster(map_shared_rank(clc_full(s), c), kClcResponseBytes);
                    } else {
                        mbar_arrive_expect_tx(clc_full(s), kClcResponseBytes);
                    }
                    clc_try_cancel<(kCluster > 1)>(clc_resp(s), clc_full(s));
                }
                __syncwarp();
                return true;
            };
            const bool requester = dyn && crank == 0;
            Cursor cur = cursor0;
            for (int j = 0; ok; ++j) {
                Work w;
                const int g = get_work(cur, w);
                if (g <= 0) {
                    ok = g == 0;
                    break;
                }
                // the last item of a list: ask for the next list now
                if (requester && cur.pos == cur.len && !(ok = request(cur.resp))) break;
                if (!GEMM_WARP_CHECK(item_ok(w), kChkWorkItem)) {
                    ok = false;
                    break;
                }
                int a_row, b_row, bt;
                operand_rows(w.tile, a_row, b_row, bt);
                if (!GEMM_WARP_CHECK(rows_ok(a_row, b_row, bt), kChkOperandRows)) {
                    ok = false;
                    break;
                }
                const int za = p.a_batched ? bt : 0, zb = p.b_batched ? bt : 0;   // batch coordinates
                int t0 = 0;
                if (j == 0) {
                    // epilogue warp 2 has issued the first item's first slots
                    const int n = preissued(w);
                    t0 = n;
                    stage = n == kStages ? 0u : (uint32_t)n;
                    phase = n == kStages ? 1u : 0u;
                }
                // Odd items walk K backwards (kReverseOddItems); the MMA warp
                // starts each sum on whatever its first slot holds.
                const bool rev = kReverseOddItems && (j & 1);
                for (int t = t0; t < w.kb_end - w.kb_begin; ++t) {
                    const int kb = rev ? w.kb_end - 1 - t : w.kb_begin + t;
                    if (!GEMM_WARP_CHECK(stage < (uint32_t)kStages && phase <= 1u, kChkRing) ||
                        !GEMM_WARP_CHECK(kb >= 0 && kb < p.k_blocks, kChkKBlock)) {
                        ok = false;
                        break;
                    }
                    const uint64_t tw = GEMM_TR_NOW();
                    if (!__all_sync(0xffffffffu,
                                    wait_bounded<(kCluster > 1), kRingWaitHintNs>(empty_bar(stage), phase ^ 1u,
                                                                                  abort_flag, p, 0, kb))) {
                        ok = false;
                        break;
                    }
                    empty_wait_ns += GEMM_TR_NOW() - tw;
                    if (issuer) issue_loads(kb, stage, a_row, b_row, za, zb);
                    __syncwarp();
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            griddep_launch_dependents();   // no more loads from this warp
            GEMM_TR_SET(kTrEmptyWaitNs, empty_wait_ns);
            if (lane == 0) GEMM_TR_SET(kTrClcWaitProducerNs, clc_wait_ns);
            (void)empty_wait_ns;
            // Every slot's last use must be released (the MMA's commit arrives
            // on this CTA's empty barriers) before the CTA may exit.
            for (int s = 0; s < kStages && ok; ++s) {
                ok = __all_sync(0xffffffffu, wait_bounded<(kCluster > 1)>(empty_bar(stage), phase ^ 1u, abort_flag, p, 1, s));
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (lane == 0) GEMM_TR(kTrProducerDone);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (leader CTA only)
        if (rank == 0) {
            const bool issuer = elect_one_sync();
            const uint32_t a_base = base, b_base = base + C::kOffB;
            // Descriptor start advance per MMA (in 16-byte units): 32 bytes along
            // a K-major row, or the MMA's K rows of 128 bytes in an MN-major tile.
            constexpr uint32_t kStepK = kMmaKBytes >> 4;
            constexpr uint32_t kStepMn = ((kMmaKBytes / (kIn == kInF8 ? 1 : 2)) * 128) >> 4;
            const uint32_t a_step = p.a_mn ? kStepMn : kStepK, b_step = p.b_mn ? kStepMn : kStepK;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int i = 0;
            uint64_t full_wait_ns = 0, acc_wait_ns = 0;   // trace builds only
            if (p.stall_test) {
                // A wait that cannot end: fix_bar(0) gets no arrival unless a
                // stream-K finisher uses it, and this launch has none.  It runs
                // out after p.wait_limit_ns and takes the kernel down the
                // timeout path (status, abort flag, orderly teardown).
                ok = __all_sync(0xffffffffu, wait_bounded<false>(fix_bar(0), 0, abort_flag, p, kRoleStallTest, 0));
            }
            Cursor cur = cursor0;
            for (; ok; ++i) {
                Work w;
                const int g = get_work(cur, w);
                if (g <= 0) {
                    ok = g == 0;
                    break;
                }
                const uint32_t b = i & 1, aphase = (i >> 1) & 1;
                if (!GEMM_WARP_CHECK(item_ok(w), kChkWorkItem) ||
                    !GEMM_WARP_CHECK(b < 2u && aphase <= 1u && b * kAccStride + kBN <= (uint32_t)kTmemCols,
                                     kChkAccumulator)) {
                    ok = false;
                    break;
                }
                const uint64_t ta = GEMM_TR_NOW();
                if (!__all_sync(0xffffffffu, wait_bounded<true>(acce_bar(b), aphase ^ 1u, abort_flag, p, 2, i))) {
                    ok = false;
                    break;
                }
                acc_wait_ns += GEMM_TR_NOW() - ta;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kAccStride;
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {   // (the producer's order may differ: counted only)
                    if (!GEMM_WARP_CHECK(stage < (uint32_t)kStages && phase <= 1u, kChkRing) ||
                        !GEMM_WARP_CHECK(kb >= 0 && kb < p.k_blocks, kChkKBlock)) {
                        ok = false;
                        break;
                    }
                    const uint64_t tf = GEMM_TR_NOW();
                    if (!__all_sync(0xffffffffu, wait_bounded<(kCluster > 1), kRingWaitHintNs>(full_bar(stage), phase,
                                                                                              abort_flag, p, 3, kb))) {
                        ok = false;
                        break;
                    }
                    full_wait_ns += GEMM_TR_NOW() - tf;
                    if (i == 0 && kb == w.kb_begin) {   // trace only
                        GEMM_TR(kTrFirstFull);
                        GEMM_TR_SET(kTrClkFirstFull, (unsigned long long)clock64());
                    }
                    const uint32_t a_addr = a_base + stage * kStageBytesA, b_addr = b_base + stage * C::kStageBytesB;
                    const uint64_t ad = p.a_mn ? smem_desc_sw128_mn(a_addr) : smem_desc_sw128(a_addr);
                    const uint64_t bd = p.b_mn ? smem_desc_sw128_mn(b_addr) : smem_desc_sw128(b_addr);
                    const uint32_t first = kb == w.kb_begin;
                    if (issuer) {
                        tc_fence_after_sync();
#pragma unroll
                        for (int j = 0; j < kBlockKBytes / kMmaKBytes; ++j) {
                            // next 16 (bf16/f16) or 32 (fp8) elements of K: a_step / b_step above
                            tc_mma<kPair, kIn == kInF8>(d_tmem, ad + a_step * j, bd + b_step * j, p.idesc,
                                                        !(first && j == 0));
                        }
                        // release the slot in every CTA whose copies write into this pair's slot
                        if constexpr (kCluster == 4) tc_commit_pair(empty_bar(stage), 0xF);
                        else if constexpr (kCluster == 2) tc_commit_pair(empty_bar(stage), 0x3);
                        else tc_commit(empty_bar(stage));
                    }
                    __syncwarp();
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (issuer) {
                    if constexpr (kPair == 2) tc_commit_pair(accf_bar(b), (uint16_t)(0x3u << leader));
                    else tc_commit(accf_bar(b));
                }
                __syncwarp();
                GEMM_TR_ITEM(kTrMmaEnd, i);
                if (i < 8) GEMM_TR_SET(kTrClkMmaEnd + i, (unsigned long long)clock64());
            }
            GEMM_TR(kTrWorkItems);
            GEMM_TR_SET(kTrFullWaitNs, full_wait_ns);
            GEMM_TR_SET(kTrAccEmptyWaitNs, acc_wait_ns);
            if (lane == 0) GEMM_TR_SET(kTrClcWaitMmaNs, clc_wait_ns);
            (void)full_wait_ns;
            (void)acc_wait_ns;
            // Every remote arrive on this CTA's barriers must land before it
            // exits: the epilogue warps of the pair release every item but the
            // last, so wait for the next-to-last item's release (the ones
            // before it were awaited before the MMAs of later items).
            for (int j = 0; j < 1 && ok; ++j, ++i) {
                ok = __all_sync(0xffffffffu, wait_bounded<true>(acce_bar(i & 1), ((i >> 1) & 1) ^ 1u, abort_flag, p, 4, j));
            }
            if (lane == 0) GEMM_TR(kTrMmaDone);
        }
        __syncwarp();
        griddep_launch_dependents();   // no more MMAs in this CTA
    } else {
        // ================= epilogue warps
        const int quad = warp & 3;                   // TMEM lanes 32*quad .. 32*quad+31
        const uint32_t staging = base + C::kOffStaging + (uint32_t)(warp - 2) * 2u * C::kSlotBytes;
        uint32_t slot = 0;

        // Convert one 32-column chunk (fp32 values of this thread's row) and
        // write it swizzled into the 32-row store box at `buf`.
        auto stage_chunk = [&](uint32_t buf, const uint32_t (&cur)[32]) {
            const uint32_t row_addr = buf + (uint32_t)lane * C::kRowBytes;
            if constexpr (kOut == kOutF32) {
                // 128-byte rows: 16-byte chunk q stored at q ^ (row % 8)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_shared_v4(row_addr + (((uint32_t)q ^ ((uint32_t)lane & 7u)) << 4), cur[4 * q], cur[4 * q + 1],
                                 cur[4 * q + 2], cur[4 * q + 3]);
            } else {
                // 64-byte rows: 16-byte chunk q stored at q ^ ((row / 2) % 4)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t w0 = pack2(__uint_as_float(cur[8 * q + 0]), __uint_as_float(cur[8 * q + 1]), kOut);
                    const uint32_t w1 = pack2(__uint_as_float(cur[8 * q + 2]), __uint_as_float(cur[8 * q + 3]), kOut);
                    const uint32_t w2 = pack2(__uint_as_float(cur[8 * q + 4]), __uint_as_float(cur[8 * q + 5]), kOut);
                    const uint32_t w3 = pack2(__uint_as_float(cur[8 * q + 6]), __uint_as_float(cur[8 * q + 7]), kOut);
                    st_shared_v4(row_addr + (((uint32_t)q ^ (((uint32_t)lane >> 1) & 3u)) << 4), w0, w1, w2, w3);
                }
            }
        };
        // Stage one chunk in this warp's two staging boxes and TMA-store it to
        // C at (ccol, row0) of batch element bt.
        auto store_chunk = [&](const uint32_t (&cur)[32], int ccol, int row0, int bt) {
            const uint32_t buf = staging + (slot & 1u) * C::kSlotBytes;
            ++slot;
            if (lane == 0) bulk_wait_group_read<1>();   // the store that last read `buf` is done
            __syncwarp();
            stage_chunk(buf, cur);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&tmC, buf, ccol, row0, bt);
                bulk_commit_group();
            }
        };

        Work w, nw;
        Cursor cur = cursor0;
        int g = get_work(cur, w), gn = 0;
        for (int i = 0; g > 0; ++i) {
            const uint32_t b = i & 1, aphase = (i >> 1) & 1;
            const bool got = wait_bounded<false, kEpiWaitHintNs>(accf_bar(b), aphase, abort_flag, p, 5, i);
            if (!__all_sync(0xffffffffu, got)) break;
            // The next item now: whether this tile is the unit's last decides
            // how it is stored.
            gn = get_work(cur, nw);
            if (gn < 0) break;
            if (warp == 2 && lane == 0) GEMM_TR_ITEM(kTrEpiStart, i);
            tc_fence_after_sync();
            if (!GEMM_WARP_CHECK(item_ok(w), kChkWorkItem)) break;
            int bt, mt, nt;
            tile_coords(p, w.tile, bt, mt, nt);
            if (!GEMM_WARP_CHECK(bt >= 0 && bt * p.tiles_per_batch < p.num_tiles && mt >= 0 && mt < p.tiles_m &&
                                     nt >= 0 && nt < p.tiles_n,
                                 kChkTileCoords))
                break;
            const int row0 = mt * C::kTileM + (int)crank * kRowsPerCta + quad * 32;
            const int col0 = nt * kBN;
            if (!GEMM_WARP_CHECK(row0 + 32 <= p.tiles_m * C::kTileM && col0 + kBN <= p.tiles_n * kBN &&
                                     b < 2u && aphase <= 1u,
                                 kChkStoreBox))
                break;
            const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + b * kAccStride;
            if (w.ncontrib == 1 && gn == 0) {
                // The last tile's loads and MMAs are done: a programmatic
                // dependent grid may be scheduled (its CTAs start as this
                // grid's exit, and wait for its completion before reading).
                griddep_launch_dependents();
                // The unit's last tile: nothing overlaps its epilogue, and its
                // operand ring is idle (no later loads, every MMA done), so each
                // chunk gets its own box there: no chunk waits for an earlier
                // store to finish reading, and each is stored as soon as it is
                // staged.
                if (row0 < p.M) {
                    const int le = kTrLastEpi + 12 * (warp - 2);   // trace builds only
                    (void)le;
                    if (lane == 0) GEMM_TR_SET(le + kLeStart, (unsigned long long)clock64());
                    const uint32_t region = base + (uint32_t)(warp - 2) * (uint32_t)(kChunks * C::kSlotBytes);
                    uint32_t ra[32], rb[32];
                    tmem_ld_32x32b_x32(t_row, ra);
                    tmem_ld_wait(ra);
                    if (lane == 0) GEMM_TR_SET(le + kLeFirstData, (unsigned long long)clock64());
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        uint32_t(&cur)[32] = (c & 1) ? rb : ra;
                        uint32_t(&nxt)[32] = (c & 1) ? ra : rb;
                        if (c + 1 < kChunks) tmem_ld_32x32b_x32(t_row + (c + 1) * kChunkCols, nxt);
                        stage_chunk(region + (uint32_t)(c * C::kSlotBytes), cur);
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0 && col0 + c * kChunkCols < p.N)
                            tma_store_3d(&tmC, region + (uint32_t)(c * C::kSlotBytes), col0 + c * kChunkCols, row0, bt);
                        if (lane == 0 && c < 8) GEMM_TR_SET(le + kLeChunk + c, (unsigned long long)clock64());
                        if (c + 1 < kChunks) tmem_ld_wait(nxt);
                    }
                    if (lane == 0) bulk_commit_group();
                    if (lane == 0) GEMM_TR_SET(le + kLeCommitted, (unsigned long long)clock64());
                }
            } else if (w.ncontrib == 1) {
                if (row0 < p.M) {
                    // Two register sets: the TMEM load of chunk c+1 is in flight
                    // while chunk c is converted, staged and stored.
                    // The stores are paced: a pause after each chunk spreads
                    // them over about a third of the next tile's K loop
                    // (~256 ns per k-block), whose operand loads share the
                    // SM's TMA unit and shared memory with them.  Issued in
                    // one burst they slowed that K loop by 1-2% (4096³:
                    // 77.7 -> 76.8 µs paced; E4M3 4096³ 45.6 -> 44.6).
                    const uint32_t pace_ns = (uint32_t)min(2000, min(p.k_blocks, 1 << 16) * 256 / (3 * kChunks));
                    uint32_t ra[32], rb[32];
                    tmem_ld_32x32b_x32(t_row, ra);
                    tmem_ld_wait(ra);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        uint32_t(&cur)[32] = (c & 1) ? rb : ra;
                        uint32_t(&nxt)[32] = (c & 1) ? ra : rb;
                        if (c + 1 < kChunks) tmem_ld_32x32b_x32(t_row + (c + 1) * kChunkCols, nxt);
                        const int ccol = col0 + c * kChunkCols;
                        if (ccol < p.N) store_chunk(cur, ccol, row0, bt);
                        if (c + 1 < kChunks && pace_ns) __nanosleep(pace_ns);
                        if (c + 1 < kChunks) tmem_ld_wait(nxt);
                    }
                }
            } else if (w.contrib == 1) {
                // Second piece of a split tile: publish the fp32 partial in
                // this unit's workspace slot, then raise this warp's flag.
                float4* mine = reinterpret_cast<float4*>(
                    p.partials + ((size_t)(w.slot * kCluster + (int)crank) * 4 + quad) * kPartialFloats);
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + c * kChunkCols, v);
                    tmem_ld_wait(v);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(&mine[(c * 8 + q) * 32 + lane],
                               make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
                }
                fence_proxy_async_global();   // the finisher reads the partial with a bulk copy
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(p.flags + (w.sk_index * kCluster + (int)crank) * 4 + quad, 1);
                if (warp == 2 && lane == 0) GEMM_TR_ITEM(kTrPartialDone, i);
            } else {
                // First piece of a split tile, the last item of this unit: its
                // operand ring is idle now that the accumulator is full.  Wait
                // for the other piece's partial, pull it into this warp's
                // 32 KB of the ring with one bulk copy, and store own + other
                // (two addends: the fp32 sum is the same in either order).
                int* flag = p.flags + (w.sk_index * kCluster + (int)crank) * 4 + quad;
                const uint32_t fix = base + (uint32_t)(warp - 2) * (uint32_t)kFixupBytes;
                const uint32_t fbar = fix_bar(warp - 2);
                bool ok = wait_flag_bounded(flag, abort_flag, p, 6, w.sk_index);
                if (ok) {
                    if (lane == 0) {
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(fbar, C::kPartialBytes);
                        bulk_copy_g2s(fix, p.partials + ((size_t)(w.slot * kCluster + (int)crank) * 4 + quad) * kPartialFloats,
                                      C::kPartialBytes, fbar);
                    }
                    ok = __all_sync(0xffffffffu, wait_bounded<false>(fbar, 0, abort_flag, p, 7, w.sk_index));
                }
                if (!ok) break;
                if (row0 < p.M) {
                    uint32_t ra[32], rb[32];
                    tmem_ld_32x32b_x32(t_row, ra);
                    tmem_ld_wait(ra);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        uint32_t(&cur)[32] = (c & 1) ? rb : ra;
                        uint32_t(&nxt)[32] = (c & 1) ? ra : rb;
                        if (c + 1 < kChunks) tmem_ld_32x32b_x32(t_row + (c + 1) * kChunkCols, nxt);
                        const int ccol = col0 + c * kChunkCols;
                        if (ccol < p.N) {
                            uint32_t sum[32];
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                uint32_t o[4];
                                ld_shared_v4(fix + (uint32_t)(((c * 8 + q) * 32 + lane) * 16), o[0], o[1], o[2], o[3]);
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    sum[4 * q + e] = __float_as_uint(__uint_as_float(cur[4 * q + e]) + __uint_as_float(o[e]));
                            }
                            store_chunk(sum, ccol, row0, bt);
                        }
                        if (c + 1 < kChunks) tmem_ld_wait(nxt);
                    }
                }
                if (lane == 0) *flag = 0;   // ready for the next launch
                if (warp == 2 && lane == 0) GEMM_TR_ITEM(kTrReduceDone, i);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (warp == 2 && lane == 0) GEMM_TR_ITEM(kTrEpiEnd, i);
            // Release the accumulator to the MMA warp, unless this was the
            // unit's last item: no MMA reuses it, and the teardown's barriers
            // order these TMEM reads before the deallocation.  (A cluster-scope
            // release there held the warp ~0.7 us behind its last stores.)
            if (lane == 0 && gn != 0) {
                if constexpr (kPair == 2) mbar_arrive_cluster(map_shared_rank(acce_bar(b), leader));
                else mbar_arrive_local(acce_bar(b));
            }
            w = nw;
            g = gn;
        }
        if (warp == 2 && lane == 0) GEMM_TR(kTrEpiLoopDone);
        griddep_launch_dependents();   // (again, if the loop ended without a last whole tile)
        // Only the staging buffers' reads must be done before shared memory
        // goes away; the writes to C complete with the grid.
        if (lane == 0) bulk_wait_group_read<0>();
        if (lane == 0) GEMM_TR_SET(kTrLastEpi + 12 * (warp - 2) + kLeStoresRead, (unsigned long long)clock64());
        __syncwarp();
        if (warp == 2 && lane == 0) GEMM_TR(kTrEpiDone);
        if (warp == 2 && lane == 0) GEMM_TR_SET(kTrClcWaitEpiNs, clc_wait_ns);
    }

    // ---- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) GEMM_TR(kTrTeardown);
    if (*abort_flag) {
        // A bounded wait gave up: let copies and MMAs already in flight land
        // (they finish in microseconds) before TMEM and shared memory go away.
        if (threadIdx.x == 0) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 2000000ull) { }
        }
        __syncthreads();
    }
    if constexpr (kCluster > 1) {
        // No CTA of the unit may leave (freeing its shared memory and TMEM)
        // while another may still touch them.  Every such access was awaited
        // in the CTA it targets before this point: operand loads and the
        // MMAs that read them through the producer's drain of every slot,
        // the MMAs' TMEM writes and commit arrives through the epilogue's
        // full-accumulator waits, the epilogue's remote releases through the
        // MMA warp's final wait.  So an execution barrier suffices; with
        // release semantics the arrive waited ~0.7 us for this CTA's C
        // stores to drain (one-wave 1024x4096x4096 f16 +1.6%, 4096^3 +0.6%).
        cluster_arrive_relaxed();
        if (threadIdx.x == 0) GEMM_TR(kTrClusterArrived);
        cluster_wait();
        if (threadIdx.x == 0) GEMM_TR(kTrClusterDone);
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<kPair>(tmem_base, kTmemCols);
        if (lane == 0) GEMM_TR(kTrDealloc);
    }
    if (threadIdx.x == 0) GEMM_TR(kTrExit);
    if (lane == 0 && warp <= 1) GEMM_TR_CLK_FLUSH();
    if (clock_owner) {
        const unsigned long long clk = (unsigned long long)clock64(), ns = global_timer_ns();
        p.clock_rec[0] = clk - clk_entry;
        p.clock_rec[1] = ns - ns_entry;
    }
}

}  // namespace gb300
