/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Operation.  C = A·Bᵀ: A is M×K row-major, B is stored transposed as N×K
 * row-major, C is M×N row-major.  Inputs are bf16, f16, E4M3 or E5M2
 * (both the same type), products are accumulated in fp32, and C is written
 * as fp32, bf16 or f16 (rounded to nearest, ties to even).  This is the problem statement of
 * "Optimizing Blackwell Matrix Multiplication in Mojo (Part 2)" (intro and
 * "Kernel 2: TMA and Tensor Core": B kept N×K so that both operands are read
 * along K), with the bf16-in / fp32-accumulate / cast-once-at-the-end
 * precision of "Chapter 7: Writing Custom Kernels with Pallas", §4.1'.
 *
 * Device.  Everything runs on one GB300 GPU.  A, B and C are device pointers
 * owned by the caller; the library never allocates, frees or retains them.
 * Each run checks, before it encodes or launches anything, that the device
 * it runs on (the plan's; for gemm_run_noalloc the current one) is current
 * and that A, B (when K > 0) and C are device memory of that device
 * (cudaPointerGetAttributes); host memory, managed memory and another
 * GPU's memory return GEMM_ERR_INVALID_ARG.  Host buffers go through
 * gemm_plan_run_host.  Work is enqueued asynchronously on the caller's
 * stream (a cudaStream_t, passed as void* so that this header needs no CUDA
 * header); 0 means the legacy default stream.
 *
 * Layout rules (checked on the host before anything is launched):
 *   - A, B, C 16-byte aligned;
 *   - K * sizeof(input element) and N * sizeof(C element) bytes multiples
 *     of 16, i.e. K % 8 == 0 (bf16/f16 in) or K % 16 == 0 (fp8 in), and
 *     N % 8 == 0 (bf16/f16 out) or N % 4 == 0 (fp32 out);
 *   - M, N, K <= 2^31 - 1024 (tile coordinates are 32-bit); larger sizes
 *     return GEMM_ERR_UNSUPPORTED.
 * Other shapes return GEMM_ERR_UNSUPPORTED: there is no slow fallback path.
 *
 * Degenerate sizes: M == 0 or N == 0 is a no-op; K == 0 writes C = 0 (the
 * empty sum) with a small fill kernel.
 *
 * Errors.  Every entry point returns a gemm_status_t.  Problems visible on
 * the host (bad arguments, alignment, a CUDA or driver call failing) are
 * returned at once and nothing is enqueued.  A wait inside the kernel that
 * outlives its bound (about two seconds; it never does in a correct run)
 * makes the kernel record GEMM_ERR_TIMEOUT in the plan's device status word
 * and return early; gemm_plan_status() reads that word after the caller has
 * synchronised the stream.
 *
 * Threads.  A plan may be used from several host threads and streams at
 * once; calls build their tensor maps on the host stack and share only
 * read-only plan state, the device status word and the last-launch record
 * (written under a lock by every run; with concurrent runs it describes one
 * of them).  Split products (GEMM_OPT_SPLIT_K) also share the plan's
 * workspace; the library orders them one after another on the GPU.
 * Exception: with the stream-K option on (off by default) runs share the
 * plan's workspace unordered, so runs that may overlap on the GPU must then
 * use different plans.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  Inputs (A and B, both the same type): BF16, F16, E4M3,
 * E5M2.  Output C: F32, BF16, F16.  E4M3 is the finite-only 8-bit format
 * (4 exponent bits, bias 7, 3 fraction bits, no infinities, S.1111.111 the
 * only NaN) and E5M2 the IEEE-style one (5 exponent bits, bias 15, 2
 * fraction bits): the float8_e4m3fn and float8_e5m2 operand types of
 * "Writing Mosaic GPU kernels with Pallas", "Blackwell (tcgen05)", "Issuing
 * the operation".  8-bit inputs are multiplied exactly and summed in fp32
 * like the 16-bit ones, at twice the tensor-core rate; no scale factors. */
typedef enum { GEMM_BF16 = 0, GEMM_F16 = 1, GEMM_F32 = 2, GEMM_E4M3 = 3, GEMM_E5M2 = 4 } gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad dtype pair, bad option,
                                    an operand that is not device memory of the run's
                                    device, or that device not current                 */
    GEMM_ERR_UNSUPPORTED = -2,   /* shape/pitch TMA cannot address (see layout rules)       */
    GEMM_ERR_MISALIGNED = -3,    /* a pointer not 16-byte aligned                            */
    GEMM_ERR_CUDA = -4,          /* a CUDA runtime call failed (launch, attribute, copy);
                                    device side: the launch's shared memory was not 1 KB
                                    aligned (see gemm_plan_status)                        */
    GEMM_ERR_DRIVER = -5,        /* the driver's tensor-map encoder failed or is missing     */
    GEMM_ERR_NO_PLAN = -6,       /* gemm_run with no plan created for the current device     */
    GEMM_ERR_TIMEOUT = -7,       /* device side: a bounded wait expired (see gemm_plan_status) */
    GEMM_ERR_NO_DEVICE = -8,     /* no usable sm_103 device                                   */
    GEMM_ERR_INTERNAL = -9       /* device side, GEMM_DEBUG builds only: a consistency check
                                    (tile coordinates, ring stage or phase, k-block range,
                                    store box) failed; the access was skipped and the kernel
                                    ended early (see gemm_plan_status)                   */
} gemm_status_t;

typedef struct gemm_plan* gemm_plan_t;

/* Operand storage for gemm_plan_run_layout (bit flags; 0 = the default of
 * every other entry point: A M×K and B N×K, both K-major).
 *   GEMM_A_MN_MAJOR: A is stored K×M row-major (a(i,k) = A[k*M + i]);
 *   GEMM_B_MN_MAJOR: B is stored K×N row-major (b(j,k) = B[k*N + j]), i.e.
 *                    C = A·B for a plain row-major K×N B, the layout of the
 *                    matmuls in "Writing Mosaic GPU kernels with Pallas" and
 *                    "Chapter 7: Writing Custom Kernels with Pallas".
 * The tensor cores read such operands in place (MN-major shared-memory
 * tiles); nothing is transposed in memory.  16-bit inputs only. */
typedef enum { GEMM_K_MAJOR = 0, GEMM_A_MN_MAJOR = 1, GEMM_B_MN_MAJOR = 2 } gemm_layout_t;

/* Plan options (gemm_plan_set_option).  For tuning sweeps and tests; the
 * defaults are what the library picks itself. */
typedef enum {
    GEMM_OPT_CTA_PAIR = 1,       /* 2: 2-CTA pairs, 256×BN tile per pair; 1: one CTA
                                    per 128×BN tile; 0 (default): pairs, except for
                                    problems under half a wave of pair tiles that fit
                                    one wave of 128×128 single-CTA tiles (there a
                                    pair's set-up costs more than it saves)         */
    GEMM_OPT_GROUP_M = 2,        /* rasterisation group height in tiles, >= 1 (0 = auto:
                                    every tile row when A is at most 48 MB, else 8)  */
    GEMM_OPT_MAX_CTAS = 3,       /* cap on resident CTAs of the persistent grid (0 = all SMs) */
    GEMM_OPT_TILE_N = 4,         /* tile width: 256, 224, 192, 160 or 128 (0 = default:
                                    chosen per problem to fill whole waves)             */
    GEMM_OPT_STREAM_K = 5,       /* 1: spread the K work of the last whole wave and a
                                    partial one over all resident units in ranges
                                    longer than a tile (a tile is split at most two
                                    ways; deterministic fix-up), or halve the tiles
                                    along K when there are fewer than half as many
                                    tiles as units, where that is predicted to pay;
                                    runs that may overlap on the GPU then need
                                    separate plans.  The unit finishing a split tile
                                    waits for a flag the other unit raises, so every
                                    unit of the launch must be resident at once: if
                                    other work on the GPU keeps some units from
                                    starting until the waiting ones end, the run ends
                                    with GEMM_ERR_TIMEOUT (after the wait bound) and C
                                    undefined, not with a result.  0 (default): whole
                                    tiles only, no unit waits for another            */
    GEMM_OPT_MULTICAST = 6,      /* with CTA pairs: 1 = two pairs per 4-CTA cluster work
                                    on vertically adjacent tiles and share their B tile
                                    through TMA multicast (512×BN per cluster); 0 = one
                                    pair per cluster; -1 (default) = multicast when the
                                    rows of A and B are not a multiple of 128 bytes.
                                    Multicast is used only while the process sees one
                                    GPU (see GEMM_OPT_VISIBLE_DEVICES): with more, the
                                    default picks pairs and 1 is GEMM_ERR_UNSUPPORTED */
    GEMM_OPT_WAIT_LIMIT_US = 7,  /* bound on any single wait inside the kernel, in µs,
                                    1..60e6 (0 = default: 2 s)                         */
    GEMM_OPT_STALL_TEST = 8,     /* tests of the timeout path only: 1 = the MMA warp
                                    first waits on a barrier nothing completes, so the
                                    run ends, after about two wait bounds, with
                                    GEMM_ERR_TIMEOUT (role 8) in the status word and
                                    C unwritten; 0 (default) = off                     */
    GEMM_OPT_DYNAMIC = 9,        /* run-time tile scheduling through cluster launch
                                    control ("Writing Mosaic GPU kernels with Pallas",
                                    "Cluster launch control"): the grid gets one
                                    cluster per list of tiles, and a unit that has
                                    done its list takes over the list of a cluster
                                    that has not started, so faster SMs do more
                                    tiles.  1: the persistent units keep their whole
                                    waves and each tile of a partial last wave is a
                                    list of its own (no effect when the tiles fill
                                    whole waves or fit in one); 2: every tile is a
                                    list.  Whole tiles only (overrides
                                    GEMM_OPT_STREAM_K).  0: the static persistent
                                    schedule.  -1 (default): 1 from six whole waves
                                    of tiles on (where it measured faster), else 0;
                                    0 on plans with GEMM_OPT_MAX_CTAS or
                                    GEMM_OPT_STREAM_K set                          */
    GEMM_OPT_FAIL_ENCODE = 10,   /* tests of the error path only: 1 = the driver's
                                    tensor-map encoder is replaced by a fake that
                                    rejects the output map, so runs on this plan
                                    return GEMM_ERR_DRIVER before any launch and
                                    leave C untouched; 0 (default) = off            */
    GEMM_OPT_CLOCK_LOG = 12,     /* measurement: keep a record of the SM clock of the
                                    last `value` launches (0..2^20; 0 = off, the
                                    default), read by gemm_plan_clock_log.  Setting it
                                    allocates (or frees) value × 16 bytes of device
                                    memory and waits for the device                  */
    GEMM_OPT_PDL = 13,           /* 1 (default): launch as a programmatic dependent of
                                    the kernel before it on the stream, so that this
                                    launch and its set-up (barriers, TMEM, first work
                                    item) overlap that kernel's end; every thread then
                                    waits for the earlier grids to complete before any
                                    access to A, B, C or the plan's device memory.  The
                                    kernel also signals its own dependents once its
                                    last tiles' loads and MMAs are issued.  A kernel
                                    launched after it without that attribute is
                                    ordered as usual.  0: plain stream order        */
    GEMM_OPT_SPLIT_K = 14,       /* K slices of a plain product with few tiles and a long
                                    K: -1 (default) = chosen per problem, 0 = never, or
                                    2, 4, 8, 16, 32 = that many where the problem allows
                                    it.  A split product runs its K slices as a batch
                                    of products over column slices of A and B, each
                                    writing an fp32 partial into the plan's stream-K
                                    workspace, then sums the partials in slice order
                                    (deterministic) and writes C.  Only for K-major
                                    operands, K a multiple of the k-block (64 16-bit or
                                    128 8-bit elements) divisible into slices of at
                                    least four k-blocks, every slice's tiles in one
                                    wave, M·N·slices floats within the workspace, and
                                    plans without stream-K or a CTA cap.  Split
                                    products of one plan are ordered one after another
                                    on the GPU, whatever their streams (an event);
                                    inside stream capture that ordering is left to the
                                    graph, so a plan whose split products are captured
                                    must not run others while the graph replays     */
    GEMM_OPT_VISIBLE_DEVICES = 11 /* GPUs the plan counts as visible to the process,
                                    1..1024 (0 = default: cudaGetDeviceCount at plan
                                    creation).  TMA multicast stays within one GPU's
                                    own memory, and the library uses it only when a
                                    single GPU is visible, so that no code of a
                                    process that may drive several GPUs multicasts;
                                    setting 2 or more here takes a one-GPU machine
                                    through that rule (tests).  A plan that runs with
                                    GEMM_OPT_MULTICAST = 1 returns GEMM_ERR_UNSUPPORTED
                                    for a value above 1                            */
} gemm_option_t;

/* Create a plan for `device` (-1 = the current device); it becomes the plan
 * gemm_run() uses on that device while it is the newest one alive.  Queries
 * the SM count and the resident cluster capacity, sets kernel attributes and
 * allocates the plan's device memory: a 16-byte status record and the
 * stream-K workspace (128 KB of fp32 partials per SM, about 19.5 MB on GB300,
 * plus a few KB of flags).  `flags` must be 0.  The caller owns the plan
 * and frees it with gemm_plan_destroy(). */
int gemm_plan_create(gemm_plan_t* plan, int device, unsigned flags);

/* Set a plan option (see gemm_option_t).  Not thread-safe with concurrent
 * runs on the same plan. */
int gemm_plan_set_option(gemm_plan_t plan, int option, int64_t value);

/* C = A·Bᵀ on `stream` with the most recently created plan of the current
 * device that is still alive (GEMM_ERR_NO_PLAN if none).  dtype: GEMM_BF16, GEMM_F16, GEMM_E4M3 or
 * GEMM_E5M2 (A and B);
 * out_dtype: GEMM_F32, GEMM_BF16 or GEMM_F16.  Asynchronous. */
int gemm_run(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
             int dtype, int out_dtype, void* stream);

/* Same, with an explicit plan.  The plan's device must be current. */
int gemm_plan_run(gemm_plan_t plan, const void* A, const void* B, void* C, int64_t M,
                  int64_t N, int64_t K, int dtype, int out_dtype, void* stream);

/* C = A·Bᵀ with the operand storage of `layout` (gemm_layout_t flags).
 * Rows of every operand must be 16-byte multiples: K for a K-major operand,
 * M (A) or N (B) for an MN-major one.  MN-major operands need 16-bit inputs
 * (GEMM_ERR_UNSUPPORTED for E4M3/E5M2).  With an MN-major B, a 4-CTA
 * multicast unit (GEMM_OPT_MULTICAST = 1) needs tile width 256
 * (GEMM_ERR_UNSUPPORTED if GEMM_OPT_TILE_N forces another); 1- and 2-CTA
 * units take every width.  Otherwise as gemm_plan_run. */
int gemm_plan_run_layout(gemm_plan_t plan, const void* A, const void* B, void* C, int64_t M, int64_t N,
                         int64_t K, int dtype, int out_dtype, int layout, void* stream);

/* A batch of products C_e = A_e·B_eᵀ, e < batch, in one persistent launch
 * over batch × tiles output tiles: A_e at A + e·stride_a, B_e at
 * B + e·stride_b, C_e at C + e·stride_c (strides in elements).  stride_a or
 * stride_b 0: every product reads the same A or B — the batched matmul with
 * a shared operand of "Chapter 7: Writing Custom Kernels with Pallas", §5.2
 * (vmap with in_axes=(0, None)).  Shapes, `layout` flags and their rules
 * as gemm_plan_run_layout, for every element.  With batch > 1: each stride
 * times its element size a multiple of 16 bytes (GEMM_ERR_UNSUPPORTED), and
 * no overlap: stride_c >= M·N, stride_a 0 or >= M·K, stride_b 0 or >= N·K
 * (GEMM_ERR_INVALID_ARG).  batch 0 is a no-op. */
int gemm_plan_run_batched(gemm_plan_t plan, const void* A, const void* B, void* C, int64_t batch, int64_t M,
                          int64_t N, int64_t K, int64_t stride_a, int64_t stride_b, int64_t stride_c, int dtype,
                          int out_dtype, int layout, void* stream);

/* End-to-end form for callers whose operands live in host memory: copies A
 * and B (host, ideally pinned) to device buffers the plan owns (grown on
 * demand and kept for reuse), runs the product, copies C back to host
 * memory, and synchronises `stream` before returning.  Copies and products
 * overlap on streams the plan owns (A and C in row chunks), ordered after
 * the work already on `stream`.  Same shape rules. */
int gemm_plan_run_host(gemm_plan_t plan, const void* A_host, const void* B_host, void* C_host,
                       int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, void* stream);

/* Read and clear the plan's device status word.  Synchronises the device.
 * *device_status receives GEMM_OK or the first device-side error code
 * recorded since the last call; after an error the stream-K flags are
 * reset too, so the plan can be used again. */
int gemm_plan_status(gemm_plan_t plan, int* device_status);

/* Number of CTAs the last run on this plan launched (for reports). */
int gemm_plan_last_grid(gemm_plan_t plan, int* ctas);

/* K slices of the last run on this plan (1: not split; see GEMM_OPT_SPLIT_K). */
int gemm_plan_last_split(gemm_plan_t plan, int* slices);

/* Tile width BN the last run on this plan used (for reports). */
int gemm_plan_last_tile_n(gemm_plan_t plan, int* tile_n);

/* Launch configuration of the last run on this plan (for reports): CTAs
 * launched, CTAs per work unit (1, 2 or 4), tile width, whole-tile waves and
 * the number of tiles split along K by the stream-K tail.  A run with a
 * dynamic work list reports its grid (one unit per list) and the whole
 * waves of the persistent units (0 when every tile is a list). */
int gemm_plan_last_launch(gemm_plan_t plan, int* ctas, int* ctas_per_unit, int* tile_n, int* dp_waves,
                          int* sk_tiles);

/* Clock log of the plan's launches since the last call (GEMM_OPT_CLOCK_LOG
 * must be set; GEMM_ERR_UNSUPPORTED otherwise): for each of the most recent
 * min(launches, option value, capacity) launches, oldest first, two words
 * go to host[2i] and host[2i+1]: the SM cycles (clock64) and the
 * nanoseconds (%globaltimer) between the entry and the exit of the launch's
 * first CTA.  cycles ÷ ns × 1000 is the SM clock in MHz the launch ran at.
 * *count receives the number of records copied; the log is then empty.
 * Launches that filled K = 0 or M/N = 0 problems record nothing.
 * Synchronises the device.  host: room for 2 × capacity words. */
int gemm_plan_clock_log(gemm_plan_t plan, uint64_t* host, int64_t capacity, int64_t* count);

/* Timeline of the last runs, for builds compiled with GEMM_TRACE (other
 * builds return GEMM_ERR_UNSUPPORTED after filling *ctas and *slots).  Copies
 * *ctas × *slots 64-bit words to `host` (at least that many bytes) and
 * clears the device buffer; synchronises the device.  Word s of CTA c is a
 * %globaltimer stamp in ns, a wait total in ns, or an SM cycle count (the
 * prologue steps and the MMA warp's per-tile stamps), per TraceSlot in the
 * kernel source. */
int gemm_plan_trace(gemm_plan_t plan, void* host, size_t bytes, int* ctas, int* slots);

/* Free the plan.  The caller must have synchronised every stream that still
 * runs work of this plan.  gemm_run() then uses the newest remaining plan of
 * the device, or returns GEMM_ERR_NO_PLAN if none is left. */
int gemm_plan_destroy(gemm_plan_t plan);

/* Allocation-free form of gemm_run(), for callers that may not allocate
 * device memory at all: services that hand all of HBM to their own pool at
 * start-up and forbid later allocations (a cudaMalloc would fail or carve
 * into memory the pool counts as its own), embedders whose device memory
 * belongs to another allocator that must account for every byte, and
 * latency-critical loops that cannot afford the device-wide synchronisation
 * a cudaFree implies.  No plan is needed and nothing is allocated, now or later (no
 * cudaMalloc, no cudaFree, no allocating library call): the kernel's only
 * scratch, its 16-byte status record, lives in a 256-byte static device
 * array that every GPU loading this library keeps until the process exits.
 * A, B, C and the layout rules are those of gemm_run(); the default
 * configuration (CTA pairs) is used.
 *   - The first call on a device sets up that device (looks up the array's
 *     device address, sets kernel attributes, queries capacity); make that
 *     first call before any stream capture.
 *   - Each call clears the status record on `stream` before launching.
 *     Every call on a device shares the array, so calls that overlap on the
 *     GPU (unordered streams) race on it.  This entry point never reads the
 *     record back: every device-side error -- a wait that outlived its bound
 *     (GEMM_ERR_TIMEOUT) and the kernel's own set-up checks (a shared-memory
 *     window not 1 KB aligned, GEMM_ERR_CUDA) -- goes unreported, and C is
 *     then undefined although the call returned GEMM_OK.  Callers that need
 *     those errors use the plan path and gemm_plan_status().
 *   - A scratch requirement beyond the array's 256 bytes is rejected with
 *     GEMM_ERR_UNSUPPORTED (the kernel needs 16 bytes whatever M, N, K).
 * The pages have no counterpart: this is a library integration entry point. */
int gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                     int dtype, int out_dtype, void* stream);

/* Tensor-core issue-rate probe (a measurement, not part of a product):
 * on the current device every SM holds one CTA (cta_pair = 1) or one CTA of
 * a pair (cta_pair = 2), and one thread per CTA (pair) issues
 * `mmas_per_sm` back-to-back tcgen05.mma of the GEMM kernel's shape --
 * 128×256 per CTA, K = 16 (dtype GEMM_BF16/GEMM_F16) or 32 (GEMM_E4M3/
 * GEMM_E5M2) -- from operand tiles already in shared memory: no loads, no
 * epilogue.  The ceiling a GEMM's K loop can reach, measured ("Optimizing
 * Blackwell Matrix Multiplication in Mojo (Part 2)" rates its kernels
 * against the tensor cores' peak).  Outputs, any of which may be NULL:
 * the dense FLOP per SM clock (median over CTAs, from the SM cycle
 * counter), the TFLOP/s of all SMs together (CUDA events around the
 * launch) and the SM clock in MHz during the stream (cycles ÷ %globaltimer
 * ns, median).  `mmas_per_sm`: a multiple of 4 in [4, 2^24].  Synchronous:
 * allocates and frees a few KB of device memory and waits for the device.
 * Errors: GEMM_ERR_INVALID_ARG, GEMM_ERR_NO_DEVICE, GEMM_ERR_CUDA,
 * GEMM_ERR_TIMEOUT (a completion wait ran out after 10 s). */
int gemm_probe_mma_rate(int dtype, int cta_pair, int64_t mmas_per_sm, double* flop_per_clk_per_sm,
                        double* tflops, double* sm_mhz);

/* The same probe with instructions of N = tile_n accumulator columns (a
 * tile width of the GEMM: 16..256 in steps of 16) instead of 256, so that
 * the tensor cores' own rate at a narrower tile can be told apart from the
 * cost of feeding that tile.  FLOP counts use tile_n.  Errors as above;
 * GEMM_ERR_INVALID_ARG for any other tile_n. */
int gemm_probe_mma_rate_n(int dtype, int cta_pair, int tile_n, int64_t mmas_per_sm, double* flop_per_clk_per_sm,
                          double* tflops, double* sm_mhz);

/* Static text for a status code. */
const char* gemm_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
