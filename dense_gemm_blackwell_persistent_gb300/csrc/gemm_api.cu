// gemm_api.cu -- host side of the library: argument checks, tensor-map
// construction, plan registry, launch of the persistent kernel, and the
// extern "C" entry points declared in include/gemm.h.
//
// The tensor map is the host-built descriptor of "Optimizing Blackwell
// Matrix Multiplication in Mojo (Part 2)", "Loading tiles into shared
// memory" (shape, strides, global address, box size and swizzle mode in one
// opaque block handed to the kernel).  It is encoded with the driver's
// cuTensorMapEncodeTiled, fetched at run time through the runtime's
// driver-entry-point query so the library does not link libcuda directly.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "kernel_table.h"
#include "launch_choice.h"

namespace {

using namespace gb300;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxExtent = (int64_t(1) << 31) - 1024;   // largest M, N or K accepted

std::mutex g_mu;
std::vector<gemm_plan*> g_plans[kMaxDevices];  // live plans per device, newest last
EncodeTiledFn g_encode = nullptr;

bool is_fp8(int dt) { return dt == GEMM_E4M3 || dt == GEMM_E5M2; }
int elem_bytes(int dt) { return dt == GEMM_F32 ? 4 : is_fp8(dt) ? 1 : 2; }
// K elements per k-block: one 128-byte swizzle row.
int64_t kblock_elems(int in_dtype) { return kBlockKBytes / elem_bytes(in_dtype); }

CUtensorMapDataType tma_dtype(int dt) {
    switch (dt) {
        case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case GEMM_E4M3:
        case GEMM_E5M2: return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // bytes moved as they are
        default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    }
}

int get_encoder(EncodeTiledFn* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_DRIVER;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return GEMM_OK;
}

// A batch of row-major matrices rows×cols (cols contiguous), `count`
// matrices `stride` elements apart, as a 3-D tensor map (cols, rows, batch);
// box = box_rows × box_cols of one matrix; zero fill outside the tensor.  A
// single matrix gets batch extent 1.  `fake_reject` (tests of the error
// path) replaces the driver's encoder by one that rejects the map.
int encode_3d(CUtensorMap* map, int dt, const void* ptr, uint64_t rows, uint64_t cols, uint64_t count,
              uint64_t stride, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle,
              CUtensorMapL2promotion promo, bool fake_reject = false, uint64_t pitch = 0) {
    EncodeTiledFn enc;
    int rc = get_encoder(&enc);
    if (rc != GEMM_OK) return rc;
    const uint64_t eb = (uint64_t)elem_bytes(dt);
    if (pitch == 0) pitch = cols;   // elements from one row to the next
    if (count <= 1) stride = rows * pitch;
    cuuint64_t dims[3] = {cols, rows, count < 1 ? 1 : count};
    cuuint64_t strides[2] = {pitch * eb, stride * eb};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fake_reject ? CUDA_ERROR_INVALID_VALUE
                             : enc(map, tma_dtype(dt), 3, const_cast<void*>(ptr), dims, strides, box, estr,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_DRIVER;
}

// A batch of products: `count` problems with A, B, C `sa`, `sb`, `sc`
// elements apart (0 for A or B: every problem uses the same matrix).  `lda`,
// `ldb`: elements from one row of a K-major A or B to the next, when larger
// than K (the K slices of a split product are column slices of A and B);
// 0 = K.
struct Batch {
    int64_t count = 1;
    int64_t sa = 0, sb = 0, sc = 0;
    int64_t lda = 0, ldb = 0;
};

// tcgen05 instruction descriptor: f32 accumulator, A and B K-major, M×N.
// Operand format field (bits 7-9 for A, 10-12 for B): kind::f16 reads
// 0 = f16, 1 = bf16; kind::f8f6f4 reads 0 = E4M3, 1 = E5M2.
uint32_t make_idesc(int in_dtype, int m, int n, int layout) {
    const uint32_t ab = (in_dtype == GEMM_BF16 || in_dtype == GEMM_E5M2) ? 1u : 0u;
    const uint32_t a_mn = (layout & GEMM_A_MN_MAJOR) ? 1u : 0u, b_mn = (layout & GEMM_B_MN_MAJOR) ? 1u : 0u;
    return (1u << 4)                   // accumulator format: f32
           | (ab << 7) | (ab << 10)    // A and B formats
           | (a_mn << 15) | (b_mn << 16)   // operand majors: 0 = K-major, 1 = MN-major
           | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// C = 0 for K == 0 (the empty sum): `count` matrices of `n16` 16-byte words,
// `stride16` words apart, in one launch.
__global__ void fill_zero_kernel(uint4* __restrict__ c, size_t n16, int64_t count, size_t stride16) {
    const size_t step = (size_t)gridDim.x * blockDim.x;
    for (int64_t e = 0; e < count; ++e) {
        uint4* m = c + (size_t)e * stride16;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += step)
            m[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// The reduction of a split product: C = Σ_s W_s, s = 0..S-1 in order (W_s
// the fp32 partial of K slice s, `slice` floats apart), converted to C's
// type (round to nearest even), four elements per thread.  Launched as a
// programmatic dependent of the slices' GEMM: it waits for that grid before
// reading the partials.
template <int kOut>
__global__ void splitk_reduce_kernel(const float4* __restrict__ w, void* __restrict__ c, size_t n4, size_t slice4,
                                     int slices) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t step = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += step) {
        float4 acc = __ldcg(w + i);
        for (int s = 1; s < slices; ++s) {
            const float4 v = __ldcg(w + (size_t)s * slice4 + i);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if constexpr (kOut == GEMM_F32) {
            reinterpret_cast<float4*>(c)[i] = acc;
        } else if constexpr (kOut == GEMM_BF16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            reinterpret_cast<uint2*>(c)[i] =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        } else {
            __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
            reinterpret_cast<uint2*>(c)[i] =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

struct gemm_plan {
    int device = 0;
    int sm_count = 0;
    int max_ctas[5] = {0, 0, 0, 0, 0};  // resident CTAs per unit size 1, 2, 4 (index by size)
    int pair = 0;                 // CTAs per MMA: 1, 2, or 0 = chosen per problem (launch_auto_pair)
    int multicast = -1;           // with pairs: share B across two pairs (1), never (0), auto (-1)
    int group_m = 0;
    int cap_ctas = 0;
    int tile_n = 0;               // 0 = 256
    int stream_k = 0;             // split the K work of a partial last wave (option)
    int dynamic = -1;             // run-time tile hand-out: 0 off, 1 the partial last wave, 2 every tile, -1 auto
    int64_t wait_limit_us = 0;    // bound on a kernel wait (0 = kWaitLimitNs)
    int stall_test = 0;           // tests of the timeout path only
    int fail_encode = 0;          // tests of the error path only: the encoder rejects every map
    int visible_devices = 1;      // GPUs the process sees (multicast only with one)
    int pdl = 1;                  // launch as a programmatic dependent of the stream's previous kernel
    int split_k = -1;             // K slices: -1 automatic (launch_split_k), 0 never, 2..32 asked for
    // Split products share the stream-K workspace: their runs are ordered
    // one after the other on the GPU, whatever stream they come from, by
    // this event (the last split product's reduction), under split_mu.
    std::mutex split_mu;
    cudaEvent_t split_ev = nullptr;
    float* d_partials = nullptr;  // stream-K workspace: one partial-tile slot per unit
    int* d_flags = nullptr;       // stream-K "partial published" flags
    unsigned long long* d_trace = nullptr;  // GEMM_TRACE builds: kTraceSlots words per CTA
    int* d_status = nullptr;      // 4 ints, see Params::status
    // Clock log (GEMM_OPT_CLOCK_LOG): a ring of clock_cap records of two
    // 64-bit words (SM cycles, ns of CTA 0's lifetime), one per launch;
    // clock_next counts the launches since the log was last read.
    unsigned long long* d_clock = nullptr;
    int64_t clock_cap = 0;
    std::atomic<int64_t> clock_next{0};
    // The last run's launch shape, for reports.  Every run writes it, so
    // runs from several host threads at once take rec_mu for it.
    std::mutex rec_mu;
    int last_grid = 0;
    int last_tile_n = 0;
    int last_unit = 0;
    int last_dp_waves = 0;
    int last_sk_tiles = 0;
    int last_split = 1;
    std::mutex host_mu;           // serialises gemm_plan_run_host's buffers
    void* hbuf[3] = {nullptr, nullptr, nullptr};
    size_t hcap[3] = {0, 0, 0};
    // gemm_plan_run_host's pipeline (created on first use): streams for the
    // copies in (B, then A), for the products and for the copies of C back;
    // events: start, B resident, and per row chunk A resident / C computed.
    cudaStream_t hstream[3] = {nullptr, nullptr, nullptr};
    cudaEvent_t hev_start = nullptr, hev_b = nullptr, hev_done = nullptr;
    cudaEvent_t hev_a[8] = {}, hev_c[8] = {};
};

namespace {

// Pure host checks, no CUDA call: shared by every run entry point.
int validate(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype,
             int layout = 0) {
    if (dtype != GEMM_BF16 && dtype != GEMM_F16 && !is_fp8(dtype)) return GEMM_ERR_INVALID_ARG;
    if (layout < 0 || layout > (GEMM_A_MN_MAJOR | GEMM_B_MN_MAJOR)) return GEMM_ERR_INVALID_ARG;
    if (out_dtype != GEMM_BF16 && out_dtype != GEMM_F16 && out_dtype != GEMM_F32) return GEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    // The kernel's tile coordinates are 32-bit and run up to one tile past
    // the last row, column or k-block: keep a margin below 2^31.
    if (M > kMaxExtent || N > kMaxExtent || K > kMaxExtent) return GEMM_ERR_UNSUPPORTED;
    if (C == nullptr) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0) return GEMM_ERR_MISALIGNED;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15u) != 0 || (reinterpret_cast<uintptr_t>(B) & 15u) != 0))
        return GEMM_ERR_MISALIGNED;
    if (layout != 0 && is_fp8(dtype)) return GEMM_ERR_UNSUPPORTED;   // MN-major: 16-bit inputs only
    // each operand's rows (K-major: K elements; MN-major: M or N) in 16-byte multiples
    const int64_t ib = elem_bytes(dtype);
    if (((layout & GEMM_A_MN_MAJOR) ? M * ib : K * ib) % 16 != 0) return GEMM_ERR_UNSUPPORTED;
    if (((layout & GEMM_B_MN_MAJOR) ? N * ib : K * ib) % 16 != 0) return GEMM_ERR_UNSUPPORTED;
    if ((N * elem_bytes(out_dtype)) % 16 != 0) return GEMM_ERR_UNSUPPORTED;
    return GEMM_OK;
}

// The operands of a run on `device`: that device must be current, and A, B
// (when K > 0) and C must be device memory of that device.  Host memory
// (pinned or not), managed memory and another GPU's memory are refused
// before anything is encoded or launched: the tensor maps would otherwise
// hand the TMA unit addresses it must not read through, and the 4-CTA unit's
// multicast copies are meant for this GPU's own memory only.  Host buffers
// go through gemm_plan_run_host.
int check_operands(int device, const void* A, const void* B, const void* C, int64_t K) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (cur != device) return GEMM_ERR_INVALID_ARG;
    const void* ptrs[3] = {C, A, B};
    for (int i = 0; i < (K > 0 ? 3 : 1); ++i) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_INVALID_ARG;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != device) return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

// CTAs the device keeps resident with the largest unit size that fits
// best; the plan's per-CTA buffers (stream-K workspace, trace) are sized
// for this many.
int max_resident_ctas(const gemm_plan* plan) {
    return std::max(plan->max_ctas[1], std::max(plan->max_ctas[2], plan->max_ctas[4]));
}

// The launch shape: the decisions themselves live in launch_choice.h
// (plain C++, also run by the CPU tests); these wrappers feed them the
// plan's options and the resident-unit counts queried on the device.
constexpr bool same_widths(int i = 0) {
    return i == kNumTileWidths || (kLaunchWidths[i] == kTileWidths[i] && same_widths(i + 1));
}
static_assert(kLaunchTileWidths == kNumTileWidths && same_widths(), "tile widths: launch choice and kernel table agree");
static_assert(kLaunchRowsPerCta == kRowsPerCta && kLaunchMnBox == kMnBoxElems, "launch choice and kernel agree");
static_assert(kErrTimeout == GEMM_ERR_TIMEOUT && kErrCuda == GEMM_ERR_CUDA && kErrInternal == GEMM_ERR_INTERNAL,
              "device-side status codes are the header's");

// CTAs per MMA for this problem: the plan's choice, or automatic (a forced
// multicast unit is made of pairs).
int cta_pair(const gemm_plan* plan, int64_t M, int64_t N, int64_t batch) {
    if (plan->pair > 0) return plan->pair;
    if (plan->multicast == 1) return 2;
    return launch_auto_pair(M, N, batch, plan->max_ctas[2] / 2, plan->max_ctas[1]);
}

int unit_ctas(const gemm_plan* plan, int pair, int64_t K, int in_dtype, int layout) {
    return launch_unit_ctas(pair, plan->multicast, plan->visible_devices, K, elem_bytes(in_dtype), layout);
}

// Resident units a launch may use.
int resident_units(const gemm_plan* plan, int cluster) {
    int units = plan->max_ctas[cluster] / cluster;
    if (plan->cap_ctas > 0) units = std::min(units, std::max(1, plan->cap_ctas / cluster));
    return std::max(1, units);
}

int choose_tile_n(const gemm_plan* plan, int64_t M, int64_t N, int cluster, int layout, int64_t batch = 1) {
    return launch_tile_n(plan->tile_n, M, N, cluster, layout, batch, resident_units(plan, cluster));
}

bool dynamic_lists(const gemm_plan* plan, int64_t tiles, int64_t resident, int* units, int* waves) {
    return launch_dynamic_lists(plan->dynamic, plan->cap_ctas > 0, plan->stream_k != 0, tiles, resident, units,
                                waves);
}

int launch_split(gemm_plan* plan, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                 int dtype, int out_dtype, cudaStream_t stream, int slices, int pair);
size_t partials_bytes(const gemm_plan* plan);

int launch(gemm_plan* plan, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype,
           int out_dtype, cudaStream_t stream, int layout = 0, const Batch& batch = Batch(), int pair_forced = 0) {
    if (K == 0) {
        // N·out_bytes and, for batches, the C stride in bytes are 16-byte multiples (checked by the callers)
        const size_t n16 = (size_t)M * (size_t)N * elem_bytes(out_dtype) / 16;
        const size_t stride16 = batch.count > 1 ? (size_t)batch.sc * elem_bytes(out_dtype) / 16 : 0;
        const int blocks = (int)std::min<size_t>((n16 + 255) / 256, (size_t)plan->sm_count * 8);
        fill_zero_kernel<<<std::max(blocks, 1), 256, 0, stream>>>(reinterpret_cast<uint4*>(C), n16, batch.count,
                                                                  stride16);
        return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    const int pair = pair_forced > 0 ? pair_forced : cta_pair(plan, M, N, batch.count);
    if (pair == 2 && plan->multicast == 1 && plan->visible_devices != 1) return GEMM_ERR_UNSUPPORTED;
    const int cluster = unit_ctas(plan, pair, K, dtype, layout);
    const int bn = choose_tile_n(plan, M, N, cluster, layout, batch.count);
    if (bn == 0) return GEMM_ERR_UNSUPPORTED;
    // Few tiles and a long K: split K over more units (one plain product,
    // K-major operands, the workspace free of stream-K).
    if (batch.count == 1 && layout == 0 && plan->split_k != 0 && !plan->stream_k && plan->d_partials != nullptr &&
        plan->cap_ctas == 0) {
        const int64_t tile_m = (int64_t)kRowsPerCta * cluster;
        const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + bn - 1) / bn);
        const int64_t kbe = kblock_elems(dtype);
        const int64_t kb = (K + kbe - 1) / kbe;
        const int slices = K % kbe == 0 ? launch_split_k(plan->split_k, tiles, resident_units(plan, cluster), kb,
                                                         M * N, (int64_t)(partials_bytes(plan) / sizeof(float)))
                                        : 1;
        if (slices > 1) return launch_split(plan, A, B, C, M, N, K, dtype, out_dtype, stream, slices, pair);
    }
    const bool pad = (layout & GEMM_B_MN_MAJOR) && !launch_b_boxes_exact(bn, cluster);
    const KernelInfo ki = kernel_info(cluster, bn, out_dtype, is_fp8(dtype) ? 1 : 0, pad);
    if (ki.fn == nullptr) return GEMM_ERR_INVALID_ARG;
    const int tile_m = kRowsPerCta * cluster;
    Params p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.tiles_m = (int)((M + tile_m - 1) / tile_m);
    p.tiles_n = (int)((N + bn - 1) / bn);
    const int64_t kbe = kblock_elems(dtype);
    p.k_blocks = (int)((K + kbe - 1) / kbe);
    // the tile space (batch elements × tiles) must fit the kernel's 32-bit tile indices
    const int64_t tiles_per_batch = (int64_t)p.tiles_m * p.tiles_n;
    if (tiles_per_batch >= (int64_t(1) << 31) || tiles_per_batch * batch.count >= (int64_t(1) << 31))
        return GEMM_ERR_UNSUPPORTED;
    p.tiles_per_batch = (int)tiles_per_batch;
    p.num_tiles = (int)(p.tiles_per_batch * batch.count);
    p.a_batched = batch.count > 1 && batch.sa != 0;
    p.b_batched = batch.count > 1 && batch.sb != 0;
    p.group_m = launch_group_m(plan->group_m, p.tiles_m, M * K * elem_bytes(dtype));
    p.fd_batch = make_fastdiv((uint32_t)p.tiles_per_batch);
    p.fd_group = make_fastdiv((uint32_t)(p.group_m * p.tiles_n));
    p.fd_gm = make_fastdiv((uint32_t)p.group_m);
    p.fd_gm_last = make_fastdiv((uint32_t)(p.tiles_m % p.group_m != 0 ? p.tiles_m % p.group_m : p.group_m));
    p.idesc = make_idesc(dtype, kRowsPerCta * pair, bn, layout);   // one MMA covers a pair's 256 rows
    p.a_mn = (layout & GEMM_A_MN_MAJOR) ? 1 : 0;
    p.b_mn = (layout & GEMM_B_MN_MAJOR) ? 1 : 0;
    p.status = plan->d_status;
    // Stream-K spreads a partial last wave over every resident unit; with
    // whole tiles only, never launch more units than tiles.  A dynamic work
    // list launches one cluster per list (clusters that do not start are
    // cancelled by running ones, which do their lists).
    const int resident = resident_units(plan, cluster);
    int dyn_units = 0, dyn_waves = 0;
    bool dyn = dynamic_lists(plan, p.num_tiles, resident, &dyn_units, &dyn_waves);
    // one cluster per list: keep the grid within the launch limit (x < 2^31), else stay static
    if (dyn && (int64_t)dyn_list_count(p.num_tiles, dyn_units, dyn_waves) * cluster >= (int64_t(1) << 31))
        dyn = false;
    const bool sk = !dyn && plan->stream_k && plan->d_partials != nullptr && plan->d_flags != nullptr;
    p.sched = make_schedule(p.num_tiles, resident, p.k_blocks, sk);
    p.dynamic = dyn ? 1 : 0;
    p.dyn_units = dyn_units;
    p.dyn_waves = dyn_waves;
    p.partials = plan->d_partials;
    p.flags = plan->d_flags;
    p.wait_limit_ns = plan->wait_limit_us > 0 ? (unsigned long long)plan->wait_limit_us * 1000ull : kWaitLimitNs;
    p.stall_test = plan->stall_test;
    p.trace = plan->d_trace;
    p.trace_ctas = max_resident_ctas(plan);
    p.clock_rec = nullptr;

    CUtensorMap tmA, tmB, tmC;
    // K-major operand: rows of K, box {one 128-byte row of K, rows}.  MN-major
    // (A stored K×M, B stored K×N): rows of M or N, box {64 elements, the
    // k-block's K rows}, several boxes per stage.
    // L2 promotion: a miss brings 256 bytes, i.e. also the row's next
    // k-block, except for A when its rows are not a multiple of 128 bytes
    // (each box row then straddles two lines); there 128-byte promotion
    // measured 4000×4000×5000 106.8 → 98.6 µs and 8000×8000×5000 399 → 376
    // (4000×3000×5000 level), while on aligned rows 256 bytes is faster
    // (1024×4096×4096: 28.7 vs 29.7 µs).  B keeps 256 bytes either way.
    const int64_t a_pitch = ((layout & GEMM_A_MN_MAJOR) ? M : (batch.lda > 0 ? batch.lda : K)) * elem_bytes(dtype);
    const CUtensorMapL2promotion promo_a =
        a_pitch % 128 != 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    const uint64_t na = p.a_batched ? (uint64_t)batch.count : 1, nb = p.b_batched ? (uint64_t)batch.count : 1;
    int rc = (layout & GEMM_A_MN_MAJOR)
                 ? encode_3d(&tmA, dtype, A, (uint64_t)K, (uint64_t)M, na, (uint64_t)batch.sa, (uint32_t)kbe,
                             kMnBoxElems, CU_TENSOR_MAP_SWIZZLE_128B, promo_a)
                 : encode_3d(&tmA, dtype, A, (uint64_t)M, (uint64_t)K, na, (uint64_t)batch.sa, kRowsPerCta,
                             (uint32_t)kbe, CU_TENSOR_MAP_SWIZZLE_128B, promo_a, false, (uint64_t)batch.lda);
    if (rc == GEMM_OK)
        rc = (layout & GEMM_B_MN_MAJOR)
                 ? encode_3d(&tmB, dtype, B, (uint64_t)K, (uint64_t)N, nb, (uint64_t)batch.sb, (uint32_t)kbe,
                             kMnBoxElems, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
                 : encode_3d(&tmB, dtype, B, (uint64_t)N, (uint64_t)K, nb, (uint64_t)batch.sb,
                             (uint32_t)(bn / cluster), (uint32_t)kbe, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, false, (uint64_t)batch.ldb);
    // C: 32-row × 32-column store boxes; 128-byte rows (fp32) or 64-byte rows (16-bit)
    if (rc == GEMM_OK)
        rc = encode_3d(&tmC, out_dtype, C, (uint64_t)M, (uint64_t)N, (uint64_t)batch.count, (uint64_t)batch.sc, 32,
                       kChunkCols, out_dtype == GEMM_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                       CU_TENSOR_MAP_L2_PROMOTION_NONE, plan->fail_encode != 0);
    if (rc != GEMM_OK) return rc;

    // clusters launched: the static schedule's units, or one per dynamic list
    const int units = dyn ? dyn_list_count(p.num_tiles, dyn_units, dyn_waves) : p.sched.units;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * cluster), 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)ki.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the grid may be scheduled before the
    // stream's previous kernel has finished, so that its launch and set-up
    // overlap that kernel's end; the kernel waits (griddepcontrol.wait) for
    // the previous grids before touching global memory.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan->pdl ? 2 : 1;
    if (plan->d_clock != nullptr) {
        const int64_t slot = plan->clock_next.fetch_add(1) % plan->clock_cap;
        p.clock_rec = plan->d_clock + 2 * slot;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, ki.fn, tmA, tmB, tmC, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(plan->rec_mu);
    plan->last_grid = units * cluster;
    plan->last_tile_n = bn;
    plan->last_unit = cluster;
    plan->last_dp_waves = dyn ? (dyn_units == p.num_tiles ? 0 : dyn_waves) : p.sched.dp_waves;
    plan->last_sk_tiles = p.sched.sk_tiles;
    plan->last_split = 1;
    return GEMM_OK;
}

// A split product: the K slices are a batch of `slices` products over column
// slices of A and B (K / slices columns each, rows still K apart), each
// writing its fp32 partial into the plan's workspace, on units of `pair` CTAs
// per MMA as the unsplit product would use; then the reduction sums the
// partials in slice order into C.  Split products of one plan share the
// workspace, so each waits on the GPU for the previous one's reduction
// (plan->split_ev) unless the stream is being captured into a graph.
int launch_split(gemm_plan* plan, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                 int dtype, int out_dtype, cudaStream_t stream, int slices, int pair) {
    std::lock_guard<std::mutex> lk(plan->split_mu);
    if (plan->split_ev == nullptr &&
        cudaEventCreateWithFlags(&plan->split_ev, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        plan->split_ev = nullptr;
        return GEMM_ERR_CUDA;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    const bool ordered = cap == cudaStreamCaptureStatusNone;
    if (ordered && cudaStreamWaitEvent(stream, plan->split_ev, 0) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    Batch bt;
    bt.count = slices;
    bt.sa = bt.sb = K / slices;
    bt.sc = M * N;
    bt.lda = bt.ldb = K;
    int rc = launch(plan, A, B, plan->d_partials, M, N, K / slices, dtype, GEMM_F32, stream, 0, bt, pair);
    if (rc != GEMM_OK) return rc;
    const size_t n4 = (size_t)M * (size_t)N / 4;
    const int blocks = (int)std::max<size_t>(1, std::min<size_t>((n4 + 255) / 256, (size_t)plan->sm_count * 4));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan->pdl ? 1 : 0;
    const float4* w = reinterpret_cast<const float4*>(plan->d_partials);
    cudaError_t e;
    if (out_dtype == GEMM_F32)
        e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<GEMM_F32>, w, C, n4, n4, slices);
    else if (out_dtype == GEMM_BF16)
        e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<GEMM_BF16>, w, C, n4, n4, slices);
    else
        e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<GEMM_F16>, w, C, n4, n4, slices);
    if (e != cudaSuccess || (ordered && cudaEventRecord(plan->split_ev, stream) != cudaSuccess)) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lr(plan->rec_mu);
    plan->last_split = slices;
    return GEMM_OK;
}

// One partial slot per unit: 4 epilogue warps × 32 rows × 256 fp32 per CTA.
size_t partials_bytes(const gemm_plan* plan) {
    const int ctas = max_resident_ctas(plan);
    return (size_t)ctas * 4 * kPartialFloats * sizeof(float);
}
// One flag per (split tile, CTA of the unit, epilogue warp); the stream-K
// part has fewer than twice as many tiles as units.
size_t flags_bytes(const gemm_plan* plan) {
    const int ctas = max_resident_ctas(plan);
    return (size_t)ctas * 2 * 4 * sizeof(int);
}

size_t trace_bytes(const gemm_plan* plan) {
    const int ctas = max_resident_ctas(plan);
    return (size_t)ctas * kTraceSlots * sizeof(unsigned long long);
}

int query_capacity(gemm_plan* plan, int cluster) {
    int max_smem = 0;
    KernelFn probe = nullptr;
    for (int v = 0; v < 9; ++v) {   // output type × (operand width, or the padded MN-major-B form)
        for (int i = 0; i < kNumTileWidths; ++i) {
            const KernelInfo ki = kernel_info(cluster, kTileWidths[i], v % 3, v / 3 == 1 ? 1 : 0, v / 3 == 2);
            if (ki.fn == nullptr) continue;
            if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem_bytes) !=
                cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            if (ki.smem_bytes > max_smem) {
                max_smem = ki.smem_bytes;
                probe = ki.fn;
            }
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(plan->sm_count / cluster * cluster), 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)max_smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (probe == nullptr || cudaOccupancyMaxActiveClusters(&clusters, probe, &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        clusters = plan->sm_count / cluster;  // one CTA per SM is what the shared-memory budget allows
    }
    plan->max_ctas[cluster] = clusters * cluster;
    return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_plan_create(gemm_plan_t* out, int device, unsigned flags) {
    if (out == nullptr || flags != 0u) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (device < 0 && cudaGetDevice(&device) != cudaSuccess) return GEMM_ERR_CUDA;
    if (device >= count || device >= kMaxDevices) return GEMM_ERR_INVALID_ARG;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_NO_DEVICE;  // built for sm_103a only
    int prev = 0;
    cudaGetDevice(&prev);
    if (cudaSetDevice(device) != cudaSuccess) return GEMM_ERR_CUDA;
    gemm_plan* plan = new (std::nothrow) gemm_plan();
    if (!plan) return GEMM_ERR_CUDA;
    plan->device = device;
    plan->sm_count = prop.multiProcessorCount;
    plan->visible_devices = count;
    int rc = query_capacity(plan, 1);
    if (rc == GEMM_OK) rc = query_capacity(plan, 2);
    if (rc == GEMM_OK) rc = query_capacity(plan, 4);
    if (rc == GEMM_OK && cudaMalloc(&plan->d_status, 4 * sizeof(int)) != cudaSuccess) rc = GEMM_ERR_CUDA;
    if (rc == GEMM_OK && cudaMemset(plan->d_status, 0, 4 * sizeof(int)) != cudaSuccess) rc = GEMM_ERR_CUDA;
    if (rc == GEMM_OK && cudaMalloc(&plan->d_partials, partials_bytes(plan)) != cudaSuccess) rc = GEMM_ERR_CUDA;
    if (rc == GEMM_OK && cudaMalloc(&plan->d_flags, flags_bytes(plan)) != cudaSuccess) rc = GEMM_ERR_CUDA;
    if (rc == GEMM_OK && cudaMemset(plan->d_flags, 0, flags_bytes(plan)) != cudaSuccess) rc = GEMM_ERR_CUDA;
#ifdef GEMM_TRACE
    if (rc == GEMM_OK && cudaMalloc(&plan->d_trace, trace_bytes(plan)) != cudaSuccess) rc = GEMM_ERR_CUDA;
    if (rc == GEMM_OK && cudaMemset(plan->d_trace, 0, trace_bytes(plan)) != cudaSuccess) rc = GEMM_ERR_CUDA;
#endif
    if (rc != GEMM_OK) {
        cudaGetLastError();
        if (plan->d_status) cudaFree(plan->d_status);
        if (plan->d_partials) cudaFree(plan->d_partials);
        if (plan->d_flags) cudaFree(plan->d_flags);
        delete plan;
        cudaSetDevice(prev);
        return rc;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_plans[device].push_back(plan);
    }
    cudaSetDevice(prev);
    *out = plan;
    return GEMM_OK;
}

int gemm_plan_set_option(gemm_plan_t plan, int option, int64_t value) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    switch (option) {
        case GEMM_OPT_CTA_PAIR:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            plan->pair = (int)value;
            return GEMM_OK;
        case GEMM_OPT_GROUP_M:
            if (value < 0 || value > (1 << 20)) return GEMM_ERR_INVALID_ARG;
            plan->group_m = (int)value;
            return GEMM_OK;
        case GEMM_OPT_MAX_CTAS:
            if (value < 0 || value > (1 << 20)) return GEMM_ERR_INVALID_ARG;
            plan->cap_ctas = (int)value;
            return GEMM_OK;
        case GEMM_OPT_MULTICAST:
            if (value < -1 || value > 1) return GEMM_ERR_INVALID_ARG;
            plan->multicast = (int)value;
            return GEMM_OK;
        case GEMM_OPT_STREAM_K:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            plan->stream_k = (int)value;
            return GEMM_OK;
        case GEMM_OPT_WAIT_LIMIT_US:
            if (value < 0 || value > 60000000) return GEMM_ERR_INVALID_ARG;
            plan->wait_limit_us = value;
            return GEMM_OK;
        case GEMM_OPT_STALL_TEST:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            plan->stall_test = (int)value;
            return GEMM_OK;
        case GEMM_OPT_DYNAMIC:
            if (value < -1 || value > 2) return GEMM_ERR_INVALID_ARG;
            plan->dynamic = (int)value;
            return GEMM_OK;
        case GEMM_OPT_FAIL_ENCODE:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            plan->fail_encode = (int)value;
            return GEMM_OK;
        case GEMM_OPT_VISIBLE_DEVICES: {
            if (value < 0 || value > 1024) return GEMM_ERR_INVALID_ARG;
            int n = (int)value;
            if (n == 0 && cudaGetDeviceCount(&n) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            plan->visible_devices = n;
            return GEMM_OK;
        }
        case GEMM_OPT_SPLIT_K:
            if (value != -1 && value != 0 && value != 2 && value != 4 && value != 8 && value != 16 && value != 32)
                return GEMM_ERR_INVALID_ARG;
            plan->split_k = (int)value;
            return GEMM_OK;
        case GEMM_OPT_PDL:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            plan->pdl = (int)value;
            return GEMM_OK;
        case GEMM_OPT_CLOCK_LOG: {
            if (value < 0 || value > (1 << 20)) return GEMM_ERR_INVALID_ARG;
            int prev = 0;
            cudaGetDevice(&prev);
            if (cudaSetDevice(plan->device) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            int rc = GEMM_OK;
            if (plan->d_clock) {
                cudaFree(plan->d_clock);   // waits for the device: no launch still writes it
                plan->d_clock = nullptr;
            }
            plan->clock_cap = 0;
            plan->clock_next = 0;
            if (value > 0) {
                const size_t bytes = (size_t)value * 2 * sizeof(unsigned long long);
                if (cudaMalloc(&plan->d_clock, bytes) != cudaSuccess ||
                    cudaMemset(plan->d_clock, 0, bytes) != cudaSuccess) {
                    cudaGetLastError();
                    if (plan->d_clock) cudaFree(plan->d_clock);
                    plan->d_clock = nullptr;
                    rc = GEMM_ERR_CUDA;
                } else {
                    plan->clock_cap = value;
                }
            }
            cudaSetDevice(prev);
            return rc;
        }
        case GEMM_OPT_TILE_N: {
            if (value == 0) {
                plan->tile_n = 0;
                return GEMM_OK;
            }
            for (int i = 0; i < kNumTileWidths; ++i)
                if (value == kTileWidths[i]) {
                    plan->tile_n = (int)value;
                    return GEMM_OK;
                }
            return GEMM_ERR_INVALID_ARG;
        }
        default: return GEMM_ERR_INVALID_ARG;
    }
}

int gemm_plan_run(gemm_plan_t plan, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                  int dtype, int out_dtype, void* stream) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    int rc = validate(A, B, C, M, N, K, dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    rc = check_operands(plan->device, A, B, C, K);
    if (rc != GEMM_OK) return rc;
    return launch(plan, A, B, C, M, N, K, dtype, out_dtype, static_cast<cudaStream_t>(stream));
}

int gemm_plan_run_layout(gemm_plan_t plan, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         int dtype, int out_dtype, int layout, void* stream) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    int rc = validate(A, B, C, M, N, K, dtype, out_dtype, layout);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    rc = check_operands(plan->device, A, B, C, K);
    if (rc != GEMM_OK) return rc;
    return launch(plan, A, B, C, M, N, K, dtype, out_dtype, static_cast<cudaStream_t>(stream), layout);
}

int gemm_plan_run_batched(gemm_plan_t plan, const void* A, const void* B, void* C, int64_t batch, int64_t M,
                          int64_t N, int64_t K, int64_t stride_a, int64_t stride_b, int64_t stride_c, int dtype,
                          int out_dtype, int layout, void* stream) {
    if (!plan || batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0) return GEMM_ERR_INVALID_ARG;
    int rc = validate(A, B, C, M, N, K, dtype, out_dtype, layout);
    if (rc != GEMM_OK || M == 0 || N == 0 || batch == 0) return rc;
    if (batch > 1) {
        // batch strides: 16-byte multiples (TMA), and no element shared by two outputs
        const int64_t ib = elem_bytes(dtype), ob = elem_bytes(out_dtype);
        if ((stride_a * ib) % 16 != 0 || (stride_b * ib) % 16 != 0 || (stride_c * ob) % 16 != 0)
            return GEMM_ERR_UNSUPPORTED;
        if (stride_c < M * N || (stride_a != 0 && stride_a < M * K) || (stride_b != 0 && stride_b < N * K))
            return GEMM_ERR_INVALID_ARG;
    }
    rc = check_operands(plan->device, A, B, C, K);
    if (rc != GEMM_OK) return rc;
    Batch bt;
    bt.count = batch;
    bt.sa = stride_a;
    bt.sb = stride_b;
    bt.sc = stride_c;
    return launch(plan, A, B, C, M, N, K, dtype, out_dtype, static_cast<cudaStream_t>(stream), layout, bt);
}

int gemm_run(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype,
             void* stream) {
    int rc = validate(A, B, C, M, N, K, dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    gemm_plan* plan = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (dev >= 0 && dev < kMaxDevices && !g_plans[dev].empty()) plan = g_plans[dev].back();
    }
    if (!plan) return GEMM_ERR_NO_PLAN;
    rc = check_operands(plan->device, A, B, C, K);
    if (rc != GEMM_OK) return rc;
    return launch(plan, A, B, C, M, N, K, dtype, out_dtype, static_cast<cudaStream_t>(stream));
}

// Streams and events of gemm_plan_run_host's pipeline, created on first use
// (the caller holds host_mu).
bool host_pipeline_ready(gemm_plan* plan) {
    if (plan->hstream[0]) return true;
    bool ok = true;
    for (int i = 0; i < 3 && ok; ++i) ok = cudaStreamCreateWithFlags(&plan->hstream[i], cudaStreamNonBlocking) == cudaSuccess;
    cudaEvent_t* evs[3] = {&plan->hev_start, &plan->hev_b, &plan->hev_done};
    for (int i = 0; i < 3 && ok; ++i) ok = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 8 && ok; ++i)
        ok = cudaEventCreateWithFlags(&plan->hev_a[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&plan->hev_c[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        for (int i = 0; i < 3; ++i)
            if (plan->hstream[i]) cudaStreamDestroy(plan->hstream[i]);
        for (int i = 0; i < 3; ++i) plan->hstream[i] = nullptr;
    }
    return ok;
}

int gemm_plan_run_host(gemm_plan_t plan, const void* A_host, const void* B_host, void* C_host, int64_t M,
                       int64_t N, int64_t K, int dtype, int out_dtype, void* stream) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    int rc = validate(A_host, B_host, C_host, M, N, K, dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (cur != plan->device) return GEMM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes[3] = {(size_t)M * (size_t)K * elem_bytes(dtype), (size_t)N * (size_t)K * elem_bytes(dtype),
                             (size_t)M * (size_t)N * (size_t)elem_bytes(out_dtype)};
    std::lock_guard<std::mutex> lk(plan->host_mu);
    for (int i = 0; i < 3; ++i) {
        if (bytes[i] > plan->hcap[i]) {
            if (plan->hbuf[i]) {
                cudaStreamSynchronize(s);
                cudaFree(plan->hbuf[i]);
                plan->hbuf[i] = nullptr;
                plan->hcap[i] = 0;
            }
            if (cudaMalloc(&plan->hbuf[i], bytes[i]) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            plan->hcap[i] = bytes[i];
        }
    }
    if (!host_pipeline_ready(plan)) return GEMM_ERR_CUDA;
    // The pipeline: B, then A in row chunks, on one copy stream (every
    // chunk's product needs all of B, so B goes first); the product of each
    // chunk starts as soon as its rows are resident, and its rows of C go
    // back on another stream while later chunks are copied and computed.
    // Chunks are whole 256-row tiles (a CTA pair's tile height).  One chunk
    // per 1024 rows, at most 8, and at least two from 512 rows on: smaller
    // chunks shorten the tail (the last chunk's product and copy back), but
    // below ~1024 rows a chunk's product no longer fills a wave of tiles and
    // the extra copies and launches cost more than the tail saves (4096³:
    // 8 chunks of 512 rows 293 vs 300 TFLOP/s end to end), except where one
    // chunk would be the whole product (1024×4096×4096: 2 chunks 126 vs 118).  The host link bounds it: measured on
    // GB300 ~208 GB/s in and ~192 GB/s out one way at a time, ~165 GB/s each
    // way at once, the same whether the copy engines or SM loads and stores
    // move the bytes; 4096³ bf16 runs at ~300 TFLOP/s end to end (234
    // unpipelined), 8192³ at ~675.
    int64_t want = std::min<int64_t>(8, M / 1024);
    if (want < 2) want = M >= 512 ? 2 : 1;
    int64_t rows = ((M + want - 1) / want + 255) / 256 * 256;
    const int nch = (int)((M + rows - 1) / rows);
    const size_t a_row_bytes = (size_t)K * elem_bytes(dtype), c_row_bytes = (size_t)N * elem_bytes(out_dtype);
    cudaStream_t sA = plan->hstream[0], sX = plan->hstream[1], sC = plan->hstream[2];   // copies in, products, copies out
    bool ok = cudaEventRecord(plan->hev_start, s) == cudaSuccess;   // after the caller's earlier work
    for (int i = 0; i < 3 && ok; ++i) ok = cudaStreamWaitEvent(plan->hstream[i], plan->hev_start, 0) == cudaSuccess;
    if (ok && K > 0)
        ok = cudaMemcpyAsync(plan->hbuf[1], B_host, bytes[1], cudaMemcpyHostToDevice, sA) == cudaSuccess &&
             cudaEventRecord(plan->hev_b, sA) == cudaSuccess && cudaStreamWaitEvent(sX, plan->hev_b, 0) == cudaSuccess;
    for (int c = 0; c < nch && ok; ++c) {
        const int64_t r0 = c * rows, mc = std::min(rows, M - r0);
        const char* a_src = static_cast<const char*>(A_host) + (size_t)r0 * a_row_bytes;
        char* a_dev = static_cast<char*>(plan->hbuf[0]) + (size_t)r0 * a_row_bytes;
        char* c_dev = static_cast<char*>(plan->hbuf[2]) + (size_t)r0 * c_row_bytes;
        if (K > 0)
            ok = cudaMemcpyAsync(a_dev, a_src, (size_t)mc * a_row_bytes, cudaMemcpyHostToDevice, sA) == cudaSuccess &&
                 cudaEventRecord(plan->hev_a[c], sA) == cudaSuccess &&
                 cudaStreamWaitEvent(sX, plan->hev_a[c], 0) == cudaSuccess;
        if (ok) {
            rc = launch(plan, a_dev, plan->hbuf[1], c_dev, mc, N, K, dtype, out_dtype, sX);
            ok = rc == GEMM_OK;
        }
        ok = ok && cudaEventRecord(plan->hev_c[c], sX) == cudaSuccess &&
             cudaStreamWaitEvent(sC, plan->hev_c[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(static_cast<char*>(C_host) + (size_t)r0 * c_row_bytes, c_dev, (size_t)mc * c_row_bytes,
                             cudaMemcpyDeviceToHost, sC) == cudaSuccess;
    }
    // the caller's stream resumes after the last copy; the call is synchronous
    ok = ok && cudaEventRecord(plan->hev_done, sC) == cudaSuccess &&
         cudaStreamWaitEvent(s, plan->hev_done, 0) == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess;
    if (!ok) {
        // Copies queued before the failure may still read the caller's host
        // buffers or write the plan's: the call is synchronous, so they end
        // before it returns, whatever failed.
        cudaGetLastError();
        for (int i = 0; i < 3; ++i) cudaStreamSynchronize(plan->hstream[i]);
        cudaGetLastError();
        return rc != GEMM_OK ? rc : GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

int gemm_plan_status(gemm_plan_t plan, int* device_status) {
    if (!plan || !device_status) return GEMM_ERR_INVALID_ARG;
    int h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, plan->d_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(plan->d_status, 0, sizeof(h)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    *device_status = h[0];
    // A run that gave up part-way may leave stream-K flags raised.
    if (h[0] != 0 && plan->d_flags != nullptr &&
        cudaMemset(plan->d_flags, 0, flags_bytes(plan)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

int gemm_plan_last_grid(gemm_plan_t plan, int* ctas) {
    if (!plan || !ctas) return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(plan->rec_mu);
    *ctas = plan->last_grid;
    return GEMM_OK;
}

int gemm_plan_last_launch(gemm_plan_t plan, int* ctas, int* ctas_per_unit, int* tile_n, int* dp_waves,
                          int* sk_tiles) {
    if (!plan || !ctas || !ctas_per_unit || !tile_n || !dp_waves || !sk_tiles) return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(plan->rec_mu);
    *ctas = plan->last_grid;
    *ctas_per_unit = plan->last_unit;
    *tile_n = plan->last_tile_n;
    *dp_waves = plan->last_dp_waves;
    *sk_tiles = plan->last_sk_tiles;
    return GEMM_OK;
}

int gemm_plan_last_split(gemm_plan_t plan, int* slices) {
    if (!plan || !slices) return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(plan->rec_mu);
    *slices = plan->last_split;
    return GEMM_OK;
}

int gemm_plan_last_tile_n(gemm_plan_t plan, int* tile_n) {
    if (!plan || !tile_n) return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(plan->rec_mu);
    *tile_n = plan->last_tile_n;
    return GEMM_OK;
}

int gemm_plan_clock_log(gemm_plan_t plan, uint64_t* host, int64_t capacity, int64_t* count) {
    if (!plan || !count || capacity < 0 || (capacity > 0 && host == nullptr)) return GEMM_ERR_INVALID_ARG;
    *count = 0;
    if (plan->d_clock == nullptr) return GEMM_ERR_UNSUPPORTED;
    const int64_t cap = plan->clock_cap;
    std::vector<unsigned long long> ring((size_t)cap * 2);
    int prev = 0;
    cudaGetDevice(&prev);
    if (cudaSetDevice(plan->device) != cudaSuccess ||
        cudaMemcpy(ring.data(), plan->d_clock, ring.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) !=
            cudaSuccess) {
        cudaGetLastError();
        cudaSetDevice(prev);
        return GEMM_ERR_CUDA;
    }
    cudaSetDevice(prev);
    const int64_t launched = plan->clock_next.exchange(0);
    const int64_t kept = std::min(launched, cap), n = std::min(kept, capacity);
    // the last n launches, oldest first: launch j went to slot j % cap
    for (int64_t i = 0; i < n; ++i) {
        const int64_t slot = (launched - n + i) % cap;
        host[2 * i] = ring[(size_t)(2 * slot)];
        host[2 * i + 1] = ring[(size_t)(2 * slot + 1)];
    }
    *count = n;
    return GEMM_OK;
}

int gemm_plan_trace(gemm_plan_t plan, void* host, size_t bytes, int* ctas, int* slots) {
    if (!plan || !ctas || !slots) return GEMM_ERR_INVALID_ARG;
    *ctas = max_resident_ctas(plan);
    *slots = kTraceSlots;
    if (plan->d_trace == nullptr) return GEMM_ERR_UNSUPPORTED;
    const size_t need = trace_bytes(plan);
    if (host == nullptr || bytes < need) return GEMM_ERR_INVALID_ARG;
    if (cudaMemcpy(host, plan->d_trace, need, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(plan->d_trace, 0, need) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

int gemm_plan_destroy(gemm_plan_t plan) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (plan->device >= 0 && plan->device < kMaxDevices) {
            auto& v = g_plans[plan->device];
            for (size_t i = 0; i < v.size(); ++i)
                if (v[i] == plan) { v.erase(v.begin() + (long)i); break; }
        }
    }
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(plan->device);
    if (plan->d_status) cudaFree(plan->d_status);
    if (plan->d_partials) cudaFree(plan->d_partials);
    if (plan->d_flags) cudaFree(plan->d_flags);
    if (plan->d_trace) cudaFree(plan->d_trace);
    if (plan->d_clock) cudaFree(plan->d_clock);
    for (int i = 0; i < 3; ++i)
        if (plan->hbuf[i]) cudaFree(plan->hbuf[i]);
    for (int i = 0; i < 3; ++i)
        if (plan->hstream[i]) cudaStreamDestroy(plan->hstream[i]);
    if (plan->split_ev) cudaEventDestroy(plan->split_ev);
    cudaEvent_t evs[3] = {plan->hev_start, plan->hev_b, plan->hev_done};
    for (cudaEvent_t e : evs)
        if (e) cudaEventDestroy(e);
    for (int i = 0; i < 8; ++i) {
        if (plan->hev_a[i]) cudaEventDestroy(plan->hev_a[i]);
        if (plan->hev_c[i]) cudaEventDestroy(plan->hev_c[i]);
    }
    cudaSetDevice(prev);
    delete plan;
    return GEMM_OK;
}

const char* gemm_strerror(int status) {
    switch (status) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "unsupported shape or pitch (K % 8, N * out_bytes % 16, or size >= 2^31)";
        case GEMM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case GEMM_ERR_CUDA: return "CUDA runtime call failed";
        case GEMM_ERR_DRIVER: return "tensor-map encoding failed or driver entry point missing";
        case GEMM_ERR_NO_PLAN: return "no plan created for the current device";
        case GEMM_ERR_TIMEOUT: return "a bounded wait in the kernel expired";
        case GEMM_ERR_NO_DEVICE: return "no usable sm_103 device";
        case GEMM_ERR_INTERNAL: return "an internal consistency check of a GEMM_DEBUG build failed";
        default: return "unknown status";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers may not allocate device memory at all: services that reserve
// every byte of HBM for their own pool at start-up and forbid allocations
// afterwards, embedders whose memory is owned by another allocator that must
// see every device allocation, and latency-critical loops that cannot take
// the device-wide synchronisation a cudaFree implies.  gemm_plan_create() allocates the plan's
// 16-byte status record with cudaMalloc, so those callers use
// gemm_run_noalloc() instead.  It launches the same kernel, but the kernel's
// only scratch -- the status record its bounded waits write on timeout --
// lives in the file-scope array below, which the library's module reserves
// on every GPU that loads it until the process exits.
//
// Limits and sharing: the array holds kNoallocScratchBytes (256 bytes); the
// kernel needs 16 of them for any M, N, K, and a request beyond the array is
// rejected with GEMM_ERR_UNSUPPORTED.  Every call on a device shares the same
// array and it keeps the last call's contents, so each call first clears the
// status record on its stream; calls that overlap on the GPU (different
// streams, no ordering between them) race on that record.  The record is not
// read back by this entry point: device-side timeouts are reported only by
// the plan path (gemm_plan_status).
namespace {

constexpr size_t kNoallocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocDevice {
    std::once_flag once;
    int rc = GEMM_OK;
    gemm_plan state;   // host-side launch parameters only; d_status points into the static array
};
NoallocDevice g_noalloc[kMaxDevices];

// Bytes of scratch one launch of the kernel needs: its status record.  It
// does not depend on the problem size.
size_t noalloc_scratch_bytes(int64_t, int64_t, int64_t) { return 4 * sizeof(int); }

// Once per device, with that device current: fetch the array's device
// address (a host-side reference to g_noalloc_scratch is only a stand-in and
// must never reach a kernel) and query the launch capacity.  No allocation.
void noalloc_setup(NoallocDevice* d, int device) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        cudaGetLastError();
        d->rc = GEMM_ERR_CUDA;
        return;
    }
    if (prop.major != 10 || prop.minor != 3) {
        d->rc = GEMM_ERR_NO_DEVICE;
        return;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        d->rc = GEMM_ERR_CUDA;
        return;
    }
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        cudaGetLastError();
        d->rc = GEMM_ERR_CUDA;
        return;
    }
    d->state.device = device;
    d->state.sm_count = prop.multiProcessorCount;
    d->state.visible_devices = count;
    d->state.d_status = static_cast<int*>(ptr);
    d->state.stream_k = 0;   // no workspace here: whole tiles only
    int rc = query_capacity(&d->state, 1);
    if (rc == GEMM_OK) rc = query_capacity(&d->state, 2);
    if (rc == GEMM_OK) rc = query_capacity(&d->state, 4);
    d->rc = rc;
}

}  // namespace

extern "C" int gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                int dtype, int out_dtype, void* stream) {
    int rc = validate(A, B, C, M, N, K, dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    if (noalloc_scratch_bytes(M, N, K) > kNoallocScratchBytes) return GEMM_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_INVALID_ARG;
    NoallocDevice* d = &g_noalloc[dev];
    std::call_once(d->once, noalloc_setup, d, dev);
    if (d->rc != GEMM_OK) return d->rc;
    rc = check_operands(dev, A, B, C, K);
    if (rc != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(d->state.d_status, 0, noalloc_scratch_bytes(M, N, K), s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return launch(&d->state, A, B, C, M, N, K, dtype, out_dtype, s);
}
