// mma_probe.cu -- tensor-core issue-rate probe.
//
// Every SM holds one CTA (alone, or one of a CTA pair) whose operand tiles
// are already in shared memory; one thread issues back-to-back tcgen05.mma
// into a TMEM accumulator, with no loads and no epilogue.  The SM cycle
// counter around the stream gives the dense FLOP/clk/SM the tensor cores
// sustain; CUDA events around the launch give the rate of all SMs at the
// clocks the launch ran at.  This is the ceiling of a GEMM's K loop: the
// "tensor-core roofline" of "Optimizing Blackwell Matrix Multiplication in
// Mojo (Part 2)" (the kernels are measured against the tensor cores' peak),
// taken on the GPU itself rather than from a data sheet.
//
// The instruction stream is the persistent GEMM's: 128×N×16 (bf16/f16,
// kind::f16) or 128×N×32 (8-bit, kind::f8f6f4) per CTA and instruction,
// M = 256 across a pair, K-major 128-byte-swizzled operands, four
// instructions per 128-byte k-block; N is 256 or any tile width asked for.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "kernel_table.h"

namespace gb300 {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeN = 256;                        // accumulator columns
constexpr int kProbeA = kRowsPerCta * kBlockKBytes; // 16 KB: 128 rows × one 128-byte k-block
constexpr int kProbeB = kProbeN * kBlockKBytes;     // 32 KB: the B rows an instruction may read
// More than half of the SM's shared memory, so that no two probe CTAs share
// an SM.
constexpr int kProbeSmem = 160 * 1024;

// out[2*cta] = SM cycles from the first issue to the last completion seen by
// the issuing CTA, out[2*cta+1] = the same interval in %globaltimer ns.
template <int kPair, bool kF8>
__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_probe_kernel(int64_t k_blocks, uint32_t idesc, unsigned long long* out, int* status,
                     unsigned long long wait_limit_ns) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {
        if (threadIdx.x == 0) atomicCAS(status, 0, kErrCuda);
        return;
    }
    const uint32_t a_tile = base, b_tile = base + kProbeA;
    const uint32_t bar = base + kProbeA + kProbeB;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem_raw + kProbeA + kProbeB + 8);
    const uint32_t rank = kPair == 2 ? cluster_cta_rank() : 0u;

    // Operands: a fixed pattern of small bf16/f16 (or 8-bit) values with
    // varied bits, so that the multipliers toggle as in a real product.
    uint32_t* words = reinterpret_cast<uint32_t*>(smem_raw);
    for (int i = threadIdx.x; i < (kProbeA + kProbeB) / 4; i += kProbeThreads) {
        uint32_t h = (uint32_t)i * 2654435761u + blockIdx.x * 40503u;
        h ^= h >> 15;
        words[i] = kF8 ? (h & 0x3B3B3B3Bu) : (h & 0x3FFF3FFFu) ^ 0x00800080u;
    }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init_cluster();
    }
    fence_proxy_async_shared();   // the operand writes, before the tensor cores read them
    if constexpr (kPair == 2) {
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        tmem_alloc<kPair>(smem_addr(tmem_holder), kProbeN);
        tmem_relinquish<kPair>();
    }
    tc_fence_before_sync();
    if constexpr (kPair == 2) {
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    unsigned long long c0 = 0, n0 = 0;
    if (threadIdx.x == 0 && rank == 0) {
        const uint64_t ad = smem_desc_sw128(a_tile), bd = smem_desc_sw128(b_tile);
        c0 = (unsigned long long)clock64();
        n0 = global_timer_ns();
        for (int64_t kb = 0; kb < k_blocks; ++kb) {
#pragma unroll
            for (int j = 0; j < kBlockKBytes / kMmaKBytes; ++j)
                tc_mma<kPair, kF8>(tmem, ad + 2 * j, bd + 2 * j, idesc, (kb | j) != 0);
        }
        if constexpr (kPair == 2) tc_commit_pair(bar, 0x3);
        else tc_commit(bar);
    }
    // every CTA waits for the completion of the stream that writes its TMEM
    bool done = false;
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        while (!(done = mbar_try_wait(bar, 0))) {
            if (global_timer_ns() - t0 > wait_limit_ns) {
                atomicCAS(status, 0, kErrTimeout);
                break;
            }
        }
        if (rank == 0) {
            out[2 * blockIdx.x] = (unsigned long long)clock64() - c0;
            out[2 * blockIdx.x + 1] = global_timer_ns() - n0;
        }
        if (!done) {   // let any instruction still in flight finish before TMEM goes away
            const uint64_t t1 = global_timer_ns();
            while (global_timer_ns() - t1 < 2000000ull) { }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kPair == 2) {
        cluster_arrive();
        cluster_wait();
    }
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<kPair>(tmem, kProbeN);
    }
}

template <int kPair, bool kF8>
int run_probe(int sm_count, int64_t k_blocks, uint32_t idesc, std::vector<unsigned long long>& host, float* ms) {
    auto fn = mma_probe_kernel<kPair, kF8>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    const int ctas = sm_count / kPair * kPair;
    unsigned long long* d_out = nullptr;
    int* d_status = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = GEMM_OK;
    if (cudaMalloc(&d_out, sizeof(unsigned long long) * 2 * ctas) != cudaSuccess ||
        cudaMalloc(&d_status, sizeof(int)) != cudaSuccess || cudaMemset(d_status, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(d_out, 0, sizeof(unsigned long long) * 2 * ctas) != cudaSuccess ||
        cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
        rc = GEMM_ERR_CUDA;
    if (rc == GEMM_OK) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas, 1, 1);
        cfg.blockDim = dim3(kProbeThreads, 1, 1);
        cfg.dynamicSmemBytes = kProbeSmem;
        cfg.stream = nullptr;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)kPair;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const unsigned long long limit = 10000000000ull;   // 10 s: far above any probe length accepted
        if (cudaEventRecord(e0, nullptr) != cudaSuccess ||
            cudaLaunchKernelEx(&cfg, fn, k_blocks, idesc, d_out, d_status, limit) != cudaSuccess ||
            cudaEventRecord(e1, nullptr) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess)
            rc = GEMM_ERR_CUDA;
    }
    int status = 0;
    if (rc == GEMM_OK) {
        host.assign(2 * ctas, 0ull);
        if (cudaMemcpy(host.data(), d_out, sizeof(unsigned long long) * 2 * ctas, cudaMemcpyDeviceToHost) !=
                cudaSuccess ||
            cudaMemcpy(&status, d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
            cudaEventElapsedTime(ms, e0, e1) != cudaSuccess)
            rc = GEMM_ERR_CUDA;
        else if (status != 0)
            rc = status;
    }
    if (rc == GEMM_ERR_CUDA) cudaGetLastError();
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (d_out) cudaFree(d_out);
    if (d_status) cudaFree(d_status);
    return rc;
}

// Instruction descriptor of the probe's MMA: n accumulator columns (the
// instruction's N, the GEMM's tile width), M = 128 per CTA.
uint32_t probe_idesc(int dtype, int pair, int n) {
    const uint32_t ab = (dtype == GEMM_BF16 || dtype == GEMM_E5M2) ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)((kRowsPerCta * pair) >> 4) << 24);
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_probe_mma_rate(int dtype, int cta_pair, int64_t mmas_per_sm, double* flop_per_clk_per_sm,
                                   double* tflops, double* sm_mhz) {
    return gemm_probe_mma_rate_n(dtype, cta_pair, kProbeN, mmas_per_sm, flop_per_clk_per_sm, tflops, sm_mhz);
}

extern "C" int gemm_probe_mma_rate_n(int dtype, int cta_pair, int tile_n, int64_t mmas_per_sm,
                                     double* flop_per_clk_per_sm, double* tflops, double* sm_mhz) {
    if (dtype != GEMM_BF16 && dtype != GEMM_F16 && dtype != GEMM_E4M3 && dtype != GEMM_E5M2)
        return GEMM_ERR_INVALID_ARG;
    if (cta_pair != 1 && cta_pair != 2) return GEMM_ERR_INVALID_ARG;
    // N of an M = 128 (one CTA) or M = 256 (pair) instruction: 16..256 in steps of 16;
    // the operand and TMEM buffers are sized for 256.
    if (tile_n < 16 || tile_n > kProbeN || tile_n % 16 != 0) return GEMM_ERR_INVALID_ARG;
    const int per_block = kBlockKBytes / kMmaKBytes;
    if (mmas_per_sm < per_block || mmas_per_sm > (int64_t(1) << 24) || mmas_per_sm % per_block != 0)
        return GEMM_ERR_INVALID_ARG;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_NO_DEVICE;
    const bool f8 = dtype == GEMM_E4M3 || dtype == GEMM_E5M2;
    const uint32_t idesc = probe_idesc(dtype, cta_pair, tile_n);
    const int64_t k_blocks = mmas_per_sm / per_block;
    std::vector<unsigned long long> out;
    float ms = 0.f;
    int rc;
    if (cta_pair == 2) rc = f8 ? run_probe<2, true>(prop.multiProcessorCount, k_blocks, idesc, out, &ms)
                               : run_probe<2, false>(prop.multiProcessorCount, k_blocks, idesc, out, &ms);
    else rc = f8 ? run_probe<1, true>(prop.multiProcessorCount, k_blocks, idesc, out, &ms)
                 : run_probe<1, false>(prop.multiProcessorCount, k_blocks, idesc, out, &ms);
    if (rc != GEMM_OK) return rc;
    // per SM and instruction: 128 rows × tile_n columns × K (16, or 32 for 8-bit) multiply-adds
    const double flop_per_mma = 2.0 * kRowsPerCta * tile_n * (f8 ? 32 : 16);
    std::vector<double> fpc, mhz;
    for (size_t c = 0; c + 1 < out.size(); c += 2) {
        if (out[c] == 0 || out[c + 1] == 0) continue;   // a pair's second CTA records nothing
        fpc.push_back(flop_per_mma * (double)mmas_per_sm / (double)out[c]);
        mhz.push_back((double)out[c] / (double)out[c + 1] * 1e3);
    }
    if (fpc.empty()) return GEMM_ERR_CUDA;
    std::sort(fpc.begin(), fpc.end());
    std::sort(mhz.begin(), mhz.end());
    const int ctas = prop.multiProcessorCount / cta_pair * cta_pair;
    if (flop_per_clk_per_sm) *flop_per_clk_per_sm = fpc[fpc.size() / 2];
    if (sm_mhz) *sm_mhz = mhz[mhz.size() / 2];
    if (tflops) *tflops = flop_per_mma * (double)mmas_per_sm * (double)ctas / ((double)ms * 1e-3) / 1e12;
    return GEMM_OK;
}
