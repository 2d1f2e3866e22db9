// kernel_table.h -- the instantiated variants of the persistent GEMM kernel.
//
// kernels_inst.cu is compiled once per (CTA pairing, output type); each
// object defines one lookup function over the tile widths.  The host side
// (gemm_api.cu) picks a variant through gb300::kernel_info().
#pragma once
#include <cuda.h>

namespace gb300 {

struct Params;
using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, Params);

struct KernelInfo {
    KernelFn fn;      // nullptr if the combination is not instantiated
    int smem_bytes;   // dynamic shared memory the launch must request
    int stages;       // depth of the shared-memory ring
};

constexpr int kNumTileWidths = 5;
constexpr int kTileWidths[kNumTileWidths] = {256, 224, 192, 160, 128};

KernelInfo kernel_info_p1_o0(int bn);
KernelInfo kernel_info_p1_o1(int bn);
KernelInfo kernel_info_p1_o2(int bn);
KernelInfo kernel_info_p2_o0(int bn);
KernelInfo kernel_info_p2_o1(int bn);
KernelInfo kernel_info_p2_o2(int bn);

inline KernelInfo kernel_info(int pair, int bn, int out) {
    if (pair == 1) {
        switch (out) {
            case 0: return kernel_info_p1_o0(bn);
            case 1: return kernel_info_p1_o1(bn);
            default: return kernel_info_p1_o2(bn);
        }
    }
    switch (out) {
        case 0: return kernel_info_p2_o0(bn);
        case 1: return kernel_info_p2_o1(bn);
        default: return kernel_info_p2_o2(bn);
    }
}

}  // namespace gb300
