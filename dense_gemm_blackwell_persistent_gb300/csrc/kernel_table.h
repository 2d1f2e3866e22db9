// kernel_table.h -- the instantiated variants of the persistent GEMM kernel.
//
// kernels_inst.cu is compiled once per (CTAs per unit, output type, operand
// width); each object defines one lookup function over the tile widths.  The host side
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

KernelInfo kernel_info_c1_o0_i0_p0(int bn);
KernelInfo kernel_info_c1_o0_i1_p0(int bn);
KernelInfo kernel_info_c1_o1_i0_p0(int bn);
KernelInfo kernel_info_c1_o1_i1_p0(int bn);
KernelInfo kernel_info_c1_o2_i0_p0(int bn);
KernelInfo kernel_info_c1_o2_i1_p0(int bn);
KernelInfo kernel_info_c2_o0_i0_p0(int bn);
KernelInfo kernel_info_c2_o0_i1_p0(int bn);
KernelInfo kernel_info_c2_o1_i0_p0(int bn);
KernelInfo kernel_info_c2_o1_i1_p0(int bn);
KernelInfo kernel_info_c2_o2_i0_p0(int bn);
KernelInfo kernel_info_c2_o2_i1_p0(int bn);
KernelInfo kernel_info_c4_o0_i0_p0(int bn);
KernelInfo kernel_info_c4_o0_i1_p0(int bn);
KernelInfo kernel_info_c4_o1_i0_p0(int bn);
KernelInfo kernel_info_c4_o1_i1_p0(int bn);
KernelInfo kernel_info_c4_o2_i0_p0(int bn);
KernelInfo kernel_info_c4_o2_i1_p0(int bn);
KernelInfo kernel_info_c1_o0_i0_p1(int bn);
KernelInfo kernel_info_c1_o1_i0_p1(int bn);
KernelInfo kernel_info_c1_o2_i0_p1(int bn);
KernelInfo kernel_info_c2_o0_i0_p1(int bn);
KernelInfo kernel_info_c2_o1_i0_p1(int bn);
KernelInfo kernel_info_c2_o2_i0_p1(int bn);

// cluster: CTAs per work unit (1, 2 or 4); out: 0 bf16, 1 f16, 2 fp32;
// in: 0 bf16/f16 operands, 1 E4M3/E5M2 operands; pad: the padded
// MN-major-B form (1- and 2-CTA units, 16-bit operands only).
inline KernelInfo kernel_info(int cluster, int bn, int out, int in, bool pad = false) {
#define GB300_PICK(C, P)                                                                                \
    (in == 0 ? (out == 0 ? kernel_info_c##C##_o0_i0_p##P(bn) : out == 1 ? kernel_info_c##C##_o1_i0_p##P(bn) \
                                                                   : kernel_info_c##C##_o2_i0_p##P(bn))     \
             : (out == 0 ? kernel_info_c##C##_o0_i1_p0(bn) : out == 1 ? kernel_info_c##C##_o1_i1_p0(bn)     \
                                                                   : kernel_info_c##C##_o2_i1_p0(bn)))
    if (pad) {
        if (in != 0) return KernelInfo{nullptr, 0, 0};
        switch (cluster) {
            case 1: return GB300_PICK(1, 1);
            case 2: return GB300_PICK(2, 1);
            default: return KernelInfo{nullptr, 0, 0};
        }
    }
    switch (cluster) {
        case 1: return GB300_PICK(1, 0);
        case 2: return GB300_PICK(2, 0);
        case 4: return GB300_PICK(4, 0);
        default: return KernelInfo{nullptr, 0, 0};
    }
#undef GB300_PICK
}

}  // namespace gb300
