// kernels_inst.cu -- instantiates gemm_tn_persistent for one unit size
// (GEMM_INST_CLUSTER = 1, 2 or 4 CTAs), one output type (GEMM_INST_OUT =
// 0 bf16, 1 f16, 2 fp32), one operand width (GEMM_INST_IN = 0 bf16/f16,
// 1 E4M3/E5M2) and, with GEMM_INST_BMN = 1, the padded MN-major-B form
// (1- and 2-CTA units, 16-bit operands), over every tile width of
// kernel_table.h.  The build compiles
// this file once per combination, in parallel.
#include "gemm_kernel.cuh"
#include "kernel_table.h"

#ifndef GEMM_INST_CLUSTER
#error "GEMM_INST_CLUSTER must be defined"
#endif
#ifndef GEMM_INST_OUT
#error "GEMM_INST_OUT must be defined"
#endif
#ifndef GEMM_INST_IN
#error "GEMM_INST_IN must be defined"
#endif
#ifndef GEMM_INST_BMN
#define GEMM_INST_BMN 0   // 1: the padded MN-major-B variants (see Cfg::kBMnPad)
#endif

#define GEMM_CAT2(a, b, c, d) kernel_info_c##a##_o##b##_i##c##_p##d
#define GEMM_CAT(a, b, c, d) GEMM_CAT2(a, b, c, d)
#define GEMM_INFO_FN GEMM_CAT(GEMM_INST_CLUSTER, GEMM_INST_OUT, GEMM_INST_IN, GEMM_INST_BMN)

namespace gb300 {

template <int kBN>
static KernelInfo make_info() {
    using C = Cfg<GEMM_INST_CLUSTER, kBN, GEMM_INST_OUT, GEMM_INST_IN, GEMM_INST_BMN != 0>;
    return KernelInfo{gemm_tn_persistent<GEMM_INST_CLUSTER, kBN, GEMM_INST_OUT, GEMM_INST_IN, GEMM_INST_BMN != 0>,
                      C::kSmemBytes, C::kStages};
}

KernelInfo GEMM_INFO_FN(int bn) {
    switch (bn) {
        case 256: return make_info<256>();
        case 224: return make_info<224>();
        case 192: return make_info<192>();
        case 160: return make_info<160>();
        case 128: return make_info<128>();
        default: return KernelInfo{nullptr, 0, 0};
    }
}

}  // namespace gb300
