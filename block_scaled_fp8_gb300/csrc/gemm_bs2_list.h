// The compiled instantiations of the CTA-pair kernel: (BLOCK_N, with C, rows per
// pair tile, FP32 D, operand layouts: bit 0 A MN-major, bit 1 B MN-major).  The
// bf16-output NT ones are instantiated in gemm_bs2_inst.cu, the FP32-output ones
// in gemm_bs2_inst_f32.cu, the NN/TN/TT ones in gemm_bs2_inst_mn.cu.
#pragma once

#define DG_BS2_LIST_BF16(X)                                                                        \
    X(128, false, 256, false, 0) X(128, true, 256, false, 0) X(192, false, 256, false, 0)                   \
    X(192, true, 256, false, 0) X(224, false, 256, false, 0) X(224, true, 256, false, 0)                    \
    X(240, false, 256, false, 0) X(240, true, 256, false, 0) X(256, false, 256, false, 0)                   \
    X(32, false, 128, false, 0) X(64, false, 128, false, 0) X(96, false, 128, false, 0)                     \
    X(128, false, 128, false, 0) X(384, false, 256, false, 0)

#define DG_BS2_LIST_F32(X)                                                                         \
    X(128, false, 256, true, 0) X(128, true, 256, true, 0) X(224, false, 256, true, 0) X(224, true, 256, true, 0)

// NN (B MN-major), TN (both), TT (A MN-major): 256 columns without C, 224 (two
// accumulators) with C; the last one is the K-grouped weight-gradient GEMM (TN,
// FP32 C and D)
#define DG_BS2_LIST_MN(X)                                                                          \
    X(256, false, 256, false, 2) X(224, true, 256, false, 2) X(256, false, 256, false, 3)          \
    X(224, true, 256, false, 3) X(256, false, 256, false, 1) X(224, true, 256, false, 1)           \
    X(224, true, 256, true, 3)

#define DG_BS2_LIST(X) DG_BS2_LIST_BF16(X) DG_BS2_LIST_F32(X) DG_BS2_LIST_MN(X)
