// The compiled instantiations of the CTA-pair kernel: (BLOCK_N, with C, rows per
// pair tile, FP32 D, operand layouts: bit 0 A MN-major, bit 1 B MN-major, bit 2
// B FP4, bit 3 A and B scales every 32 K).  The bf16-output NT ones are instantiated in gemm_bs2_inst.cu, the
// FP32-output ones in gemm_bs2_inst_f32.cu, the NN/TN/TT and K-grouped ones in
// gemm_bs2_inst_mn.cu, the FP8 x FP4 ones in gemm_bs2_inst_fp4.cu.
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
// accumulators) with C; the last two are the K-grouped weight-gradient GEMM (TN,
// FP32 C and D), with scales every 128 rows of K (224 columns) or every 32 (layout
// bit 3, 192 columns)
#define DG_BS2_LIST_MN(X)                                                                          \
    X(256, false, 256, false, 2) X(224, true, 256, false, 2) X(256, false, 256, false, 3)          \
    X(224, true, 256, false, 3) X(256, false, 256, false, 1) X(224, true, 256, false, 1)           \
    X(224, true, 256, true, 3) X(192, true, 256, true, 11)

// FP8 x FP4 (layout bit 2: B is E2M1 with one scale per 32 K): 256-row pairs with
// 128 or 256 columns without C, 128 with C; 128-row pairs (M <= 128, no C) with 32,
// 96 or 128 columns
#define DG_BS2_LIST_FP4(X)                                                                         \
    X(256, false, 256, false, 4) X(128, false, 256, false, 4) X(128, true, 256, false, 4)          \
    X(32, false, 128, false, 4) X(96, false, 128, false, 4) X(128, false, 128, false, 4)

#define DG_BS2_LIST(X) DG_BS2_LIST_BF16(X) DG_BS2_LIST_F32(X) DG_BS2_LIST_MN(X) DG_BS2_LIST_FP4(X)
