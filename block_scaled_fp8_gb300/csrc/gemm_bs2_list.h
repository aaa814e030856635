// The compiled instantiations of the CTA-pair kernel: (BLOCK_N, with C, rows per
// pair tile, FP32 D).  The bf16-output ones are instantiated in gemm_bs2_inst.cu,
// the FP32-output ones in gemm_bs2_inst_f32.cu.
#pragma once

#define DG_BS2_LIST_BF16(X)                                                                        \
    X(128, false, 256, false) X(128, true, 256, false) X(192, false, 256, false)                   \
    X(192, true, 256, false) X(224, false, 256, false) X(224, true, 256, false)                    \
    X(240, false, 256, false) X(240, true, 256, false) X(256, false, 256, false)                   \
    X(32, false, 128, false) X(64, false, 128, false) X(96, false, 128, false)                     \
    X(128, false, 128, false) X(384, false, 256, false)

#define DG_BS2_LIST_F32(X)                                                                         \
    X(128, false, 256, true) X(128, true, 256, true) X(224, false, 256, true) X(224, true, 256, true)

#define DG_BS2_LIST(X) DG_BS2_LIST_BF16(X) DG_BS2_LIST_F32(X)
