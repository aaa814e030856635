"""GB300-native block-scaled FP8 GEMM (D = C + A @ B^T, 1x128 / 128x128 scales, bf16 out)."""
