"""GB300-native block-scaled FP8 GEMM: D = C + A @ B^T with 1x128 (A) and
128x128 (B) scales, FP32 accumulation, bf16 output, plus the M-grouped MoE
variants and the scale-layout transform.  The compute runs in the CUDA
library built from csrc/ (C ABI in include/dg.h); ``binding`` marshals torch
tensors into it.  ``inputs`` generates seeded synthetic problems."""
from . import binding  # noqa: F401  (loading the .so is deferred to the first call)
from .binding import (DGError, dg_fp8_gemm_nt, dg_m_grouped_fp8_gemm_nt_contiguous,  # noqa: F401
                      dg_m_grouped_fp8_gemm_nt_masked, dg_transform_sf, transform_sf)
