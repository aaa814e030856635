"""FP32-output GEMM (dg_fp8_gemm_nt_f32, 256-row CTA pairs) against the FP32
oracle, and against the bf16 GEMM: rounding the FP32 result to bf16 must give
the bf16 GEMM's output bit for bit (same accumulator, C = 0)."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


def _packed(case):
    M, N, K = case.shape
    return (case.a.to(DEV), binding.transform_sf(case.sfa.to(DEV), 1, M), case.b.to(DEV),
            binding.transform_sf(case.sfb.to(DEV), 128, N))


def _close_f32(got, ref, what):
    """Per element |g - o| <= 1e-4 |o| + 1e-4 rms(o): the FP32 accumulation over
    K (tensor-core adders, order fixed by K) against the fp64 sum rounded once;
    100x tighter than the bf16 bar, whose own rounding step is 2^-9."""
    o = ref.astype(np.float64)
    g = got.astype(np.float64)
    assert np.isfinite(g).all(), what
    rms = float(np.sqrt(np.mean(o * o))) if o.size else 0.0
    bad = np.abs(g - o) > 1e-4 * np.abs(o) + 1e-4 * rms
    assert not bad.any(), f"{what}: {int(bad.sum())} of {g.size} out of tolerance"


@pytest.mark.parametrize("M,N,K,with_c", [(128, 256, 512, False), (256, 264, 640, True),
                                          (300, 1000, 336, False), (1000, 2048, 1536, True),
                                          (17, 96, 128, True)])
def test_f32_matches_oracle(orc, M, N, K, with_c):
    case = inputs.dense_case(M, N, K, seed=M + N + K, b_scale_exp_range=(-8, 4))
    a, sfa, b, sfb = _packed(case)
    c = (torch.randn(M, N, generator=torch.Generator().manual_seed(M)) if with_c else None)
    d = torch.full((M, N), 7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nt_f32(a, sfa, b, sfb, d, c=None if c is None else c.to(DEV), status=status)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert cfg["kind"] == 2 and cfg["block_m"] == 256, cfg
    ref = orc.gemm_nt_f32(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, N),
                          c=None if c is None else c.numpy())
    _close_f32(d.cpu().numpy(), ref, f"f32 {M}x{N}x{K}")


def test_f32_rounds_to_the_bf16_gemm():
    M, N, K = 512, 768, 1024
    case = inputs.dense_case(M, N, K, seed=23)
    a, sfa, b, sfb = _packed(case)
    d32 = torch.empty(M, N, dtype=torch.float32, device=DEV)
    d16 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    binding.dg_fp8_gemm_nt_f32(a, sfa, b, sfb, d32)
    binding.dg_fp8_gemm_nt(a, sfa, b, sfb, d16)
    torch.cuda.synchronize()
    assert torch.equal(d32.to(torch.bfloat16), d16)


@pytest.mark.parametrize("M,N,K", [(300, 1000, 384), (4096, 7168, 2048)])
def test_f32_in_place_equals_separate(M, N, K):
    """c = d (accumulated into D at L2 by TMA reduce-add) gives the same bits
    as C in its own buffer (added in registers)."""
    case = inputs.dense_case(M, N, K, seed=M + K, b_scale_exp_range=(-8, 4))
    a, sfa, b, sfb = _packed(case)
    c0 = torch.randn(M, N, generator=torch.Generator().manual_seed(M)).to(DEV)
    d_sep = torch.full((M, N), 7.0, dtype=torch.float32, device=DEV)
    binding.dg_fp8_gemm_nt_f32(a, sfa, b, sfb, d_sep, c=c0)
    d_in = c0.clone()
    binding.dg_fp8_gemm_nt_f32(a, sfa, b, sfb, d_in, c=d_in)
    torch.cuda.synchronize()
    assert torch.equal(d_sep, d_in)


def test_f32_in_place_accumulation_and_k_zero(orc):
    """c aliasing d accumulates in place; K = 0 gives D = C."""
    M, N, K = 256, 512, 768
    case = inputs.dense_case(M, N, K, seed=31)
    a, sfa, b, sfb = _packed(case)
    c0 = torch.randn(M, N, generator=torch.Generator().manual_seed(4))
    d = c0.to(DEV).clone()
    binding.dg_fp8_gemm_nt_f32(a, sfa, b, sfb, d, c=d)
    torch.cuda.synchronize()
    ref = orc.gemm_nt_f32(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, N),
                          c=c0.numpy())
    _close_f32(d.cpu().numpy(), ref, "in place")
    e = torch.empty(M, N, dtype=torch.float32, device=DEV)
    empty = torch.empty(M, 0, dtype=torch.float8_e4m3fn, device=DEV)
    sf0 = torch.empty(0, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nt_f32(empty, sf0, torch.empty(N, 0, dtype=torch.float8_e4m3fn, device=DEV), sf0,
                               e, c=c0.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(e.cpu(), c0)
