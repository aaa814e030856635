"""NN / TN / TT GEMMs ("DeepSeek V4 源码剖析 第13章" §13.3: D = C + A @ B, the
suffix letters giving the transpose state of A and B) against the oracle, and
bit for bit against the NT GEMM on the same operands stored K-contiguous: the
storage order changes what TMA loads, not the products or their order."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
CALLS = {"nn": binding.dg_fp8_gemm_nn, "tn": binding.dg_fp8_gemm_tn, "tt": binding.dg_fp8_gemm_tt}


def _stored(case, layout, pad=0):
    """A as [M, K] or [K, M], B as [N, K] or [K, N], on the device, each a
    view of a buffer whose leading dimension is the row length rounded up to
    16 bytes plus `pad` (the copies' 16-byte stride rule)."""
    def lay(x, transpose):
        x = x.view(torch.uint8)
        x = x.t().contiguous() if transpose else x.contiguous()
        rows, cols = x.shape
        ld = (cols + 15) // 16 * 16 + pad
        wide = torch.zeros(rows, ld, dtype=torch.uint8)
        wide[:, :cols] = x
        return wide.to(DEV)[:, :cols].view(torch.float8_e4m3fn)
    return lay(case.a, layout[0] == "t"), lay(case.b, layout[1] == "n")


def _run(layout, case, c=None, pad=0, d_init=7.0):
    M, N, K = case.shape
    a, b = _stored(case, layout, pad)
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.full((M, N), d_init, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    CALLS[layout](a, sfa, b, sfb, d, c=c, status=status)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d, cfg


def _nt(case, c=None):
    M, N, K = case.shape
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    binding.dg_fp8_gemm_nt(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d, c=c)
    torch.cuda.synchronize()
    return d


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
@pytest.mark.parametrize("M,N,K,with_c,pad", [(256, 256, 512, False, 0), (300, 1000, 384, True, 0),
                                              (1000, 2048, 1536, False, 32), (17, 96, 128, True, 0),
                                              (513, 264, 896, False, 16)])
def test_layout_matches_oracle_and_nt(orc, layout, M, N, K, with_c, pad):
    case = inputs.dense_case(M, N, K, seed=M + 3 * N + K, with_c=with_c)
    c = case.c.to(DEV) if with_c else None
    d, cfg = _run(layout, case, c=c, pad=pad)
    # with C, 224-column tiles (two TMEM accumulators); without, 256
    assert cfg["kind"] == 2 and cfg["block_m"] == 256 and cfg["block_n"] == (224 if with_c else 256), cfg
    a_st, b_st = _stored(case, layout)
    ref = orc.gemm(layout, u8(a_st.cpu()), case.sfa.double().numpy(), u8(b_st.cpu()),
                   sb_rows(case.sfb, N), c=None if c is None else bf16_bits(case.c))
    assert_close(bf16_bits(d), ref, f"{layout} {M}x{N}x{K}")
    assert torch.equal(d, _nt(case, c=c)), f"{layout} {M}x{N}x{K}: differs from the NT GEMM"


def test_tn_k_not_multiple_of_16(orc):
    """Both operands M/N-contiguous: K needs no alignment (rows past K are
    zero-filled by the loads)."""
    M, N, K = 320, 512, 200
    case = inputs.dense_case(M, N, K, seed=77)
    d, _ = _run("tn", case)
    a_st, b_st = _stored(case, "tn")
    ref = orc.gemm("tn", u8(a_st.cpu()), case.sfa.double().numpy(), u8(b_st.cpu()), sb_rows(case.sfb, N))
    assert_close(bf16_bits(d), ref, "tn K=200")


def test_layout_in_place_and_k_zero():
    M, N, K = 256, 512, 768
    case = inputs.dense_case(M, N, K, seed=5, with_c=True)
    ref = _nt(case, c=case.c.to(DEV))
    d = case.c.to(DEV).clone()
    a, b = _stored(case, "tt")
    binding.dg_fp8_gemm_tt(a, binding.transform_sf(case.sfa.to(DEV), 1, M), b,
                           binding.transform_sf(case.sfb.to(DEV), 128, N), d, c=d)
    torch.cuda.synchronize()
    assert torch.equal(d, ref)
    e = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    sf0 = torch.empty(0, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nn(torch.empty(M, 0, dtype=torch.float8_e4m3fn, device=DEV), sf0,
                           torch.empty(0, N, dtype=torch.float8_e4m3fn, device=DEV), sf0, e,
                           c=case.c.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(e.cpu(), case.c)


def test_layout_rejects_short_leading_dimension():
    M, N, K = 256, 256, 256
    case = inputs.dense_case(M, N, K, seed=6)
    a, b = _stored(case, "nn")
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    lib = binding.lib()
    p = binding._p
    st = lib.dg_fp8_gemm_nn(p(a), a.stride(0), p(sfa), 1, p(b), N - 16, p(sfb), 1, None, 0, p(d), N, M, N, K,
                            None, None)
    assert st == 1   # DG_ERR_INVALID_ARG: ldb < n for an N-contiguous B
