"""Parity of the CUDA library (called through the C ABI) with the oracle.

Small problems are compared element by element in full; the workload-sized
problems on sampled elements the oracle computes one by one, plus properties
that hold at any size.  Integer/byte results (scale packing, integer-exact
GEMMs, batch invariance) must match bit for bit.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _run_dense(case, c=None, d=None, status=None):
    M, N, K = case.shape
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    if d is None:
        d = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    binding.dg_fp8_gemm_nt(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d, c=c, status=status)
    return d


def _oracle_dense(orc, case, rows=None, cols=None):
    M, N, K = case.shape
    sa = case.sfa.double().numpy()
    sbr = sb_rows(case.sfb, N)
    c = None if case.c is None else bf16_bits(case.c)
    if rows is None:
        return orc.gemm_nt(u8(case.a), sa, u8(case.b), sbr, c=c)
    return orc.gemm_nt_sampled(u8(case.a), sa, u8(case.b), sbr, rows, cols, c=c)


# ------------------------------------------------------------------ scale transform

@pytest.mark.parametrize("batch,mn,sf_k,gran", [(1, 5, 6, 1), (1, 4096, 128, 1), (1, 2112, 56, 128),
                                                (32, 256, 56, 1), (8, 4096, 56, 128),
                                                (1, 30, 3, 1), (3, 130, 9, 128)])
def test_transform_sf_bit_exact(orc, batch, mn, sf_k, gran):
    g = inputs.generator(batch * 1000 + mn)
    rows = -(-mn // gran)
    e = torch.randint(-20, 10, (batch, rows, sf_k), generator=g)
    sf = torch.ldexp(torch.ones(batch, rows, sf_k, dtype=torch.float64), e).float()
    status = _status()
    got = binding.transform_sf(sf.to(DEV), gran, mn, status=status)
    ref, inexact = orc.transform_sf(sf.numpy(), gran, mn)
    assert inexact == 0 and int(status.item()) == 0
    assert np.array_equal(got.cpu().numpy(), ref)
    got32 = binding.transform_sf(sf.to(DEV), gran, mn, packed=False)
    ref32, _ = orc.transform_sf(sf.numpy(), gran, mn, packed=False)
    assert np.array_equal(got32.cpu().numpy(), ref32)


def test_transform_sf_truncates_and_flags_inexact(orc):
    sf = torch.tensor([[0.75, 3.0, 1.0, 2.0 ** -9, 5.5]], dtype=torch.float32)
    status = _status()
    got = binding.transform_sf(sf.to(DEV), 1, 1, status=status)
    ref, inexact = orc.transform_sf(sf.numpy(), 1, 1)
    assert np.array_equal(got.cpu().numpy(), ref)
    assert inexact == 3
    assert int(status.item()) & binding.DG_DEV_INEXACT_SCALE


# ------------------------------------------------------------------ dense GEMM

@pytest.mark.parametrize("M,N,K", [(128, 256, 512),     # the small workload, in full
                                   (200, 2112, 640),     # ragged M, N with a half 128-block
                                   (1, 16, 128), (129, 264, 336),   # K % 128 != 0
                                   (300, 520, 1024), (64, 7168, 256)])
def test_dense_full_compare(orc, M, N, K):
    case = inputs.dense_case(M, N, K, seed=M + N + K)
    status = _status()
    d = _run_dense(case, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(bf16_bits(d), _oracle_dense(orc, case), f"{M}x{N}x{K}")


def test_dense_integer_exact_bitwise(orc):
    case = inputs.integer_exact_case(256, 384, 1024, seed=3)
    d = _run_dense(case)
    ref = _oracle_dense(orc, case)
    assert np.array_equal(bf16_bits(d), ref)


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (130, 264, 384)])
def test_dense_with_c_and_spread_scales(orc, M, N, K):
    case = inputs.dense_case(M, N, K, seed=7, with_c=True, b_scale_exp_range=(-8, 4))
    c = case.c.to(DEV)
    d = _run_dense(case, c=c)
    ref = _oracle_dense(orc, case)
    assert_close(bf16_bits(d), ref, "with C")
    # in place: c is d
    d2 = c.clone()
    _run_dense(case, c=d2, d=d2)
    assert np.array_equal(bf16_bits(d2), bf16_bits(d))


def test_dense_strided_operands(orc):
    """Leading dimensions larger than the logical widths."""
    M, N, K = 150, 136, 384
    case = inputs.dense_case(M, N, K, seed=9, with_c=True)
    a_big = torch.zeros(M, K + 64, dtype=torch.float8_e4m3fn)
    a_big[:, :K] = case.a
    b_big = torch.zeros(N, K + 32, dtype=torch.float8_e4m3fn)
    b_big[:, :K] = case.b
    c_big = torch.zeros(M, N + 24, dtype=torch.bfloat16)
    c_big[:, :N] = case.c
    d_big = torch.full((M, N + 40), 7.0, dtype=torch.bfloat16, device=DEV)
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    a_dev, b_dev, c_dev = a_big.to(DEV), b_big.to(DEV), c_big.to(DEV)
    binding.dg_fp8_gemm_nt(a_dev[:, :K], sfa, b_dev[:, :K], sfb, d_big[:, :N], c=c_dev[:, :N])
    assert_close(bf16_bits(d_big[:, :N]), _oracle_dense(orc, case), "strided")
    assert bool((d_big[:, N:] == 7.0).all()), "wrote outside [M, N]"


@pytest.mark.parametrize("M,N,K,with_c", [(128, 256, 512, False), (200, 264, 640, True),
                                          (300, 520, 1024, False), (64, 2112, 7168, True),
                                          (129, 136, 336, False)])
def test_dense_fp32_scales_promotion(orc, M, N, K, with_c):
    """FP32 scales that are not powers of two: the two-level promotion kernel
    honours them exactly (no UE8M0 truncation)."""
    case = inputs.dense_case(M, N, K, seed=M * 7 + K, with_c=with_c)
    g = inputs.generator(5)
    mult = torch.tensor([0.75, 1.0, 3.0, 1.1, 0.6])
    sfa = case.sfa * mult[torch.randint(0, 5, case.sfa.shape, generator=g)]
    sfb = case.sfb * mult[torch.randint(0, 5, case.sfb.shape, generator=g)]
    case.sfa, case.sfb = sfa, sfb
    d = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    status = _status()
    binding.dg_fp8_gemm_nt(case.a.to(DEV), sfa.to(DEV), case.b.to(DEV), sfb.to(DEV), d,
                           c=None if case.c is None else case.c.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert binding.last_config()["kind"] == 1
    assert_close(bf16_bits(d), _oracle_dense(orc, case), f"fp32 scales {M}x{N}x{K}")


def test_fp32_and_packed_paths_agree_on_pow2_scales():
    """With power-of-two scales both kernels compute the same GEMM; results
    agree to within the accumulation-order tolerance."""
    case = inputs.dense_case(256, 512, 2048, seed=21)
    a, b = case.a.to(DEV), case.b.to(DEV)
    d1 = torch.empty(256, 512, dtype=torch.bfloat16, device=DEV)
    d2 = torch.empty_like(d1)
    binding.dg_fp8_gemm_nt(a, case.sfa.to(DEV), b, case.sfb.to(DEV), d1)
    binding.dg_fp8_gemm_nt(a, binding.transform_sf(case.sfa.to(DEV), 1, 256), b,
                           binding.transform_sf(case.sfb.to(DEV), 128, 512), d2)
    assert_close(bf16_bits(d1), bf16_bits(d2), "fp32 vs packed")


def test_dense_k_zero_gives_c():
    c = torch.randn(40, 64, device=DEV).to(torch.bfloat16)
    d = torch.empty_like(c)
    a = torch.empty(40, 0, dtype=torch.float8_e4m3fn, device=DEV)
    b = torch.empty(64, 0, dtype=torch.float8_e4m3fn, device=DEV)
    sf = torch.empty(1, 64, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nt(a, sf, b, sf, d, c=c)
    assert torch.equal(d, c)


@pytest.mark.parametrize("M", [128, 4096])
@pytest.mark.parametrize("N,K", inputs.V3_NK)
def test_dense_workload_shapes_sampled(orc, M, N, K):
    """The V3-like workload (six GEMMs) at full size, 3000 sampled elements
    against the oracle, plus every element finite."""
    case = inputs.dense_case(M, N, K, seed=0)
    status = _status()
    d = _run_dense(case, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(M + N)
    rows = rng.integers(0, M, 3000)
    cols = rng.integers(0, N, 3000)
    # always include the corners and the ragged N tail
    rows[:4] = [0, 0, M - 1, M - 1]
    cols[:4] = [0, N - 1, 0, N - 1]
    ref = _oracle_dense(orc, case, rows, cols)
    got = bf16_bits(d)
    assert_close(got[rows, cols], ref, f"{M}x{N}x{K} sampled")
    assert bool(torch.isfinite(d.float()).all())


def test_batch_invariance_bitwise():
    """Rows [0, M) of a problem with M rows are bit-identical to the same rows
    of the M=4096 problem (C-accumulate workload, spread B scales)."""
    M, N, K = 4096, 7168, 2048
    case = inputs.dense_case(M, N, K, seed=2, with_c=True, b_scale_exp_range=(-8, 4))
    a, b, c = case.a.to(DEV), case.b.to(DEV), case.c.to(DEV)
    sfa_full = case.sfa.to(DEV)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d_full = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    binding.dg_fp8_gemm_nt(a, binding.transform_sf(sfa_full, 1, M), b, sfb, d_full, c=c)
    seen = set()
    for m in [1, 2, 7, 64, 127, 128, 129, 255, 1000, 2048, 4095]:
        d = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
        binding.dg_fp8_gemm_nt(a[:m], binding.transform_sf(sfa_full[:m].contiguous(), 1, m), b,
                               sfb, d, c=c[:m])
        seen.add(binding.last_config()["block_n"])
        assert torch.equal(d, d_full[:m]), f"rows differ at M={m}"
    assert len(seen) >= 2, "the sweep should exercise more than one tile shape"


# ------------------------------------------------------------------ grouped GEMMs

def _contiguous(case):
    M_total = case.a.shape[0]
    E, N, K = case.b.shape
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M_total)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.full((M_total, N), 3.0, dtype=torch.bfloat16, device=DEV)
    status = _status()
    binding.dg_m_grouped_fp8_gemm_nt_contiguous(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d,
                                                case.grouped_layout.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d


def test_contiguous_small_full(orc):
    case = inputs.contiguous_case(4, 264, 512, seed=4, m_per_expert=[5, 130, 0, 128])
    d = _contiguous(case)
    layout = case.grouped_layout.numpy()
    valid = layout >= 0
    ref = orc.m_grouped_contiguous(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                                   sb_rows(case.sfb, 264), layout)
    assert_close(bf16_bits(d)[valid], ref[valid], "contiguous")


def test_contiguous_padding_block_skipped(orc):
    """A 128-row block whose first row is -1 is skipped: D keeps its contents."""
    case = inputs.contiguous_case(3, 136, 256, seed=8, m_per_expert=[128, 128, 128])
    case.grouped_layout[128:256] = -1
    d = _contiguous(case)
    layout = case.grouped_layout.numpy()
    assert bool((d[128:256] == 3.0).all())
    ref = orc.m_grouped_contiguous(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                                   sb_rows(case.sfb, 136), layout)
    valid = layout >= 0
    assert_close(bf16_bits(d)[valid], ref[valid], "contiguous with a padding block")


def test_contiguous_workload_sampled(orc):
    for (N, K) in [(4096, 7168), (7168, 2048)]:
        case = inputs.contiguous_case(8, N, K, seed=1)
        d = _contiguous(case)
        layout = case.grouped_layout.numpy()
        rng = np.random.default_rng(N)
        valid_rows = np.nonzero(layout >= 0)[0]
        rows = valid_rows[rng.integers(0, len(valid_rows), 3000)]
        cols = rng.integers(0, N, 3000)
        got = bf16_bits(d)[rows, cols]
        a, sa = u8(case.a), case.sfa.double().numpy()
        sbr = sb_rows(case.sfb, N)
        ref = np.empty(3000, dtype=np.uint16)
        for e in range(8):
            sel = np.nonzero(layout[rows] == e)[0]
            if len(sel):
                ref[sel] = orc.gemm_nt_sampled(a, sa, u8(case.b[e]), sbr[e], rows[sel], cols[sel])
        assert_close(got, ref, f"contiguous N={N} K={K}")


def test_contiguous_bad_expert_flagged():
    case = inputs.contiguous_case(2, 128, 256, seed=5, m_per_expert=[128, 128])
    case.grouped_layout[128:] = 7       # out of range
    M_total = case.a.shape[0]
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M_total)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, 128)
    d = torch.full((M_total, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    status = _status()
    binding.dg_m_grouped_fp8_gemm_nt_contiguous(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d,
                                                case.grouped_layout.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.DG_DEV_BAD_GROUP
    assert bool((d[128:] == 3.0).all())


def _masked(case, canary=5.0):
    E, max_m, K = case.a.shape
    N = case.b.shape[1]
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, max_m)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.full((E, max_m, N), canary, dtype=torch.bfloat16, device=DEV)
    status = _status()
    binding.dg_m_grouped_fp8_gemm_nt_masked(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d,
                                            case.masked_m.to(DEV), case.expected_m, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d


def test_masked_small_full(orc):
    case = inputs.masked_case(5, 200, 264, 384, seed=6, masked_m=[0, 200, 7, 128, 129])
    d = _masked(case)
    ref = orc.m_grouped_masked(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                               sb_rows(case.sfb, 264), case.masked_m.numpy())
    got = bf16_bits(d)
    for e, m in enumerate(case.masked_m.tolist()):
        if m:
            assert_close(got[e, :m], ref[e, :m], f"masked expert {e}")
        assert bool((d[e, m:] == 5.0).all()), f"expert {e} wrote rows past masked_m"


def test_masked_workload_sampled(orc):
    case = inputs.masked_case(32, 256, 4096, 7168, seed=0)
    d = _masked(case)
    mm = case.masked_m.numpy()
    rng = np.random.default_rng(0)
    got = bf16_bits(d)
    a, sa = u8(case.a), case.sfa.double().numpy()
    sbr = sb_rows(case.sfb, 4096)
    for e in range(32):
        if mm[e]:
            rows = rng.integers(0, mm[e], 60)
            cols = rng.integers(0, 4096, 60)
            ref = orc.gemm_nt_sampled(a[e], sa[e], u8(case.b[e]), sbr[e], rows, cols)
            assert_close(got[e][rows, cols], ref, f"masked expert {e}")
        assert bool((d[e, mm[e]:] == 5.0).all())
