"""The CTA-pair kernels (tcgen05 cta_group::2; 256- and 128-row tiles) against the oracle
and, bit for bit, against the single-CTA kernel on the same inputs.

Dense GEMMs with more than 128 rows, contiguous grouped GEMMs and masked ones
with many rows per expert run on 256-row pairs, skinny dense GEMMs on 128-row
pairs; DG_DEBUG_SINGLE_CTA forces the single-CTA kernel, so the two paths can
be compared directly.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


def _gemm(case, single_cta, c=None, flags=0):
    M, N, K = case.shape
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.full((M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.set_debug_flags((binding.DG_DEBUG_SINGLE_CTA if single_cta else 0) | flags)
    try:
        binding.dg_fp8_gemm_nt(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d, c=c, status=status)
        cfg = binding.last_config()
    finally:
        binding.set_debug_flags(0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d, cfg


# ragged M (one pair half empty, a tail pair), ragged N (half a 128-block),
# K not a multiple of 128 or of the 4-block scale group
SHAPES = [(256, 256, 512), (257, 200, 640), (300, 520, 1024), (384, 72, 128),
          (640, 1000, 336), (1000, 7168, 1536), (4096, 2112, 7168)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_matches_single_cta_bitwise(M, N, K):
    case = inputs.dense_case(M, N, K, seed=M * 3 + N + K, b_scale_exp_range=(-8, 4))
    d_pair, cfg_pair = _gemm(case, single_cta=False)
    d_one, cfg_one = _gemm(case, single_cta=True)
    assert cfg_pair["kind"] == 2 and cfg_pair["block_m"] == 256
    assert cfg_one["kind"] == 0 and cfg_one["block_m"] == 128
    assert torch.equal(d_pair, d_one), f"{M}x{N}x{K}: pair and single-CTA results differ"


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (300, 520, 1024), (1000, 264, 768)])
def test_pair_with_c_full_compare(orc, M, N, K):
    case = inputs.dense_case(M, N, K, seed=M + 11, with_c=True)
    d, cfg = _gemm(case, single_cta=False, c=case.c.to(DEV))
    assert cfg["kind"] == 2
    ref = orc.gemm_nt(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, N),
                      c=bf16_bits(case.c))
    assert_close(bf16_bits(d), ref, f"pair with C {M}x{N}x{K}")
    d_one, _ = _gemm(case, single_cta=True, c=case.c.to(DEV))
    assert torch.equal(d, d_one)


def test_pair_integer_exact_bitwise(orc):
    case = inputs.integer_exact_case(512, 640, 1024, seed=5)
    d, cfg = _gemm(case, single_cta=False)
    assert cfg["kind"] == 2
    ref = orc.gemm_nt(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, 640))
    assert np.array_equal(bf16_bits(d), ref)


def test_pair_full_compare_several_waves(orc):
    """More pair tiles than co-resident pairs: every pair runs several tiles
    (accumulator double-buffering and the scale ring wrap many times)."""
    M, N, K = 2048, 4096, 640
    case = inputs.dense_case(M, N, K, seed=17)
    d, cfg = _gemm(case, single_cta=False)
    assert cfg["kind"] == 2
    tiles = (M // 256) * -(-N // cfg["block_n"])
    assert tiles > cfg["grid"] // 2
    rng = np.random.default_rng(1)
    rows = rng.integers(0, M, 4000)
    cols = rng.integers(0, N, 4000)
    ref = orc.gemm_nt_sampled(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                              sb_rows(case.sfb, N), rows, cols)
    assert_close(bf16_bits(d)[rows, cols], ref, "pair several waves")


# ------------------------------------------------------------------ 384-column pair tiles

@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (300, 520, 1024), (512, 1000, 336), (1000, 7168, 1536),
                                   (2048, 4096, 640)])
def test_wide_pair_matches_single_cta_and_oracle(orc, M, N, K):
    """384-column tiles: two MMAs per K step (256 and 128 columns), each CTA
    holding half of each one's B rows; one TMEM accumulator, so tiles after
    the first wait for the epilogue.  Ragged N leaves the second MMA's rows
    partly or wholly past the end of B; K=336 is not a multiple of 128."""
    case = inputs.dense_case(M, N, K, seed=M + 2 * N + K, b_scale_exp_range=(-8, 4))
    d_wide, cfg = _gemm(case, single_cta=False, flags=binding.DG_DEBUG_WIDE_PAIR)
    d_one, _ = _gemm(case, single_cta=True)
    assert cfg["kind"] == 2 and cfg["block_m"] == 256 and cfg["block_n"] == 384, cfg
    assert torch.equal(d_wide, d_one), f"{M}x{N}x{K}: 384-column pairs and single CTAs differ"
    rng = np.random.default_rng(M + N)
    rows = rng.integers(0, M, 3000)
    cols = rng.integers(0, N, 3000)
    rows[:4] = [0, 0, M - 1, M - 1]
    cols[:4] = [0, N - 1, 0, N - 1]
    ref = orc.gemm_nt_sampled(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                              sb_rows(case.sfb, N), rows, cols)
    assert_close(bf16_bits(d_wide)[rows, cols], ref, f"wide pair {M}x{N}x{K}")


# ------------------------------------------------------------------ grouped layouts on pairs

def _contiguous(case, single_cta):
    M_total = case.a.shape[0]
    E, N, K = case.b.shape
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M_total)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.full((M_total, N), 3.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.set_debug_flags(binding.DG_DEBUG_SINGLE_CTA if single_cta else 0)
    try:
        binding.dg_m_grouped_fp8_gemm_nt_contiguous(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d,
                                                    case.grouped_layout.to(DEV), status=status)
        cfg = binding.last_config()
    finally:
        binding.set_debug_flags(0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d, cfg


@pytest.mark.parametrize("m_per_expert", [[5, 130, 0, 128, 300, 1], [256, 384, 129], [1, 1, 1, 1, 1]])
def test_contiguous_pair_matches_single_cta_and_oracle(orc, m_per_expert):
    """Expert segments (padded to 128 rows) of odd and even block counts, so
    256-row pairs both share an expert and straddle two."""
    E, N, K = len(m_per_expert), 264, 512
    case = inputs.contiguous_case(E, N, K, seed=sum(m_per_expert), m_per_expert=m_per_expert)
    d_pair, cfg = _contiguous(case, single_cta=False)
    d_one, cfg_one = _contiguous(case, single_cta=True)
    assert cfg["kind"] == 2 and cfg_one["kind"] == 0
    layout = case.grouped_layout.numpy()
    valid = layout >= 0
    assert torch.equal(d_pair[torch.from_numpy(valid).to(DEV)], d_one[torch.from_numpy(valid).to(DEV)])
    ref = orc.m_grouped_contiguous(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                                   sb_rows(case.sfb, N), layout)
    assert_close(bf16_bits(d_pair)[valid], ref[valid], f"contiguous pairs {m_per_expert}")
    # 128-row blocks that start with padding are left untouched by both
    for mb in range(len(layout) // 128):
        if layout[mb * 128] < 0:
            assert bool((d_pair[mb * 128:(mb + 1) * 128] == 3.0).all())


def _masked(case, single_cta, expected_m=None):
    E, max_m, K = case.a.shape
    N = case.b.shape[1]
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, max_m)
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d = torch.full((E, max_m, N), 5.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.set_debug_flags(binding.DG_DEBUG_SINGLE_CTA if single_cta else 0)
    try:
        binding.dg_m_grouped_fp8_gemm_nt_masked(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d,
                                                case.masked_m.to(DEV), expected_m or case.expected_m,
                                                status=status)
        cfg = binding.last_config()
    finally:
        binding.set_debug_flags(0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d, cfg


@pytest.mark.parametrize("max_m", [384, 520, 300])
def test_masked_pair_matches_single_cta_and_oracle(orc, max_m):
    """Masked layouts that expect more than 256 rows per expert run on pairs.
    Valid-row counts on both sides of 128 and 256 (a half-filled pair, a pair
    whose peer rows end inside its block); rows past masked_m keep their
    canary value."""
    mm = [m for m in [0, 1, 100, 128, 129, 200, 255, 256, 300, 384, 511, 520] if m <= max_m]
    N, K = 136, 384
    case = inputs.masked_case(len(mm), max_m, N, K, seed=max_m, masked_m=mm)
    d_pair, cfg = _masked(case, single_cta=False, expected_m=max_m)
    d_one, cfg_one = _masked(case, single_cta=True, expected_m=max_m)
    assert cfg["kind"] == 2 and cfg_one["kind"] == 0
    ref = orc.m_grouped_masked(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                               sb_rows(case.sfb, N), case.masked_m.numpy())
    got = bf16_bits(d_pair)
    for e, m in enumerate(mm):
        assert torch.equal(d_pair[e, :m], d_one[e, :m]), f"expert {e}: pair and single-CTA differ"
        if m:
            assert_close(got[e, :m], ref[e, :m], f"masked pairs expert {e}")
        assert bool((d_pair[e, m:] == 5.0).all()), f"expert {e} wrote rows past masked_m"


# ------------------------------------------------------------------ 128-row pairs (skinny M)

@pytest.mark.parametrize("M,N,K", [(128, 2112, 1024), (100, 7168, 640), (1, 2112, 384), (64, 7168, 2048),
                                   (128, 7168, 336)])
def test_skinny_pair_matches_single_cta_and_oracle(orc, M, N, K):
    """M <= 128 runs on 128-row pairs (64 rows of A per CTA; D columns split
    across TMEM lane halves) when the load model prefers them; the result is
    bit-identical to the single-CTA kernel and matches the oracle."""
    case = inputs.dense_case(M, N, K, seed=M + N + K, b_scale_exp_range=(-8, 4))
    d_pair, cfg = _gemm(case, single_cta=False)
    d_one, cfg_one = _gemm(case, single_cta=True)
    assert cfg["kind"] == 2 and cfg["block_m"] == 128, cfg
    assert cfg_one["kind"] == 0
    assert torch.equal(d_pair, d_one), f"{M}x{N}x{K}: 128-row pair and single-CTA results differ"
    rng = np.random.default_rng(M + K)
    rows = rng.integers(0, M, 3000)
    cols = rng.integers(0, N, 3000)
    rows[:4] = [0, 0, M - 1, M - 1]
    cols[:4] = [0, N - 1, 0, N - 1]
    ref = orc.gemm_nt_sampled(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                              sb_rows(case.sfb, N), rows, cols)
    assert_close(bf16_bits(d_pair)[rows, cols], ref, f"skinny pair {M}x{N}x{K}")
