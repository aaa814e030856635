"""The contiguous grouped GEMM with PSUM offsets (256-row CTA pairs) against
the oracle and, bit for bit on the experts' rows, against the per-row-id
contiguous GEMM on the same inputs.

Expert e's rows are [S_e, S_e + m_e), S_0 = 0, S_{e+1} = S_e + align128(m_e):
the physical layout of the contiguous test cases, whose padding rows are the
gap rows here.  Gap rows must come back 0; rows past the last segment keep
their canary.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
CANARY = 7.0


def _with_slack(case, extra_blocks):
    """The case's A and FP32 A scales with extra_blocks * 128 rows appended."""
    if extra_blocks == 0:
        return case.a, case.sfa
    g = torch.Generator().manual_seed(99)
    rows = extra_blocks * 128
    codes = torch.randint(0, 0x7E, (rows, case.a.shape[1]), generator=g, dtype=torch.uint8)
    a = torch.cat([case.a.view(torch.uint8), codes]).view(torch.float8_e4m3fn)
    sfa = torch.cat([case.sfa, torch.ones(rows, case.sfa.shape[1])])
    return a, sfa


def _run_psum(a, sfa32, b, sfb32, psum, N):
    M = a.shape[0]
    sfa = binding.transform_sf(sfa32.to(DEV), 1, M)
    sfb = binding.transform_sf(sfb32.to(DEV), 128, N)
    d = torch.full((M, N), CANARY, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_m_grouped_fp8_gemm_nt_contiguous_psum(
        a.to(DEV), sfa, b.to(DEV), sfb, d, torch.tensor(psum, dtype=torch.int32, device=DEV),
        status=status)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    return d, int(status.item()), cfg


@pytest.mark.parametrize("m_per_expert,extra", [([5, 130, 0, 128, 300, 1], 0), ([256, 384, 129], 1),
                                                ([1, 1, 1, 1, 1], 2), ([0, 0, 7], 0)])
def test_psum_matches_oracle_and_row_id_layout(orc, m_per_expert, extra):
    E, N, K = len(m_per_expert), 264, 512
    case = inputs.contiguous_case(E, N, K, seed=7 + sum(m_per_expert), m_per_expert=m_per_expert)
    a, sfa32 = _with_slack(case, extra)
    psum = np.cumsum(m_per_expert).tolist()
    d, status, cfg = _run_psum(a, sfa32, case.b, case.sfb, psum, N)
    assert status == 0
    assert cfg["kind"] == 2 and cfg["block_m"] == 256, cfg
    ref = orc.m_grouped_contiguous_psum(u8(a), sfa32.double().numpy(), u8(case.b), sb_rows(case.sfb, N),
                                        psum, d_init=bf16_bits(torch.full((a.shape[0], N), CANARY,
                                                                          dtype=torch.bfloat16)))
    starts, counts = orc.psum_segments(psum, a.shape[0])
    got = bf16_bits(d)
    valid = np.zeros(a.shape[0], dtype=bool)
    for e, m in enumerate(counts):
        valid[starts[e]:starts[e] + m] = True
    if valid.any():
        assert_close(got[valid], ref[valid], f"psum {m_per_expert}")
    # gap rows are exactly 0, rows past the last segment keep the canary
    assert np.array_equal(got[~valid], ref[~valid])
    # the experts' rows are bit-identical to the per-row-id layout's
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, case.a.shape[0])
    sfb = binding.transform_sf(case.sfb.to(DEV), 128, N)
    d2 = torch.full(tuple(case.a.shape[:1]) + (N,), CANARY, dtype=torch.bfloat16, device=DEV)
    binding.dg_m_grouped_fp8_gemm_nt_contiguous(case.a.to(DEV), sfa, case.b.to(DEV), sfb, d2,
                                                case.grouped_layout.to(DEV))
    torch.cuda.synchronize()
    rows = np.nonzero(valid[:case.a.shape[0]])[0]
    assert torch.equal(d[:case.a.shape[0]][torch.from_numpy(rows).to(DEV)],
                       d2[torch.from_numpy(rows).to(DEV)])


def test_psum_workload_sampled(orc):
    """Config-3 sizes (8 experts, N=4096, K=7168) on sampled outputs, gap rows in full."""
    case = inputs.contiguous_case(8, 4096, 7168, seed=3)
    N = 4096
    psum = np.cumsum(case.m_per_expert).tolist()
    d, status, _ = _run_psum(case.a, case.sfa, case.b, case.sfb, psum, N)
    assert status == 0
    starts, counts = orc.psum_segments(psum, case.a.shape[0])
    got = bf16_bits(d)
    layout = np.full(case.a.shape[0], -1)
    for e, m in enumerate(counts):
        layout[starts[e]:starts[e] + m] = e
    assert np.all(got[layout < 0] == 0)
    rng = np.random.default_rng(11)
    rows = rng.choice(np.nonzero(layout >= 0)[0], 4000)
    cols = rng.integers(0, N, 4000)
    a = u8(case.a)
    sa = case.sfa.double().numpy()
    b = u8(case.b)
    sbr = sb_rows(case.sfb, N)
    ref = np.empty(len(rows), dtype=np.uint16)
    for e in range(8):
        sel = np.nonzero(layout[rows] == e)[0]
        if len(sel):
            ref[sel] = orc.gemm_nt_sampled(a, sa, b[e], sbr[e], rows[sel], cols[sel])
    assert_close(got[rows, cols], ref, "psum workload")


def test_psum_decreasing_offsets_flagged():
    E, N, K = 3, 136, 256
    case = inputs.contiguous_case(E, N, K, seed=5, m_per_expert=[100, 50, 10])
    # 100 then 90: the second count is negative (taken as 0) and reported
    _, status, _ = _run_psum(case.a, case.sfa, case.b, case.sfb, [100, 90, 100], N)
    assert status & binding.DG_DEV_BAD_GROUP
