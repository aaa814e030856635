"""FP8 x FP4 GEMM ("DeepSeek V4 源码剖析 第13章" §13.1 reason 2, §13.5: E2M1
weights with one scale per 32 K, the mixed operands fed to the tensor cores)
against the oracle, and bit for bit against the FP8 GEMM when the weights'
32-K scales are equal within each 128-K block (the E2M1 codes re-encoded as
E4M3, exactly): the same products in the same order."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _b_device(b: torch.Tensor, pad: int = 0) -> torch.Tensor:
    """Packed codes [N, K/2] on the device, rows 32-byte aligned (+ pad bytes)."""
    n, kb = b.shape
    ld = (kb + 31) // 32 * 32 + pad
    wide = torch.zeros(n, ld, dtype=torch.uint8)
    wide[:, :kb] = b
    return wide.to(DEV)[:, :kb]


def _run(case, c=None, pad=0):
    M, N, K = case.shape
    sfa = binding.transform_sf(case.sfa.to(DEV), 1, M)
    sfb = binding.transform_sf(case.sfb.to(DEV), 1, N)     # [N, K/32] -> [K/128, align4(N)]
    d = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_fp8_fp4_gemm_nt(case.a.to(DEV), sfa, _b_device(case.b, pad), sfb, d, c=c, status=status)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d, cfg


@pytest.mark.parametrize("M,N,K,with_c,pad", [(256, 256, 512, False, 0), (300, 1000, 384, True, 32),
                                              (17, 96, 128, False, 0), (1000, 2048, 1536, True, 0),
                                              (513, 264, 896, False, 64), (128, 7168, 2048, False, 0),
                                              (64, 2112, 1024, False, 0), (100, 24576, 384, False, 32),
                                              (128, 520, 640, True, 0)])
def test_fp4_matches_oracle(orc, M, N, K, with_c, pad):
    case = inputs.fp4_case(M, N, K, seed=M + N + K, with_c=with_c)
    c = case.c.to(DEV) if with_c else None
    d, cfg = _run(case, c=c, pad=pad)
    # M <= 128 without C: 128-row pairs; otherwise 256-row pairs
    assert cfg["kind"] == 2 and cfg["block_m"] == (128 if M <= 128 and not with_c else 256), cfg
    ref = orc.gemm_fp8_fp4_nt(u8(case.a), case.sfa.double().numpy(), case.b.numpy(), case.sfb.double().numpy(),
                              c=None if c is None else bf16_bits(case.c))
    assert_close(bf16_bits(d), ref, f"fp4 {M}x{N}x{K}")


def test_fp4_batch_invariance_bitwise():
    """Rows [0, m) of a call with m rows equal the same rows of the m=4096 call
    bit for bit, across the 128-row pair tiles (m <= 128) and the 256-row ones."""
    M, N, K = 4096, 2112, 1536
    case = inputs.fp4_case(M, N, K, seed=77)
    a = case.a.to(DEV)
    b = _b_device(case.b)
    sfb = binding.transform_sf(case.sfb.to(DEV), 1, N)
    d_full = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    binding.dg_fp8_fp4_gemm_nt(a, binding.transform_sf(case.sfa.to(DEV), 1, M), b, sfb, d_full)
    seen = set()
    for m in [1, 17, 128, 129, 1000]:
        d = torch.empty(m, N, dtype=torch.bfloat16, device=DEV)
        binding.dg_fp8_fp4_gemm_nt(a[:m], binding.transform_sf(case.sfa[:m].contiguous().to(DEV), 1, m), b,
                                   sfb, d)
        cfg = binding.last_config()
        seen.add((cfg["block_m"], cfg["block_n"]))
        torch.cuda.synchronize()
        assert torch.equal(d, d_full[:m]), f"rows differ at m={m} ({cfg})"
    assert {bm for bm, _ in seen} == {128, 256}, seen


def test_fp4_equals_fp8_gemm_on_the_same_values():
    M, N, K = 512, 768, 1024
    case = inputs.fp4_case(M, N, K, seed=91)
    # one scale per 128-K block of each row, repeated over its four 32-K blocks
    s128 = case.sfb[:, ::4].contiguous()
    case.sfb = s128.repeat_interleave(4, dim=1).contiguous()
    d4, _ = _run(case)
    codes = torch.stack([case.b & 0xF, case.b >> 4], dim=-1).reshape(N, K).long()
    b8 = E2M1[codes].to(torch.float8_e4m3fn)
    assert torch.equal(b8.float(), E2M1[codes])
    d8 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    binding.dg_fp8_gemm_nt(case.a.to(DEV), binding.transform_sf(case.sfa.to(DEV), 1, M), b8.to(DEV),
                           binding.transform_sf(s128.to(DEV), 1, N), d8)
    torch.cuda.synchronize()
    assert torch.equal(d4, d8)


def test_fp4_workload_sampled(orc):
    """4096 x 7168 x 16384 (the largest V3-like shape with FP4 weights) on sampled outputs."""
    M, N, K = 4096, 7168, 16384
    case = inputs.fp4_case(M, N, K, seed=92)
    d, _ = _run(case)
    rng = np.random.default_rng(7)
    rows, cols = rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    ref = orc.gemm_fp8_fp4_nt_sampled(u8(case.a), case.sfa.double().numpy(), case.b.numpy(),
                                      case.sfb.double().numpy(), rows, cols)
    assert_close(bf16_bits(d)[rows, cols], ref, "fp4 workload")


def test_fp4_rejects_k_not_multiple_of_128():
    lib = binding.lib()
    P = binding._p
    a = torch.empty(128, 192, dtype=torch.float8_e4m3fn, device=DEV)
    b = torch.empty(128, 96, dtype=torch.uint8, device=DEV)
    sf = torch.empty(64, dtype=torch.int32, device=DEV)
    d = torch.empty(128, 128, dtype=torch.bfloat16, device=DEV)
    st = lib.dg_fp8_fp4_gemm_nt(P(a), 192, P(sf), P(b), 96, P(sf), None, 0, P(d), 128, 128, 128, 192, None, None)
    assert st == 2   # DG_ERR_ALIGNMENT


def _experts(E, N, K, seed):
    cases = [inputs.fp4_case(1, N, K, seed=seed + e) for e in range(E)]
    return torch.stack([c.b for c in cases]), torch.stack([c.sfb for c in cases])


@pytest.mark.parametrize("m_per_expert,N,K", [([5, 130, 0, 256, 300], 264, 512), ([128] * 4, 7168, 2048),
                                              ([1000, 17], 520, 1152)])
def test_fp4_contiguous_matches_oracle(orc, m_per_expert, N, K):
    E = len(m_per_expert)
    base = inputs.contiguous_case(E, 8, K, seed=sum(m_per_expert), m_per_expert=m_per_expert)
    b, sfb = _experts(E, N, K, seed=95)
    M = base.a.shape[0]
    sfa_p = binding.transform_sf(base.sfa.to(DEV), 1, M)
    sfb_p = binding.transform_sf(sfb.contiguous().to(DEV), 1, N)
    d = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(base.a.to(DEV), sfa_p, b.to(DEV), sfb_p, d,
                                                    base.grouped_layout.to(DEV), status=status)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and cfg["kind"] == 2 and cfg["block_m"] == 256, cfg
    init = bf16_bits(torch.full((M, N), 7.0, dtype=torch.bfloat16))
    ref = orc.m_grouped_fp8_fp4_contiguous(u8(base.a), base.sfa.double().numpy(), b.numpy(),
                                           sfb.double().numpy(), base.grouped_layout.numpy(), d_init=init)
    got = bf16_bits(d)
    layout = base.grouped_layout.numpy()
    valid = layout >= 0
    if valid.any():
        assert_close(got[valid], ref[valid], f"fp4 contiguous {m_per_expert}")
    # 128-row blocks that start with padding are left untouched (as in the FP8 layout;
    # padding rows inside an expert's block are computed from their A rows)
    for mb in range(len(layout) // 128):
        if layout[mb * 128] < 0:
            assert np.array_equal(got[mb * 128:(mb + 1) * 128], init[mb * 128:(mb + 1) * 128])
    # each expert's rows equal the dense FP8 x FP4 GEMM of those rows, bit for bit
    for e in range(E):
        rows = np.nonzero(base.grouped_layout.numpy() == e)[0]
        if len(rows) == 0:
            continue
        ae = base.a.view(torch.uint8)[torch.from_numpy(rows)].view(torch.float8_e4m3fn)
        de = torch.empty(len(rows), N, dtype=torch.bfloat16, device=DEV)
        binding.dg_fp8_fp4_gemm_nt(ae.to(DEV), binding.transform_sf(base.sfa[torch.from_numpy(rows)].to(DEV), 1,
                                                                    len(rows)),
                                   b[e].to(DEV), binding.transform_sf(sfb[e].contiguous().to(DEV), 1, N), de)
        torch.cuda.synchronize()
        if binding.last_config()["block_m"] == 256:
            assert torch.equal(de, d[torch.from_numpy(rows).to(DEV)]), e


@pytest.mark.parametrize("masked_m,max_m,N,K", [([0, 256, 17, 300], 320, 264, 512), ([5, 128, 64], 128, 7168, 1024)])
def test_fp4_masked_matches_oracle(orc, masked_m, max_m, N, K):
    E = len(masked_m)
    base = inputs.masked_case(E, max_m, 8, K, seed=sum(masked_m), masked_m=masked_m)
    b, sfb = _experts(E, N, K, seed=97)
    sfa_p = binding.transform_sf(base.sfa.to(DEV), 1, max_m)
    sfb_p = binding.transform_sf(sfb.contiguous().to(DEV), 1, N)
    d = torch.full((E, max_m, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_m_grouped_fp8_fp4_gemm_nt_masked(base.a.to(DEV), sfa_p, b.to(DEV), sfb_p, d,
                                                base.masked_m.to(DEV), base.expected_m, status=status)
    torch.cuda.synchronize()
    clamped = [min(m, max_m) for m in masked_m]
    flag = binding.DG_DEV_BAD_GROUP if any(m > max_m for m in masked_m) else 0
    assert int(status.item()) == flag
    init = bf16_bits(torch.full((E, max_m, N), 7.0, dtype=torch.bfloat16))
    ref = orc.m_grouped_fp8_fp4_masked(u8(base.a), base.sfa.double().numpy(), b.numpy(), sfb.double().numpy(),
                                       clamped, d_init=init)
    got = bf16_bits(d)
    for e in range(E):
        m = clamped[e]
        if m:
            assert_close(got[e, :m], ref[e, :m], f"fp4 masked expert {e}")
        assert np.array_equal(got[e, m:], ref[e, m:])
