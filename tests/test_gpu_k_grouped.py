"""K-grouped FP8 GEMM for MoE weight gradients (PaperTrace DeepGEMM §5.2,
§3.3): D[e] = C[e] + A_e^T B_e with the groups concatenated along K, against
the oracle; its packed scales bit for bit against the oracle's packing; and
bit for bit against the TN GEMM on each group's slice (C = 0, D rounded to
bf16): the group's K range changes where the loads start, not the products."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


def _padded(x: torch.Tensor, pad: int = 0) -> torch.Tensor:
    """x [rows, cols] float8 on the device as a view of a buffer whose row
    stride is cols rounded up to 16 bytes, plus pad."""
    rows, cols = x.shape
    ld = (cols + 15) // 16 * 16 + pad
    wide = torch.zeros(rows, ld, dtype=torch.uint8)
    wide[:, :cols] = x.view(torch.uint8)
    return wide.to(DEV)[:, :cols].view(torch.float8_e4m3fn)


def _close_f32(got, ref, what):
    """Per element |g - o| <= 1e-4 |o| + 1e-4 rms(o) (the FP32-output bar)."""
    o = ref.astype(np.float64)
    g = got.astype(np.float64)
    assert np.isfinite(g).all(), what
    rms = float(np.sqrt(np.mean(o * o))) if o.size else 0.0
    bad = np.abs(g - o) > 1e-4 * np.abs(o) + 1e-4 * rms
    assert not bad.any(), f"{what}: {int(bad.sum())} of {g.size} out of tolerance"


def _run(case, pad=0, in_place=False, status=None):
    E = len(case.ks)
    M, N = case.a.shape[1], case.b.shape[1]
    a, b = _padded(case.a, pad), _padded(case.b, pad)
    sfa = binding.dg_transform_sf_k_grouped(case.sfa.to(DEV), case.ks)
    sfb = binding.dg_transform_sf_k_grouped(case.sfb.to(DEV), case.ks)
    c = case.c.to(DEV)
    d = c if in_place else torch.full((E, M, N), 7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV) if status is None else status
    binding.dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, d, case.ks, c=c, status=st)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    return d, sfa, sfb, int(st.item()), cfg


@pytest.mark.parametrize("E,M,N,ks,pad", [(3, 256, 256, [128, 256, 384], 0),
                                          (4, 320, 264, [256, 0, 640, 128], 0),
                                          (2, 1000, 520, [1152, 128], 32),
                                          (1, 128, 128, [512], 0),
                                          (5, 64, 1032, [128, 128, 0, 0, 896], 16)])
def test_k_grouped_matches_oracle(orc, E, M, N, ks, pad):
    case = inputs.k_grouped_case(E, M, N, seed=E + M + N, ks=ks)
    d, sfa, sfb, status, cfg = _run(case, pad)
    assert status == 0
    assert cfg["kind"] == 2 and cfg["block_m"] == 256 and cfg["block_n"] == 224, cfg
    assert np.array_equal(sfa.cpu().numpy(), orc.k_grouped_pack_sf(case.sfa.numpy(), ks))
    assert np.array_equal(sfb.cpu().numpy(), orc.k_grouped_pack_sf(case.sfb.numpy(), ks))
    ref = orc.k_grouped_gemm_tn(u8(case.a), case.sfa.double().numpy(), u8(case.b), case.sfb.double().numpy(),
                                ks, case.c.numpy())
    got = d.cpu().numpy()
    for e in range(E):
        if ks[e] == 0:
            assert np.array_equal(got[e], case.c[e].numpy()), f"empty group {e}: D must be C"
        else:
            _close_f32(got[e], ref[e], f"group {e} of {ks}")


def test_k_grouped_in_place(orc):
    ks = [384, 128, 256]
    case = inputs.k_grouped_case(3, 256, 512, seed=71, ks=ks)
    d, _, _, status, _ = _run(case, in_place=True)
    assert status == 0
    ref = orc.k_grouped_gemm_tn(u8(case.a), case.sfa.double().numpy(), u8(case.b), case.sfb.double().numpy(),
                                ks, case.c.numpy())
    _close_f32(d.cpu().numpy(), ref, "in place")


@pytest.mark.parametrize("E,M,N,ks", [(4, 320, 264, [256, 0, 384, 128]), (2, 1000, 520, [1152, 128])])
def test_k_grouped_in_place_equals_separate(E, M, N, ks):
    """C passed as D itself is accumulated into D at L2 (TMA reduce-add; rows at
    the M edge by the owning thread); C in a buffer of its own is added in
    registers.  Both are one FP32 addition of C and the same sum: the same bits."""
    case = inputs.k_grouped_case(E, M, N, seed=E * M + N, ks=ks)
    d_sep, _, _, st_sep, _ = _run(case)
    d_in, _, _, st_in, _ = _run(case, in_place=True)
    assert st_sep == 0 and st_in == 0
    assert torch.equal(d_sep, d_in)
    for e, k in enumerate(ks):
        if k == 0:
            assert torch.equal(d_in[e].cpu(), case.c[e]), f"empty group {e}: D must stay C"


def test_k_grouped_equals_tn_per_group():
    ks = [256, 384, 128]
    E, M, N = 3, 512, 768
    case = inputs.k_grouped_case(E, M, N, seed=72, ks=ks)
    case.c.zero_()
    d, _, _, status, _ = _run(case)
    assert status == 0
    a, b = _padded(case.a), _padded(case.b)
    k0 = 0
    for e, k in enumerate(ks):
        s0, s1 = k0 // 128, (k0 + k) // 128
        # the TN GEMM on the group's rows, its scales packed per row of M and of N
        sfa = binding.transform_sf(case.sfa[s0:s1].t().contiguous().to(DEV), 1, M)
        sfb = binding.transform_sf(case.sfb[s0:s1].t().contiguous().to(DEV), 1, N)
        d16 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        binding.dg_fp8_gemm_tn(a[k0:k0 + k], sfa, b[k0:k0 + k], sfb, d16)
        torch.cuda.synchronize()
        assert torch.equal(d[e].to(torch.bfloat16), d16), f"group {e}"
        k0 += k


def test_k_grouped_all_empty_gives_c():
    case = inputs.k_grouped_case(2, 128, 256, seed=73, ks=[0, 0])
    c = case.c.to(DEV)
    d = torch.empty_like(c)
    empty = torch.empty(0, 128, dtype=torch.float8_e4m3fn, device=DEV)
    sf0 = torch.empty(0, 128, dtype=torch.int32, device=DEV)
    binding.dg_k_grouped_fp8_gemm_tn_contiguous(empty, sf0, torch.empty(0, 256, dtype=torch.float8_e4m3fn,
                                                                        device=DEV),
                                                torch.empty(0, 256, dtype=torch.int32, device=DEV), d, [0, 0], c=c)
    torch.cuda.synchronize()
    assert torch.equal(d, c)


def test_k_grouped_bad_device_sizes_flagged():
    """A device size that is not a multiple of 128 counts as 0 and is reported;
    nothing is read or written out of bounds."""
    ks = [128, 256]
    case = inputs.k_grouped_case(2, 256, 256, seed=74, ks=ks)
    a, b = _padded(case.a), _padded(case.b)
    sfa = binding.dg_transform_sf_k_grouped(case.sfa.to(DEV), ks)
    sfb = binding.dg_transform_sf_k_grouped(case.sfb.to(DEV), ks)
    c = case.c.to(DEV)
    d = torch.empty_like(c)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, d, ks, c=c, status=st,
                                                ks_dev=torch.tensor([128, 200], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert int(st.item()) & binding.DG_DEV_BAD_GROUP
    assert torch.equal(d[1], c[1])   # the group taken as empty: D = C


def test_k_grouped_workload_sampled(orc):
    """The weight-gradient workload (8 groups, M=4096, N=7168, sizes from the
    MoE token-count recipe) on sampled outputs."""
    E, M, N = 8, 4096, 7168
    case = inputs.k_grouped_case(E, M, N, seed=3)
    d, _, _, status, _ = _run(case, in_place=True)
    assert status == 0
    rng = np.random.default_rng(5)
    es, ms, ns = rng.integers(0, E, 3000), rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    ref = orc.k_grouped_gemm_tn_sampled(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                                        case.sfb.double().numpy(), case.ks, case.c.numpy(), es, ms, ns)
    got = d[torch.from_numpy(es).to(DEV), torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)].cpu().numpy()
    _close_f32(got, ref, "weight-gradient workload")


# ---------------------------------------------------------------- scales at a K granularity of 32

def _run32(case, pad=0, in_place=False):
    E = len(case.ks)
    M, N = case.a.shape[1], case.b.shape[1]
    a, b = _padded(case.a, pad), _padded(case.b, pad)
    sfa = binding.dg_transform_sf_k_grouped_k32(case.sfa.to(DEV), case.ks)
    sfb = binding.dg_transform_sf_k_grouped_k32(case.sfb.to(DEV), case.ks)
    c = case.c.to(DEV)
    d = c if in_place else torch.full((E, M, N), 7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_k_grouped_fp8_gemm_tn_contiguous_k32(a, sfa, b, sfb, d, case.ks, c=c, status=st)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    return d, sfa, sfb, int(st.item()), cfg


@pytest.mark.parametrize("E,M,N,ks,pad", [(3, 256, 256, [128, 256, 384], 0),
                                          (4, 320, 264, [256, 0, 640, 128], 0),
                                          (2, 1000, 520, [1152, 128], 32),
                                          (5, 64, 1032, [128, 128, 0, 0, 896], 16)])
def test_k_grouped_k32_matches_oracle(orc, E, M, N, ks, pad):
    """Scales every 32 rows of K (PaperTrace DeepGEMM §3.3): packing bit for bit
    against the oracle's, D against the oracle at the FP32 bar, in place and not."""
    case = inputs.k_grouped_case(E, M, N, seed=E + M + N + 32, ks=ks, gran_k=32)
    d, sfa, sfb, status, cfg = _run32(case, pad)
    assert status == 0
    assert cfg["kind"] == 2 and cfg["block_m"] == 256 and cfg["block_n"] == 192, cfg
    assert np.array_equal(sfa.cpu().numpy(), orc.k_grouped_pack_sf(case.sfa.numpy(), ks, gran_k=32))
    assert np.array_equal(sfb.cpu().numpy(), orc.k_grouped_pack_sf(case.sfb.numpy(), ks, gran_k=32))
    ref = orc.k_grouped_gemm_tn_k32(u8(case.a), case.sfa.double().numpy(), u8(case.b), case.sfb.double().numpy(),
                                    ks, case.c.numpy())
    got = d.cpu().numpy()
    for e in range(E):
        if ks[e] == 0:
            assert np.array_equal(got[e], case.c[e].numpy()), f"empty group {e}: D must be C"
        else:
            _close_f32(got[e], ref[e], f"group {e} of {ks}")
    d_in, _, _, st_in, _ = _run32(case, pad, in_place=True)
    assert st_in == 0 and torch.equal(d_in, d)


def test_k_grouped_k32_equals_k128_on_equal_scales():
    """32-row scales whose four rows in each 128-row block are equal give the
    128-row GEMM's result bit for bit (the same products in the same order; the
    two calls run different tile widths)."""
    ks = [256, 384, 0, 128]
    E, M, N = 4, 512, 776
    case = inputs.k_grouped_case(E, M, N, seed=76, ks=ks)
    d128, _, _, st128, _ = _run(case)
    case32 = inputs.KGroupedCase(case.a, case.sfa.repeat_interleave(4, 0).contiguous(), case.b,
                                 case.sfb.repeat_interleave(4, 0).contiguous(), case.c, ks)
    d32, _, _, st32, cfg = _run32(case32)
    assert st128 == 0 and st32 == 0 and cfg["block_n"] == 192
    assert torch.equal(d32, d128)


def test_k_grouped_k32_workload_sampled(orc):
    """The weight-gradient workload (8 groups, M=4096, N=7168) with 32-row scales,
    in place, on sampled outputs."""
    E, M, N = 8, 4096, 7168
    case = inputs.k_grouped_case(E, M, N, seed=33, gran_k=32)
    d, _, _, status, _ = _run32(case, in_place=True)
    assert status == 0
    rng = np.random.default_rng(6)
    es, ms, ns = rng.integers(0, E, 3000), rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    ref = orc.k_grouped_gemm_tn_k32_sampled(u8(case.a), case.sfa.double().numpy(), u8(case.b),
                                            case.sfb.double().numpy(), case.ks, case.c.numpy(), es, ms, ns)
    got = d[torch.from_numpy(es).to(DEV), torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)].cpu().numpy()
    _close_f32(got, ref, "weight-gradient workload, 32-row scales")
