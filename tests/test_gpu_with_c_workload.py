"""The C-accumulate workload at its own size against the oracle.

D = C + A @ B^T ("DeepSeek V4 源码剖析 第13章" §13.3) with M=4096, N=7168,
K=2048, C ~ N(0,1) in bf16 and every 128x128 B block scale replaced by 2^u,
u uniform in [-8, 4].  The launch is the one the benchmark times (256-row CTA
pairs, the 224-column tile with C).  3000 sampled elements, the four corners
among them, are compared with the oracle's one-by-one sums, for the bf16 NT
GEMM, the FP32-output GEMM (FP32 C) and the NN / TN / TT layouts; the layouts
must also equal the NT result bit for bit.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
M, N, K = 4096, 7168, 2048
NSAMP = 3000


@pytest.fixture(scope="module")
def work():
    case = inputs.dense_case(M, N, K, seed=2, with_c=True, b_scale_exp_range=(-8, 4))
    rng = np.random.default_rng(2)
    rows = rng.integers(0, M, NSAMP)
    cols = rng.integers(0, N, NSAMP)
    rows[:4] = [0, 0, M - 1, M - 1]
    cols[:4] = [0, N - 1, 0, N - 1]
    dev = {
        "a": case.a.to(DEV), "b": case.b.to(DEV), "c": case.c.to(DEV),
        "sfa": binding.transform_sf(case.sfa.to(DEV), 1, M),
        "sfb": binding.transform_sf(case.sfb.to(DEV), 128, N),
    }
    host = {"a": u8(case.a), "b": u8(case.b), "sa": case.sfa.double().numpy(),
            "sbr": sb_rows(case.sfb, N), "c": bf16_bits(case.c)}
    return case, dev, host, rows, cols


@pytest.fixture(scope="module")
def nt_result(work):
    case, dev, host, rows, cols = work
    d = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nt(dev["a"], dev["sfa"], dev["b"], dev["sfb"], d, c=dev["c"], status=status)
    cfg = binding.last_config()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return d, cfg


def test_with_c_workload_nt_sampled(orc, work, nt_result):
    case, dev, host, rows, cols = work
    d, cfg = nt_result
    assert cfg["kind"] == 2 and cfg["block_m"] == 256, cfg
    ref = orc.gemm_nt_sampled(host["a"], host["sa"], host["b"], host["sbr"], rows, cols, c=host["c"])
    got = bf16_bits(d)
    assert_close(got[rows, cols], ref, f"{M}x{N}x{K} + C, sampled")
    assert bool(torch.isfinite(d.float()).all())


def test_with_c_workload_f32_sampled(orc, work):
    """FP32 C (the bf16 C widened) and FP32 D: per element within
    1e-4 |o| + 1e-4 rms(o) of the oracle rounded once to FP32."""
    case, dev, host, rows, cols = work
    c32 = dev["c"].float()
    d = torch.full((M, N), 7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nt_f32(dev["a"], dev["sfa"], dev["b"], dev["sfb"], d, c=c32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = orc.gemm_nt_f32_sampled(host["a"], host["sa"], host["b"], host["sbr"], rows, cols,
                                  c=c32.cpu().numpy())
    got = d.cpu().numpy()[rows, cols].astype(np.float64)
    o = ref.astype(np.float64)
    rms = float(np.sqrt(np.mean(o * o)))
    bad = np.abs(got - o) > 1e-4 * np.abs(o) + 1e-4 * rms
    assert not bad.any(), f"{int(bad.sum())} of {NSAMP} FP32 samples out of tolerance"
    assert bool(torch.isfinite(d).all())


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
def test_with_c_workload_layouts(orc, work, nt_result, layout):
    """A stored [K, M] for "t", B stored [K, N] for "n": the same products in
    the same order as NT, so the same bits; and the oracle's samples."""
    case, dev, host, rows, cols = work
    d_nt, _ = nt_result
    a = dev["a"].view(torch.uint8).t().contiguous().view(torch.float8_e4m3fn) if layout[0] == "t" else dev["a"]
    b = dev["b"].view(torch.uint8).t().contiguous().view(torch.float8_e4m3fn) if layout[1] == "n" else dev["b"]
    call = {"nn": binding.dg_fp8_gemm_nn, "tn": binding.dg_fp8_gemm_tn, "tt": binding.dg_fp8_gemm_tt}[layout]
    d = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    call(a, dev["sfa"], b, dev["sfb"], d, c=dev["c"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(d, d_nt), f"{layout} differs from NT"
    ref = orc.gemm_nt_sampled(host["a"], host["sa"], host["b"], host["sbr"], rows, cols, c=host["c"])
    assert_close(bf16_bits(d)[rows, cols], ref, f"{layout} {M}x{N}x{K} + C, sampled")
