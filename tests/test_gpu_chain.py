"""GEMMs launched back to back on one stream, each reading the previous one's
output as its C.

The kernels are launched as programmatic dependents of the stream's previous
grid: their prologue may overlap it, but every thread waits for it to finish
before touching global memory.  A read of C (or a write of D) that ran ahead
of the previous GEMM would pick up the canary value D started with.
"""
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


@pytest.mark.parametrize("M,N,K,flags", [
    (1024, 2048, 2048, 0),                          # 256-row CTA pairs
    (1024, 2304, 2048, binding.DG_DEBUG_WIDE_PAIR),  # first GEMM on 384-column tiles
    (128, 2048, 4096, 0),                           # 128-row pairs, then single CTAs with C
])
def test_chain_reads_previous_output_as_c(orc, M, N, K, flags):
    cases = [inputs.dense_case(M, N, K, seed=100 + i) for i in range(3)]
    packed = [(c.a.to(DEV), binding.transform_sf(c.sfa.to(DEV), 1, M), c.b.to(DEV),
               binding.transform_sf(c.sfb.to(DEV), 128, N)) for c in cases]
    ds = [torch.full((M, N), 1000.0, dtype=torch.bfloat16, device=DEV) for _ in cases]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    binding.set_debug_flags(flags)
    try:
        for i, (a, sfa, b, sfb) in enumerate(packed):
            binding.dg_fp8_gemm_nt(a, sfa, b, sfb, ds[i], c=ds[i - 1] if i else None, status=status)
    finally:
        binding.set_debug_flags(0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    prev = None
    for i, case in enumerate(cases):
        ref = orc.gemm_nt(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, N),
                          c=prev)
        got = bf16_bits(ds[i])
        assert_close(got, ref, f"chain step {i} {M}x{N}x{K}")
        prev = got   # the next step's C is this step's GPU output
