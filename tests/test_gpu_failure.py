"""Failure detection without a GPU fault: a bounded device wait runs out.

The host asks the library to drop one operand load of the next GEMM
(DG_DEBUG_DROP_ONE_LOAD); the consumer's wait then runs out after the
configured limit, the kernel reports DG_DEV_TIMEOUT in the status word and
returns (nothing traps or hangs), and the context stays usable.
"""
import pytest
import torch

from block_scaled_fp8_gb300 import binding, inputs
from tests._util import assert_close, bf16_bits, sb_rows, u8

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _gemm(case, status):
    M, N, K = case.shape
    d = torch.full((M, N), 9.0, dtype=torch.bfloat16, device="cuda")
    binding.dg_fp8_gemm_nt(case.a.cuda(), binding.transform_sf(case.sfa.cuda(), 1, M),
                           case.b.cuda(), binding.transform_sf(case.sfb.cuda(), 128, N), d,
                           status=status)
    return d


def test_dropped_load_times_out_and_context_survives(orc):
    case = inputs.dense_case(256, 512, 1024, seed=31)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.set_wait_timeout_ms(100)
    try:
        binding.set_debug_flags(binding.DG_DEBUG_DROP_ONE_LOAD)
        _gemm(case, status)
        torch.cuda.synchronize()
        assert int(status.item()) & binding.DG_DEV_TIMEOUT
    finally:
        binding.set_debug_flags(0)
        binding.set_wait_timeout_ms(2000)
    # the flag cleared itself; the next GEMM is complete and correct
    status.zero_()
    d = _gemm(case, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = orc.gemm_nt(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, 512))
    assert_close(bf16_bits(d), ref, "after timeout")
