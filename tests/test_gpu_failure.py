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


@pytest.mark.parametrize("M,N,K,single_cta,kind,block_m", [
    (256, 512, 1024, False, 2, 256),    # 256-row CTA pairs
    (128, 2112, 1024, False, 2, 128),   # 128-row CTA pairs
    (256, 512, 1024, True, 0, 128),     # single CTA
])
def test_dropped_load_times_out_and_context_survives(orc, M, N, K, single_cta, kind, block_m):
    case = inputs.dense_case(M, N, K, seed=31)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    keep = binding.DG_DEBUG_SINGLE_CTA if single_cta else 0
    binding.set_wait_timeout_ms(100)
    try:
        binding.set_debug_flags(binding.DG_DEBUG_DROP_ONE_LOAD | keep)
        _gemm(case, status)
        cfg = binding.last_config()
        torch.cuda.synchronize()
        assert (cfg["kind"], cfg["block_m"]) == (kind, block_m)
        assert int(status.item()) & binding.DG_DEV_TIMEOUT
        # the drop flag cleared itself; the next GEMM is complete and correct
        status.zero_()
        d = _gemm(case, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    finally:
        binding.set_debug_flags(0)
        binding.set_wait_timeout_ms(2000)
    ref = orc.gemm_nt(u8(case.a), case.sfa.double().numpy(), u8(case.b), sb_rows(case.sfb, N))
    assert_close(bf16_bits(d), ref, "after timeout")
