"""How wide the block-scaled MMA accumulates ("02 · DeepGEMM 技术解析" §2.1-2.2;
"DeepSeek V4 源码剖析 第13章" §13.3 pt 1).

Hopper's FP8 MMA kept about 14 bits of its running sum, which is why the SM90
kernels promote every 128-K result on CUDA cores.  These rows are built from
power-of-two E4M3 values with unit scales, so every product and the exact sum
are known in closed form, and the FP32-output GEMM shows the accumulator itself:

  - in one 128-K block, one 2^10 (or 2^14) product and 127 products of +-2^-8
    sum exactly, wherever the large product sits (first, last, at the end of a
    32-K step): the sum needs up to 23 significant bits, and 14-bit accumulation
    would drop every small term;
  - 2^14 with 127 products of 2^-12 (27 bits) loses the small terms, so the
    MMA aligns its inputs to fewer than 27 bits;
  - over K = 1024 and 16384 the running sum is FP32: each 32-K MMA step can
    lose less than one unit in the last place of the sum, and every result lies
    on the zero side of the exact value (truncation, not rounding to nearest).

So one level of FP32 accumulation in TMEM over all of K is what the kernels use
for power-of-two scales; FP32 scales go through the promotion kernel.
"""
import math

import pytest
import torch

from block_scaled_fp8_gb300 import binding

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
M = N = 256

# row r of A and of B: (large value, small value, position of the large one in
# each 128-K block, sign of B's small values); D[r, r] is the probe
PATTERNS = {
    0: (32.0, 2.0 ** -4, 0, +1),
    1: (32.0, 2.0 ** -4, 127, +1),
    2: (32.0, 2.0 ** -4, 0, -1),
    3: (128.0, 2.0 ** -4, 0, +1),
    4: (128.0, 2.0 ** -6, 0, +1),
    5: (32.0, 2.0 ** -4, 31, +1),
}


def _operands(K):
    a = torch.zeros(M, K, dtype=torch.float32)
    b = torch.zeros(N, K, dtype=torch.float32)
    exact = {}
    for r, (big, small, pos, sign) in PATTERNS.items():
        j = torch.arange(K) % 128
        a[r] = torch.where(j == pos, big, small)
        b[r] = torch.where(j == pos, big, sign * small)
        # closed form: K/128 blocks of big^2 + 127 * sign * small^2 (all powers of two)
        exact[r] = (K // 128) * (big * big + 127 * sign * small * small)
    return a, b, exact


def _run(K):
    a, b, exact = _operands(K)
    a8, b8 = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
    assert torch.equal(a8.float(), a) and torch.equal(b8.float(), b)
    sfa = binding.transform_sf(torch.ones(M, K // 128, device=DEV), 1, M)
    sfb = binding.transform_sf(torch.ones((N + 127) // 128, K // 128, device=DEV), 128, N)
    d = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.dg_fp8_gemm_nt_f32(a8.to(DEV), sfa, b8.to(DEV), sfb, d, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return {r: float(d[r, r]) for r in PATTERNS}, exact


def _ulp32(x):
    return 2.0 ** (math.floor(math.log2(abs(x))) - 23)


def test_one_block_sums_exactly_to_23_bits():
    got, exact = _run(128)
    for r in (0, 1, 2, 3, 5):
        assert got[r] == exact[r], f"row {r}: {got[r]!r} != exact {exact[r]!r}"
    # 27 significant bits: the 2^-12 terms are dropped, nothing else is lost
    assert exact[4] - 2.0 ** -5 <= got[4] <= exact[4]


@pytest.mark.parametrize("K", [1024, 16384])
def test_long_k_is_fp32_accumulation_truncated_per_step(K):
    got, exact = _run(K)
    steps = K // 32
    for r in PATTERNS:
        err = got[r] - exact[r]
        assert abs(err) <= steps * _ulp32(exact[r]), f"K={K} row {r}: error {err!r}"
        assert err <= 0.0, f"K={K} row {r}: above the exact value ({err!r})"
    # the 1024-scale rows stay within a part in 2^18 even at K = 16384
    for r in (0, 1, 2, 5):
        assert abs(got[r] - exact[r]) <= abs(exact[r]) * 2.0 ** -18
