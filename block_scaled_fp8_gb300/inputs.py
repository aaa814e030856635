"""Seeded synthetic inputs for the block-scaled FP8 GEMM.

Shared by the tests, the smoke check and the benchmark, for both the CUDA
library and the CPU oracle.  It holds none of the GEMM's arithmetic: it only
plays the upstream quantiser that the pages leave to the caller ("DeepGEMM
does not cast; it consumes already-quantised FP8 tensors and their scales",
PaperTrace DeepGEMM §1.1), on CPU with a seeded ``torch.Generator``.

Quantisation recipe (one reading of the pages):
  * activations: one FP32 scale per 1x128 K-group of each row; weights: one
    per 128x128 block (PaperTrace DeepGEMM §1.1);
  * scale s = 2^ceil(log2(amax/448)), i.e. absmax/448 rounded up to a power of
    two, so it is exact in UE8M0; s = 1 for an all-zero group;
  * codes q = float8_e4m3fn(x / s) with torch's CPU cast (round to nearest
    even); |x/s| <= 448 so nothing saturates.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0
GRAN = 128


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def pow2_scale(amax: torch.Tensor, qmax: float = E4M3_MAX) -> torch.Tensor:
    """Smallest power of two s (FP32, normal) with amax / s <= qmax (448 for
    E4M3, 6 for E2M1); 1 where amax == 0."""
    v = amax.double() / qmax
    mant, exp = torch.frexp(v)                      # v = mant * 2^exp, mant in [0.5, 1)
    e = torch.where(mant == 0.5, exp - 1, exp)      # ceil(log2 v)
    e = torch.clamp(e, min=-126, max=127)
    s = torch.ldexp(torch.ones_like(v), e)
    s = torch.where(amax.double() > qmax * s, s * 2, s)   # guard, never expected
    s = torch.where(amax == 0, torch.ones_like(s), s)
    return s.float()


def quantize_1x128(x: torch.Tensor):
    """x fp32 [R, K] -> (codes float8_e4m3fn [R, K], scales fp32 [R, ceil(K/128)])."""
    R, K = x.shape
    sf_k = cdiv(K, GRAN)
    xp = torch.nn.functional.pad(x, (0, sf_k * GRAN - K)).view(R, sf_k, GRAN)
    s = pow2_scale(xp.abs().amax(-1))
    q = (xp / s[..., None]).view(R, sf_k * GRAN)[:, :K].contiguous()
    return q.to(torch.float8_e4m3fn), s


def quantize_128x128(w: torch.Tensor):
    """w fp32 [N, K] -> (codes float8_e4m3fn [N, K], scales fp32 [ceil(N/128), ceil(K/128)])."""
    N, K = w.shape
    nb, kb = cdiv(N, GRAN), cdiv(K, GRAN)
    wp = torch.nn.functional.pad(w, (0, kb * GRAN - K, 0, nb * GRAN - N))
    blocks = wp.view(nb, GRAN, kb, GRAN)
    s = pow2_scale(blocks.abs().amax(dim=(1, 3)))
    q = (blocks / s[:, None, :, None]).reshape(nb * GRAN, kb * GRAN)[:N, :K].contiguous()
    return q.to(torch.float8_e4m3fn), s


def random_finite_e4m3(shape, g: torch.Generator) -> torch.Tensor:
    """Uniformly random E4M3fn codes, NaN codes (0x7f, 0xff) excluded."""
    codes = torch.randint(0, 254, shape, generator=g, dtype=torch.int32, device=g.device)
    codes = codes + (codes >= 0x7f).int()          # skip 0x7f; 0xff is never reached
    return codes.to(torch.uint8).view(torch.float8_e4m3fn)


@dataclass
class DenseCase:
    """D = C + A @ B^T inputs (NT layout, PaperTrace DeepGEMM §1.1)."""
    a: torch.Tensor          # float8_e4m3fn [M, K]
    sfa: torch.Tensor        # fp32 [M, ceil(K/128)]
    b: torch.Tensor          # float8_e4m3fn [N, K]
    sfb: torch.Tensor        # fp32 [ceil(N/128), ceil(K/128)]
    c: torch.Tensor | None   # bf16 [M, N] or None
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        return self.a.shape[0], self.b.shape[0], self.a.shape[1]


def dense_case(M: int, N: int, K: int, seed: int = 0, with_c: bool = False,
               b_scale_exp_range: tuple[int, int] | None = None, device="cpu") -> DenseCase:
    """Dense NT problem: A, B from N(0,1) quantised per 1x128 / 128x128.

    b_scale_exp_range=(lo, hi) replaces every B block scale by 2^u with u a
    uniform integer in [lo, hi] (the C-accumulate workload's spread of weight
    scale exponents over 2^-8..2^4).  device="cuda" draws and quantises on the
    GPU (a different random stream, same recipe): for workload-sized timing
    inputs whose values no test compares."""
    g = generator(seed, device)
    x = torch.randn(M, K, generator=g, dtype=torch.float32, device=device)
    w = torch.randn(N, K, generator=g, dtype=torch.float32, device=device)
    a, sfa = quantize_1x128(x)
    del x
    b, sfb = quantize_128x128(w)
    del w
    if b_scale_exp_range is not None:
        lo, hi = b_scale_exp_range
        u = torch.randint(lo, hi + 1, sfb.shape, generator=g, dtype=torch.int64, device=device)
        sfb = torch.ldexp(torch.ones(sfb.shape, dtype=torch.float64, device=device), u).float()
    c = (torch.randn(M, N, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)
         if with_c else None)
    return DenseCase(a, sfa, b, sfb, c, {"M": M, "N": N, "K": K, "seed": seed})


def integer_exact_case(M: int, N: int, K: int, seed: int = 0, max_shift: int = 2) -> DenseCase:
    """Codes for integers in [-8, 8] and scales 2^j (j in [-max_shift, 0] for A,
    [0, max_shift] for B): every partial sum is an integer multiple of
    2^-max_shift well inside 2^24, so FP32 accumulation is exact and the bf16
    result is exactly bf16_rne(integer matmul)."""
    g = generator(seed)
    ai = torch.randint(-8, 9, (M, K), generator=g).float()
    bi = torch.randint(-8, 9, (N, K), generator=g).float()
    sf_k = cdiv(K, GRAN)
    ja = torch.randint(-max_shift, 1, (M, sf_k), generator=g)
    jb = torch.randint(0, max_shift + 1, (cdiv(N, GRAN), sf_k), generator=g)
    sfa = torch.ldexp(torch.ones(M, sf_k, dtype=torch.float64), ja).float()
    sfb = torch.ldexp(torch.ones(cdiv(N, GRAN), sf_k, dtype=torch.float64), jb).float()
    a = ai.to(torch.float8_e4m3fn)
    b = bi.to(torch.float8_e4m3fn)
    return DenseCase(a, sfa, b, sfb, None, {"M": M, "N": N, "K": K, "seed": seed})


@dataclass
class ContiguousCase:
    """M-grouped contiguous MoE inputs (PaperTrace DeepGEMM §5.1)."""
    a: torch.Tensor              # float8 [M_total, K]
    sfa: torch.Tensor            # fp32 [M_total, sf_k]
    b: torch.Tensor              # float8 [E, N, K]
    sfb: torch.Tensor            # fp32 [E, ceil(N/128), sf_k]
    grouped_layout: torch.Tensor  # int32 [M_total], expert id or -1 (padding row)
    m_per_expert: list[int]
    meta: dict = field(default_factory=dict)


def contiguous_case(num_groups: int, N: int, K: int, seed: int = 0, m_lo: int = 128,
                    m_hi: int = 4096, align: int = 128,
                    m_per_expert: list[int] | None = None, device="cpu") -> ContiguousCase:
    g = generator(seed, device)
    if m_per_expert is None:
        m_per_expert = [int(v) for v in torch.randint(m_lo, m_hi + 1, (num_groups,), generator=g,
                                                      device=device)]
    padded = [cdiv(m, align) * align for m in m_per_expert]
    M_total = sum(padded)
    sf_k = cdiv(K, GRAN)
    a = torch.zeros(M_total, K, dtype=torch.float8_e4m3fn, device=device)
    sfa = torch.ones(M_total, sf_k, dtype=torch.float32, device=device)
    layout = torch.full((M_total,), -1, dtype=torch.int32, device=device)
    row = 0
    for e, (m, mp) in enumerate(zip(m_per_expert, padded)):
        if m:
            q, s = quantize_1x128(torch.randn(m, K, generator=g, dtype=torch.float32, device=device))
            a[row:row + m] = q
            sfa[row:row + m] = s
            layout[row:row + m] = e
        row += mp
    b = torch.empty(num_groups, N, K, dtype=torch.float8_e4m3fn, device=device)
    sfb = torch.empty(num_groups, cdiv(N, GRAN), sf_k, dtype=torch.float32, device=device)
    for e in range(num_groups):
        b[e], sfb[e] = quantize_128x128(torch.randn(N, K, generator=g, dtype=torch.float32,
                                                    device=device))
    return ContiguousCase(a, sfa, b, sfb, layout, m_per_expert,
                          {"E": num_groups, "N": N, "K": K, "M_total": M_total, "seed": seed})


@dataclass
class MaskedCase:
    """M-grouped masked MoE inputs (PaperTrace DeepGEMM §5.2)."""
    a: torch.Tensor          # float8 [E, max_m, K]
    sfa: torch.Tensor        # fp32 [E, max_m, sf_k]
    b: torch.Tensor          # float8 [E, N, K]
    sfb: torch.Tensor        # fp32 [E, ceil(N/128), sf_k]
    masked_m: torch.Tensor   # int32 [E]
    expected_m: int
    meta: dict = field(default_factory=dict)


def masked_case(num_groups: int, max_m: int, N: int, K: int, seed: int = 0,
                masked_m: list[int] | None = None, device="cpu") -> MaskedCase:
    """Valid rows per expert uniform in [0, max_m]; rows past masked_m[e] hold
    random finite codes and random scales (they must not affect anything)."""
    g = generator(seed, device)
    if masked_m is None:
        mm = torch.randint(0, max_m + 1, (num_groups,), generator=g, dtype=torch.int32, device=device)
    else:
        mm = torch.tensor(masked_m, dtype=torch.int32, device=device)
    sf_k = cdiv(K, GRAN)
    a = random_finite_e4m3((num_groups, max_m, K), g)
    sfa = torch.ldexp(torch.ones(num_groups, max_m, sf_k, dtype=torch.float64, device=device),
                      torch.randint(-10, 4, (num_groups, max_m, sf_k), generator=g,
                                    device=device)).float()
    for e in range(num_groups):
        m = int(mm[e])
        if m:
            q, s = quantize_1x128(torch.randn(m, K, generator=g, dtype=torch.float32, device=device))
            a[e, :m] = q
            sfa[e, :m] = s
    b = torch.empty(num_groups, N, K, dtype=torch.float8_e4m3fn, device=device)
    sfb = torch.empty(num_groups, cdiv(N, GRAN), sf_k, dtype=torch.float32, device=device)
    for e in range(num_groups):
        b[e], sfb[e] = quantize_128x128(torch.randn(N, K, generator=g, dtype=torch.float32,
                                                    device=device))
    expected_m = max(1, math.ceil(float(mm.float().mean())))
    return MaskedCase(a, sfa, b, sfb, mm, expected_m,
                      {"E": num_groups, "max_m": max_m, "N": N, "K": K, "seed": seed})


# Workload shapes of the pages' models ("DeepSeek V4 源码剖析 第13章" §13.16:
# the test tables carry DeepSeek's real shapes such as (24576, 1536) and
# (7168, 16384)).
V3_NK = [(2112, 7168), (24576, 1536), (7168, 16384)]
V3_M = [128, 4096]


@dataclass
class KGroupedCase:
    """K-grouped weight-gradient inputs (PaperTrace DeepGEMM §3.3, §5.2): the
    groups' K rows are concatenated; group e owns rows [K_e, K_e + ks[e]) of A
    and B and scale rows [K_e/gran_k, (K_e + ks[e])/gran_k), gran_k = 128 or 32."""
    a: torch.Tensor      # float8 [K_total, M] (M contiguous)
    sfa: torch.Tensor    # fp32 [K_total/gran_k, M], one scale per (gran_k-row K block, m)
    b: torch.Tensor      # float8 [K_total, N] (N contiguous)
    sfb: torch.Tensor    # fp32 [K_total/gran_k, N]
    c: torch.Tensor      # fp32 [E, M, N]
    ks: list[int]
    meta: dict = field(default_factory=dict)


def quantize_1xg(x: torch.Tensor, gran: int):
    """x fp32 [R, K] with K % gran == 0 -> (codes float8_e4m3fn [R, K], scales
    fp32 [R, K/gran]): the 1x128 recipe with groups of `gran` elements."""
    R, K = x.shape
    xg = x.view(R, K // gran, gran)
    s = pow2_scale(xg.abs().amax(-1))
    return (xg / s[..., None]).view(R, K).to(torch.float8_e4m3fn), s


def k_grouped_case(num_groups: int, M: int, N: int, seed: int = 0, ks: list[int] | None = None,
                   k_lo: int = 128, k_hi: int = 4096, align: int = 128, device="cpu",
                   gran_k: int = 128) -> KGroupedCase:
    """Group sizes uniform in [k_lo, k_hi] rounded up to `align` (the token
    counts per expert of the MoE shapes, stored padded), unless given.  Each
    group's A and B come from N(0,1), quantised with one scale per gran_k rows
    of K (128, or 32 for the pages' pre-packed form) and per column (the 1x128
    recipe applied along K); sfa, sfb are then [K_total/gran_k, M or N]."""
    g = generator(seed, device)
    if ks is None:
        ks = [cdiv(int(v), align) * align
              for v in torch.randint(k_lo, k_hi + 1, (num_groups,), generator=g, device=device)]
    assert all(k % GRAN == 0 and k >= 0 for k in ks)
    k_total = sum(ks)
    a = torch.empty(k_total, M, dtype=torch.float8_e4m3fn, device=device)
    b = torch.empty(k_total, N, dtype=torch.float8_e4m3fn, device=device)
    sfa = torch.empty(k_total // gran_k, M, dtype=torch.float32, device=device)
    sfb = torch.empty(k_total // gran_k, N, dtype=torch.float32, device=device)
    k0 = 0
    for k in ks:
        if k:
            for x_out, s_out, mn in ((a, sfa, M), (b, sfb, N)):
                x = torch.randn(mn, k, generator=g, dtype=torch.float32, device=device)
                q, s = quantize_1x128(x) if gran_k == GRAN else quantize_1xg(x, gran_k)
                x_out[k0:k0 + k] = q.t()
                s_out[k0 // gran_k:(k0 + k) // gran_k] = s.t()
        k0 += k
    c = torch.randn(num_groups, M, N, generator=g, dtype=torch.float32, device=device)
    return KGroupedCase(a, sfa, b, sfb, c, list(ks),
                        {"E": num_groups, "M": M, "N": N, "K_total": k_total, "seed": seed, "gran_k": gran_k})


# E2M1 magnitudes by code (low 3 bits) and the midpoints between neighbours
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_e2m1_1x32(w: torch.Tensor):
    """w fp32 [N, K] (K % 32 == 0) -> (packed uint8 [N, K/2], scales fp32 [N, K/32]):
    one power-of-two scale per 32 consecutive K of a row (amax / s <= 6), each
    value rounded to the nearest E2M1 magnitude (a tie goes to the smaller),
    two codes per byte with the even-k element in the low nibble."""
    N, K = w.shape
    assert K % 32 == 0
    blocks = w.view(N, K // 32, 32)
    s = pow2_scale(blocks.abs().amax(-1), 6.0)
    x = blocks / s[..., None]
    mid = torch.tensor(_E2M1_MIDPOINTS, dtype=x.dtype, device=x.device)
    code = torch.bucketize(x.abs().contiguous(), mid).to(torch.uint8)
    code |= (x < 0).to(torch.uint8) << 3
    code = code.view(N, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, s


@dataclass
class Fp4Case:
    """FP8 x FP4 GEMM inputs ("DeepSeek V4 源码剖析 第13章" §13.1, §13.5): FP8
    activations with 1x128 scales, FP4 (E2M1) weights with one scale per 32 K."""
    a: torch.Tensor          # float8_e4m3fn [M, K]
    sfa: torch.Tensor        # fp32 [M, K/128]
    b: torch.Tensor          # uint8 [N, K/2], two E2M1 codes per byte (even k low)
    sfb: torch.Tensor        # fp32 [N, K/32]
    c: torch.Tensor | None   # bf16 [M, N] or None
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        return self.a.shape[0], self.b.shape[0], self.a.shape[1]


def fp4_case(M: int, N: int, K: int, seed: int = 0, with_c: bool = False, device="cpu") -> Fp4Case:
    """X, W from N(0,1); X quantised per 1x128 to E4M3, W per 1x32 to E2M1."""
    g = generator(seed, device)
    x = torch.randn(M, K, generator=g, dtype=torch.float32, device=device)
    w = torch.randn(N, K, generator=g, dtype=torch.float32, device=device)
    a, sfa = quantize_1x128(x)
    del x
    b, sfb = quantize_e2m1_1x32(w)
    del w
    c = (torch.randn(M, N, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)
         if with_c else None)
    return Fp4Case(a, sfa, b, sfb, c, {"M": M, "N": N, "K": K, "seed": seed})

