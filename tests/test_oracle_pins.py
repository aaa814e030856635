"""Pins: the oracle checked against things other than itself.

Each test ties an oracle function to a library routine, a worked example on
the pages, a closed form, an invariant or brute force in exact rationals, so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.  CPU only.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_fp8_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- E4M3 decode

def test_e4m3_all_codes_match_torch(orc):
    """All 256 codes against torch's float8_e4m3fn -> float64 conversion."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = orc.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}


def test_e4m3_textbook_values(orc):
    """OCP E4M3 fn: max 448, min normal 2^-6, min subnormal 2^-9, no inf."""
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0xFE) == -448.0
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0xB8) == -1.0
    assert orc.e4m3_decode(0x80) == 0.0 and math.copysign(1, orc.e4m3_decode(0x80)) == -1
    assert not any(math.isinf(orc.e4m3_decode(c)) for c in range(256))


# ---------------------------------------------------------------- UE8M0

def test_ue8m0_truncation_worked_example(orc):
    """The page's own example: packing keeps the exponent, 0.75 -> 0.5, 3 -> 2."""
    rows = _golden("ue8m0_truncation.txt")
    assert len(rows) == 2
    for s, v in rows:
        assert orc.ue8m0_decode(orc.fp32_to_ue8m0(float(s))) == float(v)
        assert not orc.fp32_is_exact_ue8m0(float(s))


def test_ue8m0_power_of_two_round_trip(orc):
    """Every normal FP32 power of two survives packing exactly and is flagged exact."""
    for e in range(-126, 128):
        s = math.ldexp(1.0, e)
        byte = orc.fp32_to_ue8m0(s)
        assert byte == e + 127
        assert orc.ue8m0_decode(byte) == s
        assert orc.fp32_is_exact_ue8m0(s)
    assert math.isnan(orc.ue8m0_decode(0xFF))
    assert orc.ue8m0_decode(0) == math.ldexp(1.0, -127)
    # sign and mantissa are what make a scale inexact
    for s in (-2.0, 1.5, 3.0, 0.3, float(np.float32(2.0 ** -127))):
        assert not orc.fp32_is_exact_ue8m0(s)


def test_scale_size_ratios_closed_form():
    """"DeepSeek V4 源码剖析 第13章" §13.3: a 128x128-block FP8 weight's (1-byte)
    scales are 1/16384 of its bytes; 1x128 activation scales 1/128."""
    M = N = K = 1024
    weight_bytes, act_bytes = N * K, M * K
    assert Fraction((N // 128) * (K // 128), weight_bytes) == Fraction(1, 16384)
    assert Fraction(M * (K // 128), act_bytes) == Fraction(1, 128)


# ---------------------------------------------------------------- transform

def test_transform_hand_worked_layout(orc):
    """Hand-worked fixture of the packed MN-major layout (PaperTrace §3.1)."""
    sf = np.array([[2.0 ** (i - k) for k in range(6)] for i in range(5)], dtype=np.float32)
    out, inexact = orc.transform_sf(sf, gran_mn=1, mn=5, packed=True)
    assert inexact == 0
    assert out.shape == (2, 8)
    expected = {int(i): int(h, 16) for i, h in _golden("sf_layout_small.txt")}
    flat = out.reshape(-1).view(np.uint32)
    assert {i: int(flat[i]) for i in range(16)} == expected


@pytest.mark.parametrize("mn,stride", [(2112, 2112), (30, 32), (4096, 4096), (5, 8), (1, 4)])
def test_transform_strides(orc, mn, stride):
    """Stride of a K-slice is align(mn, 4) int32 (16 B / sizeof(int32), §3.1)."""
    sf = np.ones((mn, 9), dtype=np.float32)
    out, _ = orc.transform_sf(sf, gran_mn=1, mn=mn)
    assert out.shape == (3, stride)
    assert np.all(out[:, mn:] == 0)


def test_transform_broadcast_and_fp32_mode(orc):
    """gran_mn=128 weights broadcast to one row per N index; the FP32 MN-major
    mode is the transpose (strides [1, align4(mn)])."""
    rng = np.random.default_rng(0)
    N, sf_k = 300, 5
    sfb = np.ldexp(1.0, rng.integers(-8, 5, (3, sf_k))).astype(np.float32)
    packed, _ = orc.transform_sf(sfb, gran_mn=128, mn=N)
    back = orc.unpack_sf(packed, N, sf_k)
    assert np.array_equal(back, sfb[np.arange(N) // 128].astype(np.float64))
    f32, _ = orc.transform_sf(sfb, gran_mn=128, mn=N, packed=False)
    assert f32.shape == (sf_k, 300)
    assert np.array_equal(f32[:, :N].T, sfb[np.arange(N) // 128])


def test_transform_counts_inexact(orc):
    sf = np.array([[0.75, 1.0, 3.0, 2.0 ** -3]], dtype=np.float32)
    out, inexact = orc.transform_sf(sf, gran_mn=1, mn=1)
    assert inexact == 2
    vals = orc.unpack_sf(out, 1, 4)[0]
    assert list(vals) == [0.5, 1.0, 2.0, 0.125]


# ---------------------------------------------------------------- bf16 rounding

def _bf16_value(h):
    return struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0]


def _bf16_nearest_bruteforce(x: Fraction) -> int:
    """Nearest bf16 to an exact rational by searching the neighbourhood of its
    float32 approximation; ties go to the even bit pattern."""
    f = float(x)
    if f == 0.0 and x == 0:
        return 0
    approx = struct.unpack("<I", struct.pack("<f", np.float32(f)))[0] >> 16
    best = None
    for h in range(approx - 3, approx + 4):
        h &= 0xFFFF
        v = _bf16_value(h)
        if math.isnan(v) or math.isinf(v):
            continue
        d = abs(Fraction(v) - x)
        key = (d, h & 1)
        if best is None or key < best[0]:
            best = (key, h)
    return best[1]


def test_bf16_rne_bruteforce(orc):
    rng = np.random.default_rng(1)
    vals = []
    for e in list(range(-140, -120)) + list(range(-10, 12)) + [100, 126, 127]:
        for _ in range(40):
            vals.append(math.ldexp(rng.uniform(1, 2), e) * rng.choice([-1, 1]))
    for x in vals:
        got = orc.bf16_from_double(x)
        want = _bf16_nearest_bruteforce(Fraction(x))
        if x < 0 and want == 0:
            want = 0x8000
        assert got == want, (x, hex(got), hex(want))


def test_bf16_rne_ties_and_overflow(orc):
    """Exact midpoints between neighbouring bf16 values go to the even one."""
    rng = np.random.default_rng(2)
    for h in rng.integers(0x0001, 0x7F7F, 400):
        lo, hi = _bf16_value(int(h)), _bf16_value(int(h) + 1)
        mid = (lo + hi) / 2  # exact in fp64
        want = int(h) if int(h) % 2 == 0 else int(h) + 1
        assert orc.bf16_from_double(mid) == want
        assert orc.bf16_from_double(-mid) == want | 0x8000
    big = _bf16_value(0x7F7F)
    assert orc.bf16_from_double(big) == 0x7F7F
    assert orc.bf16_from_double(big + math.ldexp(1, 127 - 8)) == 0x7F80   # tie -> even -> inf
    assert orc.bf16_from_double(big + math.ldexp(1, 127 - 9)) == 0x7F7F
    assert orc.bf16_from_double(float("inf")) == 0x7F80
    assert orc.bf16_from_double(math.ldexp(1, -134)) == 0x0000            # tie at half min subnormal
    assert orc.bf16_from_double(math.ldexp(1.5, -134)) == 0x0001


def test_bf16_rne_matches_torch_on_float32_values(orc):
    """For values already in float32, torch's f32 -> bf16 cast is one RNE step."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4096, generator=g) * torch.exp2(torch.randint(-30, 30, (4096,), generator=g).float())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_from_double(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- GEMM

def _decode_codes_torch(t):
    return t.view(torch.float8_e4m3fn).double().numpy()


def _exact_gemm_fractions(a_codes, sa, b_codes, sb_rows, c=None):
    """Brute force: D_pre[m][n] = C + sum_k a*sa[m][k//128] * b*sb[n][k//128] in rationals."""
    A = _decode_codes_torch(torch.from_numpy(a_codes))
    B = _decode_codes_torch(torch.from_numpy(b_codes))
    M, K = A.shape
    N = B.shape[0]
    out = [[None] * N for _ in range(M)]
    for m in range(M):
        arow = [Fraction(float(A[m, k])) * Fraction(float(sa[m, k // 128])) for k in range(K)]
        for n in range(N):
            s = Fraction(0) if c is None else Fraction(_bf16_value(int(c[m, n])))
            for k in range(K):
                if arow[k]:
                    s += arow[k] * Fraction(float(B[n, k])) * Fraction(float(sb_rows[n, k // 128]))
            out[m][n] = s
    return out


def _case_np(case):
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    return a, b


@pytest.mark.parametrize("M,N,K,seed", [(3, 4, 256, 0), (2, 130, 384, 1), (4, 3, 200, 2),
                                         (1, 1, 128, 3)])
def test_gemm_bruteforce_rationals(orc, M, N, K, seed):
    """Oracle pre-rounding sum vs exact rational sum (tiny shapes, N=130 has a
    partial 128-row block of B scales; K=200 a short last K-group), with
    non-power-of-two FP32 scales and a C term."""
    case = inputs.dense_case(M, N, K, seed=seed, with_c=True)
    a, b = _case_np(case)
    rng = np.random.default_rng(seed)
    sa = case.sfa.double().numpy() * rng.choice([1.0, 0.75, 3.0, 1.1], case.sfa.shape)
    sfb = case.sfb.double().numpy() * rng.choice([1.0, 0.625, 5.0], case.sfb.shape)
    sb_rows = sfb[np.arange(N) // 128]
    c = case.c.view(torch.int16).numpy().view(np.uint16)
    d, pre = orc.gemm_nt(a, sa, b, sb_rows, c=c, want_pre=True)
    exact = _exact_gemm_fractions(a, sa, b, sb_rows, c)
    for m in range(M):
        for n in range(N):
            ex = exact[m][n]
            # fp64 error bound: each term carries one product rounding and the
            # running sum one addition rounding -> (K + 2) * 2^-52 * sum|terms|
            bound = Fraction(K + 2, 2 ** 52) * (abs(ex) + 64)
            assert abs(Fraction(pre[m, n]) - ex) <= bound
            # the bf16 result is the single RNE of the pre-rounding value ...
            assert d[m, n] == _bf16_nearest_bruteforce(Fraction(pre[m, n]))
            # ... and equals the RNE of the exact value unless that sits within
            # the fp64 error of a bf16 rounding boundary
            want = _bf16_nearest_bruteforce(ex)
            if d[m, n] != want:
                mid = (Fraction(_bf16_value(int(d[m, n]))) + Fraction(_bf16_value(want))) / 2
                assert abs(mid - ex) <= bound, (m, n)


def test_gemm_pow2_scales_bruteforce_exact(orc):
    """With power-of-two scales every product is exact; at this size the fp64
    sum is exact too, so pre-rounding values equal the rationals exactly."""
    case = inputs.dense_case(3, 5, 384, seed=7)
    a, b = _case_np(case)
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(5) // 128]
    d, pre = orc.gemm_nt(a, sa, b, sb_rows, want_pre=True)
    exact = _exact_gemm_fractions(a, sa, b, sb_rows)
    for m in range(3):
        for n in range(5):
            assert Fraction(pre[m, n]) == exact[m][n]
            assert d[m, n] == _bf16_nearest_bruteforce(exact[m][n])


def test_gemm_integer_exact(orc):
    """Integer-valued codes and 2^j scales: D == bf16_rne(exact integer matmul),
    the exact value computed with an int64 matmul at a common denominator."""
    M, N, K = 33, 150, 640
    case = inputs.integer_exact_case(M, N, K, seed=5)
    a, b = _case_np(case)
    sa = case.sfa.double().numpy()
    sfb = case.sfb.double().numpy()
    sb_rows = sfb[np.arange(N) // 128]
    d = orc.gemm_nt(a, sa, b, sb_rows)
    ai = case.a.float().numpy().astype(np.int64)
    bi = case.b.float().numpy().astype(np.int64)
    # scale exponents times 4 -> integers; common denominator 2^4
    ea = np.log2(sa).astype(np.int64)
    eb = np.log2(sb_rows).astype(np.int64)
    kk = np.arange(K) // 128
    a_scaled = ai * (2 ** (ea[:, kk] + 2))            # [M, K] ints (ea >= -2)
    b_scaled = bi * (2 ** (eb[:, kk] + 2))            # [N, K] ints (eb >= 0)
    num = a_scaled @ b_scaled.T                       # exact int64, value = num / 16
    for m in range(M):
        for n in range(N):
            ex = Fraction(int(num[m, n]), 16)
            want = _bf16_nearest_bruteforce(ex)
            if ex < 0 and want == 0:
                want = 0x8000
            assert d[m, n] == want


def test_gemm_unit_scales_matches_torch_matmul(orc):
    """All scales 1: the definition reduces to a plain float64 matmul of the
    decoded operands (a library routine), up to fp64 summation order."""
    M, N, K = 17, 40, 512
    case = inputs.dense_case(M, N, K, seed=11)
    a, b = _case_np(case)
    sa = np.ones((M, K // 128))
    sb_rows = np.ones((N, K // 128))
    _, pre = orc.gemm_nt(a, sa, b, sb_rows, want_pre=True)
    ref = (case.a.double() @ case.b.double().T).numpy()
    assert np.allclose(pre, ref, rtol=1e-13, atol=1e-12)


def test_gemm_scaled_matches_expanded_torch_matmul(orc):
    """With scales, the definition is (A*S_A)(B*S_B)^T with the scale tables
    spread to every element (LinearQuant page) -- here via torch float64."""
    M, N, K = 20, 260, 384
    case = inputs.dense_case(M, N, K, seed=12, with_c=True, b_scale_exp_range=(-8, 4))
    a, b = _case_np(case)
    kk = torch.arange(K) // 128
    nn = torch.arange(N) // 128
    A = case.a.double() * case.sfa.double()[:, kk]
    B = case.b.double() * case.sfb.double()[nn][:, kk]
    ref = (case.c.double() + A @ B.T).numpy()
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[nn.numpy()]
    c = case.c.view(torch.int16).numpy().view(np.uint16)
    _, pre = orc.gemm_nt(a, sa, b, sb_rows, c=c, want_pre=True)
    assert np.allclose(pre, ref, rtol=1e-12, atol=1e-9)


def test_gemm_pow2_linearity(orc):
    """Scaling one row's A scales by 2^t scales that output row by 2^t exactly;
    scaling one B block row's scales scales exactly its 128 output columns."""
    M, N, K = 6, 260, 256
    case = inputs.dense_case(M, N, K, seed=13)
    a, b = _case_np(case)
    sa = case.sfa.double().numpy()
    sfb = case.sfb.double().numpy()
    sb_rows = sfb[np.arange(N) // 128]
    _, pre = orc.gemm_nt(a, sa, b, sb_rows, want_pre=True)
    sa2 = sa.copy()
    sa2[2] *= 8.0
    _, pre2 = orc.gemm_nt(a, sa2, b, sb_rows, want_pre=True)
    assert np.array_equal(pre2[2], pre[2] * 8.0)
    assert np.array_equal(np.delete(pre2, 2, 0), np.delete(pre, 2, 0))
    sfb3 = sfb.copy()
    sfb3[1] *= 0.25
    _, pre3 = orc.gemm_nt(a, sa, b, sfb3[np.arange(N) // 128], want_pre=True)
    assert np.array_equal(pre3[:, 128:256], pre[:, 128:256] * 0.25)
    assert np.array_equal(pre3[:, :128], pre[:, :128])
    assert np.array_equal(pre3[:, 256:], pre[:, 256:])


def test_gemm_single_k_group_isolated(orc):
    """Only K-group 1 of A row 0 is non-zero: the result is that group's partial
    dot product alone (catches k/128 <-> scale index mix-ups and transposes)."""
    M, N, K = 2, 3, 384
    case = inputs.dense_case(M, N, K, seed=14)
    a, b = _case_np(case)
    a = a.copy()
    a[0, :128] = 0
    a[0, 256:] = 0
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(N) // 128]
    _, pre = orc.gemm_nt(a, sa, b, sb_rows, want_pre=True)
    A = _decode_codes_torch(torch.from_numpy(a))
    B = _decode_codes_torch(torch.from_numpy(b))
    for n in range(N):
        want = sum(Fraction(float(A[0, k])) * Fraction(float(B[n, k])) for k in range(128, 256))
        want *= Fraction(float(sa[0, 1])) * Fraction(float(sb_rows[n, 1]))
        assert Fraction(pre[0, n]) == want


def test_promotion_regrouping_equals_flat_sum(orc):
    """PaperTrace §2.2: sum over 128-K blocks of sa*sb*(block dot) equals the
    flat per-element sum (checked in rationals against the oracle)."""
    M, N, K = 2, 2, 512
    case = inputs.dense_case(M, N, K, seed=15)
    a, b = _case_np(case)
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(N) // 128]
    _, pre = orc.gemm_nt(a, sa, b, sb_rows, want_pre=True)
    A = _decode_codes_torch(torch.from_numpy(a))
    B = _decode_codes_torch(torch.from_numpy(b))
    for m in range(M):
        for n in range(N):
            final = Fraction(0)
            for kb in range(K // 128):
                accum = sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k]))
                            for k in range(kb * 128, kb * 128 + 128))
                final += Fraction(float(sa[m, kb])) * Fraction(float(sb_rows[n, kb])) * accum
            assert Fraction(pre[m, n]) == final


def test_gemm_sampled_equals_full(orc):
    case = inputs.dense_case(40, 300, 640, seed=16, with_c=True)
    a, b = _case_np(case)
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(300) // 128]
    c = case.c.view(torch.int16).numpy().view(np.uint16)
    d = orc.gemm_nt(a, sa, b, sb_rows, c=c)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, 40, 500), rng.integers(0, 300, 500)
    s = orc.gemm_nt_sampled(a, sa, b, sb_rows, rows, cols, c=c)
    assert np.array_equal(s, d[rows, cols])


# ---------------------------------------------------------------- grouped

def test_contiguous_equals_dense_per_expert(orc):
    """Contiguous grouped GEMM == dense GEMM of each expert's segment; padding
    rows (-1) untouched (PaperTrace §5.1)."""
    case = inputs.contiguous_case(3, 200, 256, seed=17, m_per_expert=[5, 130, 0])
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[:, np.arange(200) // 128]
    layout = case.grouped_layout.numpy()
    sentinel = np.full((a.shape[0], 200), 0x7FC1, dtype=np.uint16)
    d = orc.m_grouped_contiguous(a, sa, b, sb_rows, layout, d_init=sentinel)
    for e in range(3):
        rows = np.nonzero(layout == e)[0]
        if len(rows):
            ref = orc.gemm_nt(a[rows], sa[rows], b[e], sb_rows[e])
            assert np.array_equal(d[rows], ref)
    assert np.all(d[layout < 0] == 0x7FC1)
    assert case.a.shape[0] == 128 + 256 + 0


def test_masked_equals_dense_per_expert(orc):
    case = inputs.masked_case(3, 40, 136, 256, seed=18, masked_m=[0, 40, 7])
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[:, np.arange(136) // 128]
    sentinel = np.full((3, 40, 136), 0x7FC1, dtype=np.uint16)
    d = orc.m_grouped_masked(a, sa, b, sb_rows, case.masked_m.numpy(), d_init=sentinel)
    for e, m in enumerate([0, 40, 7]):
        if m:
            assert np.array_equal(d[e, :m], orc.gemm_nt(a[e, :m], sa[e, :m], b[e], sb_rows[e]))
        assert np.all(d[e, m:] == 0x7FC1)


# ---------------------------------------------------------------- generator

def test_generator_recipe_scales_are_pow2_and_codes_fit():
    case = inputs.dense_case(64, 256, 384, seed=0)
    for s in (case.sfa, case.sfb):
        m, e = torch.frexp(s.double())
        assert torch.all(m == 0.5)
    x = torch.randn(64, 384, generator=inputs.generator(0))
    assert torch.equal(inputs.quantize_1x128(x)[0].view(torch.uint8), case.a.view(torch.uint8))
    assert not torch.isnan(case.a.float()).any() and not torch.isnan(case.b.float()).any()
    # amax of each group lands in (224, 448]
    deq = case.a.float().view(64, 3, 128).abs().amax(-1)
    assert torch.all(deq <= 448) and torch.all(deq > 224 - 32)


# ---------------------------------------------------------------- PSUM contiguous layout

def test_psum_segments_golden(orc):
    """Hand-worked segment starts and counts (tests/golden/psum_segments.txt)."""
    rows = _golden("psum_segments.txt")
    assert rows
    for case, m_total, psum, starts, counts in rows:
        s, c = orc.psum_segments([int(x) for x in psum.split(",")], int(m_total))
        assert s == [int(x) for x in starts.split(",")], case
        assert c == [int(x) for x in counts.split(",")], case


def test_psum_segments_rejects_bad_offsets(orc):
    with pytest.raises(ValueError):
        orc.psum_segments([10, 5], 256)       # decreasing
    with pytest.raises(ValueError):
        orc.psum_segments([100, 300], 256)    # segments end at 384 > 256


def test_psum_layout_dense_per_expert_and_gap_rows(orc):
    """Each expert's rows equal a dense GEMM of those rows with its B; gap rows
    are 0; rows past the last segment keep the initial value."""
    counts = [5, 0, 130, 1]
    psum = np.cumsum(counts).tolist()
    m_total = 128 + 256 + 128 + 128          # segments end at 512; one slack block
    E, N, K = 4, 136, 256
    rng = np.random.default_rng(5)
    a = rng.integers(0, 0x7E, (m_total, K), dtype=np.uint8)   # finite E4M3 codes
    b = rng.integers(0, 0x7E, (E, N, K), dtype=np.uint8)
    sa = np.exp2(rng.integers(-3, 3, (m_total, 2))).astype(np.float64)
    sb_rows = np.exp2(rng.integers(-3, 3, (E, N, 2))).astype(np.float64)
    sentinel = np.full((m_total, N), 0x7FC1, dtype=np.uint16)
    d = orc.m_grouped_contiguous_psum(a, sa, b, sb_rows, psum, d_init=sentinel)
    starts = [0, 128, 128, 384, 512]
    for e, m in enumerate(counts):
        r0 = starts[e]
        if m:
            ref = orc.gemm_nt(a[r0:r0 + m], sa[r0:r0 + m], b[e], sb_rows[e])
            assert np.array_equal(d[r0:r0 + m], ref), e
        assert np.all(d[r0 + m:starts[e + 1]] == 0), e
    assert np.all(d[512:] == 0x7FC1)


# ---------------------------------------------------------------- FP32 output

def test_gemm_f32_integer_exact(orc):
    """Integer codes and power-of-two scales (A's down to 2^-2): the result is
    a multiple of 1/4 below 2^22, exact in FP32, so the FP32 output must equal
    the float64 torch matmul (plus an integer C) exactly."""
    case = inputs.integer_exact_case(64, 96, 384, seed=41)
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(96) // 128]
    x = case.a.double() * torch.from_numpy(sa).repeat_interleave(128, 1)[:, :384]
    w = case.b.double() * torch.from_numpy(sb_rows).repeat_interleave(128, 1)[:, :384]
    c = torch.randint(-50, 50, (64, 96), generator=torch.Generator().manual_seed(3)).float()
    exact = (x @ w.T + c.double()).numpy()
    assert np.all(np.abs(exact) < 2 ** 22) and np.all(exact * 4 == np.round(exact * 4))
    got = orc.gemm_nt_f32(a, sa, b, sb_rows, c=c.numpy())
    assert np.array_equal(got.astype(np.float64), exact)


def test_gemm_f32_rounds_once_to_fp32(orc):
    """Random operands: the FP32 output is the fp64 pre-rounding value of the
    bf16 oracle (C = 0) rounded to FP32 by numpy, and bf16 of it matches the
    bf16 oracle except where the two roundings straddle a bf16 tie."""
    case = inputs.dense_case(40, 72, 640, seed=9)
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(72) // 128]
    _, pre = orc.gemm_nt(a, sa, b, sb_rows, want_pre=True)
    got = orc.gemm_nt_f32(a, sa, b, sb_rows)
    assert np.array_equal(got, pre.astype(np.float32))


def test_gemm_f32_sampled_equals_full(orc):
    """The sampled FP32 form takes the same fp64 steps in the same order as the
    full one, so the same FP32 bits at every sampled element (with and without
    C, over a ragged N that spans two 128-row B scale blocks)."""
    case = inputs.dense_case(37, 200, 384, seed=12, b_scale_exp_range=(-8, 4))
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(200) // 128]
    c = torch.randn(37, 200, generator=torch.Generator().manual_seed(8)).numpy()
    rng = np.random.default_rng(1)
    rows, cols = rng.integers(0, 37, 400), rng.integers(0, 200, 400)
    for cc in (None, c):
        full = orc.gemm_nt_f32(a, sa, b, sb_rows, c=cc)
        got = orc.gemm_nt_f32_sampled(a, sa, b, sb_rows, rows, cols, c=cc)
        assert np.array_equal(got.view(np.uint32), full[rows, cols].view(np.uint32))


# ---------------------------------------------------------------- NN / TN / TT layouts

@pytest.mark.parametrize("layout", ["nn", "tn", "tt", "nt"])
@pytest.mark.parametrize("M,N,K,seed", [(3, 130, 256, 51), (5, 4, 200, 52)])
def test_gemm_layouts_bruteforce_from_storage(orc, layout, M, N, K, seed):
    """"DeepSeek V4 源码剖析 第13章" §13.3 naming: D = C + A @ B with "t" meaning
    transposed, so A is stored [K, M] for "t" and B [K, N] for "n".  The brute
    force reads each element straight from that storage by index (no
    transpose); power-of-two scales keep every term exact, so the oracle's
    pre-rounding values must equal the rational sums exactly.  N=130 spans two
    128-row B scale blocks and M != N != K, so a swapped operand, index or scale
    axis changes the values or the shapes."""
    case = inputs.dense_case(M, N, K, seed=seed, with_c=True)
    a_mk, b_nk = _case_np(case)
    a = np.ascontiguousarray(a_mk.T) if layout[0] == "t" else a_mk
    b = np.ascontiguousarray(b_nk.T) if layout[1] == "n" else b_nk
    A = _decode_codes_torch(torch.from_numpy(a))
    B = _decode_codes_torch(torch.from_numpy(b))
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(N) // 128]
    c = case.c.view(torch.int16).numpy().view(np.uint16)
    d, pre = orc.gemm(layout, a, sa, b, sb_rows, c=c, want_pre=True)
    assert d.shape == (M, N)
    for m in range(M):
        for n in range(N):
            s = Fraction(_bf16_value(int(c[m, n])))
            for k in range(K):
                av = A[k, m] if layout[0] == "t" else A[m, k]
                bv = B[k, n] if layout[1] == "n" else B[n, k]
                if av and bv:
                    s += (Fraction(float(av)) * Fraction(float(sa[m, k // 128])) *
                          Fraction(float(bv)) * Fraction(float(sb_rows[n, k // 128])))
            assert Fraction(pre[m, n]) == s, (layout, m, n)
            assert d[m, n] == _bf16_nearest_bruteforce(s)


# ---------------------------------------------------------------- K-grouped GEMM

def test_k_grouped_bruteforce_from_storage(orc):
    """PaperTrace DeepGEMM §5.2 / §3.3: groups concatenated along K, one D per
    group, C mandatory.  The brute force reads A[k, m], B[k, n] and the scale
    rows straight from storage by index; power-of-two scales keep every term
    exact, so each FP32 output is the single rounding of the rational sum.
    The empty group must give D = C exactly."""
    ks = [128, 0, 256]
    M, N = 3, 5
    case = inputs.k_grouped_case(3, M, N, seed=61, ks=ks)
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    A = _decode_codes_torch(case.a.view(torch.uint8))
    B = _decode_codes_torch(case.b.view(torch.uint8))
    sa = case.sfa.double().numpy()
    sb = case.sfb.double().numpy()
    c = case.c.numpy()
    d = orc.k_grouped_gemm_tn(a, sa, b, sb, ks, c)
    assert d.shape == (3, M, N) and d.dtype == np.float32
    assert np.array_equal(d[1], c[1])
    k0 = 0
    for e, k in enumerate(ks):
        for m in range(M):
            for n in range(N):
                s = Fraction(float(c[e, m, n]))
                for kk in range(k0, k0 + k):
                    if A[kk, m] and B[kk, n]:
                        s += (Fraction(float(A[kk, m])) * Fraction(float(sa[kk // 128, m])) *
                              Fraction(float(B[kk, n])) * Fraction(float(sb[kk // 128, n])))
                assert d[e, m, n] == np.float32(float(s)), (e, m, n)
        k0 += k


def test_k_grouped_split_invariance_integer_exact(orc):
    """Integer codes and power-of-two scales make every sum exact in FP32: with
    C = 0, splitting one group of 512 rows into two of 256 and adding the two
    outputs must give the one-group output, and both must equal the float64
    matmul of the decoded operands."""
    g = torch.Generator().manual_seed(62)
    K, M, N = 512, 8, 12
    ai = torch.randint(-8, 9, (K, M), generator=g).float()
    bi = torch.randint(-8, 9, (K, N), generator=g).float()
    sa = torch.ldexp(torch.ones(K // 128, M, dtype=torch.float64), torch.randint(-2, 1, (K // 128, M), generator=g))
    sb = torch.ldexp(torch.ones(K // 128, N, dtype=torch.float64), torch.randint(0, 3, (K // 128, N), generator=g))
    a = ai.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    b = bi.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    one = orc.k_grouped_gemm_tn(a, sa.numpy(), b, sb.numpy(), [512], np.zeros((1, M, N), np.float32))
    two = orc.k_grouped_gemm_tn(a, sa.numpy(), b, sb.numpy(), [256, 256], np.zeros((2, M, N), np.float32))
    x = ai.double() * sa.repeat_interleave(128, 0)
    w = bi.double() * sb.repeat_interleave(128, 0)
    exact = (x.T @ w).numpy()
    assert np.array_equal(one[0].astype(np.float64), exact)
    assert np.array_equal(two[0].astype(np.float64) + two[1].astype(np.float64), exact)
    assert np.array_equal((x[:256].T @ w[:256]).numpy(), two[0].astype(np.float64))


def test_k_grouped_pack_hand_worked(orc):
    """PaperTrace DeepGEMM §3.3: each group packed on its own, 4 scale rows per
    int32, the last packed row of a group zero-filled past its rows.  ks =
    [256, 640, 0, 128] gives 2, 5, 0 and 1 scale rows, hence 1 + 2 + 0 + 1
    packed rows.  Scale row r, column i is 2^(r - i): UE8M0 byte 0x7F + r - i.
    The words below were worked out by hand (byte j = row 4q + j of the group)."""
    mn = 4
    sf = np.array([[2.0 ** (r - i) for i in range(mn)] for r in range(8)], dtype=np.float32)
    got = orc.k_grouped_pack_sf(sf, [256, 640, 0, 128]).view(np.uint32)
    want = np.array([
        [0x0000807F, 0x00007F7E, 0x00007E7D, 0x00007D7C],   # group 0: rows 0, 1
        [0x84838281, 0x83828180, 0x8281807F, 0x81807F7E],   # group 1: rows 2..5
        [0x00000085, 0x00000084, 0x00000083, 0x00000082],   # group 1: row 6
        [0x00000086, 0x00000085, 0x00000084, 0x00000083],   # group 3: row 7
    ], dtype=np.uint32)
    assert np.array_equal(got, want)


def test_k_grouped_k32_bruteforce_from_storage(orc):
    """PaperTrace DeepGEMM §3.3: the K-grouped layout's pre-packed scales come
    at a K granularity of 32.  The brute force reads A[k, m], B[k, n] and the
    scale rows k // 32 straight from storage; power-of-two scales keep every
    term exact, so each FP32 output is the single rounding of the rational sum.
    ks = [128, 0, 256] spans 4, 0 and 8 scale rows, so a scale row taken at the
    128 granularity, a group offset or an operand swap changes the values."""
    ks = [128, 0, 256]
    M, N = 3, 5
    case = inputs.k_grouped_case(3, M, N, seed=64, ks=ks, gran_k=32)
    assert case.sfa.shape == (12, M) and case.sfb.shape == (12, N)
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    A = _decode_codes_torch(case.a.view(torch.uint8))
    B = _decode_codes_torch(case.b.view(torch.uint8))
    sa = case.sfa.double().numpy()
    sb = case.sfb.double().numpy()
    assert len(np.unique(sa)) > 1 and len(np.unique(sb)) > 1
    c = case.c.numpy()
    d = orc.k_grouped_gemm_tn_k32(a, sa, b, sb, ks, c)
    assert np.array_equal(d[1], c[1])
    k0 = 0
    for e, k in enumerate(ks):
        for m in range(M):
            for n in range(N):
                s = Fraction(float(c[e, m, n]))
                for kk in range(k0, k0 + k):
                    if A[kk, m] and B[kk, n]:
                        s += (Fraction(float(A[kk, m])) * Fraction(float(sa[kk // 32, m])) *
                              Fraction(float(B[kk, n])) * Fraction(float(sb[kk // 32, n])))
                assert d[e, m, n] == np.float32(float(s)), (e, m, n)
        k0 += k


def test_k_grouped_k32_reduces_to_k128(orc):
    """Scales at a K granularity of 32 whose four rows in every 128-row block are
    equal give the 128-granularity GEMM bit for bit (the same terms in the same
    order); the sampled form equals the full one bit for bit."""
    ks = [256, 128, 0, 384]
    case = inputs.k_grouped_case(4, 24, 40, seed=65, ks=ks)
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa, sb, c = case.sfa.double().numpy(), case.sfb.double().numpy(), case.c.numpy()
    sa32, sb32 = np.repeat(sa, 4, axis=0), np.repeat(sb, 4, axis=0)
    d128 = orc.k_grouped_gemm_tn(a, sa, b, sb, ks, c)
    d32 = orc.k_grouped_gemm_tn_k32(a, sa32, b, sb32, ks, c)
    assert np.array_equal(d32.view(np.uint32), d128.view(np.uint32))
    rng = np.random.default_rng(2)
    es, ms, ns = rng.integers(0, 4, 300), rng.integers(0, 24, 300), rng.integers(0, 40, 300)
    got = orc.k_grouped_gemm_tn_k32_sampled(a, sa32, b, sb32, ks, c, es, ms, ns)
    assert np.array_equal(got.view(np.uint32), d32[es, ms, ns].view(np.uint32))


def test_k_grouped_pack_k32_hand_worked(orc):
    """PaperTrace DeepGEMM §3.3 at gran_k = 32: ks = [128, 256, 0] gives 4, 8
    and 0 scale rows, packed 4 per int32 per group: 1 + 2 + 0 packed rows.
    Scale row r, column i is 2^(r - i) (UE8M0 byte 0x7F + r - i); byte j of a
    word is row 4q + j of its group.  The words were worked out by hand."""
    mn = 4
    sf = np.array([[2.0 ** (r - i) for i in range(mn)] for r in range(12)], dtype=np.float32)
    got = orc.k_grouped_pack_sf(sf, [128, 256, 0], gran_k=32).view(np.uint32)
    want = np.array([
        [0x8281807F, 0x81807F7E, 0x807F7E7D, 0x7F7E7D7C],   # group 0: rows 0..3
        [0x86858483, 0x85848382, 0x84838281, 0x83828180],   # group 1: rows 4..7
        [0x8A898887, 0x89888786, 0x88878685, 0x87868584],   # group 1: rows 8..11
    ], dtype=np.uint32)
    assert np.array_equal(got, want)


def test_k_grouped_sampled_equals_full(orc):
    case = inputs.k_grouped_case(3, 40, 24, seed=63, ks=[256, 0, 384])
    a = case.a.view(torch.uint8).numpy()
    b = case.b.view(torch.uint8).numpy()
    sa, sb, c = case.sfa.double().numpy(), case.sfb.double().numpy(), case.c.numpy()
    full = orc.k_grouped_gemm_tn(a, sa, b, sb, case.ks, c)
    rng = np.random.default_rng(0)
    es, ms, ns = rng.integers(0, 3, 300), rng.integers(0, 40, 300), rng.integers(0, 24, 300)
    got = orc.k_grouped_gemm_tn_sampled(a, sa, b, sb, case.ks, c, es, ms, ns)
    ref = full[es, ms, ns]
    # same fp64 order (products from 0, then C), so the same FP32 bits
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------- FP8 x FP4

# OCP Microscaling FP4 E2M1 by code: sign bit 3, then the eight magnitudes
E2M1_TEXTBOOK = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_all_codes_textbook(orc):
    for code, want in enumerate(E2M1_TEXTBOOK):
        got = orc.e2m1_decode(code)
        assert got == want and np.signbit(got) == np.signbit(want), code
    assert orc.e2m1_decode(0xF7) == 6.0      # only the low nibble is read


def _nibbles(packed_row, K):
    """Codes of one packed row, read by index: element k = byte k // 2, low nibble for even k."""
    return [(int(packed_row[k // 2]) >> (4 * (k % 2))) & 0xF for k in range(K)]


def test_fp8_fp4_bruteforce_from_packed_storage(orc):
    """"DeepSeek V4 源码剖析 第13章" §13.1 reason 2: weight scales run along K,
    one per 32 elements.  Rational sums read straight from the packed bytes
    with distinct scales per 32-K block; power-of-two scales keep every term
    exact, so the oracle's fp64 values must equal them."""
    M, N, K = 3, 5, 256
    case = inputs.fp4_case(M, N, K, seed=81, with_c=True)
    rng = np.random.default_rng(81)
    sb = np.ldexp(1.0, rng.integers(-6, 4, (N, K // 32)))
    a = case.a.view(torch.uint8).numpy()
    A = _decode_codes_torch(case.a.view(torch.uint8))
    sa = case.sfa.double().numpy()
    b = case.b.numpy()
    c = case.c.view(torch.int16).numpy().view(np.uint16)
    d, pre = orc.gemm_fp8_fp4_nt(a, sa, b, sb, c=c, want_pre=True)
    for n in range(N):
        codes = _nibbles(b[n], K)
        for m in range(M):
            s = Fraction(_bf16_value(int(c[m, n])))
            for k in range(K):
                if A[m, k] and codes[k] & 7:
                    s += (Fraction(float(A[m, k])) * Fraction(float(sa[m, k // 128])) *
                          Fraction(E2M1_TEXTBOOK[codes[k]]) * Fraction(float(sb[n, k // 32])))
            assert Fraction(pre[m, n]) == s, (m, n)
            assert d[m, n] == _bf16_nearest_bruteforce(s)


def test_fp8_fp4_reduces_to_fp8_nt(orc):
    """With each row's four 32-K scales of a 128-K block equal, the FP8 x FP4
    GEMM is the NT GEMM of the same values: the E2M1 weights re-encoded as
    E4M3 (exact) with those scales as per-row 128-K scales."""
    M, N, K = 20, 24, 384
    case = inputs.fp4_case(M, N, K, seed=82)
    rng = np.random.default_rng(82)
    s128 = np.ldexp(1.0, rng.integers(-5, 5, (N, K // 128)))
    sb = np.repeat(s128, 4, axis=1)
    b = case.b.numpy()
    vals = np.array([[E2M1_TEXTBOOK[cd] for cd in _nibbles(b[n], K)] for n in range(N)])
    b8 = torch.from_numpy(vals).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(torch.from_numpy(b8).view(torch.float8_e4m3fn).double().numpy(), vals)
    a = case.a.view(torch.uint8).numpy()
    sa = case.sfa.double().numpy()
    got = orc.gemm_fp8_fp4_nt(a, sa, b, sb)
    want = orc.gemm_nt(a, sa, b8, s128)
    assert np.array_equal(got, want)


def test_m_grouped_fp4_oracles_bruteforce(orc):
    """The grouped FP8 x FP4 oracles against the packed-storage brute force on a
    few elements of every expert: the expert's own weights and scales, and
    untouched rows outside the groups."""
    E, N, K = 3, 6, 128
    cases = [inputs.fp4_case(8, N, K, seed=83 + e) for e in range(E)]
    b = np.stack([c.b.numpy() for c in cases])
    sb = np.stack([c.sfb.double().numpy() for c in cases])
    a_all = torch.cat([c.a for c in cases]).view(torch.uint8).numpy()[:20]
    sa_all = torch.cat([c.sfa for c in cases]).double().numpy()[:20]
    layout = np.array([0] * 5 + [-1] * 3 + [2] * 7 + [1] * 5)
    init = np.full((20, N), 0x7FC1, dtype=np.uint16)
    d = orc.m_grouped_fp8_fp4_contiguous(a_all, sa_all, b, sb, layout, d_init=init)
    A = _decode_codes_torch(torch.from_numpy(a_all))
    for m in range(20):
        e = layout[m]
        for n in range(N):
            if e < 0:
                assert d[m, n] == 0x7FC1
                continue
            codes = _nibbles(b[e, n], K)
            s = Fraction(0)
            for k in range(K):
                if A[m, k] and codes[k] & 7:
                    s += (Fraction(float(A[m, k])) * Fraction(float(sa_all[m, k // 128])) *
                          Fraction(E2M1_TEXTBOOK[codes[k]]) * Fraction(float(sb[e, n, k // 32])))
            assert d[m, n] == _bf16_nearest_bruteforce(s), (m, n)
    # masked: the same rows as experts' first rows
    am = np.stack([a_all[0:5], a_all[8:13], a_all[15:20]])
    sam = np.stack([sa_all[0:5], sa_all[8:13], sa_all[15:20]])
    dm = orc.m_grouped_fp8_fp4_masked(am, sam, b[[0, 2, 1]], sb[[0, 2, 1]], [5, 3, 0],
                                      d_init=np.full((3, 5, N), 0x7FC1, dtype=np.uint16))
    assert np.array_equal(dm[0], d[0:5]) and np.array_equal(dm[1, :3], d[8:11])
    assert np.all(dm[1, 3:] == 0x7FC1) and np.all(dm[2] == 0x7FC1)


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
def test_gemm_layouts_integer_exact_matmul(orc, layout):
    """Integer codes and power-of-two scales make every sum exact: the layout
    oracle must equal bf16_rne of the float64 matmul op(A) op(B) of the decoded
    stored operands, at a size (96 x 160 x 384) that spans several scale blocks."""
    M, N, K = 96, 160, 384
    case = inputs.integer_exact_case(M, N, K, seed=84)
    a_mk = case.a.view(torch.uint8).numpy()
    b_nk = case.b.view(torch.uint8).numpy()
    a = np.ascontiguousarray(a_mk.T) if layout[0] == "t" else a_mk
    b = np.ascontiguousarray(b_nk.T) if layout[1] == "n" else b_nk
    sa = case.sfa.double().numpy()
    sb_rows = case.sfb.double().numpy()[np.arange(N) // 128]
    A = _decode_codes_torch(torch.from_numpy(a))
    B = _decode_codes_torch(torch.from_numpy(b))
    A_mk = (A.T if layout[0] == "t" else A) * np.repeat(sa, 128, axis=1)[:, :K]
    B_kn = (B if layout[1] == "n" else B.T) * np.repeat(sb_rows, 128, axis=1)[:, :K].T
    exact = A_mk @ B_kn
    got = orc.gemm(layout, a, sa, b, sb_rows)
    want = np.array([[_bf16_nearest_bruteforce(Fraction(float(v))) for v in row] for row in exact],
                    dtype=np.uint16)
    assert np.array_equal(got, want)


def test_fp8_fp4_matches_float64_matmul(orc):
    """At 64 x 96 x 512 the decoded products of the seeded case span under 40
    bits, so any order of fp64 summation is exact: the FP4 oracle must equal
    bf16_rne of numpy's float64 matmul of the scale-expanded operands."""
    M, N, K = 64, 96, 512
    case = inputs.fp4_case(M, N, K, seed=85)
    a = case.a.view(torch.uint8).numpy()
    A = _decode_codes_torch(case.a.view(torch.uint8)) * np.repeat(case.sfa.double().numpy(), 128, axis=1)
    codes = np.stack([case.b.numpy() & 0xF, case.b.numpy() >> 4], axis=-1).reshape(N, K)
    B = np.array(E2M1_TEXTBOOK)[codes] * np.repeat(case.sfb.double().numpy(), 32, axis=1)
    exact = A @ B.T
    got = orc.gemm_fp8_fp4_nt(a, case.sfa.double().numpy(), case.b.numpy(), case.sfb.double().numpy())
    want = np.array([[_bf16_nearest_bruteforce(Fraction(float(v))) for v in row] for row in exact],
                    dtype=np.uint16)
    assert np.array_equal(got, want)
