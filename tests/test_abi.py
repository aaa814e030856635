"""The C-ABI library loads and exports every symbol include/dg.h declares, and
its host-side validation answers without a GPU (no compute is run here)."""
import ctypes
import os
import re

import pytest

from block_scaled_fp8_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_scaled_fp8_gb300 import build
    build.build()
    return binding.lib()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "dg.h")).read()
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(binding.EXPORTS) == _declared_symbols()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_layout_helpers(lib):
    assert binding.get_mk_alignment_for_contiguous_layout() == 128
    assert binding.get_tma_aligned_size(30, 4) == 32
    assert binding.get_tma_aligned_size(2112, 4) == 2112
    assert binding.get_tma_aligned_size(3, 2) == 8
    # batch * ceil(ceil(K/128)/4) * align4(mn)
    assert binding.packed_sf_words(1, 4096, 16384) == 32 * 4096
    assert binding.packed_sf_words(32, 256, 7168) == 32 * 14 * 256
    assert binding.packed_sf_words(1, 30, 128) == 32
    assert lib.dg_status_string(3) == b"DG_ERR_LAYOUT"


def _gemm(lib, **kw):
    args = dict(a=16, lda=128, sfa=16, sfa_fmt=1, b=16, ldb=128, sfb=16, sfb_fmt=1, c=None,
                ldc=0, d=16, ldd=64, m=8, n=64, k=128)
    args.update(kw)
    P = ctypes.c_void_p
    return lib.dg_fp8_gemm_nt(P(args["a"]), args["lda"], P(args["sfa"]), args["sfa_fmt"],
                              P(args["b"]), args["ldb"], P(args["sfb"]), args["sfb_fmt"],
                              P(args["c"]), args["ldc"], P(args["d"]), args["ldd"], args["m"],
                              args["n"], args["k"], None, None)


def test_host_validation_without_gpu(lib):
    """Bad arguments are rejected before any CUDA call (the pointers here are
    never dereferenced)."""
    assert _gemm(lib, m=-1) == 1                       # DG_ERR_INVALID_ARG
    assert _gemm(lib, sfa_fmt=5) == 1
    assert _gemm(lib, sfa_fmt=0) == 4                  # mixed formats: DG_ERR_UNSUPPORTED
    assert _gemm(lib, m=0) == 0                        # empty problem: no-op
    assert _gemm(lib, n=0) == 0
    assert _gemm(lib, d=24) == 2                       # misaligned D: DG_ERR_ALIGNMENT
    assert _gemm(lib, ldd=60) == 2
    assert _gemm(lib, n=60, ldd=64) == 2               # N % 8 != 0
    assert _gemm(lib, k=120, lda=128, ldb=128) == 2    # K % 16 != 0
    assert _gemm(lib, lda=120) == 1                    # lda < K
    assert _gemm(lib, lda=136, k=128) == 2             # lda % 16 != 0
    assert _gemm(lib, a=0) == 1                        # null A
    P = ctypes.c_void_p
    # transform: granularity and row-count rules
    assert lib.dg_transform_sf(P(16), 1, 4, 2, 2, 4, 1, P(16), None, None) == 4
    assert lib.dg_transform_sf(P(16), 1, 5, 2, 128, 300, 1, P(16), None, None) == 3
    assert lib.dg_transform_sf(P(16), 1, 4, 2, 1, 4, 9, P(16), None, None) == 1
    assert lib.dg_transform_sf(P(16), 0, 0, 2, 1, 0, 1, P(16), None, None) == 0
    # grouped
    assert lib.dg_m_grouped_fp8_gemm_nt_contiguous(P(16), 128, P(16), 1, P(16), 128, P(16), 1,
                                                   P(16), 64, P(16), 100, 64, 128, 2, None,
                                                   None) == 3   # M_total % 128 != 0
    assert lib.dg_m_grouped_fp8_gemm_nt_masked(P(16), P(16), 1, P(16), P(16), 1, P(16), P(16),
                                               2000, 64, 32, 64, 128, None, None) == 4
    assert lib.dg_m_grouped_fp8_gemm_nt_masked(P(16), P(16), 0, P(16), P(16), 0, P(16), P(16),
                                               2, 64, 32, 64, 128, None, None) == 4


def test_k_grouped_host_validation_without_gpu(lib):
    P = ctypes.c_void_p
    ks = (ctypes.c_int * 4)(256, 640, 0, 128)
    assert lib.dg_k_grouped_packed_sf_rows(ks, 4) == 4      # 1 + 2 + 0 + 1
    bad = (ctypes.c_int * 2)(128, 130)
    assert lib.dg_k_grouped_packed_sf_rows(bad, 2) == -1
    assert lib.dg_k_grouped_packed_sf_rows(ks, 256) == -1     # more than 255 groups
    assert lib.dg_k_grouped_packed_sf_rows(None, 0) == 0

    def call(m=256, n=256, c=16, ks_arr=ks, groups=4, lda=256, ldb=256):
        return lib.dg_k_grouped_fp8_gemm_tn_contiguous(P(16), lda, P(16), P(16), ldb, P(16), P(c), P(16), m, n,
                                                       ks_arr, P(16), groups, None, None)
    assert call(c=0) == 1            # C is required
    assert call(ks_arr=bad, groups=2) == 1
    assert call(m=258) == 3          # packed scales need mn % 4 == 0
    assert call(n=0) == 0            # empty
    assert call(groups=0) == 0
    assert call(m=-4) == 1
    assert lib.dg_transform_sf_k_grouped(P(16), 6, ks, 4, P(16), None, None) == 3
    assert lib.dg_transform_sf_k_grouped(P(16), 8, bad, 2, P(16), None, None) == 1
    # the same rules for the scales at a K granularity of 32
    def call32(m=256, n=256, c=16, ks_arr=ks, groups=4):
        return lib.dg_k_grouped_fp8_gemm_tn_contiguous_k32(P(16), 256, P(16), P(16), 256, P(16), P(c), P(16), m,
                                                           n, ks_arr, P(16), groups, None, None)
    assert call32(c=0) == 1
    assert call32(ks_arr=bad, groups=2) == 1
    assert call32(n=258) == 3
    assert call32(m=0) == 0
    assert lib.dg_transform_sf_k_grouped_k32(P(16), 6, ks, 4, P(16), None, None) == 3
    assert lib.dg_transform_sf_k_grouped_k32(P(16), 8, bad, 2, P(16), None, None) == 1


def test_fp4_and_layout_host_validation_without_gpu(lib):
    P = ctypes.c_void_p

    def fp4(a=32, lda=256, sfa=16, b=32, ldb=128, sfb=16, c=None, ldc=0, d=16, ldd=64, m=8, n=64, k=256):
        return lib.dg_fp8_fp4_gemm_nt(P(a), lda, P(sfa), P(b), ldb, P(sfb), P(c), ldc, P(d), ldd, m, n, k,
                                      None, None)
    assert fp4(m=-1) == 1
    assert fp4(m=0) == 0
    assert fp4(k=192, lda=256) == 2          # K % 128 != 0 (the 4-bit loads' rule)
    assert fp4(b=48) == 2                    # B not 32-byte aligned
    assert fp4(ldb=112) == 2                 # B row stride not a multiple of 32 bytes
    assert fp4(ldb=96, k=256) == 1           # ldb < k/2
    assert fp4(n=60, ldd=64) == 2            # N % 8 != 0
    assert fp4(sfb=0) == 1

    def lay(fn, a=16, lda=64, b=16, ldb=64, m=64, n=64, k=128):
        return getattr(lib, fn)(P(a), lda, P(16), 1, P(b), ldb, P(16), 1, None, 0, P(16), 64, m, n, k, None, None)
    # nn: A [m][k] K-contiguous, B [k][n]; tn: A [k][m], B [k][n]; tt: A [k][m], B [n][k]
    assert lay("dg_fp8_gemm_nn", lda=128, ldb=48) == 1    # N-contiguous B: ldb < n
    assert lay("dg_fp8_gemm_nn", lda=112, ldb=64) == 1    # K-contiguous A: lda < k
    assert lay("dg_fp8_gemm_tn", lda=48, ldb=64) == 1     # M-contiguous A: lda < m
    assert lay("dg_fp8_gemm_tt", lda=72, ldb=128) == 2    # lda % 16 != 0
    assert lay("dg_fp8_gemm_nn", lda=128, ldb=64, k=120) == 2   # K-contiguous A: K % 16 != 0
    assert lay("dg_fp8_gemm_tt", m=0) == 0
