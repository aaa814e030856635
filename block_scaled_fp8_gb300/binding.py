"""Thin Python binding of the C ABI in include/dg.h (argument marshalling only).

Every function takes torch tensors that already live on the current CUDA
device, passes their data pointers and the current torch stream to the
library, and raises DGError on a non-OK status.  All arithmetic happens in
the library's CUDA kernels; nothing here computes.  The library must have
been built (block_scaled_fp8_gb300.build) -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdg_gb300.so")

DG_SF_FP32 = 0
DG_SF_UE8M0_PACKED = 1
DG_DEV_TIMEOUT = 1
DG_DEV_INEXACT_SCALE = 2
DG_DEV_BAD_GROUP = 4
DG_DEBUG_DROP_ONE_LOAD = 1
DG_DEBUG_PRINT_CONFIGS = 2
DG_DEBUG_SINGLE_CTA = 4
DG_DEBUG_WIDE_PAIR = 8

# Every symbol include/dg.h declares.
EXPORTS = (
    "dg_fp8_gemm_nt", "dg_fp8_gemm_nt_f32", "dg_fp8_gemm_nn", "dg_fp8_gemm_tn", "dg_fp8_gemm_tt",
    "dg_fp8_fp4_gemm_nt", "dg_m_grouped_fp8_fp4_gemm_nt_contiguous", "dg_m_grouped_fp8_fp4_gemm_nt_masked",
    "dg_transform_sf", "dg_m_grouped_fp8_gemm_nt_contiguous", "dg_m_grouped_fp8_gemm_nt_contiguous_psum",
    "dg_k_grouped_fp8_gemm_tn_contiguous", "dg_transform_sf_k_grouped", "dg_k_grouped_packed_sf_rows",
    "dg_k_grouped_fp8_gemm_tn_contiguous_k32", "dg_transform_sf_k_grouped_k32",
    "dg_m_grouped_fp8_gemm_nt_masked", "dg_get_mk_alignment_for_contiguous_layout",
    "dg_get_tma_aligned_size", "dg_packed_sf_words", "dg_set_num_sms", "dg_get_num_sms",
    "dg_set_wait_timeout_ms", "dg_set_debug_flags", "dg_status_string", "dg_get_last_config",
)


class DGError(RuntimeError):
    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status
        self.name = name


_lock = threading.Lock()
_lib = None


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library not built: {LIB_PATH} is missing "
                    "(run block_scaled_fp8_gb300.build.build())")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32
            L.dg_fp8_gemm_nt.argtypes = [P, i64, P, i32, P, i64, P, i32, P, i64, P, i64, i32, i32,
                                         i32, P, P]
            for f in ("dg_fp8_gemm_nt_f32", "dg_fp8_gemm_nn", "dg_fp8_gemm_tn", "dg_fp8_gemm_tt"):
                getattr(L, f).argtypes = L.dg_fp8_gemm_nt.argtypes
            L.dg_transform_sf.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P, P]
            L.dg_m_grouped_fp8_gemm_nt_contiguous.argtypes = [P, i64, P, i32, P, i64, P, i32, P,
                                                              i64, P, i32, i32, i32, i32, P, P]
            L.dg_m_grouped_fp8_gemm_nt_contiguous_psum.argtypes = \
                L.dg_m_grouped_fp8_gemm_nt_contiguous.argtypes
            L.dg_m_grouped_fp8_gemm_nt_masked.argtypes = [P, P, i32, P, P, i32, P, P, i32, i32,
                                                          i32, i32, i32, P, P]
            L.dg_fp8_fp4_gemm_nt.argtypes = [P, i64, P, P, i64, P, P, i64, P, i64, i32, i32, i32, P, P]
            L.dg_fp8_fp4_gemm_nt.restype = i32
            L.dg_m_grouped_fp8_fp4_gemm_nt_contiguous.argtypes = [P, i64, P, P, i64, P, P, i64, P, i32, i32, i32,
                                                                  i32, P, P]
            L.dg_m_grouped_fp8_fp4_gemm_nt_masked.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, P, P]
            for f in ("dg_m_grouped_fp8_fp4_gemm_nt_contiguous", "dg_m_grouped_fp8_fp4_gemm_nt_masked"):
                getattr(L, f).restype = i32
            L.dg_k_grouped_fp8_gemm_tn_contiguous.argtypes = [P, i64, P, P, i64, P, P, P, i32, i32, P, P, i32,
                                                              P, P]
            L.dg_transform_sf_k_grouped.argtypes = [P, i32, P, i32, P, P, P]
            L.dg_k_grouped_fp8_gemm_tn_contiguous_k32.argtypes = L.dg_k_grouped_fp8_gemm_tn_contiguous.argtypes
            L.dg_transform_sf_k_grouped_k32.argtypes = L.dg_transform_sf_k_grouped.argtypes
            L.dg_k_grouped_packed_sf_rows.restype = i64
            L.dg_k_grouped_packed_sf_rows.argtypes = [P, i32]
            for f in ("dg_k_grouped_fp8_gemm_tn_contiguous", "dg_transform_sf_k_grouped",
                      "dg_k_grouped_fp8_gemm_tn_contiguous_k32", "dg_transform_sf_k_grouped_k32"):
                getattr(L, f).restype = i32
            for f in ("dg_fp8_gemm_nt", "dg_fp8_gemm_nt_f32", "dg_fp8_gemm_nn", "dg_fp8_gemm_tn",
                      "dg_fp8_gemm_tt", "dg_transform_sf",
                      "dg_m_grouped_fp8_gemm_nt_contiguous",
                      "dg_m_grouped_fp8_gemm_nt_contiguous_psum", "dg_m_grouped_fp8_gemm_nt_masked"):
                getattr(L, f).restype = i32
            L.dg_get_mk_alignment_for_contiguous_layout.restype = i32
            L.dg_get_mk_alignment_for_contiguous_layout.argtypes = []
            L.dg_get_tma_aligned_size.restype = i64
            L.dg_get_tma_aligned_size.argtypes = [i64, i32]
            L.dg_packed_sf_words.restype = i64
            L.dg_packed_sf_words.argtypes = [i32, i32, i32]
            L.dg_set_num_sms.restype = None
            L.dg_set_num_sms.argtypes = [i32]
            L.dg_get_num_sms.restype = i32
            L.dg_get_num_sms.argtypes = []
            L.dg_set_wait_timeout_ms.restype = None
            L.dg_set_wait_timeout_ms.argtypes = [i32]
            L.dg_set_debug_flags.restype = None
            L.dg_set_debug_flags.argtypes = [u32]
            L.dg_status_string.restype = ctypes.c_char_p
            L.dg_status_string.argtypes = [i32]
            L.dg_get_last_config.restype = None
            L.dg_get_last_config.argtypes = [ctypes.POINTER(ctypes.c_int)]
            _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise DGError(fn, status, lib().dg_status_string(status).decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _sf_fmt(t):
    return DG_SF_FP32 if t.dtype == torch.float32 else DG_SF_UE8M0_PACKED


# --------------------------------------------------------------------- utilities

def get_mk_alignment_for_contiguous_layout() -> int:
    return int(lib().dg_get_mk_alignment_for_contiguous_layout())


def get_tma_aligned_size(mn: int, elem_size: int) -> int:
    return int(lib().dg_get_tma_aligned_size(mn, elem_size))


def packed_sf_words(batch: int, mn: int, k: int) -> int:
    return int(lib().dg_packed_sf_words(batch, mn, k))


def set_num_sms(n: int):
    lib().dg_set_num_sms(n)


def get_num_sms() -> int:
    return int(lib().dg_get_num_sms())


def set_wait_timeout_ms(ms: int):
    lib().dg_set_wait_timeout_ms(ms)


def set_debug_flags(flags: int):
    lib().dg_set_debug_flags(flags)


def last_config() -> dict:
    arr = (ctypes.c_int * 6)()
    lib().dg_get_last_config(arr)
    return {"block_m": arr[0], "block_n": arr[1], "stages": arr[2], "grid": arr[3],
            "kind": arr[4], "launches": arr[5]}


# --------------------------------------------------------------------- entry points

def dg_transform_sf(sf: torch.Tensor, gran_mn: int, mn: int, out: torch.Tensor,
                    packed: bool = True, status: torch.Tensor | None = None, stream=None):
    """sf: float32 [batch?, mn_rows, sf_k] -> out (int32 packed [batch?, psf_k, align4(mn)]
    or float32 [batch?, sf_k, align4(mn)])."""
    assert sf.dtype == torch.float32 and sf.is_contiguous() and out.is_contiguous()
    s = sf if sf.dim() == 3 else sf.unsqueeze(0)
    batch, mn_rows, sf_k = s.shape
    _check("dg_transform_sf", lib().dg_transform_sf(
        _p(s), batch, mn_rows, sf_k, gran_mn, mn, DG_SF_UE8M0_PACKED if packed else DG_SF_FP32,
        _p(out), _p(status), _stream(stream)))
    return out


def transform_sf(sf: torch.Tensor, gran_mn: int, mn: int, packed: bool = True,
                 status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Allocates the output with torch and calls dg_transform_sf."""
    batch = () if sf.dim() == 2 else (sf.shape[0],)
    sf_k = sf.shape[-1]
    stride = (mn + 3) // 4 * 4
    if packed:
        out = torch.empty(*batch, (sf_k + 3) // 4, stride, dtype=torch.int32, device=sf.device)
    else:
        out = torch.empty(*batch, sf_k, stride, dtype=torch.float32, device=sf.device)
    return dg_transform_sf(sf, gran_mn, mn, out, packed=packed, status=status, stream=stream)


def dg_fp8_gemm_nt(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                   d: torch.Tensor, c: torch.Tensor | None = None,
                   status: torch.Tensor | None = None, stream=None):
    """D = C + A @ B^T.  a [M, K] and b [N, K] float8_e4m3fn (row stride = stride(0));
    sfa/sfb packed int32 (MN-major) or float32 ([M, sf_k] / [ceil(N/128), sf_k]);
    d (and c) bf16 [M, N] with unit column stride."""
    M, K = a.shape
    N = b.shape[0]
    assert a.stride(1) == 1 and b.stride(1) == 1 and d.stride(1) == 1
    assert d.dtype == torch.bfloat16 and (c is None or (c.dtype == torch.bfloat16 and c.stride(1) == 1))
    _check("dg_fp8_gemm_nt", lib().dg_fp8_gemm_nt(
        _p(a), a.stride(0), _p(sfa), _sf_fmt(sfa), _p(b), b.stride(0), _p(sfb), _sf_fmt(sfb),
        _p(c), 0 if c is None else c.stride(0), _p(d), d.stride(0), M, N, K, _p(status),
        _stream(stream)))
    return d


def dg_fp8_gemm_nt_f32(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                       d: torch.Tensor, c: torch.Tensor | None = None,
                       status: torch.Tensor | None = None, stream=None):
    """D = C + A @ B^T with FP32 d (and c) [M, N], unit column stride; scales packed."""
    M, K = a.shape
    N = b.shape[0]
    assert a.stride(1) == 1 and b.stride(1) == 1 and d.stride(1) == 1
    assert d.dtype == torch.float32 and (c is None or (c.dtype == torch.float32 and c.stride(1) == 1))
    _check("dg_fp8_gemm_nt_f32", lib().dg_fp8_gemm_nt_f32(
        _p(a), a.stride(0), _p(sfa), _sf_fmt(sfa), _p(b), b.stride(0), _p(sfb), _sf_fmt(sfb),
        _p(c), 0 if c is None else c.stride(0), _p(d), d.stride(0), M, N, K, _p(status),
        _stream(stream)))
    return d


def _gemm_layout(fn: str, a_mn: bool, b_mn: bool, a, sfa, b, sfb, d, c, status, stream):
    # a is [M, K] (K-contiguous) or [K, M] (M-contiguous); b is [N, K] or [K, N]
    M = a.shape[1] if a_mn else a.shape[0]
    K = a.shape[0] if a_mn else a.shape[1]
    N = b.shape[1] if b_mn else b.shape[0]
    assert (b.shape[0] if b_mn else b.shape[1]) == K
    assert a.stride(1) == 1 and b.stride(1) == 1 and d.stride(1) == 1
    assert d.dtype == torch.bfloat16 and (c is None or (c.dtype == torch.bfloat16 and c.stride(1) == 1))
    _check(fn, getattr(lib(), fn)(
        _p(a), a.stride(0), _p(sfa), _sf_fmt(sfa), _p(b), b.stride(0), _p(sfb), _sf_fmt(sfb),
        _p(c), 0 if c is None else c.stride(0), _p(d), d.stride(0), M, N, K, _p(status),
        _stream(stream)))
    return d


def dg_fp8_gemm_nn(a, sfa, b, sfb, d, c=None, status=None, stream=None):
    """D = C + A @ B: a [M, K], b [K, N] (N contiguous); packed scales as for the NT call."""
    return _gemm_layout("dg_fp8_gemm_nn", False, True, a, sfa, b, sfb, d, c, status, stream)


def dg_fp8_gemm_tn(a, sfa, b, sfb, d, c=None, status=None, stream=None):
    """D = C + A^T @ B: a [K, M] (M contiguous), b [K, N] (N contiguous)."""
    return _gemm_layout("dg_fp8_gemm_tn", True, True, a, sfa, b, sfb, d, c, status, stream)


def dg_fp8_gemm_tt(a, sfa, b, sfb, d, c=None, status=None, stream=None):
    """D = C + A^T @ B^T: a [K, M] (M contiguous), b [N, K] (K contiguous)."""
    return _gemm_layout("dg_fp8_gemm_tt", True, False, a, sfa, b, sfb, d, c, status, stream)


def dg_fp8_fp4_gemm_nt(a, sfa, b, sfb, d, c=None, status=None, stream=None):
    """D = C + A @ B^T with FP8 A [M, K] (packed 1x128 scales) and FP4 B: b uint8
    [N, K/2], two E2M1 codes per byte (even k in the low nibble), row stride =
    stride(0) bytes; sfb packed int32 [K/128, align4(N)] (4 x 32 K per word)."""
    M, K = a.shape
    N = b.shape[0]
    assert b.dtype == torch.uint8 and b.shape[1] * 2 == K and b.stride(1) == 1
    assert a.stride(1) == 1 and d.stride(1) == 1 and d.dtype == torch.bfloat16
    assert c is None or (c.dtype == torch.bfloat16 and c.stride(1) == 1)
    _check("dg_fp8_fp4_gemm_nt", lib().dg_fp8_fp4_gemm_nt(
        _p(a), a.stride(0), _p(sfa), _p(b), b.stride(0), _p(sfb), _p(c), 0 if c is None else c.stride(0), _p(d),
        d.stride(0), M, N, K, _p(status), _stream(stream)))
    return d


def dg_m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, d, grouped_layout, status=None, stream=None):
    """a [M_total, K] E4M3; b uint8 [E, N, K/2] packed E2M1 (row stride = stride(1)
    bytes, expert stride N * stride(1)); sfa packed [ceil(K/512), align4(M_total)];
    sfb packed [E, K/128, align4(N)]; d bf16 [M_total, N]; grouped_layout int32 [M_total]."""
    M, K = a.shape
    E, N, _ = b.shape
    assert b.dtype == torch.uint8 and b.stride(0) == N * b.stride(1) and b.stride(2) == 1
    assert a.stride(1) == 1 and d.stride(1) == 1
    _check("dg_m_grouped_fp8_fp4_gemm_nt_contiguous", lib().dg_m_grouped_fp8_fp4_gemm_nt_contiguous(
        _p(a), a.stride(0), _p(sfa), _p(b), b.stride(1), _p(sfb), _p(d), d.stride(0), _p(grouped_layout), M, N, K,
        E, _p(status), _stream(stream)))
    return d


def dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, d, masked_m, expected_m, status=None, stream=None):
    """a [E, max_m, K] E4M3 contiguous; b uint8 [E, N, K/2] contiguous; sfa packed
    [E, ceil(K/512), align4(max_m)]; sfb packed [E, K/128, align4(N)]; d bf16 [E, max_m, N]."""
    E, max_m, K = a.shape
    N = b.shape[1]
    assert a.is_contiguous() and b.is_contiguous() and d.is_contiguous() and b.dtype == torch.uint8
    _check("dg_m_grouped_fp8_fp4_gemm_nt_masked", lib().dg_m_grouped_fp8_fp4_gemm_nt_masked(
        _p(a), _p(sfa), _p(b), _p(sfb), _p(d), _p(masked_m), E, max_m, int(expected_m), N, K, _p(status),
        _stream(stream)))
    return d


def _ks_host(ks):
    arr = (ctypes.c_int * max(1, len(ks)))(*[int(k) for k in ks])
    return arr


def k_grouped_packed_sf_rows(ks) -> int:
    """Packed scale rows of the K-grouped layout for group sizes ks (-1 if invalid)."""
    return int(lib().dg_k_grouped_packed_sf_rows(_ks_host(ks), len(ks)))


def dg_transform_sf_k_grouped(sf: torch.Tensor, ks, out: torch.Tensor | None = None,
                              status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """sf FP32 [sum(ks)/128, mn] -> packed int32 [k_grouped_packed_sf_rows(ks), mn]."""
    assert sf.dtype == torch.float32 and sf.is_contiguous()
    mn = sf.shape[1]
    if out is None:
        out = torch.empty(max(0, k_grouped_packed_sf_rows(ks)), mn, dtype=torch.int32, device=sf.device)
    _check("dg_transform_sf_k_grouped", lib().dg_transform_sf_k_grouped(
        _p(sf), mn, _ks_host(ks), len(ks), _p(out), _p(status), _stream(stream)))
    return out


def dg_transform_sf_k_grouped_k32(sf: torch.Tensor, ks, out: torch.Tensor | None = None,
                                  status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """sf FP32 [sum(ks)/32, mn] (one scale row per 32 rows of K) -> packed int32
    [sum(ks)/128, mn]."""
    assert sf.dtype == torch.float32 and sf.is_contiguous()
    mn = sf.shape[1]
    if out is None:
        out = torch.empty(sum(ks) // 128, mn, dtype=torch.int32, device=sf.device)
    _check("dg_transform_sf_k_grouped_k32", lib().dg_transform_sf_k_grouped_k32(
        _p(sf), mn, _ks_host(ks), len(ks), _p(out), _p(status), _stream(stream)))
    return out


def dg_k_grouped_fp8_gemm_tn_contiguous_k32(a, sfa, b, sfb, d, ks, ks_dev=None, c=None,
                                            status: torch.Tensor | None = None, stream=None):
    """As dg_k_grouped_fp8_gemm_tn_contiguous with scales every 32 rows of K:
    sfa/sfb packed int32 [sum(ks)/128, M] / [sum(ks)/128, N]."""
    K, M = a.shape
    N = b.shape[1]
    assert a.stride(1) == 1 and b.stride(1) == 1 and d.is_contiguous() and d.dtype == torch.float32
    assert c is not None and c.is_contiguous() and c.dtype == torch.float32
    if ks_dev is None:
        ks_dev = torch.tensor(list(ks), dtype=torch.int32, device=d.device)
    _check("dg_k_grouped_fp8_gemm_tn_contiguous_k32", lib().dg_k_grouped_fp8_gemm_tn_contiguous_k32(
        _p(a), a.stride(0), _p(sfa), _p(b), b.stride(0), _p(sfb), _p(c), _p(d), M, N, _ks_host(ks),
        _p(ks_dev), len(ks), _p(status), _stream(stream)))
    return d


def dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, d, ks, ks_dev=None, c=None,
                                        status: torch.Tensor | None = None, stream=None):
    """D[e] = C[e] + A_e^T B_e.  a [K_total, M] and b [K_total, N] float8_e4m3fn
    (unit column stride, row stride = stride(0)); sfa/sfb packed int32
    [P, M] / [P, N]; c (required, may be d) and d FP32 [E, M, N] contiguous;
    ks host list of group sizes (multiples of 128); ks_dev the same as a
    device int32 tensor (made here if not given)."""
    K, M = a.shape
    N = b.shape[1]
    assert a.stride(1) == 1 and b.stride(1) == 1 and d.is_contiguous() and d.dtype == torch.float32
    assert c is not None and c.is_contiguous() and c.dtype == torch.float32
    if ks_dev is None:
        ks_dev = torch.tensor(list(ks), dtype=torch.int32, device=d.device)
    _check("dg_k_grouped_fp8_gemm_tn_contiguous", lib().dg_k_grouped_fp8_gemm_tn_contiguous(
        _p(a), a.stride(0), _p(sfa), _p(b), b.stride(0), _p(sfb), _p(c), _p(d), M, N, _ks_host(ks),
        _p(ks_dev), len(ks), _p(status), _stream(stream)))
    return d


def dg_m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, d, grouped_layout,
                                        status: torch.Tensor | None = None, stream=None):
    """a [M_total, K]; b [E, N, K]; sfa packed [psf_k, align4(M_total)];
    sfb packed [E, psf_k, align4(N)]; d bf16 [M_total, N]; grouped_layout int32 [M_total]."""
    M, K = a.shape
    E, N, _ = b.shape
    assert b.stride(0) == N * b.stride(1) and b.stride(2) == 1
    _check("dg_m_grouped_fp8_gemm_nt_contiguous", lib().dg_m_grouped_fp8_gemm_nt_contiguous(
        _p(a), a.stride(0), _p(sfa), _sf_fmt(sfa), _p(b), b.stride(1), _p(sfb), _sf_fmt(sfb),
        _p(d), d.stride(0), _p(grouped_layout), M, N, K, E, _p(status), _stream(stream)))
    return d


def dg_m_grouped_fp8_gemm_nt_contiguous_psum(a, sfa, b, sfb, d, psum,
                                             status: torch.Tensor | None = None, stream=None):
    """As dg_m_grouped_fp8_gemm_nt_contiguous, with psum int32 [E] (device):
    inclusive prefix sums of the experts' row counts; each expert's rows start
    on a multiple of 128 after the previous expert's; gap rows of D get 0."""
    M, K = a.shape
    E, N, _ = b.shape
    assert b.stride(0) == N * b.stride(1) and b.stride(2) == 1
    _check("dg_m_grouped_fp8_gemm_nt_contiguous_psum", lib().dg_m_grouped_fp8_gemm_nt_contiguous_psum(
        _p(a), a.stride(0), _p(sfa), _sf_fmt(sfa), _p(b), b.stride(1), _p(sfb), _sf_fmt(sfb),
        _p(d), d.stride(0), _p(psum), M, N, K, E, _p(status), _stream(stream)))
    return d


def dg_m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, d, masked_m, expected_m: int,
                                    status: torch.Tensor | None = None, stream=None):
    """a [E, max_m, K]; b [E, N, K]; sfa packed [E, psf_k, align4(max_m)];
    sfb packed [E, psf_k, align4(N)]; d bf16 [E, max_m, N]; masked_m int32 [E] (device)."""
    E, max_m, K = a.shape
    N = b.shape[1]
    assert a.is_contiguous() and b.is_contiguous() and d.is_contiguous()
    _check("dg_m_grouped_fp8_gemm_nt_masked", lib().dg_m_grouped_fp8_gemm_nt_masked(
        _p(a), _p(sfa), _sf_fmt(sfa), _p(b), _p(sfb), _sf_fmt(sfb), _p(d), _p(masked_m), E, max_m,
        expected_m, N, K, _p(status), _stream(stream)))
    return d
