"""Oracle: plain fp64 CPU restatement of the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``block_scaled_fp8_gb300``) and never imports it;
the library never imports this.

The arithmetic lives in ``oracle.c`` (built here with gcc into
``oracle/_build/liboracle.so``); this module only marshals numpy arrays.
Every function cites the page passage it restates; see ``oracle.c`` for the
readings taken where the pages are silent.

Pins (tests that tie the oracle to something other than itself) are in
``tests/test_oracle_pins.py``.  Parity status: every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_ue8m0_decode.restype = ctypes.c_double
            lib.orc_ue8m0_decode.argtypes = [ctypes.c_uint8]
            lib.orc_fp32_to_ue8m0.restype = ctypes.c_uint8
            lib.orc_fp32_to_ue8m0.argtypes = [ctypes.c_float]
            lib.orc_fp32_is_exact_ue8m0.restype = ctypes.c_int
            lib.orc_fp32_is_exact_ue8m0.argtypes = [ctypes.c_float]
            lib.orc_bf16_from_double.restype = ctypes.c_uint16
            lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
            lib.orc_bf16_decode.restype = ctypes.c_double
            lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
            lib.orc_transform_sf.restype = i64
            lib.orc_transform_sf.argtypes = [P, i32, i32, i32, i32, i32, i32, P]
            lib.orc_unpack_sf.restype = None
            lib.orc_unpack_sf.argtypes = [P, i32, i32, i32, P]
            lib.orc_expand_block_rows.restype = None
            lib.orc_expand_block_rows.argtypes = [P, i32, i32, P]
            lib.orc_gemm_nt.restype = None
            lib.orc_gemm_nt.argtypes = [i32, i32, i32, P, i64, P, P, i64, P, P, i64, P, i64, P, i32]
            lib.orc_gemm_nt_f32.restype = None
            lib.orc_gemm_nt_f32.argtypes = [i32, i32, i32, P, i64, P, P, i64, P, P, i64, P, i64, i32]
            lib.orc_gemm_nt_sampled.restype = None
            lib.orc_gemm_nt_sampled.argtypes = [i32, P, i64, P, P, i64, P, P, i64, i64, P, P, P, P,
                                                i32]
            lib.orc_m_grouped_contiguous.restype = None
            lib.orc_m_grouped_contiguous.argtypes = [i32, i32, i32, i32, P, i64, P, P, i64, P, P, P,
                                                     i64, i32]
            lib.orc_m_grouped_masked.restype = None
            lib.orc_m_grouped_masked.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, i32]
            lib.orc_e2m1_decode.restype = ctypes.c_double
            lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.orc_gemm_fp8_fp4_nt.restype = None
            lib.orc_gemm_fp8_fp4_nt.argtypes = [i32, i32, i32, P, i64, P, P, i64, P, P, i64, P, i64, P, i32]
            lib.orc_gemm_fp8_fp4_nt_sampled.restype = None
            lib.orc_gemm_fp8_fp4_nt_sampled.argtypes = [i32, P, i64, P, P, i64, P, i64, P, P, P, i32]
            lib.orc_gemm_nt_f32_gk.restype = None
            lib.orc_gemm_nt_f32_gk.argtypes = [i32, i32, i32, i32, P, i64, P, P, i64, P, P, i64, P, i64, i32]
            lib.orc_gemm_nt_gk_pre_sampled.restype = None
            lib.orc_gemm_nt_gk_pre_sampled.argtypes = [i32, i32, P, i64, P, P, i64, P, i64, P, P, P, i32]
            lib.orc_max_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        a = a.view(np.uint8) if a.itemsize == 1 else a.astype(np.uint8)
    return a


def max_threads() -> int:
    return int(_get().orc_max_threads())


# --- number formats --------------------------------------------------------

def e4m3_decode(code: int) -> float:
    """OCP FP8 E4M3fn code -> value ("FP8 e4m3" of the pages; torch.float8_e4m3fn)."""
    return float(_get().orc_e4m3_decode(int(code) & 0xFF))


def e2m1_decode(code: int) -> float:
    """OCP MX FP4 E2M1 code (low 4 bits) -> value ("DeepSeek V4 源码剖析 第13章" §13.5)."""
    return float(_get().orc_e2m1_decode(code))


def e4m3_table() -> np.ndarray:
    """All 256 decoded E4M3fn values, indexed by code."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def ue8m0_decode(e: int) -> float:
    """UE8M0 byte -> 2^(e-127); 0xff is NaN (PaperTrace DeepGEMM §3.1)."""
    return float(_get().orc_ue8m0_decode(int(e) & 0xFF))


def fp32_to_ue8m0(s: float) -> int:
    """Byte kept when an FP32 scale is packed: its exponent bits (>>23), per
    "DeepSeek V4 源码剖析 第13章" §13.3; 0.75 -> 0.5, 3 -> 2."""
    return int(_get().orc_fp32_to_ue8m0(float(s)))


def fp32_is_exact_ue8m0(s: float) -> bool:
    """(bits & 0x807fffff) == 0: a positive normal power of two (§3.1)."""
    return bool(_get().orc_fp32_is_exact_ue8m0(float(s)))


def bf16_from_double(x: float) -> int:
    """Single round-to-nearest-even of an fp64 value to bf16 bits."""
    return int(_get().orc_bf16_from_double(float(x)))


def bf16_decode(h: int) -> float:
    return float(_get().orc_bf16_decode(int(h) & 0xFFFF))


# --- scale layout ------------------------------------------------------------

def align4(x: int) -> int:
    return (x + 3) // 4 * 4


def transform_sf(sf: np.ndarray, gran_mn: int, mn: int, packed: bool = True):
    """FP32 scales [batch?, mn_rows, sf_k] -> MN-major TMA-aligned layout.

    PaperTrace DeepGEMM §3.1-3.2: packed UE8M0 (4 K-groups per int32,
    little-endian by K), shape [mn, psf_k] with strides [1, align(mn,4)],
    batch stride psf_k*align(mn,4); rows broadcast from gran_mn to 1.
    Returns (out, n_inexact) with out int32 [batch, psf_k, align4(mn)] (packed)
    or float32 [batch, sf_k, align4(mn)].
    """
    sf = np.ascontiguousarray(sf, dtype=np.float32)
    squeeze = sf.ndim == 2
    if squeeze:
        sf = sf[None]
    batch, mn_rows, sf_k = sf.shape
    if packed:
        out = np.empty((batch, (sf_k + 3) // 4, align4(mn)), dtype=np.int32)
    else:
        out = np.empty((batch, sf_k, align4(mn)), dtype=np.float32)
    n = _get().orc_transform_sf(_ptr(sf), batch, mn_rows, sf_k, gran_mn, mn, 1 if packed else 0,
                                _ptr(out))
    return (out[0] if squeeze else out), int(n)


def unpack_sf(packed: np.ndarray, mn: int, sf_k: int) -> np.ndarray:
    """Packed MN-major UE8M0 int32 -> fp64 scales [batch?, mn, sf_k]."""
    p = np.ascontiguousarray(packed)
    squeeze = p.ndim == 2
    if squeeze:
        p = p[None]
    batch = p.shape[0]
    assert p.shape[1:] == ((sf_k + 3) // 4, align4(mn)), p.shape
    out = np.empty((batch, mn, sf_k), dtype=np.float64)
    _get().orc_unpack_sf(_ptr(p.view(np.uint32)), batch, mn, sf_k, _ptr(out))
    return out[0] if squeeze else out


def expand_block_rows(sb: np.ndarray, n_rows: int) -> np.ndarray:
    """128x128 block scales [ceil(N/128), sf_k] -> one row per N index."""
    sb = np.ascontiguousarray(sb, dtype=np.float64)
    out = np.empty((n_rows, sb.shape[1]), dtype=np.float64)
    _get().orc_expand_block_rows(_ptr(sb), n_rows, sb.shape[1], _ptr(out))
    return out


# --- GEMM --------------------------------------------------------------------

def gemm_nt(a: np.ndarray, sa: np.ndarray, b: np.ndarray, sb_rows: np.ndarray,
            c: np.ndarray | None = None, want_pre: bool = False, nthreads: int = 0):
    """D = C + A @ B^T with per-element expanded scales, fp64 sum, one RNE to bf16.

    a: uint8 E4M3 codes [M, K]; sa: fp64 [M, sf_k]; b: uint8 [N, K];
    sb_rows: fp64 [N, sf_k] (one row per N index); c: uint16 bf16 bits [M, N].
    Returns uint16 bf16 bits [M, N] (and the fp64 pre-rounding values).
    "DeepSeek V4 源码剖析 第13章" §13.3 pseudocode; LinearQuant page.
    """
    a, b = _u8(a), _u8(b)
    M, K = a.shape
    N = b.shape[0]
    sf_k = (K + 127) // 128
    sa = np.ascontiguousarray(sa, dtype=np.float64)
    sb_rows = np.ascontiguousarray(sb_rows, dtype=np.float64)
    assert sa.shape == (M, sf_k) and sb_rows.shape == (N, sf_k) and b.shape[1] == K
    if c is not None:
        c = np.ascontiguousarray(c).view(np.uint16)
        assert c.shape == (M, N)
    d = np.empty((M, N), dtype=np.uint16)
    pre = np.empty((M, N), dtype=np.float64) if want_pre else None
    _get().orc_gemm_nt(M, N, K, _ptr(a), K, _ptr(sa), _ptr(b), K, _ptr(sb_rows), _ptr(c), N,
                       _ptr(d), N, _ptr(pre), nthreads)
    return (d, pre) if want_pre else d


def gemm(layout: str, a: np.ndarray, sa: np.ndarray, b: np.ndarray, sb_rows: np.ndarray,
         c: np.ndarray | None = None, want_pre: bool = False, nthreads: int = 0):
    """D = C + op(A) op(B) for the four layouts "nt", "nn", "tn", "tt".

    "DeepSeek V4 源码剖析 第13章" §13.3: the GEMMs compute D = C + A @ B, the
    two suffix letters telling whether A and B are transposed; fp8_gemm_nt is
    D = C + A @ B.T.  As stored: A is [M, K] for "n", [K, M] for "t"; B is
    [K, N] for "n", [N, K] for "t".  The scales belong to the product's
    indices, not to the storage order: sa [M, sf_k], sb_rows [N, sf_k].
    Each operand is brought to the NT form by a transpose of its storage.
    """
    assert layout in ("nt", "nn", "tn", "tt")
    a, b = _u8(a), _u8(b)
    a_mk = np.ascontiguousarray(a.T) if layout[0] == "t" else a
    b_nk = np.ascontiguousarray(b.T) if layout[1] == "n" else b
    return gemm_nt(a_mk, sa, b_nk, sb_rows, c=c, want_pre=want_pre, nthreads=nthreads)


def gemm_fp8_fp4_nt(a: np.ndarray, sa: np.ndarray, b: np.ndarray, sb: np.ndarray,
                    c: np.ndarray | None = None, want_pre: bool = False, nthreads: int = 0):
    """FP8 x FP4 GEMM ("DeepSeek V4 源码剖析 第13章" §13.1 reason 2, §13.5):
    D = C + A @ B^T with A E4M3 [M, K] and 1x128 scales sa [M, ceil(K/128)],
    B E2M1 packed two per byte [N, ceil(K/2)] (low nibble = even k) with one
    scale per 32 K of each row, sb [N, ceil(K/32)]; fp64 sum, one RNE to bf16.
    Returns uint16 bf16 bits [M, N] (and the fp64 pre-rounding values)."""
    a, b = _u8(a), _u8(b)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == (K + 1) // 2
    sa = np.ascontiguousarray(sa, dtype=np.float64)
    sb = np.ascontiguousarray(sb, dtype=np.float64)
    assert sa.shape == (M, (K + 127) // 128) and sb.shape == (N, (K + 31) // 32)
    if c is not None:
        c = np.ascontiguousarray(c).view(np.uint16)
        assert c.shape == (M, N)
    d = np.empty((M, N), dtype=np.uint16)
    pre = np.empty((M, N), dtype=np.float64) if want_pre else None
    _get().orc_gemm_fp8_fp4_nt(M, N, K, _ptr(a), K, _ptr(sa), _ptr(b), b.shape[1], _ptr(sb), _ptr(c), N,
                               _ptr(d), N, _ptr(pre), nthreads)
    return (d, pre) if want_pre else d


def gemm_fp8_fp4_nt_sampled(a, sa, b, sb, rows, cols, nthreads: int = 0) -> np.ndarray:
    """The elements (rows[i], cols[i]) of gemm_fp8_fp4_nt (C = 0), one by one."""
    a, b = _u8(a), _u8(b)
    K = a.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    sa = np.ascontiguousarray(sa, dtype=np.float64)
    sb = np.ascontiguousarray(sb, dtype=np.float64)
    out = np.empty(rows.shape[0], dtype=np.uint16)
    _get().orc_gemm_fp8_fp4_nt_sampled(K, _ptr(a), K, _ptr(sa), _ptr(b), b.shape[1], _ptr(sb), rows.shape[0],
                                       _ptr(rows), _ptr(cols), _ptr(out), nthreads)
    return out


def m_grouped_fp8_fp4_contiguous(a, sa, b, sb, grouped_layout, d_init=None, nthreads: int = 0):
    """Contiguous M-grouped FP8 x FP4 GEMM ("DeepSeek V4 源码剖析 第13章" §13.6;
    PaperTrace DeepGEMM §5.1): row m of A uses expert grouped_layout[m]'s
    weights; a row marked -1 keeps d_init.  a [M, K] E4M3, sa [M, K/128];
    b [E, N, K/2] packed E2M1, sb [E, N, K/32].  Each expert's rows are the
    dense FP8 x FP4 GEMM of those rows with that expert's weights."""
    a = _u8(a)
    layout = np.asarray(grouped_layout)
    E, N = b.shape[0], b.shape[1]
    d = (np.zeros((a.shape[0], N), dtype=np.uint16) if d_init is None
         else np.ascontiguousarray(d_init).view(np.uint16).copy())
    for e in range(E):
        rows = np.nonzero(layout == e)[0]
        if len(rows):
            d[rows] = gemm_fp8_fp4_nt(a[rows], np.asarray(sa)[rows], b[e], sb[e], nthreads=nthreads)
    return d


def m_grouped_fp8_fp4_masked(a, sa, b, sb, masked_m, d_init=None, nthreads: int = 0):
    """Masked M-grouped FP8 x FP4 GEMM (PaperTrace DeepGEMM §5.2): expert e
    computes its first masked_m[e] rows of a [E, max_m, K]; the other rows keep
    d_init.  sa [E, max_m, K/128]; b [E, N, K/2]; sb [E, N, K/32]."""
    a = _u8(a)
    E, max_m = a.shape[0], a.shape[1]
    N = b.shape[1]
    d = (np.zeros((E, max_m, N), dtype=np.uint16) if d_init is None
         else np.ascontiguousarray(d_init).view(np.uint16).copy())
    for e in range(E):
        m = int(masked_m[e])
        if m:
            d[e, :m] = gemm_fp8_fp4_nt(a[e, :m], np.asarray(sa)[e, :m], b[e], sb[e], nthreads=nthreads)
    return d


def gemm_nt_f32(a: np.ndarray, sa: np.ndarray, b: np.ndarray, sb_rows: np.ndarray,
                c: np.ndarray | None = None, nthreads: int = 0) -> np.ndarray:
    """D = C + A @ B^T as gemm_nt, with FP32 C (or none) and FP32 D: the fp64
    sum rounded once to FP32.  Returns float32 [M, N]."""
    a, b = _u8(a), _u8(b)
    M, K = a.shape
    N = b.shape[0]
    sf_k = (K + 127) // 128
    sa = np.ascontiguousarray(sa, dtype=np.float64)
    sb_rows = np.ascontiguousarray(sb_rows, dtype=np.float64)
    assert sa.shape == (M, sf_k) and sb_rows.shape == (N, sf_k) and b.shape[1] == K
    if c is not None:
        c = np.ascontiguousarray(c, dtype=np.float32)
        assert c.shape == (M, N)
    d = np.empty((M, N), dtype=np.float32)
    _get().orc_gemm_nt_f32(M, N, K, _ptr(a), K, _ptr(sa), _ptr(b), K, _ptr(sb_rows), _ptr(c), N,
                           _ptr(d), N, nthreads)
    return d


def gemm_nt_f32_sampled(a, sa, b, sb_rows, rows, cols, c=None, nthreads: int = 0) -> np.ndarray:
    """The elements (rows[i], cols[i]) of gemm_nt_f32, one by one, in its order:
    the fp64 product sum (gemm_nt_sampled, summed from 0 in increasing k), then
    the FP32 C added in fp64 (0 if c is None), rounded once to FP32.  Equals
    gemm_nt_f32 at those elements bit for bit."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    _, pre = gemm_nt_sampled(a, sa, b, sb_rows, rows, cols, want_pre=True, nthreads=nthreads)
    cv = (np.zeros(len(rows)) if c is None
          else np.asarray(c, dtype=np.float32)[rows, cols].astype(np.float64))
    return (cv + pre).astype(np.float32)


def k_grouped_pack_sf(sf: np.ndarray, ks, gran_k: int = 128) -> np.ndarray:
    """Packed scales of the K-grouped GEMM (PaperTrace DeepGEMM §3.3).

    sf: FP32 [sum_k ks/gran_k, mn], one row per gran_k-row K block (128, or 32
    for the pages' pre-packed form) of the concatenated groups, mn contiguous,
    mn % 4 == 0.  Each group is packed on its own and the results are
    concatenated: packed row q of group e holds in byte j the UE8M0 byte (the
    exponent bits, >> 23) of the group's scale row 4q + j, and 0 where the group
    has no such row.  Returns int32 [sum_e ceil(ks[e] / (4 gran_k)), mn].
    """
    sf = np.ascontiguousarray(sf, dtype=np.float32)
    mn = sf.shape[1]
    assert mn % 4 == 0
    rows = [k // gran_k for k in ks]
    assert all(k % 128 == 0 and k >= 0 for k in ks) and sum(rows) == sf.shape[0]
    exp = ((sf.view(np.uint32) >> 23) & 0xFF).astype(np.uint32)
    out = []
    r0 = 0
    for s in rows:
        for q in range((s + 3) // 4):
            word = np.zeros(mn, dtype=np.uint32)
            for j in range(4):
                if 4 * q + j < s:
                    word |= exp[r0 + 4 * q + j] << np.uint32(8 * j)
            out.append(word)
        r0 += s
    return np.array(out, dtype=np.uint32).reshape(len(out), mn).view(np.int32)


def k_grouped_gemm_tn(a: np.ndarray, sa: np.ndarray, b: np.ndarray, sb: np.ndarray, ks,
                      c: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """K-grouped GEMM for MoE weight gradients (PaperTrace DeepGEMM §5.2,
    §3.3; "DeepSeek V4 源码剖析 第13章" §13.3 naming): M and N are fixed and
    the groups are concatenated along K; for each group e

        D_e[m, n] = C_e[m, n] + sum over group e's k of A[k, m] sa(k/128, m) B[k, n] sb(k/128, n)

    a: uint8 E4M3 [K_total, M] (M contiguous, the "t" operand); b: uint8
    [K_total, N] (N contiguous, the "n" operand); sa: fp64 [K_total/128, M];
    sb: fp64 [K_total/128, N]; ks: group sizes, multiples of 128 (0 allowed);
    c: FP32 [E, M, N] (required, as the pages make C mandatory here).
    C plus the group's fp64 product sum (the products summed from 0 in increasing
    k, then C added), rounded once to FP32.  Returns FP32 [E, M, N].
    """
    a, b = _u8(a), _u8(b)
    M, N = a.shape[1], b.shape[1]
    c = np.ascontiguousarray(c, dtype=np.float32)
    E = len(ks)
    assert c.shape == (E, M, N) and a.shape[0] == b.shape[0] == sum(ks)
    d = np.empty((E, M, N), dtype=np.float32)
    k0 = 0
    for e, k in enumerate(ks):
        assert k % 128 == 0 and k >= 0
        if k == 0:
            d[e] = c[e]
        else:
            s0, s1 = k0 // 128, (k0 + k) // 128
            d[e] = gemm_nt_f32(np.ascontiguousarray(a[k0:k0 + k].T), np.ascontiguousarray(sa[s0:s1].T),
                               np.ascontiguousarray(b[k0:k0 + k].T), np.ascontiguousarray(sb[s0:s1].T),
                               c=c[e], nthreads=nthreads)
        k0 += k
    return d


def k_grouped_gemm_tn_k32(a: np.ndarray, sa: np.ndarray, b: np.ndarray, sb: np.ndarray, ks,
                          c: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """The K-grouped GEMM with scales at a K granularity of 32 (PaperTrace
    DeepGEMM §3.3: the layout's pre-packed scales come at gran_k = 32): for each
    group e

        D_e[m, n] = C_e[m, n] + sum over group e's k of A[k, m] sa(k/32, m) B[k, n] sb(k/32, n)

    a, b as for k_grouped_gemm_tn; sa: fp64 [K_total/32, M]; sb: fp64
    [K_total/32, N]; C plus the group's fp64 product sum (from 0, increasing k),
    rounded once to FP32.  Returns FP32 [E, M, N]."""
    a, b = _u8(a), _u8(b)
    M, N = a.shape[1], b.shape[1]
    c = np.ascontiguousarray(c, dtype=np.float32)
    E = len(ks)
    assert c.shape == (E, M, N) and a.shape[0] == b.shape[0] == sum(ks)
    assert sa.shape == (sum(ks) // 32, M) and sb.shape == (sum(ks) // 32, N)
    d = np.empty((E, M, N), dtype=np.float32)
    k0 = 0
    for e, k in enumerate(ks):
        assert k % 128 == 0 and k >= 0
        if k == 0:
            d[e] = c[e]
        else:
            s0, s1 = k0 // 32, (k0 + k) // 32
            at = np.ascontiguousarray(a[k0:k0 + k].T)
            bt = np.ascontiguousarray(b[k0:k0 + k].T)
            sat = np.ascontiguousarray(sa[s0:s1].T, dtype=np.float64)
            sbt = np.ascontiguousarray(sb[s0:s1].T, dtype=np.float64)
            ce = np.ascontiguousarray(c[e])
            _get().orc_gemm_nt_f32_gk(M, N, k, 32, _ptr(at), k, _ptr(sat), _ptr(bt), k, _ptr(sbt), _ptr(ce), N,
                                      _ptr(d[e]), N, nthreads)
        k0 += k
    return d


def k_grouped_gemm_tn_k32_sampled(a, sa, b, sb, ks, c, es, ms, ns, nthreads: int = 0) -> np.ndarray:
    """The elements (es[i], ms[i], ns[i]) of k_grouped_gemm_tn_k32, one by one,
    in its order (the fp64 product sum from 0, then C), rounded once to FP32."""
    a, b = _u8(a), _u8(b)
    es, ms, ns = (np.asarray(x, dtype=np.int64) for x in (es, ms, ns))
    out = np.empty(len(es), dtype=np.float32)
    k0 = 0
    for e, k in enumerate(ks):
        sel = np.nonzero(es == e)[0]
        if len(sel):
            cv = np.asarray(c[e], dtype=np.float32)[ms[sel], ns[sel]].astype(np.float64)
            if k == 0:
                out[sel] = cv.astype(np.float32)
            else:
                s0, s1 = k0 // 32, (k0 + k) // 32
                at = np.ascontiguousarray(a[k0:k0 + k].T)
                bt = np.ascontiguousarray(b[k0:k0 + k].T)
                sat = np.ascontiguousarray(sa[s0:s1].T, dtype=np.float64)
                sbt = np.ascontiguousarray(sb[s0:s1].T, dtype=np.float64)
                rows = np.ascontiguousarray(ms[sel])
                cols = np.ascontiguousarray(ns[sel])
                pre = np.empty(len(sel), dtype=np.float64)
                _get().orc_gemm_nt_gk_pre_sampled(k, 32, _ptr(at), k, _ptr(sat), _ptr(bt), k, _ptr(sbt),
                                                  len(sel), _ptr(rows), _ptr(cols), _ptr(pre), nthreads)
                out[sel] = (cv + pre).astype(np.float32)
        k0 += k
    return out


def k_grouped_gemm_tn_sampled(a, sa, b, sb, ks, c, es, ms, ns, nthreads: int = 0) -> np.ndarray:
    """The elements (es[i], ms[i], ns[i]) of k_grouped_gemm_tn, one by one, in
    the full function's order: the group's fp64 product sum (gemm_nt_sampled on
    the group's transposed slices, summed from 0 in increasing k), then C added
    in fp64, rounded once to FP32.  The result equals the full function's bit
    for bit."""
    a, b = _u8(a), _u8(b)
    es, ms, ns = (np.asarray(x, dtype=np.int64) for x in (es, ms, ns))
    out = np.empty(len(es), dtype=np.float32)
    k0 = 0
    for e, k in enumerate(ks):
        sel = np.nonzero(es == e)[0]
        if len(sel):
            cv = np.asarray(c[e], dtype=np.float64)[ms[sel], ns[sel]]
            if k == 0:
                out[sel] = cv.astype(np.float32)
            else:
                s0, s1 = k0 // 128, (k0 + k) // 128
                _, pre = gemm_nt_sampled(np.ascontiguousarray(a[k0:k0 + k].T), np.ascontiguousarray(sa[s0:s1].T),
                                         np.ascontiguousarray(b[k0:k0 + k].T), np.ascontiguousarray(sb[s0:s1].T),
                                         ms[sel], ns[sel], want_pre=True, nthreads=nthreads)
                out[sel] = (cv + pre).astype(np.float32)
        k0 += k
    return out


def gemm_nt_sampled(a, sa, b, sb_rows, rows, cols, c=None, want_pre=False, nthreads: int = 0):
    """The elements (rows[i], cols[i]) of gemm_nt, computed one by one."""
    a, b = _u8(a), _u8(b)
    M, K = a.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    sa = np.ascontiguousarray(sa, dtype=np.float64)
    sb_rows = np.ascontiguousarray(sb_rows, dtype=np.float64)
    ldc = 0
    if c is not None:
        c = np.ascontiguousarray(c).view(np.uint16)
        ldc = c.shape[1]
    out = np.empty(rows.shape[0], dtype=np.uint16)
    pre = np.empty(rows.shape[0], dtype=np.float64) if want_pre else None
    _get().orc_gemm_nt_sampled(K, _ptr(a), K, _ptr(sa), _ptr(b), K, _ptr(sb_rows), _ptr(c), ldc,
                               rows.shape[0], _ptr(rows), _ptr(cols), _ptr(out), _ptr(pre),
                               nthreads)
    return (out, pre) if want_pre else out


def m_grouped_contiguous(a, sa, b, sb_rows, grouped_layout, d_init=None, nthreads: int = 0):
    """Contiguous M-grouped GEMM (PaperTrace DeepGEMM §5.1): row m uses expert
    grouped_layout[m]; rows marked -1 are left as in d_init (default 0)."""
    a, b = _u8(a), _u8(b)
    M, K = a.shape
    E, N, _ = b.shape
    layout = np.ascontiguousarray(grouped_layout, dtype=np.int32)
    d = (np.zeros((M, N), dtype=np.uint16) if d_init is None
         else np.ascontiguousarray(d_init).view(np.uint16).copy())
    _get().orc_m_grouped_contiguous(M, N, K, E, _ptr(a), K,
                                    _ptr(np.ascontiguousarray(sa, dtype=np.float64)), _ptr(b), K,
                                    _ptr(np.ascontiguousarray(sb_rows, dtype=np.float64)),
                                    _ptr(layout), _ptr(d), N, nthreads)
    return d


def m_grouped_masked(a, sa, b, sb_rows, masked_m, d_init=None, nthreads: int = 0):
    """Masked M-grouped GEMM (PaperTrace DeepGEMM §5.2): a [E, max_m, K]; only
    rows m < masked_m[e] are computed; other rows keep d_init (default 0)."""
    a, b = _u8(a), _u8(b)
    E, max_m, K = a.shape
    N = b.shape[1]
    mm = np.ascontiguousarray(masked_m, dtype=np.int32)
    d = (np.zeros((E, max_m, N), dtype=np.uint16) if d_init is None
         else np.ascontiguousarray(d_init).view(np.uint16).copy())
    _get().orc_m_grouped_masked(E, max_m, N, K, _ptr(a),
                                _ptr(np.ascontiguousarray(sa, dtype=np.float64)), _ptr(b),
                                _ptr(np.ascontiguousarray(sb_rows, dtype=np.float64)), _ptr(mm),
                                _ptr(d), nthreads)
    return d


def psum_segments(psum, m_total: int):
    """Row segments of the PSUM contiguous layout (PaperTrace DeepGEMM §5.1: the
    per-expert prefix sums of received token counts are the group offsets; §3.1:
    groups are separated by gap rows).  Reading: psum[e] is the inclusive prefix
    sum of the token counts m_e; expert e's rows start at S_e with S_0 = 0 and
    S_{e+1} = align128(S_e + m_e); rows [S_e + m_e, S_{e+1}) are gap rows.

    Returns (starts [E+1] = S_0..S_E, counts [E]).  Raises ValueError if psum
    decreases or the segments end past m_total."""
    psum = [int(x) for x in psum]
    starts, counts, prev, s = [0], [], 0, 0
    for v in psum:
        m = v - prev
        if m < 0:
            raise ValueError("psum decreases")
        counts.append(m)
        s = (s + m + 127) // 128 * 128
        starts.append(s)
        prev = v
    if starts[-1] > m_total:
        raise ValueError("segments end past m_total")
    return starts, counts


def m_grouped_contiguous_psum(a, sa, b, sb_rows, psum, d_init=None, nthreads: int = 0):
    """Contiguous M-grouped GEMM with PSUM offsets (PaperTrace DeepGEMM §5.1,
    §3.1): expert e's rows [S_e, S_e + m_e) are computed with expert e's B; gap
    rows [S_e + m_e, S_{e+1}) are written 0; rows at or past S_E keep d_init
    (default 0).  Returns uint16 bf16 bits [m_total, N]."""
    a = _u8(a)
    M = a.shape[0]
    starts, counts = psum_segments(psum, M)
    layout = np.full(M, -1, dtype=np.int32)
    for e, m in enumerate(counts):
        layout[starts[e]:starts[e] + m] = e
    d = m_grouped_contiguous(a, sa, b, sb_rows, layout, d_init=d_init, nthreads=nthreads)
    for e, m in enumerate(counts):
        d[starts[e] + m:starts[e + 1]] = 0
    return d
