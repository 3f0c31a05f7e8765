"""CPU oracle for the dense GEMM -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline / reference leg may
import this package. The product path (``dense_tensor_core_gb300``) never imports it, and the two
share no code: this wraps ``dtc_oracle.c`` (plain C, fp64 accumulation, one RNE rounding at the
end), whose header states the definition it computes and the page passages it follows:

* 16-bit: ``C = round_out(A . Bop)``, ``Bop = B^T`` for "NT" (TileLang SM100 Support (Preview),
  "Code Example" and "Compilation and Usage") or ``Bop = B`` for "NN" (tilelang (velog), 1.1).
* MXFP8: e4m3 operands times ``2^(sf-127)`` per row per 128 K-elements (05 Blackwell TCGEN05 GEMM
  tutorial, "Advanced": gemm_blockscaled with granularity 128 for A and B).
* 2:4 structured-sparse A (the tutorial's gemm_sp, named in "An API-level note"): per group of
  4 K-elements two stored values and their positions (2-bit fields of a metadata nibble).
* The other block-scaled formats of that section, read as the OCP MX family: elements e4m3, e5m2,
  e2m3, e3m2 (fp6) or e2m1 (fp4), packed little-endian in rows; E8M0 scales per 32 or 128
  K-elements, or UE4M3 scales per 16 (NVFP4).

Arrays are numpy: 16-bit operands are passed as ``uint16`` code arrays, e4m3/E8M0 as ``uint8``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

BF16, F16 = 0, 1
NT, NN, TN, TT = 0, 1, 2, 3

_lib = None


def _bind(path):
    L = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    L.dtc_oracle_dec_bf16.restype = ctypes.c_double
    L.dtc_oracle_dec_bf16.argtypes = [ctypes.c_uint16]
    L.dtc_oracle_dec_f16.restype = ctypes.c_double
    L.dtc_oracle_dec_f16.argtypes = [ctypes.c_uint16]
    L.dtc_oracle_dec_e4m3.restype = ctypes.c_double
    L.dtc_oracle_dec_e4m3.argtypes = [ctypes.c_uint8]
    L.dtc_oracle_dec_e5m2.restype = ctypes.c_double
    L.dtc_oracle_dec_e5m2.argtypes = [ctypes.c_uint8]
    L.dtc_oracle_dec_e8m0.restype = ctypes.c_double
    L.dtc_oracle_dec_e8m0.argtypes = [ctypes.c_uint8]
    for name in ("e2m3", "e3m2", "e2m1", "ue4m3"):
        f = getattr(L, "dtc_oracle_dec_" + name)
        f.restype = ctypes.c_double
        f.argtypes = [ctypes.c_uint8]
    L.dtc_oracle_format_bits.restype = ctypes.c_int
    L.dtc_oracle_format_bits.argtypes = [ctypes.c_int]
    L.dtc_oracle_gemm_bs.restype = ctypes.c_int
    L.dtc_oracle_gemm_bs.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p,
                                     u8p, u8p, u8p, i64, i64, i64, u16p, dp, ctypes.c_int]
    L.dtc_oracle_gemm_bs_sampled.restype = ctypes.c_int
    L.dtc_oracle_gemm_bs_sampled.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, u8p, u8p, u8p, u8p, i64, i64, i64,
                                             i64p, i64p, i64, u16p, dp]
    L.dtc_oracle_enc_bf16.restype = ctypes.c_uint16
    L.dtc_oracle_enc_bf16.argtypes = [ctypes.c_double]
    L.dtc_oracle_enc_f16.restype = ctypes.c_uint16
    L.dtc_oracle_enc_f16.argtypes = [ctypes.c_double]
    L.dtc_oracle_gemm16.restype = ctypes.c_int
    L.dtc_oracle_gemm16.argtypes = [ctypes.c_int, ctypes.c_int, u16p, u16p, i64, i64, i64,
                                    u16p, dp, ctypes.c_int]
    L.dtc_oracle_gemm16_sampled.restype = ctypes.c_int
    L.dtc_oracle_gemm16_sampled.argtypes = [ctypes.c_int, ctypes.c_int, u16p, u16p, i64, i64,
                                            i64, i64p, i64p, i64, u16p, dp]
    L.dtc_oracle_gemm_mxfp8.restype = ctypes.c_int
    L.dtc_oracle_gemm_mxfp8.argtypes = [u8p, u8p, u8p, u8p, i64, i64, i64, u16p, dp,
                                        ctypes.c_int]
    L.dtc_oracle_gemm_mxfp8_sampled.restype = ctypes.c_int
    L.dtc_oracle_gemm_mxfp8_sampled.argtypes = [u8p, u8p, u8p, u8p, i64, i64, i64, i64p,
                                                i64p, i64, u16p, dp]
    L.dtc_oracle_gemm_mx.restype = ctypes.c_int
    L.dtc_oracle_gemm_mx.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p, u8p, u8p,
                                     i64, i64, i64, u16p, dp, ctypes.c_int]
    L.dtc_oracle_gemm_mx_sampled.restype = ctypes.c_int
    L.dtc_oracle_gemm_mx_sampled.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p,
                                             u8p, u8p, i64, i64, i64, i64p, i64p, i64, u16p, dp]
    L.dtc_oracle_gemm_sp.restype = ctypes.c_int
    L.dtc_oracle_gemm_sp.argtypes = [ctypes.c_int, ctypes.c_int, u16p, u8p, u16p, i64, i64, i64,
                                     u16p, dp, ctypes.c_int]
    L.dtc_oracle_default_threads.restype = ctypes.c_int
    return L


def lib():
    """The oracle library built from this directory's source.

    ``DTC_ORACLE_LIB`` may name another build of the same source; the tests use it to run the
    pins against copies with deliberately planted mistakes and check that the pins catch them."""
    global _lib
    if _lib is None:
        _lib = _bind(os.environ.get("DTC_ORACLE_LIB") or _build.build())
    return _lib


def _L():
    return lib()


def threads() -> int:
    """Worker threads the oracle uses by default: the host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return _L().dtc_oracle_default_threads()


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _dtype_code(dtype):
    return {"bf16": BF16, "f16": F16, BF16: BF16, F16: F16}[dtype]


def _layout_code(layout):
    return {"NT": NT, "NN": NN, "TN": TN, "TT": TT, NT: NT, NN: NN, TN: TN, TT: TT}[layout]


def a_shape(layout, M, K):
    """Storage shape of A: [M,K], or [K,M] when the layout's first letter is T."""
    return (K, M) if layout[0] == "T" else (M, K)


def b_shape(layout, N, K):
    """Storage shape of B: [N,K] when the layout's second letter is T, else [K,N]."""
    return (N, K) if layout[1] == "T" else (K, N)


# --- codecs -----------------------------------------------------------------------------------

def dec_bf16(codes):
    f = _L().dtc_oracle_dec_bf16
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint16).ravel()])


def dec_f16(codes):
    f = _L().dtc_oracle_dec_f16
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint16).ravel()])


def dec_e4m3(codes):
    f = _L().dtc_oracle_dec_e4m3
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def dec_e5m2(codes):
    f = _L().dtc_oracle_dec_e5m2
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def dec_e8m0(codes):
    f = _L().dtc_oracle_dec_e8m0
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def enc_bf16(values):
    f = _L().dtc_oracle_enc_bf16
    return np.array([f(float(v)) for v in np.asarray(values, dtype=np.float64).ravel()],
                    dtype=np.uint16)


def enc_f16(values):
    f = _L().dtc_oracle_enc_f16
    return np.array([f(float(v)) for v in np.asarray(values, dtype=np.float64).ravel()],
                    dtype=np.uint16)


# --- GEMM -------------------------------------------------------------------------------------

def gemm16(dtype, layout, A, B, M, N, K, *, sums=False, nthreads=None):
    """Full C (uint16 codes, [M,N]); with ``sums=True`` also the unrounded fp64 sums."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    assert A.size == M * K and B.size == N * K
    C = np.zeros((M, N), dtype=np.uint16)
    S = np.zeros((M, N), dtype=np.float64) if sums else None
    rc = _L().dtc_oracle_gemm16(_dtype_code(dtype), _layout_code(layout), _ptr(A, ctypes.c_uint16),
                                 _ptr(B, ctypes.c_uint16), M, N, K, _ptr(C, ctypes.c_uint16),
                                 _ptr(S, ctypes.c_double), nthreads or threads())
    if rc != 0:
        raise ValueError("oracle gemm16 rejected its arguments")
    return (C, S) if sums else C


def gemm16_sampled(dtype, layout, A, B, M, N, K, rows, cols):
    """C at the listed (rows[i], cols[i]) only: (codes, unrounded sums)."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    C = np.zeros(rows.size, dtype=np.uint16)
    S = np.zeros(rows.size, dtype=np.float64)
    rc = _L().dtc_oracle_gemm16_sampled(_dtype_code(dtype), _layout_code(layout),
                                         _ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), M, N,
                                         K, _ptr(rows, ctypes.c_int64), _ptr(cols, ctypes.c_int64),
                                         rows.size, _ptr(C, ctypes.c_uint16),
                                         _ptr(S, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gemm16_sampled rejected its arguments")
    return C, S


def gemm_mxfp8(A, B, sfA, sfB, M, N, K, *, sums=False, nthreads=None):
    """Block-scaled e4m3 GEMM, NT; scales are [rows, ceil(K/128)] E8M0 codes. Output bf16 codes."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
    sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
    kb = (K + 127) // 128
    assert A.size == M * K and B.size == N * K and sfA.size == M * kb and sfB.size == N * kb
    C = np.zeros((M, N), dtype=np.uint16)
    S = np.zeros((M, N), dtype=np.float64) if sums else None
    rc = _L().dtc_oracle_gemm_mxfp8(_ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                     _ptr(sfA, ctypes.c_uint8), _ptr(sfB, ctypes.c_uint8), M, N, K,
                                     _ptr(C, ctypes.c_uint16), _ptr(S, ctypes.c_double),
                                     nthreads or threads())
    if rc != 0:
        raise ValueError("oracle gemm_mxfp8 rejected its arguments")
    return (C, S) if sums else C


def gemm_mxfp8_sampled(A, B, sfA, sfB, M, N, K, rows, cols):
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
    sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    C = np.zeros(rows.size, dtype=np.uint16)
    S = np.zeros(rows.size, dtype=np.float64)
    rc = _L().dtc_oracle_gemm_mxfp8_sampled(_ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                             _ptr(sfA, ctypes.c_uint8), _ptr(sfB, ctypes.c_uint8),
                                             M, N, K, _ptr(rows, ctypes.c_int64),
                                             _ptr(cols, ctypes.c_int64), rows.size,
                                             _ptr(C, ctypes.c_uint16), _ptr(S, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gemm_mxfp8_sampled rejected its arguments")
    return C, S


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def _mx_inputs(A, B, sfA, sfB, M, N, K, block):
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
    sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
    kb = (K + block - 1) // block
    assert A.size == M * K and B.size == N * K and sfA.size == M * kb and sfB.size == N * kb
    return A, B, sfA, sfB


def gemm_mx(A, B, sfA, sfB, M, N, K, *, a_fmt="e4m3", b_fmt="e4m3", block=128, sums=False,
            nthreads=None):
    """Block-scaled fp8 GEMM, NT: A [M,K] and B [N,K] as e4m3 or e5m2 codes, scales
    [rows, ceil(K/block)] E8M0 codes with block 128 or 32. Output bf16 codes."""
    A, B, sfA, sfB = _mx_inputs(A, B, sfA, sfB, M, N, K, block)
    C = np.zeros((M, N), dtype=np.uint16)
    S = np.zeros((M, N), dtype=np.float64) if sums else None
    rc = _L().dtc_oracle_gemm_mx(FP8_FORMATS[a_fmt], FP8_FORMATS[b_fmt], block,
                                  _ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                  _ptr(sfA, ctypes.c_uint8), _ptr(sfB, ctypes.c_uint8), M, N, K,
                                  _ptr(C, ctypes.c_uint16), _ptr(S, ctypes.c_double),
                                  nthreads or threads())
    if rc != 0:
        raise ValueError("oracle gemm_mx rejected its arguments")
    return (C, S) if sums else C


def gemm_mx_sampled(A, B, sfA, sfB, M, N, K, rows, cols, *, a_fmt="e4m3", b_fmt="e4m3",
                    block=128):
    A, B, sfA, sfB = _mx_inputs(A, B, sfA, sfB, M, N, K, block)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    C = np.zeros(rows.size, dtype=np.uint16)
    S = np.zeros(rows.size, dtype=np.float64)
    rc = _L().dtc_oracle_gemm_mx_sampled(FP8_FORMATS[a_fmt], FP8_FORMATS[b_fmt], block,
                                          _ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                          _ptr(sfA, ctypes.c_uint8), _ptr(sfB, ctypes.c_uint8),
                                          M, N, K, _ptr(rows, ctypes.c_int64),
                                          _ptr(cols, ctypes.c_int64), rows.size,
                                          _ptr(C, ctypes.c_uint16), _ptr(S, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gemm_mx_sampled rejected its arguments")
    return C, S


# --- the general block-scaled family (OCP MX element formats, packed rows) ---------------------

BS_FORMATS = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4}
BS_SCALES = {"e8m0": 0, "ue4m3": 1}
FORMAT_BITS = {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}


def dec_e2m3(codes):
    f = _L().dtc_oracle_dec_e2m3
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def dec_e3m2(codes):
    f = _L().dtc_oracle_dec_e3m2
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def dec_e2m1(codes):
    f = _L().dtc_oracle_dec_e2m1
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def dec_ue4m3(codes):
    f = _L().dtc_oracle_dec_ue4m3
    return np.array([f(int(c)) for c in np.asarray(codes, dtype=np.uint8).ravel()])


def row_bytes(fmt, K):
    """Bytes of one packed row of K elements of format `fmt`."""
    return (K * FORMAT_BITS[fmt] + 7) // 8


def _bs_inputs(A, B, sfA, sfB, M, N, K, a_fmt, b_fmt, block):
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
    sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
    kb = (K + block - 1) // block
    assert A.size == M * row_bytes(a_fmt, K) and B.size == N * row_bytes(b_fmt, K)
    assert sfA.size == M * kb and sfB.size == N * kb
    return A, B, sfA, sfB


def gemm_bs(A, B, sfA, sfB, M, N, K, *, a_fmt="e4m3", b_fmt="e4m3", scale="e8m0", block=128,
            sums=False, nthreads=None):
    """Block-scaled GEMM, NT: A [M, row_bytes(a_fmt, K)] and B [N, row_bytes(b_fmt, K)] packed
    rows of element codes, scales [rows, ceil(K/block)] (E8M0 or UE4M3 codes, block 16, 32 or
    128). Output bf16 codes."""
    A, B, sfA, sfB = _bs_inputs(A, B, sfA, sfB, M, N, K, a_fmt, b_fmt, block)
    C = np.zeros((M, N), dtype=np.uint16)
    S = np.zeros((M, N), dtype=np.float64) if sums else None
    rc = _L().dtc_oracle_gemm_bs(BS_FORMATS[a_fmt], BS_FORMATS[b_fmt], BS_SCALES[scale], block,
                                  _ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                  _ptr(sfA, ctypes.c_uint8), _ptr(sfB, ctypes.c_uint8), M, N, K,
                                  _ptr(C, ctypes.c_uint16), _ptr(S, ctypes.c_double),
                                  nthreads or threads())
    if rc != 0:
        raise ValueError("oracle gemm_bs rejected its arguments")
    return (C, S) if sums else C


def gemm_bs_sampled(A, B, sfA, sfB, M, N, K, rows, cols, *, a_fmt="e4m3", b_fmt="e4m3",
                    scale="e8m0", block=128):
    A, B, sfA, sfB = _bs_inputs(A, B, sfA, sfB, M, N, K, a_fmt, b_fmt, block)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    C = np.zeros(rows.size, dtype=np.uint16)
    S = np.zeros(rows.size, dtype=np.float64)
    rc = _L().dtc_oracle_gemm_bs_sampled(BS_FORMATS[a_fmt], BS_FORMATS[b_fmt], BS_SCALES[scale],
                                          block, _ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                          _ptr(sfA, ctypes.c_uint8), _ptr(sfB, ctypes.c_uint8),
                                          M, N, K, _ptr(rows, ctypes.c_int64),
                                          _ptr(cols, ctypes.c_int64), rows.size,
                                          _ptr(C, ctypes.c_uint16), _ptr(S, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gemm_bs_sampled rejected its arguments")
    return C, S


# --- 2:4 structured-sparse A --------------------------------------------------------------------

def gemm_sp(dtype, layout, vals, meta, B, M, N, K, *, sums=False, nthreads=None):
    """Sparse-A GEMM: vals [M, K/2] 16-bit codes (two stored values per group of 4 K-elements),
    meta [M, K/8] bytes (group g's nibble at bits 4*(g % 2) of byte g/2: bits 0-1 the position of
    the group's first value, bits 2-3 of its second), B as for gemm16 ("NT" or "NN")."""
    vals = np.ascontiguousarray(vals, dtype=np.uint16)
    meta = np.ascontiguousarray(meta, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    assert vals.size == M * (K // 2) and meta.size == M * ((K // 4 + 1) // 2) and B.size == N * K
    C = np.zeros((M, N), dtype=np.uint16)
    S = np.zeros((M, N), dtype=np.float64) if sums else None
    rc = _L().dtc_oracle_gemm_sp(_dtype_code(dtype), _layout_code(layout),
                                  _ptr(vals, ctypes.c_uint16), _ptr(meta, ctypes.c_uint8),
                                  _ptr(B, ctypes.c_uint16), M, N, K, _ptr(C, ctypes.c_uint16),
                                  _ptr(S, ctypes.c_double), nthreads or threads())
    if rc != 0:
        raise ValueError("oracle gemm_sp rejected its arguments")
    return (C, S) if sums else C
