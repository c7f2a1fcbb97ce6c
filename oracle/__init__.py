"""CPU oracle for the fine-grained FP8 quantizers and block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and bench.py's CPU
baseline leg are the only callers.  The product library never imports this
package and this package never imports the product library.

The arithmetic lives in ``fp8bs_oracle.c`` (plain C, binary32 quantization,
binary64 GEMM); this module compiles it with gcc on first use and wraps it with
numpy arrays.  Grouped GEMM is the dense oracle applied expert by expert.
The MX variant (UE8M0 power-of-two scales on 1x32 groups, applied per group)
has its own quantizer and GEMM in the same file, and so does the
quantize-then-dispatch step of MoE layers (stable grouping of tokens by
expert, padding to 128 rows, 1x128 quantization of each routed row).

The GEMMs split their output elements over POSIX threads (one per online CPU
unless ``set_threads`` says otherwise); each element is computed by the same
loop in the same order whatever the thread count.

Every function cites the passage it restates in the C source's header.  Pins
(tests/test_oracle_pins.py) tie it to the OCP E4M3 format, to PyTorch's own
float8_e4m3fn conversion, to brute force and to closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bs_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
SB_BLOCK_NK, SB_BLOCK_KN, SB_PERCOL = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-Wall", "-Wextra", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.fp8bs_oracle_e4m3_decode.restype = ctypes.c_double
        lib.fp8bs_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fp8bs_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.fp8bs_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fp8bs_oracle_e4m3_encode_n.argtypes = [P, I64, P]
        lib.fp8bs_oracle_e4m3_encode_n.restype = None
        lib.fp8bs_oracle_quant_act_1x128.argtypes = [P, I, I64, I64, I64, P, I64, P, I64]
        lib.fp8bs_oracle_quant_act_128x1.argtypes = [P, I, I64, I64, I64, P, I64, P, I64]
        lib.fp8bs_oracle_quant_w_128x128.argtypes = [P, I, I64, I64, I64, P, I64, P, I64, P]
        lib.fp8bs_oracle_gemm.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I, I64, P, P]
        lib.fp8bs_oracle_gemm_elements.argtypes = [I64, P, I64, P, I64, P, I64, P, I, I64,
                                                   I64, P, P, P, P]
        lib.fp8bs_oracle_mx_quant_1x32.argtypes = [P, I, I64, I64, I64, P, I64, P, I64]
        lib.fp8bs_oracle_mx_gemm.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I64,
                                             P, P]
        lib.fp8bs_oracle_mx_gemm_elements.argtypes = [I64, P, I64, P, I64, P, I64, P, I64,
                                                      I64, P, P, P, P]
        for f in ("quant_act_1x128", "quant_act_128x1", "quant_w_128x128", "gemm",
                  "gemm_elements", "mx_quant_1x32", "mx_gemm", "mx_gemm_elements"):
            getattr(lib, "fp8bs_oracle_" + f).restype = None
        lib.fp8bs_oracle_set_threads.argtypes = [I]
        lib.fp8bs_oracle_set_threads.restype = None
        lib.fp8bs_oracle_threads.argtypes = []
        lib.fp8bs_oracle_threads.restype = I
        lib.fp8bs_oracle_dispatch.argtypes = [P, I, I64, I64, I64, P, ctypes.c_int32, I64, P, I64,
                                              P, I64, P, P, P, P]
        lib.fp8bs_oracle_dispatch.restype = I64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_input(x: np.ndarray):
    """Return (contiguous array, dtype code).  bf16 inputs arrive as uint16 bits."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"oracle input must be float32 or bf16 bits (uint16), got {x.dtype}")


def set_threads(n: int) -> None:
    """Threads the GEMMs use (n <= 0: one per online CPU)."""
    _load().fp8bs_oracle_set_threads(int(n))


def threads() -> int:
    """Threads the GEMMs use now."""
    return int(_load().fp8bs_oracle_threads())


# ------------------------------------------------------------------ E4M3

def e4m3_decode(code: int) -> float:
    return _load().fp8bs_oracle_e4m3_decode(code)


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: float) -> int:
    return _load().fp8bs_oracle_e4m3_encode(v)


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    """Encode every fp32 value on its own (no tile scaling)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, np.uint8)
    _load().fp8bs_oracle_e4m3_encode_n(_ptr(v), v.size, _ptr(out))
    return out


# ------------------------------------------------------------ quantizers

def quant_act_1x128(x: np.ndarray):
    """1x128 tiles along K.  x [M x K] (float32 or bf16 bits) ->
    (q [M x K] uint8, s [K/128 x M] float32)."""
    x, dt = _as_input(x)
    M, K = x.shape
    assert K % 128 == 0
    q = np.zeros((M, K), np.uint8)
    s = np.zeros((K // 128, M), np.float32)
    _load().fp8bs_oracle_quant_act_1x128(_ptr(x), dt, M, K, K, _ptr(q), K, _ptr(s), M)
    return q, s


def quant_act_128x1(x: np.ndarray):
    """128x1 tiles along T (tokens).  x [T x C] -> (qT [C x T] uint8,
    s [T/128 x C] float32)."""
    x, dt = _as_input(x)
    T, C = x.shape
    assert T % 128 == 0
    qT = np.zeros((C, T), np.uint8)
    s = np.zeros((T // 128, C), np.float32)
    _load().fp8bs_oracle_quant_act_128x1(_ptr(x), dt, T, C, C, _ptr(qT), T, _ptr(s), C)
    return qT, s


def quant_w_128x128(w: np.ndarray, with_transpose: bool = True):
    """128x128 blocks.  w [R x C] -> (q [R x C], qT [C x R] or None,
    s [R/128 x C/128])."""
    w, dt = _as_input(w)
    R, C = w.shape
    assert R % 128 == 0 and C % 128 == 0
    q = np.zeros((R, C), np.uint8)
    qT = np.zeros((C, R), np.uint8) if with_transpose else None
    s = np.zeros((R // 128, C // 128), np.float32)
    _load().fp8bs_oracle_quant_w_128x128(_ptr(w), dt, R, C, C, _ptr(q), C,
                                         _ptr(qT) if qT is not None else None, R, _ptr(s))
    return q, qT, s


def dequant_act_1x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Dequantized activations (fp64): dec(q[m][k]) * s[k/128][m]."""
    dec = e4m3_decode_table()
    return dec[q] * np.repeat(s.T.astype(np.float64), 128, axis=1)


def dequant_w_128x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    dec = e4m3_decode_table()
    return dec[q] * np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)


# ------------------------------------------------------------------ GEMM

def _sb_ld(sb: np.ndarray) -> int:
    return sb.shape[1]


def gemm(A: np.ndarray, sa: np.ndarray, B: np.ndarray, sb: np.ndarray, sb_mode: int):
    """Block-scaled GEMM by definition.  A [M x K] codes, sa [K/128 x M];
    B [N x K] codes; sb in the layout sb_mode names.  Returns (C_ref, S_abs),
    both float64 [M x N]."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and K % 128 == 0 and sa.shape == (K // 128, M)
    c = np.zeros((M, N), np.float64)
    a = np.zeros((M, N), np.float64)
    _load().fp8bs_oracle_gemm(M, N, K, _ptr(A), K, _ptr(sa), M, _ptr(B), K, _ptr(sb), sb_mode,
                              _sb_ld(sb), _ptr(c), _ptr(a))
    return c, a


def gemm_elements(A, sa, B, sb, sb_mode: int, rows, cols):
    """Same as gemm() at the listed (row, col) positions only."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    M, K = A.shape
    assert B.shape[1] == K and K % 128 == 0 and sa.shape == (K // 128, M)
    c = np.zeros(rows.size, np.float64)
    a = np.zeros(rows.size, np.float64)
    _load().fp8bs_oracle_gemm_elements(K, _ptr(A), K, _ptr(sa), M, _ptr(B), K, _ptr(sb), sb_mode,
                                       _sb_ld(sb), rows.size, _ptr(rows), _ptr(cols),
                                       _ptr(c), _ptr(a))
    return c, a


def grouped_gemm(offsets, A, sa, B, sb, sb_mode: int):
    """Grouped GEMM: the dense oracle per expert e over rows
    offsets[e]..offsets[e+1] with B[e], sb[e].  Rows past offsets[-1] stay 0."""
    offsets = [int(v) for v in offsets]
    M = A.shape[0]
    N = B.shape[1]
    c = np.zeros((M, N), np.float64)
    a = np.zeros((M, N), np.float64)
    for e in range(len(offsets) - 1):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        ce, ae = gemm(A[r0:r1], sa[:, r0:r1], B[e], sb[e], sb_mode)
        c[r0:r1], a[r0:r1] = ce, ae
    return c, a


def grouped_gemm_elements(offsets, A, sa, B, sb, sb_mode: int, rows, cols):
    """grouped_gemm() at the listed positions; rows must be < offsets[-1]."""
    offsets = np.asarray(offsets, np.int64)
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    expert = np.searchsorted(offsets, rows, side="right") - 1
    c = np.zeros(rows.size, np.float64)
    a = np.zeros(rows.size, np.float64)
    for e in np.unique(expert):
        sel = np.nonzero(expert == e)[0]
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        ce, ae = gemm_elements(A[r0:r1], sa[:, r0:r1], B[e], sb[e], sb_mode,
                               rows[sel] - r0, cols[sel])
        c[sel], a[sel] = ce, ae
    return c, a


# ------------------------------------------------------------ MX variant

def mx_quant_1x32(x: np.ndarray):
    """1x32 groups along K with power-of-two (UE8M0) scales.  x [R x K]
    (float32 or bf16 bits) -> (q [R x K] uint8, sf [K/128 x R x 4] uint8):
    sf[kb, r, j] = e + 127 for the group of columns 128*kb + 32*j .. +31 of
    row r, whose values were multiplied by 2^-e before the E4M3 rounding."""
    x, dt = _as_input(x)
    R, K = x.shape
    assert K % 128 == 0
    q = np.zeros((R, K), np.uint8)
    sf = np.zeros((K // 128, R, 4), np.uint8)
    _load().fp8bs_oracle_mx_quant_1x32(_ptr(x), dt, R, K, K, _ptr(q), K, _ptr(sf), R)
    return q, sf


def mx_dequant(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """dec(q[r][k]) * 2^(sf byte of (r, k/32) - 127), fp64."""
    dec = e4m3_decode_table()
    R, K = q.shape
    e = sf.transpose(1, 0, 2).reshape(R, K // 32).astype(np.int64) - 127
    return dec[q] * np.ldexp(1.0, np.repeat(e, 32, axis=1))


def mx_gemm(A: np.ndarray, sfa: np.ndarray, B: np.ndarray, sfb: np.ndarray):
    """MX GEMM by definition: C = A * B^T with each 32-deep group's product sum
    multiplied by 2^(ea + eb).  A [M x K], B [N x K] codes; sfa [K/128 x M x 4],
    sfb [K/128 x N x 4].  Returns (C_ref, S_abs), float64 [M x N]."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    sfa = np.ascontiguousarray(sfa, np.uint8)
    sfb = np.ascontiguousarray(sfb, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and K % 128 == 0
    assert sfa.shape == (K // 128, M, 4) and sfb.shape == (K // 128, N, 4)
    c = np.zeros((M, N), np.float64)
    a = np.zeros((M, N), np.float64)
    _load().fp8bs_oracle_mx_gemm(M, N, K, _ptr(A), K, _ptr(sfa), M, _ptr(B), K, _ptr(sfb), N,
                                 _ptr(c), _ptr(a))
    return c, a


def mx_gemm_elements(A, sfa, B, sfb, rows, cols):
    """mx_gemm() at the listed (row, col) positions only."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    sfa = np.ascontiguousarray(sfa, np.uint8)
    sfb = np.ascontiguousarray(sfb, np.uint8)
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    M, K = A.shape
    N = B.shape[0]
    assert sfa.shape == (K // 128, M, 4) and sfb.shape == (K // 128, N, 4)
    c = np.zeros(rows.size, np.float64)
    a = np.zeros(rows.size, np.float64)
    _load().fp8bs_oracle_mx_gemm_elements(K, _ptr(A), K, _ptr(sfa), M, _ptr(B), K, _ptr(sfb), N,
                                          rows.size, _ptr(rows), _ptr(cols), _ptr(c), _ptr(a))
    return c, a


# ------------------------------------------------- quantize-then-dispatch

def dispatch(x: np.ndarray, expert: np.ndarray, E: int):
    """Quantize-then-dispatch by its steps (see the C source): tokens grouped
    by expert in token order, each expert padded to a multiple of 128 rows,
    routed rows quantized 1x128, padding rows codes 0 / scale 1.  x [T x K]
    (float32 or bf16 bits), expert [T] ints (ids outside [0, E) are dropped).
    Returns (q [n x K], s [K/128 x n], offsets [E+1], counts [E],
    token_row [T] (-1 for dropped tokens), row_token [n] (-1 on padding rows),
    dropped), n = offsets[E]."""
    x, dt = _as_input(x)
    T, K = x.shape
    assert K % 128 == 0
    expert = np.ascontiguousarray(expert, np.int32)
    assert expert.shape == (T,)
    M_cap = (T + 127 * E + 127) // 128 * 128
    q = np.zeros((max(M_cap, 1), K), np.uint8)
    s = np.zeros((K // 128, max(M_cap, 1)), np.float32)
    offsets = np.zeros(E + 1, np.int64)
    counts = np.zeros(E, np.int64)
    token_row = np.zeros(max(T, 1), np.int64)
    row_token = np.zeros(max(M_cap, 1), np.int64)
    dropped = _load().fp8bs_oracle_dispatch(
        _ptr(x), dt, T, K, K, _ptr(expert), E, M_cap, _ptr(q), K, _ptr(s), s.shape[1],
        _ptr(offsets), _ptr(counts), _ptr(token_row), _ptr(row_token))
    assert dropped >= 0
    n = int(offsets[E])
    return (q[:n], np.ascontiguousarray(s[:, :n]), offsets, counts, token_row[:T],
            row_token[:n], int(dropped))
