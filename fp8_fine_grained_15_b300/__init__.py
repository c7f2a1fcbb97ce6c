"""Python binding of the fp8bs C ABI (include/fp8bs.h).

Argument marshalling only: every function here forwards torch tensors' device
pointers, shapes and strides to the same-named C entry point of
``libfp8bs.so`` and raises :class:`Fp8bsError` on a non-OK status.  All
arithmetic runs in the library's CUDA kernels; if the library is missing the
import of a function fails loudly -- there is no CPU fallback.

PyTorch provides device memory and streams.  The default stream argument is
torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8bs.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "fp8bs.h")

# enums (mirroring include/fp8bs.h)
FP8BS_OK = 0
FP8BS_ERR_INVALID_ARG = 1
FP8BS_ERR_MISALIGNED = 2
FP8BS_ERR_UNSUPPORTED = 3
FP8BS_ERR_CUDA = 4
FP8BS_ERR_DEVICE_TIMEOUT = 5
FP8BS_ERR_DEVICE_BAD_OFFSETS = 6
FP8BS_ERR_DEVICE_BAD_ROUTING = 7
FP8BS_F32 = 0
FP8BS_BF16 = 1
FP8BS_SB_BLOCK_NK = 0
FP8BS_SB_BLOCK_KN = 1
FP8BS_SB_PERCOL = 2

_lib = None


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"fp8bs CUDA library not found at {LIB_PATH}; build it with "
                "`python -m fp8_fine_grained_15_b300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
        L.fp8bs_quant_act_1x128.argtypes = [P, I, I64, I64, I64, P, I64, P, I64, P]
        L.fp8bs_quant_act_128x1.argtypes = [P, I, I64, I64, I64, P, I64, P, I64, P]
        L.fp8bs_quant_w_128x128.argtypes = [P, I, I64, I64, I64, P, I64, P, I64, P, I64, P]
        L.fp8bs_gemm_accumulate.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I, I64, P,
                                            I64, P, ctypes.c_size_t, P]
        L.fp8bs_quant_dispatch.argtypes = [P, I, I64, I64, I64, P, I32, P, I64, P, I64, I64, P, P,
                                           P, P, P]
        L.fp8bs_quant_act_dual.argtypes = [P, I, I64, I64, I64, P, I64, P, I64, P, I64, P, I64, P]
        L.fp8bs_gemm.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I, I64, P, I, I64, P]
        L.fp8bs_grouped_gemm.argtypes = [I32, P, I64, I64, I64, P, I64, P, I64, P, I64, P, I,
                                         I64, I64, P, I, I64, P]
        L.fp8bs_gemm_workspace_size.argtypes = [I64, I64, I64, ctypes.POINTER(ctypes.c_size_t)]
        L.fp8bs_gemm_ws.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I, I64, P, I, I64, P,
                                    ctypes.c_size_t, P]
        L.fp8bs_gemm_static_ws.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I, I64, P, I,
                                           I64, P]
        L.fp8bs_mx_quant_1x32.argtypes = [P, I, I64, I64, I64, P, I64, P, I64, P]
        L.fp8bs_mx_gemm.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, I64, P, I, I64, P]
        L.fp8bs_sync_status.argtypes = [P]
        L.fp8bs_status_string.argtypes = [I]
        L.fp8bs_status_string.restype = ctypes.c_char_p
        L.fp8bs_debug_timeout_probe.argtypes = [I64, P]
        L.fp8bs_probe_mma_f8f6f4.argtypes = [P, P, I64, P, P]
        for name in ("fp8bs_quant_act_1x128", "fp8bs_quant_act_128x1", "fp8bs_quant_w_128x128",
                     "fp8bs_gemm", "fp8bs_grouped_gemm", "fp8bs_sync_status",
                     "fp8bs_debug_timeout_probe", "fp8bs_gemm_workspace_size", "fp8bs_gemm_ws",
                     "fp8bs_gemm_static_ws", "fp8bs_quant_act_dual", "fp8bs_gemm_accumulate",
                     "fp8bs_probe_mma_f8f6f4", "fp8bs_quant_dispatch", "fp8bs_mx_quant_1x32",
                     "fp8bs_mx_gemm"):
            getattr(L, name).restype = I
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/fp8bs.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:fp8bs_status|const char\*)\s+(fp8bs_\w+)\s*\(",
                                 text, flags=re.M)))


def status_string(status: int) -> str:
    try:
        return lib().fp8bs_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FP8BS_BF16
    if t.dtype == torch.float32:
        return FP8BS_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != FP8BS_OK:
        raise Fp8bsError(st, where)


def _row_stride(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


def fp8bs_quant_act_1x128(x, q, s, stream=None):
    """x [M x K] bf16/fp32 -> q [M x K] uint8 codes, s [K/128 x lds>=M] fp32."""
    M, K = x.shape
    _check(lib().fp8bs_quant_act_1x128(_ptr(x), _dtype(x), M, K, _row_stride(x), _ptr(q),
                                       _row_stride(q), _ptr(s), _row_stride(s),
                                       _stream(stream)), "fp8bs_quant_act_1x128")


def fp8bs_quant_act_128x1(x, qT, s, stream=None):
    """x [T x C] -> qT [C x T] uint8 codes (tokens contiguous), s [T/128 x lds>=C]."""
    T, C = x.shape
    _check(lib().fp8bs_quant_act_128x1(_ptr(x), _dtype(x), T, C, _row_stride(x), _ptr(qT),
                                       _row_stride(qT), _ptr(s), _row_stride(s),
                                       _stream(stream)), "fp8bs_quant_act_128x1")


def fp8bs_quant_act_dual(x, q, s, qT, sT, stream=None):
    """x [T x C] -> q [T x C] + s [C/128 x >=T] (1x128) and qT [C x T] +
    sT [T/128 x >=C] (128x1), from one read of x."""
    T, C = x.shape
    _check(lib().fp8bs_quant_act_dual(_ptr(x), _dtype(x), T, C, _row_stride(x), _ptr(q),
                                      _row_stride(q), _ptr(s), _row_stride(s), _ptr(qT),
                                      _row_stride(qT), _ptr(sT), _row_stride(sT),
                                      _stream(stream)), "fp8bs_quant_act_dual")


def fp8bs_quant_dispatch(x, expert, E: int, q, s, offsets, counts, token_row, row_token,
                         stream=None):
    """x [T x K] -> q [M_cap x K], s [K/128 x >=M_cap] in expert-grouped rows;
    expert [T] int32 device; offsets [E+1], counts [E], token_row [T],
    row_token [M_cap] int32 device outputs."""
    T, K = x.shape
    M_cap = q.shape[0]
    _check(lib().fp8bs_quant_dispatch(_ptr(x), _dtype(x), T, K, _row_stride(x), _ptr(expert), E,
                                      _ptr(q), _row_stride(q), _ptr(s), _row_stride(s), M_cap,
                                      _ptr(offsets), _ptr(counts), _ptr(token_row),
                                      _ptr(row_token), _stream(stream)), "fp8bs_quant_dispatch")


def fp8bs_quant_w_128x128(w, q, qT, s, stream=None):
    """w [R x C] -> q [R x C] (or None), qT [C x R] (or None), s [R/128 x lds>=C/128]."""
    R, C = w.shape
    _check(lib().fp8bs_quant_w_128x128(
        _ptr(w), _dtype(w), R, C, _row_stride(w), _ptr(q), _row_stride(q) if q is not None else 0,
        _ptr(qT), _row_stride(qT) if qT is not None else 0, _ptr(s), _row_stride(s),
        _stream(stream)), "fp8bs_quant_w_128x128")


def fp8bs_gemm(A, sa, B, sb, sb_mode: int, C, stream=None):
    """C [M x N] = block-scaled A [M x K] * B [N x K]^T (see include/fp8bs.h)."""
    M, K = A.shape
    N = B.shape[0]
    _check(lib().fp8bs_gemm(M, N, K, _ptr(A), _row_stride(A), _ptr(sa), _row_stride(sa),
                            _ptr(B), _row_stride(B), _ptr(sb), sb_mode, _row_stride(sb),
                            _ptr(C), _dtype(C), _row_stride(C), _stream(stream)), "fp8bs_gemm")


def fp8bs_gemm_workspace_size(M: int, N: int, K: int) -> int:
    """Bytes of workspace fp8bs_gemm_ws can use for this shape (0: no split)."""
    n = ctypes.c_size_t(0)
    _check(lib().fp8bs_gemm_workspace_size(M, N, K, ctypes.byref(n)),
           "fp8bs_gemm_workspace_size")
    return n.value


def fp8bs_gemm_ws(A, sa, B, sb, sb_mode: int, C, workspace, stream=None):
    """fp8bs_gemm with a device workspace (uint8 tensor, or None) for the K
    split of the last wave's tiles."""
    M, K = A.shape
    N = B.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8bs_gemm_ws(M, N, K, _ptr(A), _row_stride(A), _ptr(sa), _row_stride(sa),
                               _ptr(B), _row_stride(B), _ptr(sb), sb_mode, _row_stride(sb),
                               _ptr(C), _dtype(C), _row_stride(C), _ptr(workspace), ws_bytes,
                               _stream(stream)), "fp8bs_gemm_ws")


def fp8bs_gemm_accumulate(A, sa, B, sb, sb_mode: int, C, workspace=None, stream=None):
    """C (fp32) += block-scaled A * B^T; workspace as in fp8bs_gemm_ws."""
    M, K = A.shape
    N = B.shape[0]
    if C.dtype != __import__("torch").float32:
        raise TypeError("fp8bs_gemm_accumulate needs a float32 C")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8bs_gemm_accumulate(M, N, K, _ptr(A), _row_stride(A), _ptr(sa),
                                       _row_stride(sa), _ptr(B), _row_stride(B), _ptr(sb),
                                       sb_mode, _row_stride(sb), _ptr(C), _row_stride(C),
                                       _ptr(workspace), ws_bytes, _stream(stream)),
           "fp8bs_gemm_accumulate")


def fp8bs_gemm_static_ws(A, sa, B, sb, sb_mode: int, C, stream=None):
    """fp8bs_gemm_ws with the library's own 20 MiB device array as workspace
    (allocates nothing; calls must not overlap on the GPU)."""
    M, K = A.shape
    N = B.shape[0]
    _check(lib().fp8bs_gemm_static_ws(M, N, K, _ptr(A), _row_stride(A), _ptr(sa), _row_stride(sa),
                                      _ptr(B), _row_stride(B), _ptr(sb), sb_mode, _row_stride(sb),
                                      _ptr(C), _dtype(C), _row_stride(C), _stream(stream)),
           "fp8bs_gemm_static_ws")


def fp8bs_grouped_gemm(offsets, A, sa, B, sb, sb_mode: int, C, stream=None):
    """Expert e: C[offsets[e]:offsets[e+1]] = A[rows] * B[e]^T.
    offsets: device int32 [E+1]; B [E x N x K]; sb [E x ...] (per-expert layout
    sb_mode, row stride = ldsb)."""
    E, N, K = B.shape
    M_cap = A.shape[0]
    if B.stride(2) != 1 or B.stride(0) != N * B.stride(1):
        raise ValueError("B must be [E][N][ldb] with experts N*ldb bytes apart")
    if sb.dim() != 3 or sb.stride(2) != 1:
        raise ValueError("sb must be a 3-D tensor [E x rows x ld]")
    _check(lib().fp8bs_grouped_gemm(E, _ptr(offsets), M_cap, N, K, _ptr(A), _row_stride(A),
                                    _ptr(sa), _row_stride(sa), _ptr(B), B.stride(1), _ptr(sb),
                                    sb_mode, sb.stride(1), sb.stride(0), _ptr(C), _dtype(C),
                                    _row_stride(C), _stream(stream)), "fp8bs_grouped_gemm")


def _words(sf):
    """Row stride, in 32-bit words, of an exponent-word tensor: int32 [K/128 x ld]."""
    import torch
    if sf.dtype != torch.int32 or sf.dim() != 2 or sf.stride(1) != 1:
        raise ValueError("MX exponent words must be a 2-D int32 tensor with unit column stride")
    return sf.stride(0)


def fp8bs_mx_quant_1x32(x, q, sf, stream=None):
    """x [R x K] bf16/fp32 -> q [R x K] uint8 codes and sf [K/128 x ld>=R] int32
    words of four UE8M0 group exponents (group 4kb+j in byte j)."""
    R, K = x.shape
    _check(lib().fp8bs_mx_quant_1x32(_ptr(x), _dtype(x), R, K, _row_stride(x), _ptr(q),
                                     _row_stride(q), _ptr(sf), _words(sf), _stream(stream)),
           "fp8bs_mx_quant_1x32")


def fp8bs_mx_gemm(A, sfa, B, sfb, C, stream=None):
    """C [M x N] (bf16/fp32) = A [M x K] * B [N x K]^T with the MX group
    exponents sfa [K/128 x >=M], sfb [K/128 x >=N] (int32 words)."""
    M, K = A.shape
    N = B.shape[0]
    _check(lib().fp8bs_mx_gemm(M, N, K, _ptr(A), _row_stride(A), _ptr(sfa), _words(sfa), _ptr(B),
                               _row_stride(B), _ptr(sfb), _words(sfb), _ptr(C), _dtype(C),
                               _row_stride(C), _stream(stream)),
           "fp8bs_mx_gemm")


def fp8bs_sync_status(stream=None) -> int:
    """Synchronize and return (and clear) the device error status."""
    return lib().fp8bs_sync_status(_stream(stream))


def fp8bs_probe_mma_f8f6f4(a, b, d, stream=None):
    """d [128 x 256] fp32 = a [128 x K] * b [256 x K]^T over raw E4M3 codes,
    as the tensor cores compute it (K in 32..128, multiple of 32)."""
    K = a.shape[1]
    _check(lib().fp8bs_probe_mma_f8f6f4(_ptr(a), _ptr(b), K, _ptr(d), _stream(stream)),
           "fp8bs_probe_mma_f8f6f4")


def fp8bs_debug_timeout_probe(limit_ns: int, stream=None):
    _check(lib().fp8bs_debug_timeout_probe(limit_ns, _stream(stream)),
           "fp8bs_debug_timeout_probe")
