"""Helpers shared by the GPU parity tests: run the library's entry points on
host tensors and bring the results back, and the GEMM tolerance check."""
from __future__ import annotations

import numpy as np
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
from workloads import bf16_bits

DEV = "cuda:0"


def oracle_input(x: torch.Tensor) -> np.ndarray:
    """The bytes the oracle reads: fp32 values or raw bf16 bits."""
    return bf16_bits(x) if x.dtype == torch.bfloat16 else x.contiguous().numpy()


def gpu_quant_1x128(x: torch.Tensor, pad_ld: int = 0, pad_lds: int = 0):
    M, K = x.shape
    xd = torch.zeros((M, K + pad_ld), dtype=x.dtype, device=DEV)[:, :K]
    xd.copy_(x)
    q = torch.full((M, K + pad_ld), 0xAB, dtype=torch.uint8, device=DEV)[:, :K]
    s = torch.full((K // 128, M + pad_lds), -1.0, dtype=torch.float32, device=DEV)[:, :M]
    fb.fp8bs_quant_act_1x128(xd, q, s)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return q.cpu().numpy(), s.cpu().numpy()


def gpu_quant_128x1(x: torch.Tensor):
    T, C = x.shape
    xd = x.to(DEV)
    qT = torch.full((C, T), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((T // 128, C), -1.0, dtype=torch.float32, device=DEV)
    fb.fp8bs_quant_act_128x1(xd, qT, s)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return qT.cpu().numpy(), s.cpu().numpy()


def gpu_quant_dual(x: torch.Tensor, pad: int = 0):
    """Both activation quantizers from one pass; outputs padded by `pad`
    elements in every leading dimension (pre-filled with sentinels)."""
    T, C = x.shape
    xd = torch.zeros((T, C + pad * 8), dtype=x.dtype, device=DEV)[:, :C]
    xd.copy_(x)
    q = torch.full((T, C + pad * 16), 0xAB, dtype=torch.uint8, device=DEV)[:, :C]
    s = torch.full((C // 128, T + pad), -1.0, dtype=torch.float32, device=DEV)[:, :T]
    qT = torch.full((C, T + pad * 16), 0xAB, dtype=torch.uint8, device=DEV)[:, :T]
    sT = torch.full((T // 128, C + pad), -1.0, dtype=torch.float32, device=DEV)[:, :C]
    fb.fp8bs_quant_act_dual(xd, q, s, qT, sT)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return q.cpu().numpy(), s.cpu().numpy(), qT.cpu().numpy(), sT.cpu().numpy()


def gpu_quant_w(w: torch.Tensor, want_q: bool = True, want_qT: bool = True):
    R, C = w.shape
    wd = w.to(DEV)
    q = torch.full((R, C), 0xAB, dtype=torch.uint8, device=DEV) if want_q else None
    qT = torch.full((C, R), 0xAB, dtype=torch.uint8, device=DEV) if want_qT else None
    s = torch.full((R // 128, C // 128), -1.0, dtype=torch.float32, device=DEV)
    fb.fp8bs_quant_w_128x128(wd, q, qT, s)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return (q.cpu().numpy() if q is not None else None,
            qT.cpu().numpy() if qT is not None else None, s.cpu().numpy())


def to_dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(DEV)


def to_dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def gpu_gemm(A: np.ndarray, sa: np.ndarray, B: np.ndarray, sb: np.ndarray, sb_mode: int,
             out_dtype=torch.bfloat16) -> np.ndarray:
    M = A.shape[0]
    N = B.shape[0]
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    fb.fp8bs_gemm(to_dev_u8(A), to_dev_f32(sa), to_dev_u8(B), to_dev_f32(sb), sb_mode, C)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return C.float().cpu().numpy().astype(np.float64)


def gemm_bound(c_ref: np.ndarray, s_abs: np.ndarray, bf16_out: bool) -> np.ndarray:
    """Element-wise tolerance: 2^-7 |C_ref| + 1e-5 S_abs for BF16 output,
    1e-5 S_abs for FP32 output (S_abs = sum_k |a_ik b_kj|, dequantized)."""
    if bf16_out:
        return 2.0 ** -7 * np.abs(c_ref) + 1e-5 * s_abs
    return 1e-5 * s_abs


def assert_gemm_close(c_gpu, c_ref, s_abs, bf16_out: bool, what: str = ""):
    err = np.abs(c_gpu - c_ref)
    bound = gemm_bound(c_ref, s_abs, bf16_out)
    bad = ~(err <= bound)          # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = [(tuple(i), float(c_gpu[tuple(i)]), float(c_ref[tuple(i)]),
                   float(bound[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"first (index, gpu, ref, bound): {detail}")
    return float(np.max(err / np.maximum(bound, 1e-300)))


MODES = {"KN": oracle.SB_BLOCK_KN, "NK": oracle.SB_BLOCK_NK, "PERCOL": oracle.SB_PERCOL}


def gemm_operands(M, N, K, mode, seed):
    """Oracle-quantized A [M x K] (1x128) and B [N x K] with scales in `mode` layout."""
    a = wl.random_matrix((M, K), seed=seed, dtype=torch.bfloat16)
    Aq, sa = oracle.quant_act_1x128(oracle_input(a))
    if mode == "PERCOL":
        bt = wl.random_matrix((K, N), seed=seed + 1, dtype=torch.bfloat16, std=1e-3)
        Bq, sb = oracle.quant_act_128x1(oracle_input(bt))       # [N x K], [K/128 x N]
    else:
        w = wl.random_matrix((K, N), seed=seed + 1, dtype=torch.bfloat16, std=0.02)
        Wq, WqT, sw = oracle.quant_w_128x128(oracle_input(w))   # sw [K/128 x N/128]
        Bq, sb = WqT, sw
        if mode == "NK":
            sb = np.ascontiguousarray(sw.T)                      # [N/128 x K/128]
    return Aq, sa, Bq, sb


def gpu_gemm_ws(A, sa, B, sb, sb_mode, out_dtype=torch.bfloat16, ws_bytes=None):
    """fp8bs_gemm_ws with a workspace of ws_bytes (default: the full size the
    library asks for; 0: no workspace)."""
    M, N = A.shape[0], B.shape[0]
    if ws_bytes is None:
        ws_bytes = fb.fp8bs_gemm_workspace_size(M, N, A.shape[1])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV) if ws_bytes > 0 else None
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    fb.fp8bs_gemm_ws(to_dev_u8(A), to_dev_f32(sa), to_dev_u8(B), to_dev_f32(sb), sb_mode, C, ws)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return C.float().cpu().numpy().astype(np.float64)
