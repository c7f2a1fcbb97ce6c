"""Block-scaled GEMM parity: CUDA kernel vs the CPU oracle on the same
(oracle-quantized) inputs, element-wise within
  |C_gpu - C_ref| <= 2^-7 |C_ref| + 1e-5 S_abs   (BF16 output)
  |C_gpu - C_ref| <= 1e-5 S_abs                  (FP32 output),
S_abs = sum_k |a_ik b_kj| of the dequantized operands.  Every output element
is compared: small and ragged shapes, and the layer's Fprop / Dgrad / Wgrad
at full size (4096 x 18432, 4096 x 7168 and 7168 x 18432 outputs, against the
multithreaded oracle's whole output)."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
import full_ref
from gpu_helpers import (DEV, MODES, assert_gemm_close, gemm_operands as _operands, gpu_gemm,
                         oracle_input, to_dev_f32, to_dev_u8)

pytestmark = pytest.mark.gpu

@pytest.mark.parametrize("M,N,K,mode,out", [
    (128, 256, 128, "KN", torch.bfloat16),      # one tile, one slab
    (128, 128, 128, "KN", torch.float32),       # half-width N tile
    (1, 256, 256, "KN", torch.bfloat16),        # single row
    (300, 384, 1024, "KN", torch.bfloat16),     # ragged M, N % 256 == 128
    (256, 512, 640, "NK", torch.bfloat16),
    (384, 272, 512, "PERCOL", torch.float32),   # ragged N in per-column mode
    (200, 96, 384, "PERCOL", torch.bfloat16),
    (640, 1024, 896, "NK", torch.float32),
])
def test_gemm_matches_oracle(M, N, K, mode, out):
    Aq, sa, Bq, sb = _operands(M, N, K, mode, seed=M + N + K)
    c = gpu_gemm(Aq, sa, Bq, sb, MODES[mode], out_dtype=out)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, MODES[mode])
    assert_gemm_close(c, c_ref, s_abs, out == torch.bfloat16, f"{M}x{N}x{K} {mode}")


def test_gemm_tiny_fprop():
    a, w = wl.tiny_fprop()
    Aq, sa = oracle.quant_act_1x128(a)
    Wq, WqT, sw = oracle.quant_w_128x128(w)
    c = gpu_gemm(Aq, sa, WqT, sw, oracle.SB_BLOCK_KN, torch.bfloat16)
    c_ref, s_abs = oracle.gemm(Aq, sa, WqT, sw, oracle.SB_BLOCK_KN)
    assert_gemm_close(c, c_ref, s_abs, True, "tiny Fprop")


def test_gemm_many_tiles_per_cta():
    """More output tiles than SMs: every CTA walks several tiles."""
    M, N, K = 2560, 4096, 256
    Aq, sa, Bq, sb = _operands(M, N, K, "KN", seed=5)
    c = gpu_gemm(Aq, sa, Bq, sb, oracle.SB_BLOCK_KN, torch.bfloat16)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, oracle.SB_BLOCK_KN)
    assert_gemm_close(c, c_ref, s_abs, True, "many tiles")


def test_gemm_zero_k_writes_zeros():
    C = torch.full((64, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    A = torch.zeros((64, 0), dtype=torch.uint8, device=DEV)
    B = torch.zeros((128, 0), dtype=torch.uint8, device=DEV)
    sa = torch.zeros((0, 64), dtype=torch.float32, device=DEV)
    sb = torch.zeros((0, 1), dtype=torch.float32, device=DEV)
    st = fb.lib().fp8bs_gemm(64, 128, 0, A.data_ptr(), 16, sa.data_ptr(), 64, B.data_ptr(), 16,
                             sb.data_ptr(), fb.FP8BS_SB_BLOCK_KN, 1, C.data_ptr(), fb.FP8BS_BF16,
                             128, torch.cuda.current_stream().cuda_stream)
    assert st == fb.FP8BS_OK
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    assert torch.all(C == 0)


def _tile_samples(M, N, seed, extra, bm=128, bn=256):
    """One random element in every 128 x 256 output tile, plus `extra` random
    elements and the four corners."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for m0 in range(0, M, bm):
        for n0 in range(0, N, bn):
            rows.append(rng.integers(m0, min(M, m0 + bm)))
            cols.append(rng.integers(n0, min(N, n0 + bn)))
    rows = np.concatenate([rows, rng.integers(0, M, extra), [0, 0, M - 1, M - 1]])
    cols = np.concatenate([cols, rng.integers(0, N, extra), [0, N - 1, 0, N - 1]])
    return rows.astype(np.int64), cols.astype(np.int64)


@pytest.mark.parametrize("which", ["fprop", "dgrad", "wgrad"])
def test_layer_gemm_full(which):
    """The layer's GEMM through fp8bs_gemm (no K split), every output element
    against the oracle."""
    A, sa, B, sb, mode, bf16_out = full_ref.layer_gemm_args(which)
    c = gpu_gemm(A, sa, B, sb, mode, torch.bfloat16 if bf16_out else torch.float32)
    c_ref, s_abs = full_ref.layer_reference(which)
    assert_gemm_close(c, c_ref, s_abs, bf16_out, f"layer {which} {c.shape}")
