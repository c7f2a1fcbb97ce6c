"""fp8bs_gemm_ws: the dense GEMM whose last, partial wave of tiles is split
along K over the idle CTA pairs, with the FP32 partials in a caller-provided
workspace summed by a second kernel.  Parity with the CPU oracle under the
same element-wise tolerance as fp8bs_gemm, on shapes that split (few tiles,
long K), on smaller workspaces (fewer K-ranges, then none), and at the layer
sizes on every output element; the split result is deterministic."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
from gpu_helpers import (DEV, MODES, assert_gemm_close, gemm_operands, gpu_gemm, gpu_gemm_ws,
                         to_dev_f32, to_dev_u8)
import full_ref

pytestmark = pytest.mark.gpu

PAIR_TILE = 256 * 256 * 4   # bytes of one FP32 partial tile


@pytest.mark.parametrize("M,N,K,mode,out", [
    (256, 512, 4096, "KN", torch.bfloat16),     # 2 tiles, 32 slabs: every pair gets a K-range
    (300, 272, 2048, "PERCOL", torch.float32),  # ragged M and N
    (512, 1024, 1024, "NK", torch.float32),     # 8 tiles
    (128, 256, 128, "KN", torch.bfloat16),      # one slab: a split would leave one range
])
def test_gemm_ws_matches_oracle(M, N, K, mode, out):
    Aq, sa, Bq, sb = gemm_operands(M, N, K, mode, seed=M + 2 * N + K)
    need = fb.fp8bs_gemm_workspace_size(M, N, K)
    if K // 128 >= 2:
        assert need > 0 and need % PAIR_TILE == 0
    else:
        assert need == 0
    c = gpu_gemm_ws(Aq, sa, Bq, sb, MODES[mode], out_dtype=out)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, MODES[mode])
    assert_gemm_close(c, c_ref, s_abs, out == torch.bfloat16, f"ws {M}x{N}x{K} {mode}")


@pytest.mark.parametrize("fraction", [0.5, 0.01, 0.0])
def test_gemm_ws_smaller_workspace(fraction):
    """Less workspace: fewer K-ranges (or none); the result stays in tolerance."""
    M, N, K = 256, 512, 4096
    Aq, sa, Bq, sb = gemm_operands(M, N, K, "KN", seed=77)
    need = fb.fp8bs_gemm_workspace_size(M, N, K)
    c = gpu_gemm_ws(Aq, sa, Bq, sb, oracle.SB_BLOCK_KN, ws_bytes=int(need * fraction))
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, oracle.SB_BLOCK_KN)
    assert_gemm_close(c, c_ref, s_abs, True, f"ws fraction {fraction}")


def test_gemm_ws_deterministic_and_close_to_unsplit():
    M, N, K = 512, 1024, 2048
    Aq, sa, Bq, sb = gemm_operands(M, N, K, "NK", seed=3)
    c1 = gpu_gemm_ws(Aq, sa, Bq, sb, oracle.SB_BLOCK_NK, torch.float32)
    c2 = gpu_gemm_ws(Aq, sa, Bq, sb, oracle.SB_BLOCK_NK, torch.float32)
    assert np.array_equal(c1, c2)
    c0 = gpu_gemm(Aq, sa, Bq, sb, oracle.SB_BLOCK_NK, torch.float32)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, oracle.SB_BLOCK_NK)
    assert_gemm_close(c0, c_ref, s_abs, False, "unsplit")
    assert_gemm_close(c1, c_ref, s_abs, False, "split")


def test_gemm_ws_misaligned_workspace_rejected():
    A = torch.zeros((128, 128), dtype=torch.uint8, device=DEV)
    sa = torch.ones((1, 128), dtype=torch.float32, device=DEV)
    B = torch.zeros((256, 128), dtype=torch.uint8, device=DEV)
    sb = torch.ones((1, 2), dtype=torch.float32, device=DEV)
    C = torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    st = fb.lib().fp8bs_gemm_ws(128, 256, 128, A.data_ptr(), 128, sa.data_ptr(), 128,
                                B.data_ptr(), 128, sb.data_ptr(), fb.FP8BS_SB_BLOCK_KN, 2,
                                C.data_ptr(), fb.FP8BS_BF16, 256, ws.data_ptr() + 16, 1 << 19,
                                torch.cuda.current_stream().cuda_stream)
    assert st == fb.FP8BS_ERR_MISALIGNED


@pytest.mark.parametrize("which", ["fprop", "dgrad", "wgrad"])
def test_layer_gemm_ws_full(which):
    """The layer's GEMM through fp8bs_gemm_ws (the bench's call: the last,
    partial wave split along K where the tile count leaves one -- Dgrad and
    Wgrad on a 148-SM B300, not Fprop), every output element against the
    oracle."""
    A, sa, B, sb, mode, bf16_out = full_ref.layer_gemm_args(which)
    c = gpu_gemm_ws(A, sa, B, sb, mode, torch.bfloat16 if bf16_out else torch.float32)
    c_ref, s_abs = full_ref.layer_reference(which)
    assert_gemm_close(c, c_ref, s_abs, bf16_out, f"layer {which} ws {c.shape}")
