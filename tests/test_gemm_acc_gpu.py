"""fp8bs_gemm_accumulate: C (FP32) += block-scaled A * B^T.  C_new - C_old
must match the CPU oracle's product within the FP32 GEMM tolerance, plus the
rounding of the one FP32 add:  |C_new - (C_old + C_ref)| <= 1e-5 S_abs +
2^-24 |C_new|.  Whole tiles (TMA reduce-add) and split tail tiles (partial-sum
kernel) are both covered; K == 0 leaves C unchanged."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import full_ref
from gpu_helpers import DEV, MODES, gemm_operands, to_dev_f32, to_dev_u8

pytestmark = pytest.mark.gpu


def _acc(Aq, sa, Bq, sb, mode, c0, ws_bytes):
    C = torch.from_numpy(c0).to(DEV)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV) if ws_bytes > 0 else None
    fb.fp8bs_gemm_accumulate(to_dev_u8(Aq), to_dev_f32(sa), to_dev_u8(Bq), to_dev_f32(sb),
                             MODES[mode], C, ws)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return C.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("M,N,K,mode", [
    (384, 272, 1024, "PERCOL"),    # the Wgrad form, ragged N
    (512, 1024, 2048, "NK"),
    (300, 512, 640, "KN"),
])
def test_gemm_accumulate_matches_oracle(M, N, K, mode, split):
    Aq, sa, Bq, sb = gemm_operands(M, N, K, mode, seed=M + 11 * N + K)
    rng = np.random.default_rng(M + N)
    c0 = rng.standard_normal((M, N)).astype(np.float32)
    ws_bytes = fb.fp8bs_gemm_workspace_size(M, N, K) if split else 0
    if split:
        assert ws_bytes > 0
    c1 = _acc(Aq, sa, Bq, sb, mode, c0, ws_bytes)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, MODES[mode])
    err = np.abs(c1 - (c0.astype(np.float64) + c_ref))
    bound = 1e-5 * s_abs + 2.0 ** -24 * np.abs(c1)
    assert np.all(err <= bound), f"max err/bound {np.max(err / np.maximum(bound, 1e-300))}"


def test_gemm_accumulate_twice_adds_twice():
    M, N, K = 256, 512, 1024
    Aq, sa, Bq, sb = gemm_operands(M, N, K, "PERCOL", seed=9)
    C = torch.zeros((M, N), dtype=torch.float32, device=DEV)
    A, SA, B, SB = to_dev_u8(Aq), to_dev_f32(sa), to_dev_u8(Bq), to_dev_f32(sb)
    for _ in range(2):
        fb.fp8bs_gemm_accumulate(A, SA, B, SB, fb.FP8BS_SB_PERCOL, C)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, oracle.SB_PERCOL)
    c = C.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(c - 2 * c_ref) <= 2e-5 * s_abs + 2.0 ** -23 * np.abs(c))


def test_gemm_accumulate_zero_k_leaves_c():
    C = torch.full((64, 128), 3.5, dtype=torch.float32, device=DEV)
    A = torch.zeros((64, 16), dtype=torch.uint8, device=DEV)
    B = torch.zeros((128, 16), dtype=torch.uint8, device=DEV)
    sa = torch.zeros((1, 64), dtype=torch.float32, device=DEV)
    sb = torch.zeros((1, 1), dtype=torch.float32, device=DEV)
    st = fb.lib().fp8bs_gemm_accumulate(64, 128, 0, A.data_ptr(), 16, sa.data_ptr(), 64,
                                        B.data_ptr(), 16, sb.data_ptr(), fb.FP8BS_SB_BLOCK_KN, 1,
                                        C.data_ptr(), 128, None, 0,
                                        torch.cuda.current_stream().cuda_stream)
    assert st == fb.FP8BS_OK
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    assert torch.all(C == 3.5)


def test_layer_wgrad_accumulate_full():
    """The layer's Wgrad (7168 x 18432, K = 4096 tokens) added into an FP32
    gradient buffer that already holds values, with the K split of the last
    wave: every element of C_new - C_old against the oracle."""
    A, sa, B, sb, mode, _ = full_ref.layer_gemm_args("wgrad")
    M, N = A.shape[0], B.shape[0]
    c0 = np.random.default_rng(17).standard_normal((M, N)).astype(np.float32) * np.float32(1e-2)
    c1 = _acc(A, sa, B, sb, "PERCOL", c0, fb.fp8bs_gemm_workspace_size(M, N, A.shape[1]))
    c_ref, s_abs = full_ref.layer_reference("wgrad")
    err = np.abs(c1 - (c0.astype(np.float64) + c_ref))
    bound = 1e-5 * s_abs + 2.0 ** -24 * np.abs(c1)
    assert np.all(err <= bound), f"max err/bound {np.max(err / np.maximum(bound, 1e-300))}"
