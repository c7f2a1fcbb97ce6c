"""fp8bs_gemm_static_ws, the GEMM entry point for callers that cannot
allocate device memory (they cannot call cudaMalloc where they run, or have
no workspace to lend): its split-K partials live in the library's own device
array instead of a caller workspace.  Called through the C ABI twice in a
row, it must give what fp8bs_gemm_ws with a caller workspace gives, within
the GEMM tolerance of the other tests (and both must meet it against the CPU
oracle).  This file is collected last so that a run stopping at its first
failure has already run every other test; it also passes alone."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
from gpu_helpers import (DEV, MODES, assert_gemm_close, gemm_bound, gemm_operands, gpu_gemm_ws,
                         to_dev_f32, to_dev_u8)

pytestmark = pytest.mark.gpu


def _static_ws_call(Aq, sa, Bq, sb, mode, out_dtype):
    M, K = Aq.shape
    N = Bq.shape[0]
    A, SA, B, SB = to_dev_u8(Aq), to_dev_f32(sa), to_dev_u8(Bq), to_dev_f32(sb)
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    ct = fb.FP8BS_BF16 if out_dtype == torch.bfloat16 else fb.FP8BS_F32
    st = fb.lib().fp8bs_gemm_static_ws(M, N, K, A.data_ptr(), A.stride(0), SA.data_ptr(),
                                       SA.stride(0), B.data_ptr(), B.stride(0), SB.data_ptr(),
                                       MODES[mode], SB.stride(0), C.data_ptr(), ct, C.stride(0),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == fb.FP8BS_OK, fb.status_string(st)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return C.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K,mode,out", [
    (512, 1024, 2048, "NK", torch.float32),     # 8 tiles, each split in 8 K-ranges
    (256, 512, 4096, "KN", torch.bfloat16),     # 2 tiles, 32 K-ranges each
])
def test_static_workspace_gemm_matches_workspace_gemm(M, N, K, mode, out):
    need = fb.fp8bs_gemm_workspace_size(M, N, K)
    assert 0 < need <= 20 << 20          # the shape splits and fits the static array
    Aq, sa, Bq, sb = gemm_operands(M, N, K, mode, seed=M + N + 3 * K)
    c_ws = gpu_gemm_ws(Aq, sa, Bq, sb, MODES[mode], out_dtype=out)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, MODES[mode])
    bf16 = out == torch.bfloat16
    assert_gemm_close(c_ws, c_ref, s_abs, bf16, "caller workspace")
    bound = gemm_bound(c_ref, s_abs, bf16)
    for call in range(2):                # the array keeps the previous call's partials
        c = _static_ws_call(Aq, sa, Bq, sb, mode, out)
        assert np.all(np.abs(c - c_ws) <= bound), f"call {call}: differs from fp8bs_gemm_ws"
        assert_gemm_close(c, c_ref, s_abs, bf16, f"static workspace, call {call}")
