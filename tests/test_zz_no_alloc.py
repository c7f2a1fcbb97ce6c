"""fp8bs_gemm_static_ws, the GEMM entry point for callers that cannot
allocate device memory (they cannot call cudaMalloc where they run, or have
no workspace to lend): its split-K partials live in the library's own device
array instead of a caller workspace.

Called through the C ABI twice in a row, it must give exactly what
fp8bs_gemm_ws gives with a caller workspace (the two choose the same split,
so the outputs are bit-identical), and both must meet the GEMM tolerance of
the other tests against the CPU oracle.  Between the two calls an unrelated
split shape runs through the same array, so the second call can only match
if it rewrites every partial it reads.  This file is collected last so that
a run stopping at its first failure has already run every other test; it also
passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
from gpu_helpers import (DEV, MODES, assert_gemm_close, gemm_operands, gpu_gemm_ws, to_dev_f32,
                         to_dev_u8)

pytestmark = pytest.mark.gpu

STATIC_BYTES = 20 << 20


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


@pytest.mark.parametrize("M,N,K,mode,out,other", [
    # 8 tiles, each split in 8 K-ranges; in between, 2 tiles x 32 ranges
    (512, 1024, 2048, "NK", torch.float32, (256, 512, 4096, "KN", torch.bfloat16)),
    # 2 tiles, 32 K-ranges each; in between, a ragged per-column shape
    (256, 512, 4096, "KN", torch.bfloat16, (300, 272, 2048, "PERCOL", torch.float32)),
])
def test_static_workspace_gemm_matches_workspace_gemm(M, N, K, mode, out, other):
    need = fb.fp8bs_gemm_workspace_size(M, N, K)
    assert 0 < need <= STATIC_BYTES          # the shape splits and fits the static array
    Aq, sa, Bq, sb = gemm_operands(M, N, K, mode, seed=M + N + 3 * K)
    c_ws = gpu_gemm_ws(Aq, sa, Bq, sb, MODES[mode], out_dtype=out)
    c_ref, s_abs = oracle.gemm(Aq, sa, Bq, sb, MODES[mode])
    bf16 = out == torch.bfloat16
    assert_gemm_close(c_ws, c_ref, s_abs, bf16, "caller workspace")

    oM, oN, oK, omode, oout = other
    assert fb.fp8bs_gemm_workspace_size(oM, oN, oK) > 0
    oAq, osa, oBq, osb = gemm_operands(oM, oN, oK, omode, seed=oM + oN + oK)
    for call in range(2):
        c = _static_ws_call(Aq, sa, Bq, sb, mode, out)
        assert np.array_equal(c, c_ws), f"call {call}: differs from fp8bs_gemm_ws"
        assert_gemm_close(c, c_ref, s_abs, bf16, f"static workspace, call {call}")
        if call == 0:   # leave unrelated partials in the array before the second call
            c_other = _static_ws_call(oAq, osa, oBq, osb, omode, oout)
            o_ref, o_abs = oracle.gemm(oAq, osa, oBq, osb, MODES[omode])
            assert_gemm_close(c_other, o_ref, o_abs, oout == torch.bfloat16, "interleaved shape")
