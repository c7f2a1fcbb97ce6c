"""Grouped (MoE expert) GEMM parity against the oracle applied expert by
expert, plus device-side offset validation."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
import full_ref
from gpu_helpers import DEV, assert_gemm_close, oracle_input, to_dev_f32, to_dev_u8

pytestmark = pytest.mark.gpu


def _run_grouped(offsets, Aq, sa, Bq, sb, mode, out=torch.bfloat16, sentinel=3.0):
    M_cap = Aq.shape[0]
    N = Bq.shape[1]
    C = torch.full((M_cap, N), sentinel, dtype=out, device=DEV)
    off = torch.tensor(np.asarray(offsets, np.int32), device=DEV)
    fb.fp8bs_grouped_gemm(off, to_dev_u8(Aq), to_dev_f32(sa), to_dev_u8(Bq), to_dev_f32(sb),
                          mode, C)
    st = fb.fp8bs_sync_status()
    return st, C.float().cpu().numpy().astype(np.float64)


def _experts(E, N, K, seed):
    Bq, sbs = [], []
    for e in range(E):
        w = wl.random_matrix((K, N), seed=seed + e, dtype=torch.bfloat16, std=0.02)
        _, WqT, sw = oracle.quant_w_128x128(oracle_input(w))
        Bq.append(WqT)
        sbs.append(sw)
    return np.stack(Bq), np.stack(sbs)          # [E x N x K], [E x K/128 x N/128]


def test_grouped_small_with_empty_experts():
    E, N, K = 4, 384, 512
    offsets = [0, 128, 128, 384, 512]            # expert 1 empty
    M_cap = 640                                  # rows 512.. belong to nobody
    a = wl.random_matrix((M_cap, K), seed=41, dtype=torch.bfloat16)
    Aq, sa = oracle.quant_act_1x128(oracle_input(a))
    Bq, sb = _experts(E, N, K, seed=42)
    st, c = _run_grouped(offsets, Aq, sa, Bq, sb, fb.FP8BS_SB_BLOCK_KN)
    assert st == fb.FP8BS_OK
    c_ref, s_abs = oracle.grouped_gemm(offsets, Aq, sa, Bq, sb, oracle.SB_BLOCK_KN)
    assert_gemm_close(c[:512], c_ref[:512], s_abs[:512], True, "grouped small")
    assert np.all(c[512:] == 3.0), "rows past offsets[E] must be untouched"


def test_grouped_nk_scales_fp32_out():
    E, N, K = 3, 256, 384
    offsets = [0, 256, 384, 384]                 # last expert empty
    a = wl.random_matrix((384, K), seed=43, dtype=torch.bfloat16)
    Aq, sa = oracle.quant_act_1x128(oracle_input(a))
    Bq, sb = _experts(E, N, K, seed=44)
    sb_nk = np.ascontiguousarray(np.transpose(sb, (0, 2, 1)))
    st, c = _run_grouped(offsets, Aq, sa, Bq, sb_nk, fb.FP8BS_SB_BLOCK_NK, out=torch.float32)
    assert st == fb.FP8BS_OK
    c_ref, s_abs = oracle.grouped_gemm(offsets, Aq, sa, Bq, sb_nk, oracle.SB_BLOCK_NK)
    assert_gemm_close(c, c_ref, s_abs, False, "grouped NK fp32")


def test_grouped_odd_blocks_and_many_experts():
    """Experts with odd numbers of 128-row blocks (the second half of their
    last 256-row pair tile lies past the expert and must stay untouched), and
    more experts than the pair kernel stages (300: the single-CTA kernel)."""
    N, K = 256, 256
    for E, sizes in ((5, [384, 128, 0, 640, 256]), (300, [128 if e % 97 == 0 else 0
                                                            for e in range(300)])):
        offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
        M_cap = int(offsets[-1]) + 256
        a = wl.random_matrix((M_cap, K), seed=E + 50, dtype=torch.bfloat16)
        Aq, sa = oracle.quant_act_1x128(oracle_input(a))
        Bq, sb = _experts(E, N, K, seed=E + 51)
        st, c = _run_grouped(offsets, Aq, sa, Bq, sb, fb.FP8BS_SB_BLOCK_KN)
        assert st == fb.FP8BS_OK
        n = int(offsets[-1])
        c_ref, s_abs = oracle.grouped_gemm(offsets, Aq, sa, Bq, sb, oracle.SB_BLOCK_KN)
        assert_gemm_close(c[:n], c_ref[:n], s_abs[:n], True, f"grouped E={E}")
        assert np.all(c[n:] == 3.0), "rows past offsets[E] must be untouched"


@pytest.mark.parametrize("offsets", [[0, 100, 256], [0, 256, 128], [128, 256, 384],
                                     [0, 128, 1024]])
def test_grouped_bad_offsets_reported_and_nothing_written(offsets):
    E, N, K = 2, 256, 128
    Aq = np.zeros((512, K), np.uint8)
    sa = np.ones((1, 512), np.float32)
    Bq = np.zeros((E, N, K), np.uint8)
    sb = np.ones((E, 1, 2), np.float32)
    st, c = _run_grouped(offsets, Aq, sa, Bq, sb, fb.FP8BS_SB_BLOCK_KN)
    assert st == fb.FP8BS_ERR_DEVICE_BAD_OFFSETS
    assert np.all(c == 3.0)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK      # the status was cleared


def test_grouped_moe_up_projection_full():
    """32 experts, 16384 routed rows with Zipf(1.1) counts padded to 128,
    K = 7168, N = 4096 per expert: every output element against the oracle
    (padding rows must come out as exactly 0)."""
    counts, offsets, Aq, sa, Bq, sb = full_ref.moe_operands()
    st, c = _run_grouped(offsets, Aq, sa, Bq, sb, fb.FP8BS_SB_BLOCK_KN)
    assert st == fb.FP8BS_OK
    c_ref, s_abs = full_ref.moe_reference()
    assert_gemm_close(c, c_ref, s_abs, True, "grouped MoE")
    pad = np.concatenate([np.arange(int(offsets[e]) + int(counts[e]), int(offsets[e + 1]))
                          for e in range(len(counts))])
    assert pad.size > 0 and np.all(c[pad] == 0)
