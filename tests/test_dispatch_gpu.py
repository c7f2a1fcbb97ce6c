"""Quantize-then-dispatch (fp8bs_quant_dispatch) against the CPU oracle's
dispatch (tokens grouped by expert in token order, each expert padded to a
multiple of 128 rows with quantized zero rows, routed rows quantized 1x128).
Codes, scales, offsets, counts and both row maps must match exactly; the
dispatched operands then feed the grouped GEMM."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
from gpu_helpers import DEV, assert_gemm_close, oracle_input, to_dev_f32, to_dev_u8

pytestmark = pytest.mark.gpu


def _oracle_dispatch(x, expert, E):
    q, s, offsets, counts, token_row, row_token, _ = oracle.dispatch(oracle_input(x), expert, E)
    return q, s, offsets, counts, token_row, row_token


def _gpu_dispatch(x, expert, E):
    T, K = x.shape
    M_cap = (T + 127 * E + 127) // 128 * 128
    xd = x.to(DEV)
    ed = torch.from_numpy(expert.astype(np.int32)).to(DEV)
    q = torch.full((M_cap, K), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((K // 128, M_cap), -3.0, dtype=torch.float32, device=DEV)
    offsets = torch.full((E + 1,), -9, dtype=torch.int32, device=DEV)
    counts = torch.full((E,), -9, dtype=torch.int32, device=DEV)
    token_row = torch.full((T,), -9, dtype=torch.int32, device=DEV)
    row_token = torch.full((M_cap,), -9, dtype=torch.int32, device=DEV)
    fb.fp8bs_quant_dispatch(xd, ed, E, q, s, offsets, counts, token_row, row_token)
    st = fb.fp8bs_sync_status()
    return (st, q.cpu().numpy(), s.cpu().numpy(), offsets.cpu().numpy(), counts.cpu().numpy(),
            token_row.cpu().numpy(), row_token.cpu().numpy())


def _check(x, expert, E):
    st, q, s, off, cnt, t2r, r2t = _gpu_dispatch(x, expert, E)
    assert st == fb.FP8BS_OK
    qr, sr, offr, cntr, rows, r2tr = _oracle_dispatch(x, expert, E)
    assert np.array_equal(off, offr) and np.array_equal(cnt, cntr)
    assert np.array_equal(t2r, rows)
    n = int(offr[E])
    assert np.array_equal(r2t[:n], r2tr)
    scratch = -(-x.shape[0] // 1024) * E   # row_token entries that serve as scratch
    assert np.all(r2t[max(n, scratch):] == -9), "row_token past the rows and the scratch"
    assert np.all(q[n:] == 0xAB) and np.all(s[:, n:] == -3.0), "rows past the last expert"
    if n:
        assert np.array_equal(q[:n], qr), "codes"
        assert np.array_equal(s[:, :n], sr), "scales"
    return off


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,K,E", [(300, 256, 4), (1000, 512, 7), (4096, 128, 256), (1, 128, 3)])
def test_dispatch_matches_oracle(T, K, E, dtype):
    rng = np.random.default_rng(T + K + E)
    expert = rng.integers(0, E, T)
    if E == 7:
        expert[expert == 3] = 5          # an empty expert in the middle
    x = wl.random_matrix((T, K), seed=T * 3 + K, dtype=dtype)
    _check(x, expert, E)


def test_dispatch_all_to_one_expert():
    x = wl.random_matrix((777, 256), seed=1, dtype=torch.bfloat16)
    _check(x, np.full(777, 2), 5)


def test_dispatch_moe_workload():
    """The MoE up-projection workload: 16384 tokens x 7168, 32 experts with
    Zipf(1.1) routing."""
    expert = wl.zipf_expert_ids()
    x = wl.random_matrix((expert.size, wl.HIDDEN), seed=7, dtype=torch.bfloat16)
    off = _check(x, expert, wl.EXPERTS)
    assert np.array_equal(off, wl.padded_offsets(np.bincount(expert, minlength=wl.EXPERTS)))


def test_dispatch_bad_expert_id_reported_and_dropped():
    x = wl.random_matrix((256, 128), seed=2, dtype=torch.bfloat16)
    expert = np.random.default_rng(3).integers(0, 4, 256)
    expert[5] = 4                         # outside [0, 4)
    st, q, s, off, cnt, t2r, r2t = _gpu_dispatch(x, expert, 4)
    assert st == fb.FP8BS_ERR_DEVICE_BAD_ROUTING
    assert t2r[5] == -1
    assert cnt.sum() == 255
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK   # the error word was cleared
    qr, sr, offr, cntr, rows, r2tr = _oracle_dispatch(x, expert, 4)   # the token is dropped there too
    n = int(offr[-1])
    assert np.array_equal(off, offr) and np.array_equal(cnt, cntr) and np.array_equal(t2r, rows)
    assert np.array_equal(r2t[:n], r2tr)
    assert np.array_equal(q[:n], qr) and np.array_equal(s[:, :n], sr)


def test_dispatch_then_grouped_gemm():
    """dispatch -> grouped GEMM: each token's output row equals the dense
    block-scaled product of its quantized row with its expert's weight."""
    T, K, N, E = 300, 256, 256, 4
    expert = np.random.default_rng(4).integers(0, E, T)
    x = wl.random_matrix((T, K), seed=5, dtype=torch.bfloat16)
    M_cap = (T + 127 * E + 127) // 128 * 128
    q = torch.zeros((M_cap, K), dtype=torch.uint8, device=DEV)
    s = torch.zeros((K // 128, M_cap), dtype=torch.float32, device=DEV)
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(E, dtype=torch.int32, device=DEV)
    t2r = torch.zeros(T, dtype=torch.int32, device=DEV)
    r2t = torch.zeros(M_cap, dtype=torch.int32, device=DEV)
    fb.fp8bs_quant_dispatch(x.to(DEV), torch.from_numpy(expert.astype(np.int32)).to(DEV), E, q, s,
                            off, cnt, t2r, r2t)
    Wq, Ws = [], []
    for e in range(E):
        w = wl.random_matrix((K, N), seed=20 + e, dtype=torch.bfloat16, std=0.02)
        _, wqT, sw = oracle.quant_w_128x128(oracle_input(w))
        Wq.append(wqT)
        Ws.append(sw)
    B = to_dev_u8(np.stack(Wq))
    SB = to_dev_f32(np.stack(Ws))
    C = torch.full((M_cap, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    fb.fp8bs_grouped_gemm(off, q, s, B, SB, fb.FP8BS_SB_BLOCK_KN, C)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    rows = t2r.cpu().numpy()
    c = C.float().cpu().numpy().astype(np.float64)[rows]
    xq, xs = oracle.quant_act_1x128(oracle_input(x))
    for e in range(E):
        tok = np.nonzero(expert == e)[0]
        if tok.size == 0:
            continue
        c_ref, s_abs = oracle.gemm(xq[tok], np.ascontiguousarray(xs[:, tok]), Wq[e], Ws[e],
                                   oracle.SB_BLOCK_KN)
        assert_gemm_close(c[tok], c_ref, s_abs, True, f"expert {e}")
