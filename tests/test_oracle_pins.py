"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: the OCP E4M3 format
anchors (tests/golden/e4m3_anchors.txt), PyTorch's own float8_e4m3fn conversion
(an independent library implementation), brute-force nearest-value search,
closed-form GEMM cases and invariants the method fixes (amax maps to +-448, an
all-zero tile gets scale 1).  A plausible mistake in the oracle -- a wrong
rounding direction, a dropped saturation, a transposed scale index, a wrong
tile boundary, a missing scale factor -- fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, random_matrix, tiny_fprop

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ E4M3 codec

def _anchors():
    out = []
    with open(os.path.join(GOLDEN, "e4m3_anchors.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            out.append((int(code, 16), float(val)))
    return out


def test_decode_matches_ocp_anchors():
    for code, val in _anchors():
        got = oracle.e4m3_decode(code)
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val, (hex(code), got, val)


def test_decode_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # Sign of zero survives decoding.
    assert math.copysign(1.0, got[0x80]) == -1.0


def _torch_encode(v: np.ndarray) -> np.ndarray:
    """PyTorch's RNE cast (no saturation: |v| >= 464 becomes NaN there)."""
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _encoder_probe_values(n_random: int = 400_000, seed: int = 11) -> np.ndarray:
    rng = np.random.default_rng(seed)
    # 1. every bf16 value with |v| < 464 (covers all binades down to fp32 subnormals)
    bits = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    allbf = bits.view(np.float32)
    allbf = allbf[np.isfinite(allbf) & (np.abs(allbf) < 464)]
    # 2. midpoints between neighbouring E4M3 values, and one fp32 ulp either side
    dec = oracle.e4m3_decode_table()
    pos = np.unique(dec[np.isfinite(dec) & (dec >= 0)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)   # exact in fp32
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9))])
    # 3. random fp32 bit patterns restricted to |v| < 464
    rb = rng.integers(0, 1 << 32, size=n_random * 3, dtype=np.uint64).astype(np.uint32)
    rv = rb.view(np.float32)
    rv = rv[np.isfinite(rv) & (np.abs(rv) < 464)][:n_random]
    v = np.concatenate([allbf, near, -near, rv]).astype(np.float32)
    return v


def test_encoder_matches_torch_cast_in_range():
    v = _encoder_probe_values()
    ref = _torch_encode(v)
    got = oracle.e4m3_encode_array(v)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(v[i]), int(ref[i]), int(got[i])) for i in bad[:10]]


def _brute_force_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search over the 254 finite codes;
    ties go to the code with an even mantissa; magnitudes >= 448 clamp."""
    dec = oracle.e4m3_decode_table()
    codes = np.array([c for c in range(256) if not math.isnan(dec[c])], np.int64)
    vals = dec[codes]
    out = np.empty(v.size, np.uint8)
    vd = v.astype(np.float64)
    for i, x in enumerate(vd):
        if abs(x) >= 448:
            out[i] = 0x7E | (0x80 if x < 0 else 0)
            continue
        d = np.abs(vals - x)          # exact: neighbours are within a factor 2
        best = d.min()
        cand = codes[d == best]
        # both signed zeros tie at x = 0: keep the sign of x
        if best == 0 and x == 0:
            out[i] = 0x80 if math.copysign(1.0, x) < 0 else 0x00
            continue
        cand = [c for c in cand if (c & 0x80) == (0x80 if x < 0 else 0)] or list(cand)
        even = [c for c in cand if (c & 1) == 0]
        out[i] = (even or cand)[0]
    return out


def test_encoder_matches_brute_force():
    rng = np.random.default_rng(5)
    v = _encoder_probe_values(n_random=3000, seed=6)
    v = v[rng.choice(v.size, size=8000, replace=False)]
    extra = np.array([0.0, -0.0, 448, -448, 449, 463.99, 464, 1e30, -1e30, 2**-10,
                      -(2**-10), 3 * 2**-10, 2**-12, 240, 232, 248, 0.01], np.float32)
    v = np.concatenate([v, extra])
    assert np.array_equal(oracle.e4m3_encode_array(v), _brute_force_encode(v))


def test_encoder_saturates_finite_overflow():
    v = np.array([448, 448.5, 463.9, 464, 480, 1e4, 3.4e38, np.inf], np.float32)
    assert list(oracle.e4m3_encode_array(v)) == [0x7E] * v.size
    assert list(oracle.e4m3_encode_array(-v)) == [0xFE] * v.size


# ------------------------------------------------------------------ quantizers

def _independent_tile_quant(x: np.ndarray):
    """Quantize one tile with numpy binary32 arithmetic and torch's cast
    (clamped to +-448 first, which is the saturation)."""
    x = x.astype(np.float32)
    amax = np.float32(np.max(np.abs(x)))
    with np.errstate(divide="ignore", over="ignore"):
        r = np.float32(448) / amax
    if not np.isfinite(r):
        s, r = np.float32(1), np.float32(1)
    else:
        s = amax / np.float32(448)
    y = (x * r).astype(np.float32)
    y = np.clip(y, -448, 448).astype(np.float32)
    return _torch_encode(y), s


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quant_1x128_matches_independent_tile_quant(dtype):
    x = random_matrix((5, 384), seed=21, dtype=dtype)
    xn = x.float().numpy()
    inp = bf16_bits(x) if dtype == torch.bfloat16 else xn
    q, s = oracle.quant_act_1x128(inp)
    assert s.shape == (3, 5)
    for m in range(5):
        for kb in range(3):
            qr, sr = _independent_tile_quant(xn[m, kb * 128:(kb + 1) * 128])
            assert np.array_equal(q[m, kb * 128:(kb + 1) * 128], qr)
            assert s[kb, m] == sr


def test_quant_128x128_matches_independent_block_quant():
    w = random_matrix((256, 384), seed=22, dtype=torch.bfloat16, std=0.02)
    wn = w.float().numpy()
    q, qT, s = oracle.quant_w_128x128(bf16_bits(w))
    assert s.shape == (2, 3)
    for rb in range(2):
        for cb in range(3):
            blk = wn[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
            qr, sr = _independent_tile_quant(blk.ravel())
            assert np.array_equal(q[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128].ravel(), qr)
            assert s[rb, cb] == sr
    assert np.array_equal(qT, q.T)


def test_amax_maps_to_448_and_sign_symmetry():
    x = random_matrix((64, 1024), seed=23, dtype=torch.bfloat16)
    xn = x.float().numpy()
    q, s = oracle.quant_act_1x128(bf16_bits(x))
    for m in range(64):
        for kb in range(8):
            tile = xn[m, kb * 128:(kb + 1) * 128]
            i = int(np.argmax(np.abs(tile)))
            assert q[m, kb * 128 + i] == (0xFE if tile[i] < 0 else 0x7E)
    qn, sn = oracle.quant_act_1x128(bf16_bits(-x))
    assert np.array_equal(sn, s)
    assert np.array_equal(qn, q ^ 0x80)


def test_zero_tile_gets_scale_one():
    x = np.zeros((3, 256), np.float32)
    x[1, :128] = -0.0
    x[2, 128] = 1.0           # second tile of row 2 is non-zero
    q, s = oracle.quant_act_1x128(x)
    assert s[0, 0] == 1.0 and s[1, 0] == 1.0 and s[0, 2] == 1.0 and s[1, 1] == 1.0
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80)
    assert s[1, 2] == np.float32(1.0) / np.float32(448) and q[2, 128] == 0x7E
    # amax so small that 448/amax overflows fp32: treated as an all-zero tile
    tiny = np.full((1, 128), 1e-37, np.float32)
    qt, st = oracle.quant_act_1x128(tiny)
    assert st[0, 0] == 1.0 and np.all(qt == 0)


def test_power_of_two_equivariance():
    x = random_matrix((16, 512), seed=24, dtype=torch.float32).numpy()
    q0, s0 = oracle.quant_act_1x128(x)
    for k in (-20, -3, 5, 30):
        q1, s1 = oracle.quant_act_1x128((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(q1, q0)
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** k)).astype(np.float32))


def test_128x1_is_1x128_of_transpose():
    x = random_matrix((256, 96), seed=25, dtype=torch.bfloat16)
    qT, s = oracle.quant_act_128x1(bf16_bits(x))
    q2, s2 = oracle.quant_act_1x128(bf16_bits(x.t().contiguous()))
    assert np.array_equal(qT, q2)
    assert np.array_equal(s, s2)          # both [T/128 x C]


# ------------------------------------------------------------------ GEMM

def _quantized_case(M, N, K, seed):
    a = random_matrix((M, K), seed=seed, dtype=torch.bfloat16)
    w = random_matrix((K, N), seed=seed + 1, dtype=torch.bfloat16, std=0.02)
    Aq, sa = oracle.quant_act_1x128(bf16_bits(a))
    Wq, WqT, sw = oracle.quant_w_128x128(bf16_bits(w))
    return Aq, sa, Wq, WqT, sw


def test_gemm_matches_dequantized_fp64_matmul_tiny_fprop():
    a, w = tiny_fprop()
    Aq, sa = oracle.quant_act_1x128(a)
    Wq, WqT, sw = oracle.quant_w_128x128(w)
    c, sabs = oracle.gemm(Aq, sa, WqT, sw, oracle.SB_BLOCK_KN)
    ref = oracle.dequant_act_1x128(Aq, sa) @ oracle.dequant_w_128x128(Wq, sw)
    assert np.all(np.abs(c - ref) <= 1e-12 * sabs)
    absref = np.abs(oracle.dequant_act_1x128(Aq, sa)) @ np.abs(oracle.dequant_w_128x128(Wq, sw))
    assert np.allclose(sabs, absref, rtol=1e-12, atol=0)
    # and the quantized product is close to the unquantized one (sanity of scales)
    exact = a.astype(np.float64) @ w.astype(np.float64)
    assert np.abs(c - exact).max() < 0.1 * np.abs(exact).max()


def test_gemm_scale_layouts_agree():
    Aq, sa, Wq, WqT, sw = _quantized_case(64, 384, 256, 31)
    c_kn, _ = oracle.gemm(Aq, sa, WqT, sw, oracle.SB_BLOCK_KN)
    c_nk, _ = oracle.gemm(Aq, sa, WqT, np.ascontiguousarray(sw.T), oracle.SB_BLOCK_NK)
    percol = np.repeat(sw, 128, axis=1)           # [K/128 x N]
    c_pc, _ = oracle.gemm(Aq, sa, WqT, percol, oracle.SB_PERCOL)
    assert np.array_equal(c_kn, c_nk)
    assert np.array_equal(c_kn, c_pc)


def test_gemm_integer_codes_are_exact_integer_matmul():
    rng = np.random.default_rng(32)
    dec = oracle.e4m3_decode_table()
    ints = {int(dec[c]): c for c in range(256) if not math.isnan(dec[c]) and
            dec[c] == int(dec[c]) and abs(dec[c]) <= 8 and not (c == 0x80)}
    keys = np.array(sorted(ints))
    M, N, K = 32, 48, 384
    ia = rng.choice(keys, size=(M, K))
    ib = rng.choice(keys, size=(N, K))
    A = np.vectorize(ints.get)(ia).astype(np.uint8)
    B = np.vectorize(ints.get)(ib).astype(np.uint8)
    c, _ = oracle.gemm(A, np.ones((K // 128, M), np.float32), B,
                       np.ones((K // 128, 1), np.float32), oracle.SB_BLOCK_KN)
    assert np.array_equal(c, (ia.astype(np.int64) @ ib.T.astype(np.int64)).astype(np.float64))


def test_gemm_identity_b_returns_dequantized_a():
    Aq, sa, *_ = _quantized_case(16, 128, 256, 33)
    K = 256
    B = np.zeros((K, K), np.uint8)
    B[np.arange(K), np.arange(K)] = 0x38                     # code for 1.0
    c, _ = oracle.gemm(Aq, sa, B, np.ones((K // 128, K // 128), np.float32),
                       oracle.SB_BLOCK_KN)
    assert np.array_equal(c, oracle.dequant_act_1x128(Aq, sa))


def test_gemm_single_nonzero_slab_uses_that_slab_scales():
    Aq, sa, Wq, WqT, sw = _quantized_case(8, 256, 384, 34)
    A1 = Aq.copy()
    A1[:, :128] = 0
    A1[:, 256:] = 0
    c, _ = oracle.gemm(A1, sa, WqT, sw, oracle.SB_BLOCK_KN)
    dec = oracle.e4m3_decode_table()
    for j in (0, 127, 128, 255):
        for i in (0, 7):
            p = float(np.dot(dec[A1[i, 128:256]], dec[WqT[j, 128:256]]))
            assert c[i, j] == p * float(sa[1, i]) * float(sw[1, j // 128])


def test_gemm_elements_equal_full():
    Aq, sa, Wq, WqT, sw = _quantized_case(40, 256, 384, 35)
    c, a = oracle.gemm(Aq, sa, WqT, sw, oracle.SB_BLOCK_KN)
    rows = np.array([0, 39, 17, 5]); cols = np.array([0, 255, 128, 77])
    ce, ae = oracle.gemm_elements(Aq, sa, WqT, sw, oracle.SB_BLOCK_KN, rows, cols)
    assert np.array_equal(ce, c[rows, cols]) and np.array_equal(ae, a[rows, cols])


def test_grouped_is_dense_per_expert_and_pads_zero():
    rng = np.random.default_rng(36)
    E, N, K = 3, 128, 256
    offsets = [0, 128, 128, 384]                 # expert 1 is empty
    M = 512                                      # rows 384..511 belong to no expert
    A = rng.integers(0, 0x7E, size=(M, K)).astype(np.uint8)
    sa = rng.random((K // 128, M)).astype(np.float32)
    B = rng.integers(0, 0x7E, size=(E, N, K)).astype(np.uint8)
    sb = rng.random((E, K // 128, N // 128)).astype(np.float32)
    c, _ = oracle.grouped_gemm(offsets, A, sa, B, sb, oracle.SB_BLOCK_KN)
    c2, _ = oracle.gemm(A[128:384], sa[:, 128:384], B[2], sb[2], oracle.SB_BLOCK_KN)
    assert np.array_equal(c[128:384], c2)
    assert np.all(c[384:] == 0)
    rows = np.array([0, 127, 128, 383]); cols = np.array([0, 5, 127, 64])
    ce, _ = oracle.grouped_gemm_elements(offsets, A, sa, B, sb, oracle.SB_BLOCK_KN, rows, cols)
    assert np.array_equal(ce, c[rows, cols])


def test_results_do_not_depend_on_the_thread_count():
    """Threads only split the list of tiles / output elements: one thread and
    several give bit-identical quantizer and GEMM outputs."""
    x = random_matrix((384, 640), seed=31, dtype=torch.bfloat16)
    xb = bf16_bits(x)
    outs = []
    try:
        for nt in (1, 3, 0):
            oracle.set_threads(nt)
            q, s = oracle.quant_act_1x128(xb)
            qT, sT = oracle.quant_act_128x1(xb)
            wq, wqT, ws = oracle.quant_w_128x128(xb[:384, :512])
            B, sb = np.ascontiguousarray(qT[:256]), np.ascontiguousarray(sT[:, :256])
            c, a = oracle.gemm(qT, sT, B, sb, oracle.SB_PERCOL)     # [640 x 256], K = 384
            rows, cols = np.array([0, 5, 639, 17]), np.array([0, 255, 3, 100])
            ce, ae = oracle.gemm_elements(qT, sT, B, sb, oracle.SB_PERCOL, rows, cols)
            assert np.array_equal(ce, c[rows, cols]) and np.array_equal(ae, a[rows, cols])
            mq, msf = oracle.mx_quant_1x32(xb)
            outs.append((q, s, qT, sT, wq, wqT, ws, c, a, mq, msf))
    finally:
        oracle.set_threads(0)
    for other in outs[1:]:
        for u, v in zip(outs[0], other):
            assert np.array_equal(u, v)
