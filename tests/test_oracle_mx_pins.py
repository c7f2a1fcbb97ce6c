"""Pins for the oracle's MX variant (no GPU): 1x32 groups with power-of-two
(UE8M0) scales, and the GEMM that applies them per 32-deep group.

Each test ties the oracle to something other than its own arithmetic: the
group exponent against a frexp closed form, the codes against PyTorch's
float8_e4m3fn cast, the scale at exact binade boundaries, the byte layout
through planted per-group magnitudes, and the GEMM against an FP64 matmul of
operands dequantized by PyTorch, integer-valued cases and single planted
groups.  A plausible mistake -- an exponent off by one at a boundary, a floor
where a ceiling belongs, a transposed or shifted exponent byte, a scale
applied to the wrong group -- fails one of them.
"""
import numpy as np
import torch

import oracle
from workloads import bf16_bits, random_matrix


def _frexp_exponent(amax: np.ndarray) -> np.ndarray:
    """Closed form of the smallest e with amax <= 448 * 2^e: amax = f * 2^E
    with f in [0.5, 1) and 448 = 0.875 * 2^9, so e = E - 9 + (f > 0.875);
    clamped to [-127, 127]; zero -> 0."""
    f, E = np.frexp(amax.astype(np.float64))
    e = E - 9 + (f > 0.875)
    e = np.clip(e, -127, 127)
    return np.where(amax == 0, 0, e).astype(np.int64)


def _group_amax(x: np.ndarray) -> np.ndarray:
    R, K = x.shape
    return np.abs(x.astype(np.float64)).reshape(R, K // 32, 32).max(-1)


def _sf_as_groups(sf: np.ndarray) -> np.ndarray:
    """[K/128, R, 4] bytes -> [R, K/32] exponents."""
    kb, R, _ = sf.shape
    return sf.transpose(1, 0, 2).reshape(R, kb * 4).astype(np.int64) - 127


def _torch_dequant(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    vals = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    e = _sf_as_groups(sf)
    return vals * np.exp2(np.repeat(e, 32, axis=1).astype(np.float64))


def test_mx_exponent_matches_frexp_closed_form():
    rng = np.random.default_rng(5)
    R, K = 64, 512
    x = rng.standard_normal((R, K)).astype(np.float32)
    # magnitudes spread over many binades, some groups zero, some tiny or huge
    x *= np.exp2(rng.integers(-60, 60, size=(R, K // 32))).repeat(32, axis=1).astype(np.float32)
    x[3, 64:96] = 0.0
    x[5, 0:32] = 1e-40                                  # fp32 subnormal: clamps at -127
    x[6, 32:64] = np.float32(3.0e38)                    # near FLT_MAX
    q, sf = oracle.mx_quant_1x32(x)
    assert np.array_equal(_sf_as_groups(sf), _frexp_exponent(_group_amax(x)))
    assert _sf_as_groups(sf)[3, 2] == 0 and _sf_as_groups(sf)[5, 0] == -127


def test_mx_exponent_at_binade_boundaries():
    # amax exactly 448 * 2^k keeps k; the next fp32 value above needs k + 1
    for k in (-20, -3, 0, 1, 7, 40):
        at = np.float32(np.ldexp(448.0, k))
        above = np.nextafter(at, np.float32(np.inf))
        below = np.nextafter(at, np.float32(0))
        x = np.full((3, 128), np.float32(np.ldexp(1.0, k)), np.float32)
        x[0, 5], x[1, 5], x[2, 5] = at, above, below
        q, sf = oracle.mx_quant_1x32(x)
        e = _sf_as_groups(sf)[:, 0]
        assert list(e) == [k, k + 1, k], (k, e)
        assert q[0, 5] == 0x7E                           # amax lands on 448
        assert q[2, 5] == 0x7E                           # rounds up to 448, no overflow


def test_mx_codes_match_torch_cast_of_scaled_values():
    x = random_matrix((96, 384), seed=41, dtype=torch.float32).numpy()
    q, sf = oracle.mx_quant_1x32(x)
    e = np.repeat(_sf_as_groups(sf), 32, axis=1)
    scaled = (x.astype(np.float64) * np.exp2(-e.astype(np.float64))).astype(np.float32)
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    assert np.all(np.abs(scaled) <= 448.0)


def test_mx_bf16_input_equals_fp32_of_same_values():
    xb = random_matrix((40, 256), seed=42, dtype=torch.bfloat16)
    q1, s1 = oracle.mx_quant_1x32(bf16_bits(xb))
    q2, s2 = oracle.mx_quant_1x32(xb.float().numpy())
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_mx_exponent_byte_layout():
    # group g of row r gets the planted magnitude 2^(g + r): its exponent byte
    # must sit at sf[g // 4, r, g % 4]
    R, K = 8, 512
    x = np.full((R, K), np.float32(2.0 ** -40), np.float32)   # below every planted value
    for r in range(R):
        for g in range(K // 32):
            x[r, 32 * g + 7] = np.float32(np.ldexp(448.0, g + r - 10))
    q, sf = oracle.mx_quant_1x32(x)
    for r in range(R):
        for g in range(K // 32):
            assert int(sf[g // 4, r, g % 4]) - 127 == g + r - 10


def test_mx_dequant_error_within_half_e4m3_ulp():
    x = random_matrix((32, 256), seed=43, dtype=torch.float32).numpy().astype(np.float64)
    q, sf = oracle.mx_quant_1x32(x.astype(np.float32))
    d = _torch_dequant(q, sf)
    e = np.repeat(_sf_as_groups(sf), 32, axis=1).astype(np.float64)
    # E4M3: 3 mantissa bits; subnormal spacing 2^-9 in the scaled domain
    ulp = np.maximum(np.exp2(np.floor(np.log2(np.maximum(np.abs(x) * np.exp2(-e), 1e-300))) - 3),
                     2.0 ** -9) * np.exp2(e)
    assert np.all(np.abs(d - x) <= 0.5 * ulp + 1e-300)


def test_mx_gemm_matches_fp64_matmul_of_torch_dequantized_operands():
    a = random_matrix((64, 384), seed=44, dtype=torch.float32).numpy()
    b = random_matrix((48, 384), seed=45, dtype=torch.float32, std=0.02).numpy()
    A, sfa = oracle.mx_quant_1x32(a)
    B, sfb = oracle.mx_quant_1x32(b)
    c, s_abs = oracle.mx_gemm(A, sfa, B, sfb)
    da, db = _torch_dequant(A, sfa), _torch_dequant(B, sfb)
    ref = da @ db.T
    assert np.allclose(c, ref, rtol=1e-12, atol=1e-12 * (np.abs(da) @ np.abs(db).T).max())
    assert np.allclose(s_abs, np.abs(da) @ np.abs(db).T, rtol=1e-12)


def test_mx_gemm_integer_codes_unit_scales_exact():
    rng = np.random.default_rng(46)
    enc = {float(v): c for c, v in enumerate(oracle.e4m3_decode_table()) if np.isfinite(v)}
    codes = np.array([enc[float(v)] for v in range(-8, 9)], np.uint8)
    vals = np.arange(-8, 9, dtype=np.int64)
    ia, ib = rng.integers(0, 17, (32, 256)), rng.integers(0, 17, (24, 256))
    sfa = np.full((2, 32, 4), 127, np.uint8)
    sfb = np.full((2, 24, 4), 127, np.uint8)
    c, _ = oracle.mx_gemm(codes[ia], sfa, codes[ib], sfb)
    assert np.array_equal(c, (vals[ia] @ vals[ib].T).astype(np.float64))


def test_mx_gemm_single_group_uses_that_groups_exponents():
    # only group g is non-zero; every group of A row i / B row j has its own
    # exponent, so the result names which exponent bytes were applied
    rng = np.random.default_rng(47)
    M, N, K = 4, 5, 512
    one = 0x38                                           # E4M3 code of 1.0
    sfa = rng.integers(100, 150, (K // 128, M, 4)).astype(np.uint8)
    sfb = rng.integers(100, 150, (K // 128, N, 4)).astype(np.uint8)
    for g in (0, 5, 10, 15):
        A = np.zeros((M, K), np.uint8)
        B = np.zeros((N, K), np.uint8)
        A[:, 32 * g:32 * g + 32] = one
        B[:, 32 * g:32 * g + 32] = one
        c, _ = oracle.mx_gemm(A, sfa, B, sfb)
        ea = sfa[g // 4, :, g % 4].astype(np.int64) - 127
        eb = sfb[g // 4, :, g % 4].astype(np.int64) - 127
        assert np.array_equal(c, 32.0 * np.exp2((ea[:, None] + eb[None, :]).astype(np.float64)))


def test_mx_gemm_elements_equal_full():
    a = random_matrix((40, 256), seed=48, dtype=torch.float32).numpy()
    b = random_matrix((36, 256), seed=49, dtype=torch.float32).numpy()
    A, sfa = oracle.mx_quant_1x32(a)
    B, sfb = oracle.mx_quant_1x32(b)
    c, s = oracle.mx_gemm(A, sfa, B, sfb)
    rows = np.array([0, 39, 17, 5]), np.array([0, 35, 2, 30])
    ce, se = oracle.mx_gemm_elements(A, sfa, B, sfb, rows[0], rows[1])
    assert np.array_equal(ce, c[rows]) and np.array_equal(se, s[rows])
