"""MX variant on the GPU: the 1x32 power-of-two quantizer (bit-exact against
the oracle: codes and exponent bytes) and the block-scaled MMA GEMM, whose
group exponents the tensor cores apply (within the GEMM tolerance of the
other tests: 2^-7 |C| + 1e-5 S_abs for BF16, 1e-5 S_abs for FP32; exact where
every partial sum is exactly representable)."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
from gpu_helpers import DEV, assert_gemm_close, oracle_input, to_dev_u8
import full_ref

pytestmark = pytest.mark.gpu


def _words_to_bytes(sf: torch.Tensor, rows: int) -> np.ndarray:
    """int32 words [K/128 x ld] -> the oracle's bytes [K/128 x rows x 4]."""
    w = np.ascontiguousarray(sf.cpu().numpy()[:, :rows])
    return w.view(np.uint8).reshape(w.shape[0], rows, 4)


def _bytes_to_words(sf: np.ndarray, ld: int | None = None) -> torch.Tensor:
    kb, rows, _ = sf.shape
    ld = ld or rows
    w = np.zeros((kb, ld), np.int32)
    w[:, :rows] = np.ascontiguousarray(sf).view(np.int32).reshape(kb, rows)
    return torch.from_numpy(w).to(DEV)


def gpu_mx_quant(x: torch.Tensor, pad_ld: int = 0, pad_ldsf: int = 0):
    R, K = x.shape
    xd = torch.zeros((R, K + pad_ld), dtype=x.dtype, device=DEV)[:, :K]
    xd.copy_(x)
    q = torch.full((R, K + pad_ld), 0xAB, dtype=torch.uint8, device=DEV)[:, :K]
    sf = torch.full((K // 128, R + pad_ldsf), -1, dtype=torch.int32, device=DEV)
    fb.fp8bs_mx_quant_1x32(xd, q, sf)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    if pad_ldsf:   # padding words stay untouched
        assert torch.all(sf[:, R:] == -1)
    return q.cpu().numpy(), _words_to_bytes(sf, R)


def gpu_mx_gemm(A, sfa, B, sfb, out_dtype=torch.bfloat16, ld_pad: int = 0):
    M, N = A.shape[0], B.shape[0]
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    fb.fp8bs_mx_gemm(to_dev_u8(A), _bytes_to_words(sfa, M + ld_pad), to_dev_u8(B),
                     _bytes_to_words(sfb, N + ld_pad), C)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return C.float().cpu().numpy().astype(np.float64)


# ------------------------------------------------------------------ quantizer

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,K", [(300, 1152), (8, 128), (1037, 2048), (64, 7168)])
def test_mx_quant_matches_oracle(dtype, R, K):
    x = wl.random_matrix((R, K), seed=R + K, dtype=dtype)
    q, sf = gpu_mx_quant(x)
    qr, sfr = oracle.mx_quant_1x32(oracle_input(x))
    assert np.array_equal(sf, sfr), "exponent bytes differ from the oracle"
    assert np.array_equal(q, qr), "codes differ from the oracle"


def test_mx_quant_padded_strides():
    x = wl.random_matrix((200, 640), seed=5, dtype=torch.bfloat16)
    q, sf = gpu_mx_quant(x, pad_ld=64, pad_ldsf=12)
    qr, sfr = oracle.mx_quant_1x32(oracle_input(x))
    assert np.array_equal(q, qr) and np.array_equal(sf, sfr)


def test_mx_quant_edge_groups():
    """Zero, subnormal, near-FLT_MAX groups and exact binade boundaries."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 512)).astype(np.float32)
    x[0, 0:32] = 0.0
    x[1, 32:64] = 1e-40
    x[2, 64:96] = np.float32(3.0e38)
    x[2, 70] = -np.float32(3.4e38)
    for i, k in enumerate((-20, -3, 0, 1, 7, 40)):
        at = np.float32(np.ldexp(448.0, k))
        x[3 + i, 128:160] = np.float32(np.ldexp(1.0, k))
        x[3 + i, 130] = at
        x[3 + i, 160:192] = np.float32(np.ldexp(1.0, k))
        x[3 + i, 170] = np.nextafter(at, np.float32(np.inf))
        x[3 + i, 192:224] = np.float32(np.ldexp(1.0, k))
        x[3 + i, 200] = -np.nextafter(at, np.float32(0))
    x[10, :] *= np.float32(2.0 ** -130)                 # whole row in fp32 subnormals
    q, sf = gpu_mx_quant(torch.from_numpy(x))
    qr, sfr = oracle.mx_quant_1x32(x)
    assert np.array_equal(sf, sfr)
    assert np.array_equal(q, qr)


def test_mx_quant_layer_activations_full_size():
    x = wl.layer_activations()
    q, sf = gpu_mx_quant(x)
    qr, sfr = oracle.mx_quant_1x32(oracle_input(x))
    assert np.array_equal(sf, sfr) and np.array_equal(q, qr)


# ----------------------------------------------------------------------- GEMM

@pytest.mark.parametrize("M,N", [(128, 256), (256, 256), (384, 512)])
def test_mx_gemm_single_group_applies_that_groups_exponents(M, N):
    """Only group g holds non-zero codes (all 1.0); every row of A and of B has
    its own exponent in every group, so each output is exactly
    32 * 2^(ea(m, g) + eb(n, g)) -- it names the two scale bytes the tensor
    core applied (row, column and group), on both CTAs of a pair tile and in
    both halves of B."""
    rng = np.random.default_rng(31 + M + N)
    K = 512
    sfa = rng.integers(100, 150, (K // 128, M, 4)).astype(np.uint8)
    sfb = rng.integers(100, 150, (K // 128, N, 4)).astype(np.uint8)
    for g in (0, 1, 2, 3, 6, 13):
        A = np.zeros((M, K), np.uint8)
        B = np.zeros((N, K), np.uint8)
        A[:, 32 * g:32 * g + 32] = 0x38
        B[:, 32 * g:32 * g + 32] = 0x38
        c = gpu_mx_gemm(A, sfa, B, sfb, torch.float32)
        c_ref, _ = oracle.mx_gemm(A, sfa, B, sfb)
        assert np.array_equal(c, c_ref), f"group {g}"


def test_mx_gemm_integer_codes_exact():
    rng = np.random.default_rng(32)
    enc = {float(v): c for c, v in enumerate(oracle.e4m3_decode_table()) if np.isfinite(v)}
    codes = np.array([enc[float(v)] for v in range(-4, 5)], np.uint8)
    M, N, K = 256, 512, 1024
    A = codes[rng.integers(0, 9, (M, K))]
    B = codes[rng.integers(0, 9, (N, K))]
    sfa = np.full((K // 128, M, 4), 127, np.uint8)
    sfb = np.full((K // 128, N, 4), 127, np.uint8)
    c = gpu_mx_gemm(A, sfa, B, sfb, torch.float32)
    c_ref, _ = oracle.mx_gemm(A, sfa, B, sfb)
    assert np.array_equal(c, c_ref)


def _mx_operands(M, N, K, seed):
    a = wl.random_matrix((M, K), seed=seed, dtype=torch.bfloat16)
    b = wl.random_matrix((N, K), seed=seed + 1, dtype=torch.bfloat16, std=0.02)
    A, sfa = oracle.mx_quant_1x32(oracle_input(a))
    B, sfb = oracle.mx_quant_1x32(oracle_input(b))
    return A, sfa, B, sfb


@pytest.mark.parametrize("M,N,K,out", [
    (128, 256, 128, torch.bfloat16),     # one tile, one K block
    (300, 272, 1024, torch.float32),     # ragged M and N
    (512, 1024, 2048, torch.bfloat16),   # 16 tiles
    (256, 512, 7168, torch.float32),     # long K
    (1024, 2048, 512, torch.bfloat16),   # 64 tiles: several per CTA on small grids
])
def test_mx_gemm_matches_oracle(M, N, K, out):
    A, sfa, B, sfb = _mx_operands(M, N, K, seed=M + N + K)
    c = gpu_mx_gemm(A, sfa, B, sfb, out)
    c_ref, s_abs = oracle.mx_gemm(A, sfa, B, sfb)
    assert_gemm_close(c, c_ref, s_abs, out == torch.bfloat16, f"MX {M}x{N}x{K}")


def test_mx_gemm_padded_exponent_rows():
    A, sfa, B, sfb = _mx_operands(256, 512, 512, seed=7)
    c = gpu_mx_gemm(A, sfa, B, sfb, torch.bfloat16, ld_pad=4)
    c_ref, s_abs = oracle.mx_gemm(A, sfa, B, sfb)
    assert_gemm_close(c, c_ref, s_abs, True, "padded exponent rows")


def test_mx_gemm_zero_k_writes_zeros():
    C = torch.full((64, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    st = fb.lib().fp8bs_mx_gemm(64, 128, 0, None, 0, None, 0, None, 0, None, 0, C.data_ptr(),
                                fb.FP8BS_BF16, 128, torch.cuda.current_stream().cuda_stream)
    assert st == fb.FP8BS_OK
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    assert torch.all(C == 0)


def test_mx_quant_then_gemm_chain():
    """Library quantizer straight into the library GEMM (words stay on the device)."""
    a = wl.random_matrix((384, 1536), seed=61, dtype=torch.bfloat16)
    b = wl.random_matrix((768, 1536), seed=62, dtype=torch.bfloat16, std=0.02)
    Aq = torch.empty((384, 1536), dtype=torch.uint8, device=DEV)
    Bq = torch.empty((768, 1536), dtype=torch.uint8, device=DEV)
    sfa = torch.empty((12, 384), dtype=torch.int32, device=DEV)
    sfb = torch.empty((12, 768), dtype=torch.int32, device=DEV)
    fb.fp8bs_mx_quant_1x32(a.to(DEV), Aq, sfa)
    fb.fp8bs_mx_quant_1x32(b.to(DEV), Bq, sfb)
    C = torch.empty((384, 768), dtype=torch.bfloat16, device=DEV)
    fb.fp8bs_mx_gemm(Aq, sfa, Bq, sfb, C)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    A, sa = oracle.mx_quant_1x32(oracle_input(a))
    B, sb = oracle.mx_quant_1x32(oracle_input(b))
    c_ref, s_abs = oracle.mx_gemm(A, sa, B, sb)
    assert_gemm_close(C.float().cpu().numpy().astype(np.float64), c_ref, s_abs, True, "chain")


def test_mx_layer_fprop_full():
    """The layer's Fprop (4096 tokens, 7168 -> 18432) in the MX format: X and
    W^T quantized 1x32 along K by the oracle; every output element against
    the oracle."""
    A, sfa, B, sfb = full_ref.mx_layer_operands()
    c = gpu_mx_gemm(A, sfa, B, sfb, torch.bfloat16)
    c_ref, s_abs = full_ref.mx_layer_reference()
    assert_gemm_close(c, c_ref, s_abs, True, "MX Fprop 4096x18432x7168")


def test_mx_quant_at_sweep_maximum_full():
    """65536 x 7168 bf16 through the MX quantizer (8192 x 7 CTAs): every code
    and exponent byte against the oracle."""
    x = wl.sweep_activations(65536)
    R, K = x.shape
    xd = x.to(DEV)
    q = torch.empty((R, K), dtype=torch.uint8, device=DEV)
    sf = torch.empty((K // 128, R), dtype=torch.int32, device=DEV)
    fb.fp8bs_mx_quant_1x32(xd, q, sf)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    qr, sfr = oracle.mx_quant_1x32(oracle_input(x))
    assert np.array_equal(q.cpu().numpy(), qr), "codes"
    assert np.array_equal(_words_to_bytes(sf, R), sfr), "exponents"
