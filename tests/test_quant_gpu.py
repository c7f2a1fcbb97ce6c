"""Quantizer parity: the CUDA kernels against the CPU oracle, bit-exact
(E4M3 codes and FP32 scales), at small ragged sizes, edge cases and the full
sweep sizes of the quantizer bandwidth workload."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
from gpu_helpers import (DEV, gpu_quant_1x128, gpu_quant_128x1, gpu_quant_dual, gpu_quant_w,
                         oracle_input)

pytestmark = pytest.mark.gpu


def _eq(got, ref, what):
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,K", [(1, 128), (127, 256), (129, 640), (300, 7168), (8, 1024)])
def test_quant_1x128_matches_oracle(dtype, M, K):
    x = wl.random_matrix((M, K), seed=M * 7 + K, dtype=dtype)
    q, s = gpu_quant_1x128(x)
    qr, sr = oracle.quant_act_1x128(oracle_input(x))
    _eq(q, qr, "codes")
    _eq(s, sr, "scales")


def test_quant_1x128_padded_strides():
    x = wl.random_matrix((77, 384), seed=3, dtype=torch.bfloat16)
    q, s = gpu_quant_1x128(x, pad_ld=128, pad_lds=13)
    qr, sr = oracle.quant_act_1x128(oracle_input(x))
    _eq(q, qr, "codes")
    _eq(s, sr, "scales")


def test_quant_1x128_tiny_fprop_activations():
    a, _ = wl.tiny_fprop()
    x = torch.from_numpy(a)
    q, s = gpu_quant_1x128(x)
    qr, sr = oracle.quant_act_1x128(a)
    _eq(q, qr, "codes")
    _eq(s, sr, "scales")


def test_quant_edge_tiles():
    x = np.zeros((6, 512), np.float32)
    x[1, :128] = -0.0                          # negative zeros
    x[2, 128:256] = 1e-37                      # 448/amax overflows: treated as zero
    x[3, 256] = -3.0                           # single non-zero element
    x[4, 384:] = np.float32(3.0e38)            # huge (finite in bf16 too)
    x[5, :] = np.linspace(-1e-3, 1e-3, 512, dtype=np.float32)
    for dtype in (torch.float32, torch.bfloat16):
        t = torch.from_numpy(x).to(dtype)
        q, s = gpu_quant_1x128(t)
        qr, sr = oracle.quant_act_1x128(oracle_input(t))
        _eq(q, qr, f"codes {dtype}")
        _eq(s, sr, f"scales {dtype}")
    assert s[0, 0] == 1.0 and s[1, 2] == 1.0 and q[3, 256] == 0xFE


def _probe_values(seed: int, n_random: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    bits = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    allbf = bits.view(np.float32)
    allbf = allbf[np.isfinite(allbf) & (np.abs(allbf) <= 448)]
    dec = oracle.e4m3_decode_table()
    pos = np.unique(dec[np.isfinite(dec) & (dec >= 0)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9))])
    rb = rng.integers(0, 1 << 32, size=3 * n_random, dtype=np.uint64).astype(np.uint32)
    rv = rb.view(np.float32)
    rv = rv[np.isfinite(rv) & (np.abs(rv) <= 448)][:n_random]
    return np.concatenate([allbf, near, -near, rv]).astype(np.float32)


def test_device_conversion_matches_oracle_encoder():
    """Tiles whose amax is exactly 448 have r = 1, so every other element is
    encoded as-is: this pushes every bf16 value, every rounding midpoint (and
    its neighbours) and 4M random fp32 values through the kernel's conversion."""
    v = _probe_values(17, 4_000_000)
    per = 127
    n_tiles = (v.size + per - 1) // per
    x = np.zeros((n_tiles, 128), np.float32)
    x[:, 0] = 448.0
    flat = np.zeros(n_tiles * per, np.float32)
    flat[:v.size] = v
    x[:, 1:] = flat.reshape(n_tiles, per)
    q, s = gpu_quant_1x128(torch.from_numpy(x))
    assert np.all(s == np.float32(1.0))
    ref = oracle.e4m3_encode_array(x)
    _eq(q, ref, "codes")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,C", [(128, 16), (256, 96), (384, 208), (512, 7168)])
def test_quant_128x1_matches_oracle(dtype, T, C):
    x = wl.random_matrix((T, C), seed=T + C, dtype=dtype)
    qT, s = gpu_quant_128x1(x)
    qr, sr = oracle.quant_act_128x1(oracle_input(x))
    _eq(qT, qr, "codes")
    _eq(s, sr, "scales")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,C", [(128, 128), (512, 256), (384, 1152)])
def test_quant_128x128_matches_oracle(dtype, R, C):
    w = wl.random_matrix((R, C), seed=R * 3 + C, dtype=dtype, std=0.02)
    q, qT, s = gpu_quant_w(w)
    qr, qTr, sr = oracle.quant_w_128x128(oracle_input(w))
    _eq(q, qr, "codes")
    _eq(qT, qTr, "transposed codes")
    _eq(s, sr, "scales")
    q1, _, s1 = gpu_quant_w(w, want_qT=False)
    _, qT2, s2 = gpu_quant_w(w, want_q=False)
    _eq(q1, qr, "codes (q only)")
    _eq(qT2, qTr, "transposed codes (qT only)")


def test_quant_128x128_tiny_fprop_weight():
    _, w = wl.tiny_fprop()
    q, qT, s = gpu_quant_w(torch.from_numpy(w))
    qr, qTr, sr = oracle.quant_w_128x128(w)
    _eq(q, qr, "codes")
    _eq(qT, qTr, "transposed codes")
    _eq(s, sr, "scales")


@pytest.mark.parametrize("M", [1024, 8192])
def test_quant_sweep_activation_sizes(M):
    x = wl.sweep_activations(M)
    q, s = gpu_quant_1x128(x)
    qr, sr = oracle.quant_act_1x128(oracle_input(x))
    _eq(q, qr, "1x128 codes")
    _eq(s, sr, "1x128 scales")
    qT, sT = gpu_quant_128x1(x)
    qTr, sTr = oracle.quant_act_128x1(oracle_input(x))
    _eq(qT, qTr, "128x1 codes")
    _eq(sT, sTr, "128x1 scales")


def test_quant_sweep_large_activation_full():
    """M = 65536 x 7168 (the largest sweep size): every code and scale of the
    1x128 and 128x1 quantizers against the oracle."""
    x = wl.sweep_activations(65536)
    q, s = gpu_quant_1x128(x)
    qr, sr = oracle.quant_act_1x128(oracle_input(x))
    _eq(q, qr, "1x128 codes")
    _eq(s, sr, "1x128 scales")
    del q, s, qr, sr
    qT, sT = gpu_quant_128x1(x)
    qTr, sTr = oracle.quant_act_128x1(oracle_input(x))
    _eq(qT, qTr, "128x1 codes")
    _eq(sT, sTr, "128x1 scales")


def test_quant_layer_weight_full():
    w = wl.layer_weight()
    q, qT, s = gpu_quant_w(w)
    qr, qTr, sr = oracle.quant_w_128x128(oracle_input(w))
    _eq(s, sr, "scales")
    _eq(q, qr, "codes")
    _eq(qT, qTr, "transposed codes")


def _check_dual(x, what, pad=0):
    q, s, qT, sT = gpu_quant_dual(x, pad=pad)
    qr, sr = oracle.quant_act_1x128(oracle_input(x))
    qTr, sTr = oracle.quant_act_128x1(oracle_input(x))
    _eq(q, qr, f"{what}: 1x128 codes")
    _eq(s, sr, f"{what}: 1x128 scales")
    _eq(qT, qTr, f"{what}: 128x1 codes")
    _eq(sT, sTr, f"{what}: 128x1 scales")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,C", [(128, 128), (256, 640), (384, 1152), (512, 7168)])
def test_quant_dual_matches_oracle(dtype, T, C):
    """One pass gives exactly the 1x128 and the 128x1 quantizers' outputs."""
    x = wl.random_matrix((T, C), seed=T * 5 + C, dtype=dtype)
    _check_dual(x, f"{T}x{C} {dtype}")


def test_quant_dual_padded_strides_and_edge_blocks():
    x = np.zeros((256, 512), np.float32)
    x[0:128, 0:128] = 0.0                         # all-zero block: s = 1 both ways
    x[0:128, 128:256] = 1e-37                     # amax too small for 448/amax
    x[128:256, 256:384] = np.float32(3.0e38)      # huge
    x[5, 300] = -7.0
    x[128:, 384:] = np.linspace(-2.0, 3.0, 128 * 128, dtype=np.float32).reshape(128, 128)
    for dtype in (torch.float32, torch.bfloat16):
        _check_dual(torch.from_numpy(x).to(dtype), f"edges {dtype}", pad=3)


def test_quant_dual_layer_activations_and_grads():
    """The layer step's two activation tensors, in full."""
    _check_dual(wl.layer_activations(), "X 4096x7168")
    _check_dual(wl.layer_grad_output(), "dY 4096x18432")


def test_dual_quantizer_at_sweep_maximum_full():
    """The sweep's largest case, 65536 x 7168 bf16 (56 x 512 CTAs), through the
    dual quantizer: every code and scale of both outputs against the oracle."""
    _check_dual(wl.sweep_activations(65536), "X 65536x7168")
