"""Accumulation precision of the B300 FP8 tensor cores (tcgen05 kind::f8f6f4),
measured through fp8bs_probe_mma_f8f6f4 -- the experiment the pages report for
H800 (page at why-be.why-be.co.kr, accumulation-precision passage: only about
14 bits of the accumulated sum are kept there).

Inputs are adversarial rows: one large product next to 31 (or more) small
ones, with the large product's exponent swept across columns so that the
small terms fall at every bit position of an FP32 mantissa and below it.
The reference is the exact sum of the decoded products (the oracle's E4M3
table, FP64 -- exact for these sums).

Measured behaviour, asserted here: each K=32 MMA step aligns the exact
products and the FP32 value already in TMEM to their largest exponent, keeps
each to 25 bits below that exponent (truncating toward zero), adds them
exactly and truncates the sum toward zero to FP32.  A 14-bit window does not
match: on B300 the per-slab partial sums are FP32-precise."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

T = oracle.e4m3_decode_table().astype(np.float64)
ENC = {float(T[c]): c for c in range(256) if np.isfinite(T[c])}
SMALL = np.array([c for c in range(256) if np.isfinite(T[c]) and T[c] != 0 and abs(T[c]) <= 1.0],
                 np.uint8)


def _run(A, B):
    a, b = torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)
    d = torch.empty((128, 256), dtype=torch.float32, device=DEV)
    fb.fp8bs_probe_mma_f8f6f4(a, b, d)
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    return d.cpu().numpy().astype(np.float64)


def _trunc_f32(x):
    f = x.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    return np.where(over, np.nextafter(f, np.float32(0)), f).astype(np.float64)


def _aligned_sum(vals, bits):
    """Sum of vals[..., :] after truncating each toward zero to `bits` bits
    below the largest exponent among them."""
    m = np.max(np.abs(vals), axis=-1, keepdims=True)
    e = np.floor(np.log2(np.where(m > 0, m, 1.0)))
    q = 2.0 ** (e - bits)
    return (np.trunc(vals / q) * q).sum(-1)


def _model(P, bits):
    """MMA-by-MMA accumulation of products P[..., K] in chunks of 32."""
    D = None
    for i in range(P.shape[-1] // 32):
        c = P[..., 32 * i:32 * (i + 1)]
        D = _trunc_f32(_aligned_sum(c if D is None else np.concatenate([D[..., None], c], -1),
                                    bits))
    return D


def _adversarial(K, seed):
    rng = np.random.default_rng(seed)
    A = rng.choice(SMALL, (128, K)).astype(np.uint8)
    B = np.full((256, K), ENC[1.0], np.uint8)
    for r in range(128):   # one +-448 in a random position
        A[r, rng.integers(0, K)] = ENC[448.0] if r % 2 else ENC[-448.0]
    for c in range(256):   # one power of two 2^-9 .. 2^8 in a random position
        B[c, rng.integers(0, K)] = ENC[float(2.0 ** (-9 + c % 18))]
    return A, B


@pytest.mark.parametrize("K", [32, 128])
def test_probe_integer_sums_exact(K):
    rng = np.random.default_rng(K)
    codes = np.array([ENC[float(v)] for v in range(-4, 5)], np.uint8)
    A, B = rng.choice(codes, (128, K)), rng.choice(codes, (256, K))
    assert np.array_equal(_run(A, B), T[A] @ T[B].T)


@pytest.mark.parametrize("K", [32, 64, 128])
def test_probe_accumulation_model(K):
    A, B = _adversarial(K, seed=100 + K)
    d = _run(A, B)
    P = T[A][:, None, :] * T[B][None, :, :]
    exact = P.sum(-1)
    # within two FP32 ulps of the exact sum
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(d - exact) <= 2 * ulp)
    assert np.array_equal(d, _model(P, 25)), "25-bit aligned, truncating model"
    assert not np.array_equal(d, _model(P, 14)), "a 14-bit window would lose the small terms"
    assert np.mean(_model(P, 14) == d) < 0.9
