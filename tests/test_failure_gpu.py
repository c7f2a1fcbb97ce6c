"""Failure detection on the GPU without a fault: a kernel whose wait runs out
(a barrier nothing arrives at, limit 2 ms) records a timeout in the device
error word and returns; the host reads it; the context stays usable."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_15_b300 as fb
import oracle
import workloads as wl
from gpu_helpers import gpu_quant_1x128, oracle_input

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    fb.fp8bs_debug_timeout_probe(2_000_000)
    assert fb.fp8bs_sync_status() == fb.FP8BS_ERR_DEVICE_TIMEOUT
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
    x = wl.random_matrix((64, 256), seed=1, dtype=torch.bfloat16)
    q, s = gpu_quant_1x128(x)
    qr, sr = oracle.quant_act_1x128(oracle_input(x))
    assert np.array_equal(q, qr) and np.array_equal(s, sr)


def test_invalid_arguments_launch_nothing():
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda:0")
    q = torch.zeros((4, 100), dtype=torch.uint8, device="cuda:0")
    s = torch.zeros((1, 4), dtype=torch.float32, device="cuda:0")
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8bs_quant_act_1x128(x, q, s)
    assert e.value.status == fb.FP8BS_ERR_UNSUPPORTED
    assert fb.fp8bs_sync_status() == fb.FP8BS_OK
