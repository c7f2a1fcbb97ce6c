"""Oracle results of the full-size workloads, computed once per test process
and shared by every parity test that needs them.

A full-size GEMM costs the oracle ~5e11 multiply-adds; split over the host's
cores (one thread per core) that is tens of seconds, so the layer's Fprop,
Dgrad and Wgrad references, the grouped MoE reference and the MX Fprop
reference are each computed once and kept for the process.  Nothing here does
arithmetic of its own: the operands are the oracle's quantizers applied to the
seeded workloads, the references are the oracle's GEMMs."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl
from workloads import bf16_bits

_cache: dict = {}


def _memo(key, fn):
    if key not in _cache:
        _cache[key] = fn()
    return _cache[key]


def layer_operands() -> dict:
    """The single-layer workload (4096 tokens, 7168 -> 18432) quantized by the
    oracle: Xq/Sx, Wq/WqT/Sw, dYq/Sdy (1x128 and 128x128) and XqT/SxT,
    dYqT/SdyT (128x1)."""
    def make():
        x = bf16_bits(wl.layer_activations())
        w = bf16_bits(wl.layer_weight())
        dy = bf16_bits(wl.layer_grad_output())
        d = {}
        d["Xq"], d["Sx"] = oracle.quant_act_1x128(x)
        d["Wq"], d["WqT"], d["Sw"] = oracle.quant_w_128x128(w)
        d["dYq"], d["Sdy"] = oracle.quant_act_1x128(dy)
        d["XqT"], d["SxT"] = oracle.quant_act_128x1(x)
        d["dYqT"], d["SdyT"] = oracle.quant_act_128x1(dy)
        return d
    return _memo("layer", make)


def layer_gemm_args(which: str):
    """(A, sa, B, sb, mode, bf16_out) of the layer's Fprop, Dgrad or Wgrad."""
    d = layer_operands()
    if which == "fprop":
        return d["Xq"], d["Sx"], d["WqT"], d["Sw"], oracle.SB_BLOCK_KN, True
    if which == "dgrad":
        return d["dYq"], d["Sdy"], d["Wq"], d["Sw"], oracle.SB_BLOCK_NK, True
    if which == "wgrad":
        return d["XqT"], d["SxT"], d["dYqT"], d["SdyT"], oracle.SB_PERCOL, False
    raise ValueError(which)


def layer_reference(which: str):
    """(C_ref, S_abs) of the whole output of the layer's Fprop, Dgrad or Wgrad."""
    def make():
        A, sa, B, sb, mode, _ = layer_gemm_args(which)
        return oracle.gemm(A, sa, B, sb, mode)
    return _memo(("layer_ref", which), make)


def moe_operands():
    """The MoE up-projection workload quantized by the oracle: (counts,
    offsets, Aq [rows x 7168], sa, Bq [32 x 4096 x 7168], sb [32 x 56 x 32])."""
    def make():
        counts, offsets, x, w = wl.grouped_moe()
        E, K, N = w.shape
        Aq, sa = oracle.quant_act_1x128(bf16_bits(x))
        Bq = np.empty((E, N, K), np.uint8)
        sb = np.empty((E, K // 128, N // 128), np.float32)
        for e in range(E):
            _, Bq[e], sb[e] = oracle.quant_w_128x128(bf16_bits(w[e]), with_transpose=True)
        return counts, offsets, Aq, sa, Bq, sb
    return _memo("moe", make)


def moe_reference():
    def make():
        counts, offsets, Aq, sa, Bq, sb = moe_operands()
        return oracle.grouped_gemm(offsets, Aq, sa, Bq, sb, oracle.SB_BLOCK_KN)
    return _memo("moe_ref", make)


def mx_layer_operands():
    """The layer's Fprop operands in the MX format: X and W^T quantized 1x32
    along K by the oracle."""
    def make():
        x = bf16_bits(wl.layer_activations())
        wt = bf16_bits(wl.layer_weight().t().contiguous())
        A, sfa = oracle.mx_quant_1x32(x)
        B, sfb = oracle.mx_quant_1x32(wt)
        return A, sfa, B, sfb
    return _memo("mx_layer", make)


def mx_layer_reference():
    def make():
        return oracle.mx_gemm(*mx_layer_operands())
    return _memo("mx_layer_ref", make)
