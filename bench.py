"""Benchmark of the fine-grained FP8 hot path on B300.

One step = one training pass of a linear layer (tokens 4096, K_in 7168,
N_out 18432) through every row of the path:
    quant 1x128 + 128x1 of X (one pass) -> quant 128x128 (W, with transposed
    copy) -> Fprop GEMM -> quant 1x128 + 128x1 of dY (one pass) -> Dgrad GEMM
    -> Wgrad GEMM (FP32 out)
The GEMMs split the K range of their last, partial wave (fp8bs_gemm_ws).
`value` = the three GEMMs' FLOPs (3 x 2*M*N*K) / device time of the whole step,
in TFLOPS, with inputs resident in HBM.  Per-kernel CUDA-event timings give the
roofline of the dominant kernel and of every other launch.  `e2e` repeats the
step through the same entry points from pinned host buffers, copies included.
Extras (not part of `value`): the grouped MoE up-projection and the quantizer
bandwidth sweep.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fp8bs|reference]

Under torchrun each rank runs an independent replica (no data-path collective);
the barrier / max-over-ranks timing uses torch.distributed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

TOKENS, HIDDEN, FFN = wl.TOKENS, wl.HIDDEN, wl.FFN
GEMM_FLOPS = 2.0 * TOKENS * HIDDEN * FFN          # each of Fprop, Dgrad, Wgrad
METRIC = "block-scaled FP8 GEMM TFLOPS (% of B300 FP8 peak); quantizer GB/s (% of HBM)"
WORKLOAD = ("linear-layer training step: quant 1x128/128x1/128x128 + Fprop, Dgrad, Wgrad "
            f"block-scaled FP8 GEMMs, tokens={TOKENS}, K={HIDDEN}, N={FFN}")

DATA = ("synthetic (seeded numpy: N(0,1) activations with 0.1% x100 outliers, "
        "N(0,0.02) weights, N(0,1e-3) output grads; bf16)")


def config_dict(world: int) -> dict:
    """The workload both arms report (identical in both)."""
    return {"workload": WORKLOAD, "tokens": TOKENS, "K": HIDDEN, "N": FFN,
            "l2": "inputs larger than L2 (474 MB of bf16 inputs per step)",
            "parallelism": f"replicas x{world} (no data-path collective)"}


class L2Flush:
    """Between timed launches: write 256 MB (more than the 126 MB L2), then read
    another 256 MB.  The next launch finds none of its inputs in L2 and no dirty
    lines of the flush left to write back; with the write alone a small launch
    paid for up to 126 MB of write-back (8192 x 7168 quantizers: 1x128 34.8 ->
    30.7 us, 128x1 38.9 -> 34.8 us, dual 51.2 -> 49.1 us, measured)."""

    def __init__(self, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


# Algorithmic bytes per element of the quantizers (read input, write codes, write scales).
def quant_bytes(elems: int, in_bytes: int, transposed_copy: bool = False, block=False) -> float:
    scale = 4.0 / (128 * 128) if block else 4.0 / 128
    return elems * (in_bytes + 1 + (1 if transposed_copy else 0) + scale)


def dual_bytes(elems: int, in_bytes: int) -> float:
    """One read of the input, both code copies, both scale arrays."""
    return elems * (in_bytes + 2 + 2 * 4.0 / 128)


# DRAM traffic per launch measured by ncu (dram__bytes_read.sum + write.sum), with
# the sha256 of the kernel sources it was measured on; ignored once they change.
NCU_TRAFFIC = {
    # one launch of `bench.py --case wgrad`, measured by ncu on that launch
    "gemm_wgrad": {"files": ("gemm_pair_kernel.cuh", "gemm_kernel.cuh", "ptx.cuh"),
                   "src": "b1df381dda21827f", "bytes": 156778752 + 499927808},
}


def _src_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "fp8_fine_grained_15_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, src = 6400.0, 1800.0, "fallback"
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        hbm, bf16, src = float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    # FP8 dense = 2 x BF16 dense (nominal ratio 4.5 / 2.25 PFLOP/s).
    return {"hbm_gbs": hbm, "fp8_tflops": 2.0 * bf16, "source": src}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- the step

class LayerStep:
    """Device buffers and the launch sequence of one layer training step."""

    KERNELS = ["quant_dual_X", "quant_128x128_W", "gemm_fprop", "quant_dual_dY",
               "gemm_dgrad", "gemm_wgrad"]

    def __init__(self, x, w, dy, dev):
        import fp8_fine_grained_15_b300 as fb
        self.fb = fb
        T, K = x.shape
        N = w.shape[1]
        e = lambda *s, dt=torch.uint8: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.x, self.w, self.dy = x, w, dy
        self.Xq, self.Sx = e(T, K), e(K // 128, T, dt=torch.float32)
        self.Wq, self.WqT, self.Sw = e(K, N), e(N, K), e(K // 128, N // 128, dt=torch.float32)
        self.dYq, self.Sdy = e(T, N), e(N // 128, T, dt=torch.float32)
        self.XqT, self.SxT = e(K, T), e(T // 128, K, dt=torch.float32)
        self.dYqT, self.SdyT = e(N, T), e(T // 128, N, dt=torch.float32)
        self.Y = e(T, N, dt=torch.bfloat16)
        self.dX = e(T, K, dt=torch.bfloat16)
        self.dW = e(K, N, dt=torch.float32)
        self.T, self.K, self.N = T, K, N
        # one workspace for the K split of the GEMMs' last waves (the three
        # GEMMs run in order on one stream, so they can share it)
        self.ws_need = [fb.fp8bs_gemm_workspace_size(*s) for s in ((T, N, K), (T, K, N), (K, N, T))]
        self.ws = e(max(self.ws_need)) if max(self.ws_need) > 0 else None

    def launches(self):
        fb = self.fb
        return [
            lambda s: fb.fp8bs_quant_act_dual(self.x, self.Xq, self.Sx, self.XqT, self.SxT, s),
            lambda s: fb.fp8bs_quant_w_128x128(self.w, self.Wq, self.WqT, self.Sw, s),
            lambda s: fb.fp8bs_gemm_ws(self.Xq, self.Sx, self.WqT, self.Sw, fb.FP8BS_SB_BLOCK_KN,
                                       self.Y, self.ws, s),
            lambda s: fb.fp8bs_quant_act_dual(self.dy, self.dYq, self.Sdy, self.dYqT, self.SdyT, s),
            lambda s: fb.fp8bs_gemm_ws(self.dYq, self.Sdy, self.Wq, self.Sw, fb.FP8BS_SB_BLOCK_NK,
                                       self.dX, self.ws, s),
            lambda s: fb.fp8bs_gemm_ws(self.XqT, self.SxT, self.dYqT, self.SdyT,
                                       fb.FP8BS_SB_PERCOL, self.dW, self.ws, s),
        ]

    def kernel_launches(self):
        """Library kernels one step launches: 3 quantizers, 3 GEMMs, plus the
        partial-sum kernel of each GEMM whose last wave is split."""
        return 6 + sum(1 for n in self.ws_need if n > 0)

    def work(self):
        """(kind, algorithmic amount) per launch: bytes for quantizers, FLOPs for GEMMs."""
        T, K, N = self.T, self.K, self.N
        g = 2.0 * T * K * N
        return [("hbm", dual_bytes(T * K, 2)), ("hbm", quant_bytes(K * N, 2, True, True)),
                ("tensor", g), ("hbm", dual_bytes(T * N, 2)), ("tensor", g), ("tensor", g)]


def _barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def _max_over_ranks(v: float, dist_on: bool) -> float:
    if not dist_on:
        return v
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.distributed.get_backend() == "nccl" else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_fp8bs(args, rank, world, dist_on):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = _peaks()
    # Inputs: seeded host generation (identical recipe to the parity tests),
    # one independent replica per rank (seeds offset by rank).
    x_h = wl.layer_activations(seed=0 + 10 * rank)
    w_h = wl.layer_weight(seed=1 + 10 * rank)
    dy_h = wl.layer_grad_output(seed=2 + 10 * rank)
    x, w, dy = x_h.to(dev), w_h.to(dev), dy_h.to(dev)
    step = LayerStep(x, w, dy, dev)
    stream = torch.cuda.current_stream(dev)
    fns = step.launches()
    nk = len(fns)

    for _ in range(args.warmup):
        for f in fns:
            f(stream)
    torch.cuda.synchronize(dev)
    st = step.fb.fp8bs_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {step.fb.status_string(st)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    _barrier(dist_on)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        for k in range(args.steps):
            ev[k][0].record(stream)
            for i, f in enumerate(fns):
                f(stream)
                ev[k][i + 1].record(stream)
        torch.cuda.synchronize(dev)
    _barrier(dist_on)
    if step.fb.fp8bs_sync_status(stream) != 0:
        raise RuntimeError("device error during the timed region")
    total_ms = sum(ev[k][0].elapsed_time(ev[k][nk]) for k in range(args.steps))
    per_kernel_ms = [statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1])
                                     for k in range(args.steps)) for i in range(nk)]
    ms_per_step = _max_over_ranks(total_ms / args.steps, dist_on)
    value = world * 3 * GEMM_FLOPS / (ms_per_step * 1e-3) / 1e12

    kernels = {}
    for name, ms, (kind, amount) in zip(LayerStep.KERNELS, per_kernel_ms, step.work()):
        if kind == "tensor":
            ach = amount / (ms * 1e-3) / 1e12
            kernels[name] = {"ms": round(ms, 4), "TFLOP/s": round(ach, 1),
                             "frac_fp8_peak": round(ach / peaks["fp8_tflops"], 4)}
        else:
            ach = amount / (ms * 1e-3) / 1e9
            kernels[name] = {"ms": round(ms, 4), "GB/s": round(ach, 1),
                             "frac_hbm": round(ach / peaks["hbm_gbs"], 4)}
    dom = max(range(nk), key=lambda i: per_kernel_ms[i])
    dom_name = LayerStep.KERNELS[dom]
    kind, amount = step.work()[dom]
    if kind == "tensor":
        ach = amount / (per_kernel_ms[dom] * 1e-3) / 1e12
        peak, unit = peaks["fp8_tflops"], "TFLOP/s"
    else:
        ach = amount / (per_kernel_ms[dom] * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    traffic = None
    rec = NCU_TRAFFIC.get(dom_name)
    if rec and rec["bytes"] is not None and rec["src"] == _src_hash(rec["files"]):
        traffic = rec["bytes"]
    roofline = {"bound": kind, "kernel": dom_name, "achieved": round(ach, 2),
                "peak": round(peak, 1), "unit": unit, "frac": round(ach / peak, 4),
                "traffic": traffic,
                "peak_source": f"{peaks['source']}: FP8 = 2 x bf16 burst; HBM copy"}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, x_h, w_h, dy_h, dev, stream, args, dist_on, world)
    extras = None if args.no_extras else run_extras(dev, stream, peaks)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": DATA, "config": config_dict(world),
        "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": step.kernel_launches() * args.steps, "clocks": clk.summary(), "extras": extras,
    }
    return result


def run_e2e(step, x_h, w_h, dy_h, dev, stream, args, dist_on, world):
    """The same step through the same entry points from pinned host buffers,
    copies included: every step uploads X, W, dY and downloads Y, dX, dW.
    The copies are pipelined against the compute on three streams with two
    device buffer sets (upload of step i+1 and download of step i-1 overlap
    the compute of step i; PCIe carries both directions at once)."""
    xp, wp, dyp = x_h.pin_memory(), w_h.pin_memory(), dy_h.pin_memory()
    sets = [step, LayerStep(torch.empty_like(step.x), torch.empty_like(step.w),
                            torch.empty_like(step.dy), dev)]
    outs = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (st.Y, st.dX, st.dW))
            for st in sets]
    fns = [st.launches() for st in sets]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done, out_done = {}, {}

    def one(i):
        b = i % 2
        st = sets[b]
        if i >= 2:   # buffer set b is free once step i-2 computed and was read back
            s_in.wait_event(comp_done[i - 2])
        with torch.cuda.stream(s_in):
            st.x.copy_(xp, non_blocking=True)
            st.w.copy_(wp, non_blocking=True)
            st.dy.copy_(dyp, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        stream.wait_event(in_done)
        if i >= 2:
            stream.wait_event(out_done[i - 2])
        for f in fns[b]:
            f(stream)
        comp_done[i] = torch.cuda.Event()
        comp_done[i].record(stream)
        s_out.wait_event(comp_done[i])
        with torch.cuda.stream(s_out):
            for h, d in zip(outs[b], (st.Y, st.dX, st.dW)):
                h.copy_(d, non_blocking=True)
            out_done[i] = torch.cuda.Event()
            out_done[i].record(s_out)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(dev)
    n = max(4, min(args.steps, 8))
    _barrier(dist_on)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(2, 2 + n):
        one(i)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize(dev)
    _barrier(dist_on)
    ms = _max_over_ranks(t0.elapsed_time(t1) / n, dist_on)
    h2d = sum(t.numel() * t.element_size() for t in (xp, wp, dyp))
    d2h = sum(t.numel() * t.element_size() for t in outs[0])
    if step.fb.fp8bs_sync_status(stream) != 0:
        raise RuntimeError("device error during the end-to-end run")
    return {"value": round(world * 3 * GEMM_FLOPS / (ms * 1e-3) / 1e12, 2), "unit": "TFLOPS",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "H2D / compute / D2H on three streams, two device buffer sets",
            "steps": n}


def run_extras(dev, stream, peaks):
    """Grouped MoE up-projection (32 experts, Zipf(1.1) routing of 16384 rows,
    7168 -> 4096) and the quantizer bandwidth sweep, timed with CUDA events.
    Inputs are drawn on the device with a seeded generator (timing only)."""
    import fp8_fine_grained_15_b300 as fb
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)

    def timeit(fn, reps=10, flush=None):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            if flush is not None:
                flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(s.elapsed_time(e))
        return statistics.median(ts), min(ts)

    flush = L2Flush(dev)

    # grouped GEMM
    counts = wl.zipf_counts()
    offsets = wl.padded_offsets(counts)
    E, K, N = wl.EXPERTS, wl.HIDDEN, wl.EXPERT_N
    M_cap = int(offsets[-1])
    Aq = torch.randint(0, 0x7E, (M_cap, K), dtype=torch.uint8, device=dev, generator=gen)
    sa = torch.rand((K // 128, M_cap), device=dev, generator=gen) * 1e-2
    Bq = torch.randint(0, 0x7E, (E, N, K), dtype=torch.uint8, device=dev, generator=gen)
    sb = torch.rand((E, K // 128, N // 128), device=dev, generator=gen) * 1e-3
    C = torch.empty((M_cap, N), dtype=torch.bfloat16, device=dev)
    off = torch.tensor(offsets.astype(np.int32), device=dev)
    med, best = timeit(lambda: fb.fp8bs_grouped_gemm(off, Aq, sa, Bq, sb, fb.FP8BS_SB_BLOCK_KN,
                                                     C, stream), flush=flush)
    flops_real = 2.0 * int(counts.sum()) * K * N
    flops_pad = 2.0 * M_cap * K * N
    out["grouped_moe_up"] = {
        "experts": E, "rows_routed": int(counts.sum()), "rows_padded": M_cap,
        "ms_median": round(med, 4),
        "TFLOP/s_unpadded": round(flops_real / (med * 1e-3) / 1e12, 1),
        "TFLOP/s_padded": round(flops_pad / (med * 1e-3) / 1e12, 1),
        "frac_fp8_peak_unpadded": round(flops_real / (med * 1e-3) / 1e12 / peaks["fp8_tflops"], 4)}
    del Aq, Bq, C, sa, sb

    # quantize-then-dispatch of the same routing (16384 tokens x 7168, bf16)
    expert = torch.from_numpy(wl.zipf_expert_ids().astype(np.int32)).to(dev)
    T = int(expert.numel())
    xt = torch.randn((T, K), device=dev, generator=gen).to(torch.bfloat16)
    Mc = (T + 127 * E + 127) // 128 * 128
    qd = torch.empty((Mc, K), dtype=torch.uint8, device=dev)
    sd = torch.empty((K // 128, Mc), dtype=torch.float32, device=dev)
    i32 = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    offd, cntd, t2r, r2t = i32(E + 1), i32(E), i32(T), i32(Mc)
    md, _ = timeit(lambda: fb.fp8bs_quant_dispatch(xt, expert, E, qd, sd, offd, cntd, t2r, r2t,
                                                   stream), flush=flush)
    dbytes = quant_bytes(T * K, 2) + (M_cap - T) * (K + 4 * K / 128)   # + padding rows written
    out["quant_dispatch_moe"] = {"tokens": T, "experts": E, "us": round(md * 1e3, 2),
                                 "GB/s": round(dbytes / (md * 1e-3) / 1e9, 1),
                                 "frac_hbm": round(dbytes / (md * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                 "launches": 3}
    del xt, qd, sd

    # MX variant: the layer's Fprop with 1x32 power-of-two scales applied by the
    # tensor cores, and the MX quantizer of X
    xm = torch.randn((TOKENS, HIDDEN), device=dev, generator=gen).to(torch.bfloat16)
    wm = (torch.randn((FFN, HIDDEN), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    Am = torch.empty((TOKENS, HIDDEN), dtype=torch.uint8, device=dev)
    Bm = torch.empty((FFN, HIDDEN), dtype=torch.uint8, device=dev)
    sfa = torch.empty((HIDDEN // 128, TOKENS), dtype=torch.int32, device=dev)
    sfb = torch.empty((HIDDEN // 128, FFN), dtype=torch.int32, device=dev)
    fb.fp8bs_mx_quant_1x32(wm, Bm, sfb, stream)
    mq, _ = timeit(lambda: fb.fp8bs_mx_quant_1x32(xm, Am, sfa, stream), flush=flush)
    Cm = torch.empty((TOKENS, FFN), dtype=torch.bfloat16, device=dev)
    mg, _ = timeit(lambda: fb.fp8bs_mx_gemm(Am, sfa, Bm, sfb, Cm, stream), flush=flush)
    qbytes = quant_bytes(TOKENS * HIDDEN, 2)
    flops = 2.0 * TOKENS * HIDDEN * FFN
    out["mx_variant"] = {
        "fprop_ms": round(mg, 4), "fprop_TFLOP/s": round(flops / (mg * 1e-3) / 1e12, 1),
        "fprop_frac_fp8_peak": round(flops / (mg * 1e-3) / 1e12 / peaks["fp8_tflops"], 4),
        "quant_X_us": round(mq * 1e3, 2), "quant_X_GB/s": round(qbytes / (mq * 1e-3) / 1e9, 1),
        "quant_X_frac_hbm": round(qbytes / (mq * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    del xm, wm, Am, Bm, sfa, sfb, Cm

    # quantizer sweep
    sweep = {}
    for M in (1024, 8192, 65536):
        x = torch.randn((M, wl.HIDDEN), device=dev, generator=gen).to(torch.bfloat16)
        q = torch.empty((M, wl.HIDDEN), dtype=torch.uint8, device=dev)
        s = torch.empty((wl.HIDDEN // 128, M), dtype=torch.float32, device=dev)
        qT = torch.empty((wl.HIDDEN, M), dtype=torch.uint8, device=dev)
        sT = torch.empty((M // 128, wl.HIDDEN), dtype=torch.float32, device=dev)
        nbytes = quant_bytes(M * wl.HIDDEN, 2)
        m1, _ = timeit(lambda: fb.fp8bs_quant_act_1x128(x, q, s, stream), flush=flush)
        m2, _ = timeit(lambda: fb.fp8bs_quant_act_128x1(x, qT, sT, stream), flush=flush)
        m3, _ = timeit(lambda: fb.fp8bs_quant_act_dual(x, q, s, qT, sT, stream), flush=flush)
        dbytes = dual_bytes(M * wl.HIDDEN, 2)
        sweep[f"M{M}"] = {
            "bytes": int(nbytes),
            "1x128_us": round(m1 * 1e3, 2), "1x128_GB/s": round(nbytes / (m1 * 1e-3) / 1e9, 1),
            "1x128_frac_hbm": round(nbytes / (m1 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "128x1_us": round(m2 * 1e3, 2), "128x1_GB/s": round(nbytes / (m2 * 1e-3) / 1e9, 1),
            "128x1_frac_hbm": round(nbytes / (m2 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "dual_bytes": int(dbytes), "dual_us": round(m3 * 1e3, 2),
            "dual_GB/s": round(dbytes / (m3 * 1e-3) / 1e9, 1),
            "dual_frac_hbm": round(dbytes / (m3 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        del x, q, s, qT, sT
    wgt = torch.randn((wl.HIDDEN, wl.FFN), device=dev, generator=gen).to(torch.bfloat16)
    wq = torch.empty((wl.HIDDEN, wl.FFN), dtype=torch.uint8, device=dev)
    wqT = torch.empty((wl.FFN, wl.HIDDEN), dtype=torch.uint8, device=dev)
    ws = torch.empty((wl.HIDDEN // 128, wl.FFN // 128), dtype=torch.float32, device=dev)
    for name, qq, tt, tr in (("128x128", wq, None, False), ("128x128+T", wq, wqT, True)):
        nbytes = quant_bytes(wl.HIDDEN * wl.FFN, 2, tr, True)
        m, _ = timeit(lambda: fb.fp8bs_quant_w_128x128(wgt, qq, tt, ws, stream), flush=flush)
        sweep[f"W_{name}"] = {"bytes": int(nbytes), "us": round(m * 1e3, 2),
                              "GB/s": round(nbytes / (m * 1e-3) / 1e9, 1),
                              "frac_hbm": round(nbytes / (m * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    out["quant_sweep"] = sweep
    if fb.fp8bs_sync_status(stream) != 0:
        raise RuntimeError("device error during extras")
    return out


# ------------------------------------------------------ CPU oracle baseline

# Bounded samples of the layer step for the oracle: the full K and N, fewer
# tokens (the work per token is the same, so the rate carries over).
CPU_BASELINE_TOKENS = 1024    # one run inside the fp8bs arm: ~16 s on 16 cores
REFERENCE_STEP_TOKENS = 256   # one step of the reference arm


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


_cpu_inputs_cache: dict = {}


def _cpu_inputs(tokens: int):
    if tokens not in _cpu_inputs_cache:
        from workloads import bf16_bits
        _cpu_inputs_cache[tokens] = (bf16_bits(wl.layer_activations(tokens, HIDDEN)),
                                     bf16_bits(wl.layer_weight(HIDDEN, FFN)),
                                     bf16_bits(wl.layer_grad_output(tokens, FFN)))
    return _cpu_inputs_cache[tokens]


def cpu_layer_step(tokens: int) -> float:
    """The oracle, as it stands, on the layer step restricted to `tokens`
    tokens (same eight operations: dual quantizers as 1x128 + 128x1, the
    128x128 weight quantizer with its transposed copy, Fprop, Dgrad, Wgrad),
    on every host core.  Returns the seconds it took."""
    import oracle
    x, w, dy = _cpu_inputs(tokens)
    oracle.build()
    oracle.set_threads(host_cores())
    t0 = time.perf_counter()
    Xq, Sx = oracle.quant_act_1x128(x)
    XqT, SxT = oracle.quant_act_128x1(x)
    Wq, WqT, Sw = oracle.quant_w_128x128(w)
    oracle.gemm(Xq, Sx, WqT, Sw, oracle.SB_BLOCK_KN)
    dYq, Sdy = oracle.quant_act_1x128(dy)
    dYqT, SdyT = oracle.quant_act_128x1(dy)
    oracle.gemm(dYq, Sdy, Wq, np.ascontiguousarray(Sw.T), oracle.SB_BLOCK_NK)
    oracle.gemm(XqT, SxT, dYqT, SdyT, oracle.SB_PERCOL)
    return time.perf_counter() - t0


def _cpu_sample(tokens: int) -> str:
    return (f"layer step (8 ops) on tokens={tokens} of {TOKENS}, K={HIDDEN}, N={FFN}; "
            f"C oracle with FP64 GEMM, one POSIX thread per host core")


def cpu_baseline():
    """The oracle timed on the host cores on a bounded sample of the step."""
    import oracle
    T = CPU_BASELINE_TOKENS
    dt = cpu_layer_step(T)
    return {"value": round(3 * 2.0 * T * HIDDEN * FFN / dt / 1e12, 6), "unit": "TFLOPS",
            "cores": oracle.threads(), "kind": "oracle", "seconds": round(dt, 2),
            "sample": _cpu_sample(T)}


def run_reference(args, rank, world, dist_on):
    """The reference arm: the CPU oracle, timed on the host cores, each step
    one bounded sample of the same workload (the layer step on
    REFERENCE_STEP_TOKENS tokens); rank 0 only."""
    if rank != 0:
        return None
    import oracle
    T = args.ref_tokens
    for _ in range(max(0, min(args.warmup, 1))):
        cpu_layer_step(T)
    secs = [cpu_layer_step(T) for _ in range(args.steps)]
    med = statistics.median(secs)
    v = round(3 * 2.0 * T * HIDDEN * FFN / med / 1e12, 6)
    cores = oracle.threads()
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(med * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA, "config": config_dict(world),
        "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": _cpu_sample(T) + " per step"},
        "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


CASES = ("fprop", "dgrad", "wgrad", "grouped", "quant_1x128", "quant_128x1", "quant_dual",
         "quant_128x128", "mx_fprop", "mx_quant", "quant_dispatch")


def run_case(args):
    """One kernel alone on its layer-sized operands (device-drawn, seeded):
    `--warmup` untimed launches, then `--steps` launches timed one by one with
    CUDA events.  This is the command the ncu captures under profiles/ run."""
    import fp8_fine_grained_15_b300 as fb
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    T, K, N = TOKENS, HIDDEN, FFN
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device=dev)  # noqa: E731
    f32 = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)  # noqa: E731
    c = args.case
    if c in ("fprop", "dgrad", "wgrad"):
        x = torch.randn((T, K), device=dev, generator=gen).to(torch.bfloat16)
        dy = (torch.randn((T, N), device=dev, generator=gen) * 1e-3).to(torch.bfloat16)
        w = (torch.randn((K, N), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        if c == "fprop":
            A, sa, B, sb = u8(T, K), f32(K // 128, T), u8(N, K), f32(K // 128, N // 128)
            fb.fp8bs_quant_act_1x128(x, A, sa, stream)
            fb.fp8bs_quant_w_128x128(w, None, B, sb, stream)
            out, mode = torch.empty((T, N), dtype=torch.bfloat16, device=dev), fb.FP8BS_SB_BLOCK_KN
        elif c == "dgrad":
            A, sa, B, sb = u8(T, N), f32(N // 128, T), u8(K, N), f32(K // 128, N // 128)
            fb.fp8bs_quant_act_1x128(dy, A, sa, stream)
            fb.fp8bs_quant_w_128x128(w, B, None, sb, stream)
            out, mode = torch.empty((T, K), dtype=torch.bfloat16, device=dev), fb.FP8BS_SB_BLOCK_NK
        else:
            A, sa, B, sb = u8(K, T), f32(T // 128, K), u8(N, T), f32(T // 128, N)
            fb.fp8bs_quant_act_128x1(x, A, sa, stream)
            fb.fp8bs_quant_act_128x1(dy, B, sb, stream)
            out, mode = torch.empty((K, N), dtype=torch.float32, device=dev), fb.FP8BS_SB_PERCOL
        del x, dy, w
        M_, K_ = A.shape
        need = fb.fp8bs_gemm_workspace_size(M_, B.shape[0], K_)
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
        fn = lambda: fb.fp8bs_gemm_ws(A, sa, B, sb, mode, out, ws, stream)  # noqa: E731
        amount, kind = 2.0 * T * K * N, "tensor"
    elif c == "mx_fprop":
        x = torch.randn((T, K), device=dev, generator=gen).to(torch.bfloat16)
        w = (torch.randn((N, K), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        A, B = u8(T, K), u8(N, K)
        sfa = torch.empty((K // 128, T), dtype=torch.int32, device=dev)
        sfb = torch.empty((K // 128, N), dtype=torch.int32, device=dev)
        fb.fp8bs_mx_quant_1x32(x, A, sfa, stream)
        fb.fp8bs_mx_quant_1x32(w, B, sfb, stream)
        del x, w
        out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: fb.fp8bs_mx_gemm(A, sfa, B, sfb, out, stream)  # noqa: E731
        amount, kind = 2.0 * T * K * N, "tensor"
    elif c == "quant_dispatch":
        expert = torch.from_numpy(wl.zipf_expert_ids().astype(np.int32)).to(dev)
        E, T_ = wl.EXPERTS, int(expert.numel())
        x = torch.randn((T_, K), device=dev, generator=gen).to(torch.bfloat16)
        Mc = (T_ + 127 * E + 127) // 128 * 128
        q, s = u8(Mc, K), f32(K // 128, Mc)
        i32 = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
        offd, cntd, t2r, r2t = i32(E + 1), i32(E), i32(T_), i32(Mc)
        fn = lambda: fb.fp8bs_quant_dispatch(x, expert, E, q, s, offd, cntd, t2r, r2t,  # noqa: E731
                                             stream)
        padded = int(wl.padded_offsets(wl.zipf_counts())[-1])
        amount, kind = quant_bytes(T_ * K, 2) + (padded - T_) * (K + 4 * K / 128), "hbm"
    elif c == "grouped":
        counts = wl.zipf_counts()
        offsets = wl.padded_offsets(counts)
        E, Kg, Ng = wl.EXPERTS, wl.HIDDEN, wl.EXPERT_N
        M_cap = int(offsets[-1])
        A = torch.randint(0, 0x7E, (M_cap, Kg), dtype=torch.uint8, device=dev, generator=gen)
        sa = torch.rand((Kg // 128, M_cap), device=dev, generator=gen) * 1e-2
        B = torch.randint(0, 0x7E, (E, Ng, Kg), dtype=torch.uint8, device=dev, generator=gen)
        sb = torch.rand((E, Kg // 128, Ng // 128), device=dev, generator=gen) * 1e-3
        out = torch.empty((M_cap, Ng), dtype=torch.bfloat16, device=dev)
        off = torch.tensor(offsets.astype(np.int32), device=dev)
        fn = lambda: fb.fp8bs_grouped_gemm(off, A, sa, B, sb, fb.FP8BS_SB_BLOCK_KN, out,  # noqa: E731
                                           stream)
        amount, kind = 2.0 * int(counts.sum()) * Kg * Ng, "tensor"
    else:
        M = args.case_rows
        if c == "quant_128x128":
            x = (torch.randn((K, N), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
            q, qT, s = u8(K, N), u8(N, K), f32(K // 128, N // 128)
            fn = lambda: fb.fp8bs_quant_w_128x128(x, q, qT, s, stream)  # noqa: E731
            amount = quant_bytes(K * N, 2, True, True)
        else:
            x = torch.randn((M, K), device=dev, generator=gen).to(torch.bfloat16)
            amount = quant_bytes(M * K, 2)
            if c == "quant_1x128":
                q, s = u8(M, K), f32(K // 128, M)
                fn = lambda: fb.fp8bs_quant_act_1x128(x, q, s, stream)  # noqa: E731
            elif c == "quant_128x1":
                q, s = u8(K, M), f32(M // 128, K)
                fn = lambda: fb.fp8bs_quant_act_128x1(x, q, s, stream)  # noqa: E731
            elif c == "mx_quant":
                q = u8(M, K)
                s = torch.empty((K // 128, M), dtype=torch.int32, device=dev)
                fn = lambda: fb.fp8bs_mx_quant_1x32(x, q, s, stream)  # noqa: E731
            else:
                q, s, qT, sT = u8(M, K), f32(K // 128, M), u8(K, M), f32(M // 128, K)
                fn = lambda: fb.fp8bs_quant_act_dual(x, q, s, qT, sT, stream)  # noqa: E731
                amount = dual_bytes(M * K, 2)
        kind = "hbm"
    flush = L2Flush(dev)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(args.steps):
        flush()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(ev0.elapsed_time(ev1))
    if fb.fp8bs_sync_status(stream) != 0:
        raise RuntimeError("device error in case run")
    med = statistics.median(ts)
    if kind == "tensor":
        ach, peak, unit = amount / (med * 1e-3) / 1e12, peaks["fp8_tflops"], "TFLOP/s"
    else:
        ach, peak, unit = amount / (med * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    return {"case": c, "launches": args.steps, "ms_median": round(med, 4),
            "ms_min": round(min(ts), 4), "achieved": round(ach, 1), "unit": unit,
            "peak": round(peak, 1), "frac": round(ach / peak, 4), "amount": amount}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=CASES, default=None,
                    help="time one kernel alone (profiling command); no JSON bench line")
    ap.add_argument("--case-rows", type=int, default=65536,
                    help="rows of the activation quantizer cases")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["fp8bs", "reference"], default="fp8bs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=REFERENCE_STEP_TOKENS,
                    help="tokens of the layer step the reference arm runs per step (multiple of 128)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "fp8bs":
        ap.error("at least 3 warm-up steps")
    if args.case is not None:
        print(json.dumps(run_case(args)), flush=True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist_on = world > 1
    if dist_on:
        backend = "nccl" if (torch.cuda.is_available() and args.impl == "fp8bs") else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend)

    if args.impl == "reference":
        res = run_reference(args, rank, world, dist_on)
    else:
        res = run_fp8bs(args, rank, world, dist_on)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
