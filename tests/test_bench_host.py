"""bench.py host logic without a GPU: the multi-rank timing path (barrier,
max over ranks) with two gloo ranks, the reference arm's JSON line, and the
roofline bookkeeping helpers."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._barrier(True)
    v = bench._max_over_ranks(float(rank + 1) * 1.5, True)
    q.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 3.0), (1, 3.0)]


def test_quant_bytes_accounting():
    assert bench.quant_bytes(128, 2) == 128 * (2 + 1 + 4 / 128)
    assert bench.quant_bytes(16384, 2, True, True) == 16384 * (2 + 2 + 4 / 16384)


def test_reference_arm_line_under_torchrun(tmp_path):
    """Two gloo ranks: rank 0 prints one JSON line with impl=reference and the
    other rank exits 0 without work."""
    port = _free_port()
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--ref-tokens", "128"]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["config"] == bench.config_dict(2)          # the fp8bs arm's config, unchanged
    assert d["cpu_baseline"]["cores"] == bench.host_cores()
    assert "tokens=128" in d["cpu_baseline"]["sample"]
