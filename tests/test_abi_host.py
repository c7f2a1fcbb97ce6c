"""The C-ABI library on the host (no GPU): it builds for sm_103a, loads,
exports every function include/fp8bs.h declares, and rejects invalid
arguments with the documented status before touching the device."""
import ctypes
import subprocess

import pytest

import fp8_fine_grained_15_b300 as fb
from fp8_fine_grained_15_b300 import build as fbuild


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fb.lib()


def test_header_declares_the_path_entry_points():
    names = fb.header_functions()
    for n in ("fp8bs_quant_act_1x128", "fp8bs_quant_act_128x1", "fp8bs_quant_w_128x128",
              "fp8bs_gemm", "fp8bs_grouped_gemm", "fp8bs_sync_status", "fp8bs_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.check_output(["nm", "-D", "--defined-only", fb.LIB_PATH], text=True)
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in fb.header_functions():
        assert n in exported, n
        assert getattr(L, n) is not None


def test_status_strings(L):
    for st in range(8):
        assert fb.status_string(st) not in ("", "unknown status")
    assert fb.status_string(99) == "unknown status"


NULL = None
BF16, F32 = fb.FP8BS_BF16, fb.FP8BS_F32
FAKE = 0x10000          # 16-byte aligned non-null "pointer": never dereferenced on error paths
FAKE_ODD = 0x10004


@pytest.mark.parametrize("args,expect", [
    ((NULL, BF16, 4, 100, 100, NULL, 100, NULL, 4), fb.FP8BS_ERR_UNSUPPORTED),   # K % 128
    ((NULL, BF16, -1, 128, 128, NULL, 128, NULL, 4), fb.FP8BS_ERR_INVALID_ARG),
    ((NULL, 7, 4, 128, 128, NULL, 128, NULL, 4), fb.FP8BS_ERR_INVALID_ARG),       # dtype
    ((NULL, BF16, 4, 128, 128, FAKE, 128, FAKE, 4), fb.FP8BS_ERR_INVALID_ARG),    # null x
    ((FAKE, BF16, 4, 128, 64, FAKE, 128, FAKE, 4), fb.FP8BS_ERR_INVALID_ARG),     # ldx < K
    ((FAKE, BF16, 4, 128, 128, FAKE, 128, FAKE, 2), fb.FP8BS_ERR_INVALID_ARG),    # lds < M
    ((FAKE_ODD, BF16, 4, 128, 128, FAKE, 128, FAKE, 4), fb.FP8BS_ERR_MISALIGNED),
    ((FAKE, BF16, 4, 128, 132, FAKE, 128, FAKE, 4), fb.FP8BS_ERR_MISALIGNED),     # ldx*2 % 16
    ((NULL, BF16, 0, 128, 128, NULL, 128, NULL, 4), fb.FP8BS_OK),                 # M == 0
])
def test_quant_1x128_host_checks(L, args, expect):
    assert L.fp8bs_quant_act_1x128(*args, None) == expect


def test_quant_128x1_and_w_host_checks(L):
    q1 = L.fp8bs_quant_act_128x1
    assert q1(NULL, BF16, 100, 128, 128, NULL, 128, NULL, 128, None) == fb.FP8BS_ERR_UNSUPPORTED
    assert q1(NULL, BF16, 128, 20, 32, NULL, 128, NULL, 32, None) == fb.FP8BS_ERR_UNSUPPORTED
    assert q1(FAKE, BF16, 128, 32, 32, FAKE, 64, FAKE, 32, None) == fb.FP8BS_ERR_INVALID_ARG
    qw = L.fp8bs_quant_w_128x128
    assert qw(FAKE, BF16, 128, 100, 128, FAKE, 128, NULL, 0, FAKE, 1, None) == \
        fb.FP8BS_ERR_UNSUPPORTED
    assert qw(FAKE, BF16, 128, 128, 128, NULL, 0, NULL, 0, FAKE, 1, None) == \
        fb.FP8BS_ERR_INVALID_ARG                                    # neither output
    assert qw(FAKE, BF16, 128, 128, 128, FAKE_ODD, 128, NULL, 0, FAKE, 1, None) == \
        fb.FP8BS_ERR_MISALIGNED


def _gemm(L, M=128, N=256, K=256, A=FAKE, lda=256, sa=FAKE, ldsa=128, B=FAKE, ldb=256,
          sb=FAKE, mode=fb.FP8BS_SB_BLOCK_KN, ldsb=2, C=FAKE, ct=BF16, ldc=256):
    return L.fp8bs_gemm(M, N, K, A, lda, sa, ldsa, B, ldb, sb, mode, ldsb, C, ct, ldc, None)


def test_gemm_host_checks(L):
    assert _gemm(L, K=100) == fb.FP8BS_ERR_UNSUPPORTED
    assert _gemm(L, N=200) == fb.FP8BS_ERR_UNSUPPORTED                 # block mode N % 128
    assert _gemm(L, N=200, mode=fb.FP8BS_SB_PERCOL, ldsb=200) == fb.FP8BS_ERR_UNSUPPORTED
    assert _gemm(L, mode=9) == fb.FP8BS_ERR_INVALID_ARG
    assert _gemm(L, A=NULL) == fb.FP8BS_ERR_INVALID_ARG
    assert _gemm(L, lda=128) == fb.FP8BS_ERR_INVALID_ARG
    assert _gemm(L, ldsa=64) == fb.FP8BS_ERR_INVALID_ARG
    assert _gemm(L, ldsb=1) == fb.FP8BS_ERR_INVALID_ARG                # KN needs N/128
    assert _gemm(L, mode=fb.FP8BS_SB_BLOCK_NK, ldsb=1) == fb.FP8BS_ERR_INVALID_ARG
    assert _gemm(L, lda=264) == fb.FP8BS_ERR_MISALIGNED
    assert _gemm(L, B=FAKE_ODD) == fb.FP8BS_ERR_MISALIGNED
    assert _gemm(L, ldc=260) == fb.FP8BS_ERR_MISALIGNED                # 520 bytes
    assert _gemm(L, M=0) == fb.FP8BS_OK
    assert _gemm(L, M=-1) == fb.FP8BS_ERR_INVALID_ARG


def test_grouped_host_checks(L):
    g = L.fp8bs_grouped_gemm
    base = dict(E=2, off=FAKE, M=256, N=256, K=256)

    def call(E=2, off=FAKE, M=256, N=256, K=256, sbe=4):
        return g(E, off, M, N, K, FAKE, 256, FAKE, 256, FAKE, 256, FAKE,
                 fb.FP8BS_SB_BLOCK_KN, 2, sbe, FAKE, BF16, 256, None)
    assert call(E=0) == fb.FP8BS_ERR_INVALID_ARG
    assert call(E=2000) == fb.FP8BS_ERR_INVALID_ARG
    assert call(off=NULL) == fb.FP8BS_ERR_INVALID_ARG
    assert call(M=200) == fb.FP8BS_ERR_UNSUPPORTED
    assert call(sbe=-1) == fb.FP8BS_ERR_INVALID_ARG
    assert call(K=100) == fb.FP8BS_ERR_UNSUPPORTED
    assert call(M=0) == fb.FP8BS_OK
    del base


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fb, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fb, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        fb.lib()


def test_workspace_size_host_checks(L):
    n = ctypes.c_size_t(7)
    assert L.fp8bs_gemm_workspace_size(128, 256, 128, None) == fb.FP8BS_ERR_INVALID_ARG
    assert L.fp8bs_gemm_workspace_size(-1, 256, 128, ctypes.byref(n)) == fb.FP8BS_ERR_INVALID_ARG
    assert L.fp8bs_gemm_workspace_size(128, 256, 100, ctypes.byref(n)) == fb.FP8BS_ERR_UNSUPPORTED
    assert L.fp8bs_gemm_workspace_size(0, 256, 128, ctypes.byref(n)) == fb.FP8BS_OK
    assert n.value == 0


def test_gemm_ws_host_checks(L):
    # misaligned workspace, and the fp8bs_gemm checks on the same arguments
    assert L.fp8bs_gemm_ws(128, 256, 128, FAKE, 128, FAKE, 128, FAKE, 128, FAKE,
                           fb.FP8BS_SB_BLOCK_KN, 2, FAKE, BF16, 256, FAKE + 16, 1 << 20,
                           None) == fb.FP8BS_ERR_MISALIGNED
    assert L.fp8bs_gemm_ws(128, 256, 100, FAKE, 128, FAKE, 128, FAKE, 128, FAKE,
                           fb.FP8BS_SB_BLOCK_KN, 2, FAKE, BF16, 256, NULL, 0,
                           None) == fb.FP8BS_ERR_UNSUPPORTED
    assert L.fp8bs_gemm_ws(0, 256, 128, NULL, 128, NULL, 128, NULL, 128, NULL,
                           fb.FP8BS_SB_BLOCK_KN, 2, NULL, BF16, 256, NULL, 0, None) == fb.FP8BS_OK


@pytest.mark.parametrize("kw", [
    dict(K=100), dict(N=200), dict(mode=9), dict(A=NULL), dict(lda=128), dict(ldsa=64),
    dict(ldsb=1), dict(lda=264), dict(B=FAKE_ODD), dict(ldc=260), dict(M=-1), dict(C=NULL),
    dict(ct=7), dict(M=0),
])
def test_static_ws_rejects_like_gemm_ws(L, kw):
    """The no-allocation GEMM checks its arguments on the host before anything
    else, so a bad call returns what fp8bs_gemm_ws returns for it (and never
    reaches the device: these pointers are fake)."""
    a = dict(M=128, N=256, K=256, A=FAKE, lda=256, sa=FAKE, ldsa=128, B=FAKE, ldb=256, sb=FAKE,
             mode=fb.FP8BS_SB_BLOCK_KN, ldsb=2, C=FAKE, ct=BF16, ldc=256)
    a.update(kw)
    args = (a["M"], a["N"], a["K"], a["A"], a["lda"], a["sa"], a["ldsa"], a["B"], a["ldb"],
            a["sb"], a["mode"], a["ldsb"], a["C"], a["ct"], a["ldc"])
    want = L.fp8bs_gemm_ws(*args, NULL, 0, None)
    got = L.fp8bs_gemm_static_ws(*args, None)
    assert got == want
    if a["M"] != 0:
        assert got != fb.FP8BS_OK


def test_dispatch_host_checks(L):
    args = lambda E, M_cap, K=128, T=100: (FAKE, BF16, T, K, K, FAKE, E, FAKE, K, FAKE, M_cap,  # noqa: E731
                                          M_cap, FAKE, FAKE, FAKE, FAKE, None)
    assert L.fp8bs_quant_dispatch(*args(0, 1024)) == fb.FP8BS_ERR_UNSUPPORTED       # E < 1
    assert L.fp8bs_quant_dispatch(*args(257, 40960)) == fb.FP8BS_ERR_UNSUPPORTED    # E > 256
    assert L.fp8bs_quant_dispatch(*args(4, 1024, K=100)) == fb.FP8BS_ERR_UNSUPPORTED
    assert L.fp8bs_quant_dispatch(*args(4, 512)) == fb.FP8BS_ERR_INVALID_ARG         # < T + 127 E
    assert L.fp8bs_quant_dispatch(*args(4, 1000)) == fb.FP8BS_ERR_UNSUPPORTED        # M_cap % 128
    assert L.fp8bs_quant_dispatch(*args(4, 1024, K=0)) == fb.FP8BS_ERR_UNSUPPORTED   # K == 0
    assert L.fp8bs_quant_dispatch(*args(256, 256 * 1024 * 1024, T=205 * 1024)) == \
        fb.FP8BS_ERR_UNSUPPORTED                                   # chunk counts past the plan CTA


def _mx_gemm(L, M=128, N=256, K=256, A=FAKE, lda=256, sfa=FAKE, ldsfa=128, B=FAKE, ldb=256,
             sfb=FAKE, ldsfb=256, C=FAKE, ct=BF16, ldc=256):
    return L.fp8bs_mx_gemm(M, N, K, A, lda, sfa, ldsfa, B, ldb, sfb, ldsfb, C, ct, ldc, None)


def test_mx_gemm_host_checks(L):
    assert _mx_gemm(L, K=100) == fb.FP8BS_ERR_UNSUPPORTED
    assert _mx_gemm(L, N=200, ldsfb=200, ldc=200) == fb.FP8BS_ERR_UNSUPPORTED      # N % 16
    assert _mx_gemm(L, ct=5) == fb.FP8BS_ERR_INVALID_ARG
    assert _mx_gemm(L, A=NULL) == fb.FP8BS_ERR_INVALID_ARG
    assert _mx_gemm(L, sfb=NULL) == fb.FP8BS_ERR_INVALID_ARG
    assert _mx_gemm(L, lda=128) == fb.FP8BS_ERR_INVALID_ARG
    assert _mx_gemm(L, ldsfa=64) == fb.FP8BS_ERR_INVALID_ARG
    assert _mx_gemm(L, ldsfb=128) == fb.FP8BS_ERR_INVALID_ARG
    assert _mx_gemm(L, M=130, ldsfa=130) == fb.FP8BS_ERR_MISALIGNED               # ldsfa % 4
    assert _mx_gemm(L, sfa=FAKE_ODD) == fb.FP8BS_ERR_MISALIGNED
    assert _mx_gemm(L, lda=264) == fb.FP8BS_ERR_MISALIGNED
    assert _mx_gemm(L, ldc=260) == fb.FP8BS_ERR_MISALIGNED
    assert _mx_gemm(L, M=0) == fb.FP8BS_OK
    assert _mx_gemm(L, M=-1) == fb.FP8BS_ERR_INVALID_ARG


def test_mx_quant_host_checks(L):
    q = L.fp8bs_mx_quant_1x32
    assert q(NULL, BF16, 4, 100, 100, NULL, 100, NULL, 4, None) == fb.FP8BS_ERR_UNSUPPORTED
    assert q(NULL, 9, 4, 128, 128, NULL, 128, NULL, 4, None) == fb.FP8BS_ERR_INVALID_ARG
    assert q(FAKE, BF16, 4, 128, 128, NULL, 128, FAKE, 4, None) == fb.FP8BS_ERR_INVALID_ARG
    assert q(FAKE, BF16, 4, 128, 128, FAKE, 128, FAKE, 2, None) == fb.FP8BS_ERR_INVALID_ARG
    assert q(FAKE, BF16, 4, 128, 132, FAKE, 128, FAKE, 4, None) == fb.FP8BS_ERR_MISALIGNED
    assert q(FAKE, BF16, 4, 128, 128, FAKE, 136, FAKE, 4, None) == fb.FP8BS_ERR_MISALIGNED
    assert q(FAKE, BF16, 4, 128, 128, FAKE, 128, FAKE + 2, 4, None) == fb.FP8BS_ERR_MISALIGNED
    assert q(NULL, BF16, 0, 128, 128, NULL, 128, NULL, 0, None) == fb.FP8BS_OK


def test_binding_wraps_every_declared_function():
    # the binding's wrappers keep the C names (fp8bs_status_string is status_string)
    for n in fb.header_functions():
        if n == "fp8bs_status_string":
            assert callable(fb.status_string)
        else:
            assert callable(getattr(fb, n, None)), f"no Python wrapper for {n}"
