"""Host-side tests of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments before touching the GPU (so these run on a
machine without one).  Pointers here are plain integers that are never
dereferenced: every call below fails validation first."""
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swiglu.h")


@pytest.fixture(scope="module")
def sw():
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swiglu_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_calls():
    assert declared_functions() == sorted(
        ["swiglu_gateup_fwd", "swiglu_gateup_bwd", "swiglu_silu_mul_fwd", "swiglu_silu_mul_bwd",
         "swiglu_gateup_weighted_fwd", "swiglu_gateup_weighted_bwd", "swiglu_gateup_bias_fwd",
         "swiglu_gateup_bias_bwd_workspace_size", "swiglu_gateup_bias_bwd",
         "swiglu_gateup_weighted_bias_fwd", "swiglu_gateup_weighted_bias_bwd_workspace_size",
         "swiglu_gateup_weighted_bias_bwd", "swiglu_gateup_bias_bwd_noalloc", "swiglu_fc1_fwd",
         "swiglu_fc1_timeout_flag", "swiglu_gateup_fwd_bwd_host_staging_size",
         "swiglu_gateup_fwd_bwd_host", "swiglu_status_string", "swiglu_last_cuda_error",
         "swiglu_abi_version"])


def test_library_exports_every_declared_symbol(sw):
    for name in declared_functions():
        assert hasattr(sw.lib, name), name
    assert set(sw.EXPORTS) == set(declared_functions())
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", sw.LIB_PATH], capture_output=True,
                             text=True, check=True).stdout
        for name in declared_functions():
            assert re.search(rf"\bT {name}\b", out), name


def test_status_strings(sw):
    for code in range(-7, 1):
        s = sw.status_string(code)
        assert s and s != "unknown status"
    assert sw.status_string(-99) == "unknown status"
    assert sw.lib.swiglu_abi_version() == 5
    assert sw.lib.swiglu_last_cuda_error() == 0


# fake, never-dereferenced device addresses, 256-byte aligned and far apart
X, Y, DY, DX = 0x10_0000_0000, 0x20_0000_0000, 0x30_0000_0000, 0x40_0000_0000
F32, BF16 = 0, 1


def fwd(sw, x=X, y=Y, rows=4, n=8, sx=16, sy=8, dt=BF16):
    return sw.lib.swiglu_gateup_fwd(x, y, rows, n, sx, sy, dt, None)


def bwd(sw, dy=DY, x=X, dx=DX, rows=4, n=8, sdy=8, sx=16, sdx=16, dt=BF16, ip=0):
    return sw.lib.swiglu_gateup_bwd(dy, x, dx, rows, n, sdy, sx, sdx, dt, ip, None)


def test_empty_calls_are_noops(sw):
    assert fwd(sw, x=None, y=None, rows=0) == 0
    assert fwd(sw, x=None, y=None, n=0) == 0
    assert bwd(sw, dy=None, x=None, dx=None, rows=0) == 0
    assert bwd(sw, dy=None, x=None, dx=None, n=0, ip=1) == 0


def test_fwd_rejections(sw):
    assert fwd(sw, dt=7) == -2
    assert fwd(sw, dt=-1) == -2
    assert fwd(sw, rows=-1) == -3
    assert fwd(sw, n=-1) == -3
    assert fwd(sw, n=(1 << 30) + 1, sx=1 << 32, sy=1 << 31) == -3
    assert fwd(sw, x=None) == -1
    assert fwd(sw, y=None) == -1
    assert fwd(sw, sx=15) == -4
    assert fwd(sw, sy=7) == -4
    # extent overflows int64
    assert fwd(sw, rows=1 << 40, sx=1 << 40) == -3
    # y inside x's span, or x inside y's
    assert fwd(sw, y=X + 2 * 16 * 3) == -5
    assert fwd(sw, y=X - 2) == -5


def test_bwd_rejections(sw):
    assert bwd(sw, dt=3) == -2
    assert bwd(sw, rows=-5) == -3
    assert bwd(sw, dy=None) == -1
    assert bwd(sw, x=None) == -1
    assert bwd(sw, dx=None) == -1
    assert bwd(sw, sdy=7) == -4
    assert bwd(sw, sx=15) == -4
    assert bwd(sw, sdx=10) == -4
    # out of place: dx may not overlap x or dy
    assert bwd(sw, dx=X) == -5
    assert bwd(sw, dx=X + 8) == -5
    assert bwd(sw, dx=DY + 4) == -5
    # in place: dx must be x (or NULL) with x's stride, dy may not overlap x
    assert bwd(sw, ip=1, dx=DX) == -5
    assert bwd(sw, ip=1, dx=X, sdx=24) == -4
    assert bwd(sw, ip=1, dx=X, dy=X + 16) == -5


def test_pointers_must_sit_on_elements(sw):
    """A pointer off its element size is refused before anything is launched
    (the kernels load and store whole elements)."""
    assert fwd(sw, x=X + 1) == -4
    assert fwd(sw, y=Y + 1) == -4
    assert fwd(sw, x=X + 2, dt=F32) == -4
    assert fwd(sw, y=Y + 6, dt=F32) == -4
    assert bwd(sw, dy=DY + 1) == -4
    assert bwd(sw, dx=DX + 3) == -4
    assert bwd(sw, x=X + 2, dt=F32) == -4
    assert bwd(sw, ip=1, dx=X + 1, x=X + 1) == -4


A, B, C, DA, DB = X, Y, DY, DX, 0x50_0000_0000


def mfwd(sw, a=A, b=B, c=C, rows=4, n=8, sa=8, sb=8, sc=8, dt=BF16):
    return sw.lib.swiglu_silu_mul_fwd(a, b, c, rows, n, sa, sb, sc, dt, None)


def mbwd(sw, dc=DY, a=A, b=B, da=DA, db=DB, rows=4, n=8, s=(8, 8, 8, 8, 8), dt=BF16):
    return sw.lib.swiglu_silu_mul_bwd(dc, a, b, da, db, rows, n, *s, dt, None)


def test_two_tensor_rejections(sw):
    assert mfwd(sw, a=None, rows=0) == 0
    assert mfwd(sw, dt=5) == -2
    assert mfwd(sw, n=-2) == -3
    assert mfwd(sw, b=None) == -1
    assert mfwd(sw, sb=7) == -4
    assert mfwd(sw, c=A + 16) == -5
    assert mfwd(sw, c=B) == -5
    assert mbwd(sw, rows=0, da=None) == 0
    assert mbwd(sw, db=None) == -1
    assert mbwd(sw, s=(8, 8, 8, 7, 8)) == -4
    # outputs: no overlap with each other, with dc, or with the other input
    assert mbwd(sw, db=DA + 8) == -5
    assert mbwd(sw, da=DY) == -5
    assert mbwd(sw, da=B) == -5
    assert mbwd(sw, db=A + 2) == -5
    # da partially over a is rejected; exactly a (same stride) is the in-place form
    assert mbwd(sw, da=A + 2) == -5
    assert mbwd(sw, da=A, s=(8, 8, 8, 16, 8)) == -5


W, DW, BIAS, DBIAS, WS = 0x60_0000_0000, 0x70_0000_0000, 0x80_0000_0000, 0x90_0000_0000, 0xA0_0000_0000


def test_weighted_rejections(sw):
    f = lambda **k: sw.lib.swiglu_gateup_weighted_fwd(  # noqa: E731
        k.get("x", X), k.get("w", W), k.get("y", Y), k.get("rows", 4), 8, 16, 8, BF16, None)
    b = lambda **k: sw.lib.swiglu_gateup_weighted_bwd(  # noqa: E731
        DY, X, k.get("w", W), k.get("dx", DX), k.get("dw", DW), k.get("rows", 4), k.get("n", 8),
        8, 16, 16, BF16, k.get("ip", 0), None)
    assert f(w=None) == -1
    assert f(rows=-1) == -3
    assert f(y=W - 4) == -5          # y over w
    assert b(rows=0, w=None) == 0
    assert b(dw=None) == -1
    assert b(w=None) == -1
    assert b(dw=W + 4) == -5         # dw over w
    assert b(dw=X + 8) == -5         # dw over x
    assert b(dw=DX + 8) == -5        # dw over dx
    assert b(w=DX) == -5             # w under the written dx
    assert b(ip=1, dx=DX) == -5      # the in-place contract still holds


def test_bias_rejections(sw):
    import ctypes

    out = ctypes.c_size_t(123)
    assert sw.lib.swiglu_gateup_bias_bwd_workspace_size(0, 8, ctypes.byref(out)) == 0
    assert out.value == 0
    assert sw.lib.swiglu_gateup_bias_bwd_workspace_size(-1, 8, ctypes.byref(out)) == -3
    assert sw.lib.swiglu_gateup_bias_bwd_workspace_size(4, 8, None) == -1
    f = lambda **k: sw.lib.swiglu_gateup_bias_fwd(  # noqa: E731
        X, k.get("bias", BIAS), k.get("y", Y), 4, 8, 16, 8, BF16, None)
    assert f(bias=None) == -1
    assert f(y=BIAS + 4) == -5
    b = lambda **k: sw.lib.swiglu_gateup_bias_bwd(  # noqa: E731
        DY, X, k.get("bias", BIAS), k.get("dx", DX), k.get("dbias", DBIAS), k.get("ws", WS),
        k.get("wsb", 1 << 20), k.get("rows", 4), 8, 8, 16, 16, BF16, k.get("ip", 0), None)
    assert b(bias=None) == -1
    assert b(dbias=None) == -1
    assert b(ws=None) == -1
    assert b(dbias=BIAS + 2) == -5       # dbias over bias
    assert b(dbias=X + 2) == -5          # dbias over x
    assert b(ws=DX + 16) == -5           # workspace over dx
    assert b(ws=BIAS) == -5              # workspace over bias
    assert b(bias=DX) == -5              # bias under the written dx
    assert b(ws=WS + 4) == -7            # misaligned workspace


def test_weighted_bias_rejections(sw):
    import ctypes

    out = ctypes.c_size_t(123)
    assert sw.lib.swiglu_gateup_weighted_bias_bwd_workspace_size(4, 0, ctypes.byref(out)) == 0
    assert out.value == 0
    assert sw.lib.swiglu_gateup_weighted_bias_bwd_workspace_size(4, -8, ctypes.byref(out)) == -3
    assert sw.lib.swiglu_gateup_weighted_bias_bwd_workspace_size(4, 8, None) == -1
    f = lambda **k: sw.lib.swiglu_gateup_weighted_bias_fwd(  # noqa: E731
        X, k.get("bias", BIAS), k.get("w", W), k.get("y", Y), 4, 8, 16, 8, BF16, None)
    assert f(bias=None) == -1
    assert f(w=None) == -1
    assert f(y=BIAS + 4) == -5           # y over bias
    assert f(y=W + 4) == -5              # y over w
    b = lambda **k: sw.lib.swiglu_gateup_weighted_bias_bwd(  # noqa: E731
        DY, X, k.get("bias", BIAS), k.get("w", W), k.get("dx", DX), k.get("dbias", DBIAS),
        k.get("dw", DW), k.get("ws", WS), k.get("wsb", 1 << 20), k.get("rows", 4), k.get("n", 8),
        8, 16, 16, BF16, k.get("ip", 0), None)
    assert b(rows=0, w=None, dw=None, dbias=None) == -1   # dbias still needed (set to zero)
    assert b(n=0, rows=0) == 0
    assert b(w=None) == -1
    assert b(dw=None) == -1
    assert b(bias=None) == -1
    assert b(ws=None) == -1
    assert b(dw=W + 4) == -5             # dw over w
    assert b(dw=DBIAS) == -5             # dw over dbias
    assert b(dw=WS + 64) == -5           # dw over the workspace
    assert b(dw=X + 8) == -5             # dw over x
    assert b(w=DX) == -5                 # w under the written dx
    assert b(w=DBIAS) == -5              # w under the written dbias
    assert b(w=WS) == -5                 # w under the workspace
    assert b(bias=DX) == -5              # bias under the written dx
    assert b(ws=DX + 16) == -5           # workspace over dx
    assert b(ws=WS + 4) == -7            # misaligned workspace
    assert b(ip=1, dx=DX) == -5          # the in-place contract still holds


def test_fc1_rejections(sw):
    f = lambda **k: sw.lib.swiglu_fc1_fwd(  # noqa: E731
        k.get("x", X), k.get("w", W), k.get("y", Y), k.get("xo", None), k.get("M", 256),
        k.get("n", 256), k.get("K", 512), k.get("dt", BF16), None)
    assert f(dt=F32) == -2
    assert f(M=-1) == -3
    assert f(M=0, x=None) == 0
    assert f(n=100) == -3          # n must be a multiple of 8
    assert f(K=70) == -3           # K must be a multiple of 8
    assert f(K=0) == -3
    assert f(x=None) == -1
    assert f(w=None) == -1
    assert f(y=None) == -1
    assert f(x=X + 8) == -4        # 16-byte alignment
    assert f(xo=DX + 2) == -4
    assert f(y=X + 4096) == -5     # y inside X
    assert f(y=W) == -5
    assert f(xo=Y + 64) == -5      # x_out over y
    assert f(xo=X) == -5
    assert sw.lib.swiglu_fc1_timeout_flag(None) == -1


def test_host_pipeline_rejections(sw):
    """swiglu_gateup_fwd_bwd_host checks everything before its first CUDA call
    (the host addresses below are never touched)."""
    import ctypes

    HX, HDY, HY, HDX, ST = 0x1000_0000, 0x2000_0000, 0x3000_0000, 0x4000_0000, 0x50_0000_0000
    size = ctypes.c_size_t(0)
    assert sw.lib.swiglu_gateup_fwd_bwd_host_staging_size(16, 8, BF16, 3, ctypes.byref(size)) == 0
    # three slots of x [16, 16], dy [16, 8], y [16, 8] bf16, each region 256-byte rounded
    assert size.value == 3 * (512 + 256 + 256)
    assert sw.lib.swiglu_gateup_fwd_bwd_host_staging_size(0, 8, BF16, 3, ctypes.byref(size)) == -3
    assert sw.lib.swiglu_gateup_fwd_bwd_host_staging_size(16, 8, BF16, 9, ctypes.byref(size)) == -3
    assert sw.lib.swiglu_gateup_fwd_bwd_host_staging_size(16, 8, 4, 3, ctypes.byref(size)) == -2
    assert sw.lib.swiglu_gateup_fwd_bwd_host_staging_size(16, 8, BF16, 3, None) == -1
    need = 3 * (512 + 256 + 256)

    def h(**k):
        return sw.lib.swiglu_gateup_fwd_bwd_host(
            k.get("x", HX), k.get("dy", HDY), k.get("y", HY), k.get("dx", HDX), k.get("rows", 40),
            k.get("n", 8), k.get("dt", BF16), k.get("st", ST), k.get("bytes", need),
            k.get("chunk", 16), k.get("depth", 3), None, None, None)

    assert h(rows=0, x=None, st=None) == 0
    assert h(dt=9) == -2
    assert h(n=-1) == -3
    assert h(x=None) == -1
    assert h(dx=None) == -1
    assert h(st=None) == -1
    assert h(chunk=0) == -3
    assert h(depth=0) == -3
    assert h(depth=9) == -3
    assert h(bytes=need - 1) == -7          # staging too small
    assert h(st=ST + 16) == -7              # staging not 256-byte aligned
    assert h(y=HX + 64) == -5               # y inside x
    assert h(dx=HDY) == -5                  # dx over dy
    assert h(dx=HY + 32) == -5              # outputs overlap each other


def test_import_fails_loudly_without_the_library(tmp_path):
    pkg = os.path.join(ROOT, "gate_up_swiglu_gb300")
    dst = tmp_path / "gate_up_swiglu_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
    code = "import gate_up_swiglu_gb300"
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0
    assert "libswiglu.so is not built" in r.stderr
