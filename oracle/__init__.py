"""The oracle: a plain fp64 CPU statement of the fused gate-up SwiGLU.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``gate_up_swiglu_gb300``) never imports it and shares no code with
it.

``swiglu_oracle.c`` holds the arithmetic (cited there); this module compiles it
with gcc into ``oracle/_build/liboracle_swiglu.so`` and marshals torch CPU
tensors to it.  Parity status: forward and both backward variants are pinned by
``tests/test_oracle.py`` (closed forms, the Lambert-W stationary point,
finite differences, torch float64 autograd on the two-tensor formulation,
brute-force rounding checks and planted-mistake tests).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swiglu_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_swiglu.so")

F32, BF16, F64 = 0, 1, 2
_CODE = {torch.float32: F32, torch.bfloat16: BF16, torch.float64: F64}

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C source into a shared library; return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_library()
    return _LIB


def load(path: str = None):
    """Load (building first if needed) the oracle library and declare its calls."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_swiglu_fwd.argtypes = [vp, vp, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_swiglu_fwd.restype = ctypes.c_int
        lib.oracle_swiglu_bwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_swiglu_bwd.restype = ctypes.c_int
        lib.oracle_silu_mul_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_silu_mul_fwd.restype = ctypes.c_int
        lib.oracle_silu_mul_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                            ctypes.c_int]
        lib.oracle_silu_mul_bwd.restype = ctypes.c_int
        lib.oracle_swiglu_weighted_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_swiglu_weighted_fwd.restype = ctypes.c_int
        lib.oracle_swiglu_weighted_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                   ctypes.c_int]
        lib.oracle_swiglu_weighted_bwd.restype = ctypes.c_int
        lib.oracle_swiglu_bias_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_swiglu_bias_fwd.restype = ctypes.c_int
        lib.oracle_swiglu_bias_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                               ctypes.c_int]
        lib.oracle_swiglu_bias_bwd.restype = ctypes.c_int
        lib.oracle_swiglu_weighted_bias_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64,
                                                        ctypes.c_int]
        lib.oracle_swiglu_weighted_bias_fwd.restype = ctypes.c_int
        lib.oracle_swiglu_weighted_bias_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64,
                                                        i64, i64, i64, ctypes.c_int]
        lib.oracle_swiglu_weighted_bias_bwd.restype = ctypes.c_int
        lib.oracle_fc1_swiglu_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_int]
        lib.oracle_fc1_swiglu_fwd.restype = ctypes.c_int
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        if path is None:
            _lib = lib
        return lib


def _rowmajor(t: torch.Tensor, name: str) -> None:
    if t.device.type != "cpu":
        raise ValueError(f"oracle: {name} must be a CPU tensor")
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"oracle: {name} must be 2D with unit column stride")


def fwd(x: torch.Tensor, y: torch.Tensor = None, lib=None) -> torch.Tensor:
    """y[r, j] = silu(x[r, j]) * x[r, n + j], rounded once to x's dtype."""
    lib = lib or load()
    _rowmajor(x, "x")
    rows, two_n = x.shape
    n = two_n // 2
    if y is None:
        y = torch.empty((rows, n), dtype=x.dtype)
    _rowmajor(y, "y")
    rc = lib.oracle_swiglu_fwd(x.data_ptr(), y.data_ptr(), rows, n, x.stride(0), y.stride(0),
                               _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_fwd rejected its arguments")
    return y


def bwd(dy: torch.Tensor, x: torch.Tensor, dx: torch.Tensor = None, lib=None) -> torch.Tensor:
    """dx[:, :n] = d(gate), dx[:, n:] = d(up); pass dx=x for the in-place form."""
    lib = lib or load()
    _rowmajor(x, "x")
    _rowmajor(dy, "dy")
    rows, two_n = x.shape
    n = two_n // 2
    if dx is None:
        dx = torch.empty((rows, 2 * n), dtype=x.dtype)
    _rowmajor(dx, "dx")
    rc = lib.oracle_swiglu_bwd(dy.data_ptr(), x.data_ptr(), dx.data_ptr(), rows, n, dy.stride(0),
                               x.stride(0), dx.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_bwd rejected its arguments")
    return dx


def silu_mul_fwd(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor = None, lib=None) -> torch.Tensor:
    """Two-tensor form: c = silu(a) * b, rounded once to a's dtype."""
    lib = lib or load()
    for t, nm in ((a, "a"), (b, "b")):
        _rowmajor(t, nm)
    rows, n = a.shape
    if c is None:
        c = torch.empty((rows, n), dtype=a.dtype)
    _rowmajor(c, "c")
    rc = lib.oracle_silu_mul_fwd(a.data_ptr(), b.data_ptr(), c.data_ptr(), rows, n, a.stride(0),
                                 b.stride(0), c.stride(0), _CODE[a.dtype])
    if rc != 0:
        raise ValueError("oracle_silu_mul_fwd rejected its arguments")
    return c


def silu_mul_bwd(dc, a, b, da=None, db=None, lib=None):
    """Two-tensor form: returns (da, db); pass da=a, db=b for the in-place form."""
    lib = lib or load()
    for t, nm in ((dc, "dc"), (a, "a"), (b, "b")):
        _rowmajor(t, nm)
    rows, n = a.shape
    da = torch.empty((rows, n), dtype=a.dtype) if da is None else da
    db = torch.empty((rows, n), dtype=a.dtype) if db is None else db
    rc = lib.oracle_silu_mul_bwd(dc.data_ptr(), a.data_ptr(), b.data_ptr(), da.data_ptr(),
                                 db.data_ptr(), rows, n, dc.stride(0), a.stride(0), b.stride(0),
                                 da.stride(0), db.stride(0), _CODE[a.dtype])
    if rc != 0:
        raise ValueError("oracle_silu_mul_bwd rejected its arguments")
    return da, db


def _vec(t: torch.Tensor, name: str, dtype, size: int) -> None:
    if t.device.type != "cpu" or t.dtype != dtype or t.dim() != 1 or t.numel() != size or \
            (size > 1 and t.stride(0) != 1):
        raise ValueError(f"oracle: {name} must be a contiguous CPU {dtype} vector of {size}")


def weighted_fwd(x: torch.Tensor, w: torch.Tensor, lib=None) -> torch.Tensor:
    """y[r, j] = w[r] * silu(x[r, j]) * x[r, n + j]; w fp32 [rows]."""
    lib = lib or load()
    _rowmajor(x, "x")
    rows, two_n = x.shape
    n = two_n // 2
    _vec(w, "w", torch.float32, rows)
    y = torch.empty((rows, n), dtype=x.dtype)
    rc = lib.oracle_swiglu_weighted_fwd(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, n,
                                        x.stride(0), y.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_weighted_fwd rejected its arguments")
    return y


def weighted_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, dx: torch.Tensor = None,
                 lib=None):
    """Returns (dx, dw): dx of the weighted activation, dw fp32 [rows]."""
    lib = lib or load()
    _rowmajor(x, "x")
    _rowmajor(dy, "dy")
    rows, two_n = x.shape
    n = two_n // 2
    _vec(w, "w", torch.float32, rows)
    dx = torch.empty((rows, 2 * n), dtype=x.dtype) if dx is None else dx
    dw = torch.empty(rows, dtype=torch.float32)
    rc = lib.oracle_swiglu_weighted_bwd(dy.data_ptr(), x.data_ptr(), w.data_ptr(), dx.data_ptr(),
                                        dw.data_ptr(), rows, n, dy.stride(0), x.stride(0),
                                        dx.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_weighted_bwd rejected its arguments")
    return dx, dw


def bias_fwd(x: torch.Tensor, bias: torch.Tensor, lib=None) -> torch.Tensor:
    """y = silu(g + bias[:n]) * (u + bias[n:]); bias [2n] in x's dtype."""
    lib = lib or load()
    _rowmajor(x, "x")
    rows, two_n = x.shape
    n = two_n // 2
    _vec(bias, "bias", x.dtype, 2 * n)
    y = torch.empty((rows, n), dtype=x.dtype)
    rc = lib.oracle_swiglu_bias_fwd(x.data_ptr(), bias.data_ptr(), y.data_ptr(), rows, n,
                                    x.stride(0), y.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_bias_fwd rejected its arguments")
    return y


def bias_bwd(dy: torch.Tensor, x: torch.Tensor, bias: torch.Tensor, dx: torch.Tensor = None,
             lib=None):
    """Returns (dx, dbias): dbias[k] = sum over rows of the exact dx[:, k]."""
    lib = lib or load()
    _rowmajor(x, "x")
    _rowmajor(dy, "dy")
    rows, two_n = x.shape
    n = two_n // 2
    _vec(bias, "bias", x.dtype, 2 * n)
    dx = torch.empty((rows, 2 * n), dtype=x.dtype) if dx is None else dx
    dbias = torch.empty(2 * n, dtype=x.dtype)
    acc = torch.empty(2 * n, dtype=torch.float64)
    rc = lib.oracle_swiglu_bias_bwd(dy.data_ptr(), x.data_ptr(), bias.data_ptr(), dx.data_ptr(),
                                    dbias.data_ptr(), acc.data_ptr(), rows, n, dy.stride(0),
                                    x.stride(0), dx.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_bias_bwd rejected its arguments")
    return dx, dbias


def weighted_bias_fwd(x: torch.Tensor, bias: torch.Tensor, w: torch.Tensor, lib=None) -> torch.Tensor:
    """y = w[r] * silu(g + bias[:n]) * (u + bias[n:])."""
    lib = lib or load()
    _rowmajor(x, "x")
    rows, two_n = x.shape
    n = two_n // 2
    _vec(bias, "bias", x.dtype, 2 * n)
    _vec(w, "w", torch.float32, rows)
    y = torch.empty((rows, n), dtype=x.dtype)
    rc = lib.oracle_swiglu_weighted_bias_fwd(x.data_ptr(), bias.data_ptr(), w.data_ptr(), y.data_ptr(),
                                             rows, n, x.stride(0), y.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_weighted_bias_fwd rejected its arguments")
    return y


def weighted_bias_bwd(dy: torch.Tensor, x: torch.Tensor, bias: torch.Tensor, w: torch.Tensor,
                      lib=None):
    """Returns (dx, dbias, dw)."""
    lib = lib or load()
    _rowmajor(x, "x")
    _rowmajor(dy, "dy")
    rows, two_n = x.shape
    n = two_n // 2
    _vec(bias, "bias", x.dtype, 2 * n)
    _vec(w, "w", torch.float32, rows)
    dx = torch.empty((rows, 2 * n), dtype=x.dtype)
    dbias = torch.empty(2 * n, dtype=x.dtype)
    dw = torch.empty(rows, dtype=torch.float32)
    acc = torch.empty(2 * n, dtype=torch.float64)
    rc = lib.oracle_swiglu_weighted_bias_bwd(dy.data_ptr(), x.data_ptr(), bias.data_ptr(),
                                             w.data_ptr(), dx.data_ptr(), dbias.data_ptr(),
                                             dw.data_ptr(), acc.data_ptr(), rows, n, dy.stride(0),
                                             x.stride(0), dx.stride(0), _CODE[x.dtype])
    if rc != 0:
        raise ValueError("oracle_swiglu_weighted_bias_bwd rejected its arguments")
    return dx, dbias, dw


def fc1_swiglu_fwd(X: torch.Tensor, Wt: torch.Tensor, want_fc1: bool = False, lib=None):
    """y = silu((X W^T)[:, :n]) * (X W^T)[:, n:] with W: [2n, K]; returns y, or
    (y, fc1) with want_fc1.  Exact dot products, one rounding."""
    lib = lib or load()
    for t, nm in ((X, "X"), (Wt, "W")):
        if t.device.type != "cpu" or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"oracle: {nm} must be a contiguous 2D CPU tensor")
    M, K = X.shape
    two_n, K2 = Wt.shape
    if K2 != K or two_n % 2 or Wt.dtype != X.dtype:
        raise ValueError("oracle: W must be [2n, K] with X's K and dtype")
    n = two_n // 2
    y = torch.empty((M, n), dtype=X.dtype)
    fc1 = torch.empty((M, two_n), dtype=X.dtype) if want_fc1 else None
    acc = torch.empty(two_n, dtype=torch.float64)
    rc = lib.oracle_fc1_swiglu_fwd(X.data_ptr(), Wt.data_ptr(), y.data_ptr(),
                                   fc1.data_ptr() if want_fc1 else None, acc.data_ptr(), M, n, K,
                                   _CODE[X.dtype])
    if rc != 0:
        raise ValueError("oracle_fc1_swiglu_fwd rejected its arguments")
    return (y, fc1) if want_fc1 else y


def bf16_from_double(v: float, lib=None) -> int:
    """Bits of the bf16 nearest to ``v`` (ties to even)."""
    lib = lib or load()
    return int(lib.oracle_bf16_from_double(float(v)))
