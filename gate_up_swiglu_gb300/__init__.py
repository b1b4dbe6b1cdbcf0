"""Python binding of libswiglu, the GB300 fused gate-up SwiGLU.

Argument marshalling only: every element of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/swiglu.h``.  There is no CPU or
eager fallback: if ``libswiglu.so`` has not been built, importing this package
raises.

    y  = swiglu_gateup_fwd(x)                       # x: [..., 2n] CUDA tensor
    dx = swiglu_gateup_bwd(dy, x)                   # new [..., 2n] gradient
    swiglu_gateup_bwd(dy, x, in_place=True)         # gradient written over x

``x`` is Megatron's ``linear_fc1`` output, gate in columns ``[0, n)`` and up in
``[n, 2n)`` (Liger-Kernel Megatron SwiGLU page, §Background).  2D
``[tokens, 2n]`` and 3D ``[s, b, 2n]`` tensors are flattened to rows without a
copy (§Megatron feature compatibility).
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libswiglu.so")

SWIGLU_F32, SWIGLU_BF16 = 0, 1
_DTYPE = {torch.float32: SWIGLU_F32, torch.bfloat16: SWIGLU_BF16}

STATUS = {0: "SWIGLU_OK", -1: "SWIGLU_ERR_NULL", -2: "SWIGLU_ERR_DTYPE", -3: "SWIGLU_ERR_SHAPE",
          -4: "SWIGLU_ERR_STRIDE", -5: "SWIGLU_ERR_ALIAS", -6: "SWIGLU_ERR_CUDA",
          -7: "SWIGLU_ERR_WORKSPACE"}

# every symbol include/swiglu.h declares
EXPORTS = ("swiglu_gateup_fwd", "swiglu_gateup_bwd", "swiglu_silu_mul_fwd", "swiglu_silu_mul_bwd",
           "swiglu_gateup_weighted_fwd", "swiglu_gateup_weighted_bwd", "swiglu_gateup_bias_fwd",
           "swiglu_gateup_bias_bwd_workspace_size", "swiglu_gateup_bias_bwd",
           "swiglu_gateup_weighted_bias_fwd", "swiglu_gateup_weighted_bias_bwd_workspace_size",
           "swiglu_gateup_weighted_bias_bwd", "swiglu_gateup_bias_bwd_noalloc", "swiglu_fc1_fwd",
           "swiglu_fc1_timeout_flag", "swiglu_gateup_fwd_bwd_host_staging_size",
           "swiglu_gateup_fwd_bwd_host", "swiglu_status_string", "swiglu_last_cuda_error",
           "swiglu_abi_version")


class SwigluError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libswiglu.so is not built ({LIB_PATH} missing); build it with "
            "`python gate_up_swiglu_gb300/build.py` or __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.swiglu_gateup_fwd.argtypes = [vp, vp, i64, i64, i64, i64, i32, vp]
    lib.swiglu_gateup_fwd.restype = i32
    lib.swiglu_gateup_bwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, vp]
    lib.swiglu_gateup_bwd.restype = i32
    lib.swiglu_silu_mul_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
    lib.swiglu_silu_mul_fwd.restype = i32
    lib.swiglu_silu_mul_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i32, vp]
    lib.swiglu_silu_mul_bwd.restype = i32
    lib.swiglu_gateup_weighted_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp]
    lib.swiglu_gateup_weighted_fwd.restype = i32
    lib.swiglu_gateup_weighted_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, i32,
                                               vp]
    lib.swiglu_gateup_weighted_bwd.restype = i32
    lib.swiglu_gateup_bias_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp]
    lib.swiglu_gateup_bias_fwd.restype = i32
    lib.swiglu_gateup_bias_bwd_workspace_size.argtypes = [i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.swiglu_gateup_bias_bwd_workspace_size.restype = i32
    lib.swiglu_gateup_bias_bwd.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i64, i64, i64,
                                           i64, i64, i32, i32, vp]
    lib.swiglu_gateup_bias_bwd.restype = i32
    lib.swiglu_gateup_bias_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32,
                                                   i32, vp]
    lib.swiglu_gateup_bias_bwd_noalloc.restype = i32
    lib.swiglu_gateup_weighted_bias_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i32, vp]
    lib.swiglu_gateup_weighted_bias_fwd.restype = i32
    lib.swiglu_gateup_weighted_bias_bwd_workspace_size.argtypes = [i64, i64,
                                                                   ctypes.POINTER(ctypes.c_size_t)]
    lib.swiglu_gateup_weighted_bias_bwd_workspace_size.restype = i32
    lib.swiglu_gateup_weighted_bias_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                                    i64, i64, i64, i64, i64, i32, i32, vp]
    lib.swiglu_gateup_weighted_bias_bwd.restype = i32
    lib.swiglu_fc1_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp]
    lib.swiglu_fc1_fwd.restype = i32
    lib.swiglu_fc1_timeout_flag.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.swiglu_fc1_timeout_flag.restype = i32
    lib.swiglu_gateup_fwd_bwd_host_staging_size.argtypes = [i64, i64, i32, i32,
                                                            ctypes.POINTER(ctypes.c_size_t)]
    lib.swiglu_gateup_fwd_bwd_host_staging_size.restype = i32
    lib.swiglu_gateup_fwd_bwd_host.argtypes = [vp, vp, vp, vp, i64, i64, i32, vp, ctypes.c_size_t,
                                               i64, i32, vp, vp, vp]
    lib.swiglu_gateup_fwd_bwd_host.restype = i32
    lib.swiglu_status_string.argtypes = [i32]
    lib.swiglu_status_string.restype = ctypes.c_char_p
    lib.swiglu_last_cuda_error.argtypes = []
    lib.swiglu_last_cuda_error.restype = i32
    lib.swiglu_abi_version.argtypes = []
    lib.swiglu_abi_version.restype = i32
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.swiglu_status_string(int(status)).decode()


def _rows_view(t: torch.Tensor, name: str):
    """(rows, cols, row_stride) of a [..., cols] tensor whose leading dims
    flatten to evenly strided rows of unit-stride elements, without a copy."""
    if t.dim() < 1:
        raise ValueError(f"{name} must have at least one dimension")
    cols = t.shape[-1]
    if cols > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    lead = t.shape[:-1]
    rows = 1
    for d in lead:
        rows *= d
    if t.dim() == 1:
        return 1, cols, cols
    # the leading dims must collapse into one stride: stride[i] = stride[i+1] * shape[i+1]
    stride = t.stride(-2)
    for i in range(t.dim() - 3, -1, -1):
        if t.shape[i] > 1 and t.stride(i) != t.stride(i + 1) * t.shape[i + 1]:
            raise ValueError(f"{name}: leading dimensions do not flatten to evenly strided rows")
    if rows <= 1:
        stride = max(stride, cols)
    return rows, cols, stride


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(t: torch.Tensor, stream) -> int:
    """The cudaStream_t to launch on: `stream` (a torch stream or a raw
    handle), else the current stream of t's device."""
    if stream is None:
        if _raw_stream is not None:
            return int(_raw_stream(t.device.index))
        stream = torch.cuda.current_stream(t.device)
    return int(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


def _on_device(dev):
    """Make `dev` current for the call (the library launches on the current
    device); a no-op when it already is, which is the common case and saves
    the context switch on every call."""
    if dev.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def _check_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("libswiglu operates on CUDA tensors only")
    dev = ts[0].device
    for t in ts[1:]:
        if t.device != dev:
            raise ValueError("all tensors must be on the same CUDA device")
    if ts[0].dtype not in _DTYPE or any(t.dtype != ts[0].dtype for t in ts):
        raise ValueError("tensors must all be float32 or all bfloat16")


def swiglu_gateup_fwd(x: torch.Tensor, y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """y[..., j] = silu(x[..., j]) * x[..., n + j]; returns y ([..., n])."""
    if y is None:
        y = torch.empty((*x.shape[:-1], x.shape[-1] // 2), dtype=x.dtype, device=x.device)
    _check_cuda(x, y)
    if x.shape[-1] % 2:
        raise ValueError("x's last dimension must be even (gate and up halves)")
    rows, two_n, sx = _rows_view(x, "x")
    yrows, n, sy = _rows_view(y, "y")
    if yrows != rows or n * 2 != two_n:
        raise ValueError("y must be [..., n] with the rows of x")
    with _on_device(x.device):
        st = lib.swiglu_gateup_fwd(x.data_ptr(), y.data_ptr(), rows, n, sx, sy, _DTYPE[x.dtype],
                                   _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_fwd")
    return y


def swiglu_gateup_bwd(dy: torch.Tensor, x: torch.Tensor, dx: torch.Tensor = None,
                      in_place: bool = False, stream=None) -> torch.Tensor:
    """Gradient of silu(gate) * up w.r.t. x; d gate in [..., :n], d up in [..., n:].

    ``in_place=True`` writes the gradient over ``x`` and returns ``x``."""
    if in_place:
        if dx is not None and dx.data_ptr() != x.data_ptr():
            raise ValueError("in_place=True writes over x; dx must be None or x")
        dx = x
    elif dx is None:
        dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    _check_cuda(dy, x, dx)
    rows, two_n, sx = _rows_view(x, "x")
    dyrows, n, sdy = _rows_view(dy, "dy")
    dxrows, dxcols, sdx = _rows_view(dx, "dx")
    if two_n % 2 or dyrows != rows or n * 2 != two_n or dxrows != rows or dxcols != two_n:
        raise ValueError("shapes must be dy [..., n], x [..., 2n], dx [..., 2n] over the same rows")
    with _on_device(x.device):
        st = lib.swiglu_gateup_bwd(dy.data_ptr(), x.data_ptr(), dx.data_ptr(), rows, n, sdy, sx, sdx,
                                   _DTYPE[x.dtype], 1 if in_place else 0, _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_bwd")
    return dx


def swiglu_silu_mul_fwd(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor = None,
                        stream=None) -> torch.Tensor:
    """Two-tensor form: c = silu(a) * b for [..., n] tensors a, b."""
    if c is None:
        c = torch.empty(a.shape, dtype=a.dtype, device=a.device)
    _check_cuda(a, b, c)
    rows, n, sa = _rows_view(a, "a")
    (rb, nb, sb), (rc, nc, sc) = _rows_view(b, "b"), _rows_view(c, "c")
    if (rb, nb) != (rows, n) or (rc, nc) != (rows, n):
        raise ValueError("a, b and c must have the same [..., n] shape")
    with _on_device(a.device):
        st = lib.swiglu_silu_mul_fwd(a.data_ptr(), b.data_ptr(), c.data_ptr(), rows, n, sa, sb, sc,
                                     _DTYPE[a.dtype], _stream_handle(a, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_silu_mul_fwd")
    return c


def swiglu_silu_mul_bwd(dc: torch.Tensor, a: torch.Tensor, b: torch.Tensor, da=None, db=None,
                        in_place: bool = False, stream=None):
    """Two-tensor form: returns (da, db).  ``in_place=True`` writes da over a
    and db over b."""
    if in_place:
        da, db = a, b
    da = torch.empty(a.shape, dtype=a.dtype, device=a.device) if da is None else da
    db = torch.empty(b.shape, dtype=b.dtype, device=b.device) if db is None else db
    _check_cuda(dc, a, b, da, db)
    views = [_rows_view(t, nm) for t, nm in ((dc, "dc"), (a, "a"), (b, "b"), (da, "da"), (db, "db"))]
    rows, n = views[1][0], views[1][1]
    if any((v[0], v[1]) != (rows, n) for v in views):
        raise ValueError("dc, a, b, da and db must have the same [..., n] shape")
    with _on_device(a.device):
        st = lib.swiglu_silu_mul_bwd(dc.data_ptr(), a.data_ptr(), b.data_ptr(), da.data_ptr(),
                                     db.data_ptr(), rows, n, *[v[2] for v in views],
                                     _DTYPE[a.dtype], _stream_handle(a, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_silu_mul_bwd")
    return da, db


def _vector(t: torch.Tensor, name: str, numel: int, dtype) -> None:
    if t.dtype != dtype or t.numel() != numel or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of {numel} elements")


def swiglu_gateup_weighted_fwd(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor = None,
                               stream=None) -> torch.Tensor:
    """y = w[row] * silu(gate) * up; w: fp32, one weight per row of x."""
    if y is None:
        y = torch.empty((*x.shape[:-1], x.shape[-1] // 2), dtype=x.dtype, device=x.device)
    _check_cuda(x, y)
    rows, two_n, sx = _rows_view(x, "x")
    yrows, n, sy = _rows_view(y, "y")
    if yrows != rows or 2 * n != two_n:
        raise ValueError("y must be [..., n] with the rows of x")
    _vector(w, "w", rows, torch.float32)
    with _on_device(x.device):
        st = lib.swiglu_gateup_weighted_fwd(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, n, sx,
                                            sy, _DTYPE[x.dtype], _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_weighted_fwd")
    return y


def swiglu_gateup_weighted_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, dx=None,
                               dw=None, in_place: bool = False, stream=None):
    """Returns (dx, dw): the input gradient and the fp32 per-row weight gradient."""
    if in_place:
        dx = x
    elif dx is None:
        dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    rows, two_n, sx = _rows_view(x, "x")
    if dw is None:
        dw = torch.empty(w.shape, dtype=torch.float32, device=x.device)
    _check_cuda(dy, x, dx)
    dyrows, n, sdy = _rows_view(dy, "dy")
    dxrows, dxcols, sdx = _rows_view(dx, "dx")
    if dyrows != rows or 2 * n != two_n or dxrows != rows or dxcols != two_n:
        raise ValueError("shapes must be dy [..., n], x [..., 2n], dx [..., 2n] over the same rows")
    _vector(w, "w", rows, torch.float32)
    _vector(dw, "dw", rows, torch.float32)
    with _on_device(x.device):
        st = lib.swiglu_gateup_weighted_bwd(dy.data_ptr(), x.data_ptr(), w.data_ptr(), dx.data_ptr(),
                                            dw.data_ptr(), rows, n, sdy, sx, sdx, _DTYPE[x.dtype],
                                            1 if in_place else 0, _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_weighted_bwd")
    return dx, dw


def swiglu_gateup_bias_fwd(x: torch.Tensor, bias: torch.Tensor, y: torch.Tensor = None,
                           stream=None) -> torch.Tensor:
    """y = silu(gate + bias[:n]) * (up + bias[n:]); bias: [2n] in x's dtype."""
    if y is None:
        y = torch.empty((*x.shape[:-1], x.shape[-1] // 2), dtype=x.dtype, device=x.device)
    _check_cuda(x, y, bias)
    rows, two_n, sx = _rows_view(x, "x")
    yrows, n, sy = _rows_view(y, "y")
    if yrows != rows or 2 * n != two_n:
        raise ValueError("y must be [..., n] with the rows of x")
    _vector(bias, "bias", two_n, x.dtype)
    with _on_device(x.device):
        st = lib.swiglu_gateup_bias_fwd(x.data_ptr(), bias.data_ptr(), y.data_ptr(), rows, n, sx, sy,
                                        _DTYPE[x.dtype], _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_bias_fwd")
    return y


def bias_bwd_workspace_bytes(rows: int, n: int) -> int:
    """Workspace the bias backward needs on the current device."""
    out = ctypes.c_size_t(0)
    st = lib.swiglu_gateup_bias_bwd_workspace_size(rows, n, ctypes.byref(out))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_bias_bwd_workspace_size")
    return int(out.value)


def swiglu_gateup_bias_bwd(dy: torch.Tensor, x: torch.Tensor, bias: torch.Tensor, dx=None,
                           dbias=None, workspace: torch.Tensor = None, in_place: bool = False,
                           stream=None):
    """Returns (dx, dbias).  `workspace` (a CUDA byte tensor of at least
    bias_bwd_workspace_bytes(rows, n)) is allocated here when not given."""
    if in_place:
        dx = x
    elif dx is None:
        dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    if dbias is None:
        dbias = torch.empty_like(bias)
    _check_cuda(dy, x, dx, bias, dbias)
    rows, two_n, sx = _rows_view(x, "x")
    dyrows, n, sdy = _rows_view(dy, "dy")
    dxrows, dxcols, sdx = _rows_view(dx, "dx")
    if dyrows != rows or 2 * n != two_n or dxrows != rows or dxcols != two_n:
        raise ValueError("shapes must be dy [..., n], x [..., 2n], dx [..., 2n] over the same rows")
    _vector(bias, "bias", two_n, x.dtype)
    _vector(dbias, "dbias", two_n, x.dtype)
    with _on_device(x.device):
        if workspace is None:
            workspace = torch.empty(max(16, bias_bwd_workspace_bytes(rows, n)), dtype=torch.uint8,
                                    device=x.device)
        st = lib.swiglu_gateup_bias_bwd(dy.data_ptr(), x.data_ptr(), bias.data_ptr(), dx.data_ptr(),
                                        dbias.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                        rows, n, sdy, sx, sdx, _DTYPE[x.dtype], 1 if in_place else 0,
                                        _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_bias_bwd")
    return dx, dbias


def swiglu_gateup_weighted_bias_fwd(x: torch.Tensor, bias: torch.Tensor, w: torch.Tensor,
                                    y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """y = w[row] * silu(gate + bias[:n]) * (up + bias[n:]); bias: [2n] in x's
    dtype, w: fp32, one weight per row of x."""
    if y is None:
        y = torch.empty((*x.shape[:-1], x.shape[-1] // 2), dtype=x.dtype, device=x.device)
    _check_cuda(x, y, bias)
    rows, two_n, sx = _rows_view(x, "x")
    yrows, n, sy = _rows_view(y, "y")
    if yrows != rows or 2 * n != two_n:
        raise ValueError("y must be [..., n] with the rows of x")
    _vector(bias, "bias", two_n, x.dtype)
    _vector(w, "w", rows, torch.float32)
    with _on_device(x.device):
        st = lib.swiglu_gateup_weighted_bias_fwd(x.data_ptr(), bias.data_ptr(), w.data_ptr(),
                                                 y.data_ptr(), rows, n, sx, sy, _DTYPE[x.dtype],
                                                 _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_weighted_bias_fwd")
    return y


def weighted_bias_bwd_workspace_bytes(rows: int, n: int) -> int:
    """Workspace the weighted bias backward needs on the current device."""
    out = ctypes.c_size_t(0)
    st = lib.swiglu_gateup_weighted_bias_bwd_workspace_size(rows, n, ctypes.byref(out))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_weighted_bias_bwd_workspace_size")
    return int(out.value)


def swiglu_gateup_weighted_bias_bwd(dy: torch.Tensor, x: torch.Tensor, bias: torch.Tensor,
                                    w: torch.Tensor, dx=None, dbias=None, dw=None,
                                    workspace: torch.Tensor = None, in_place: bool = False,
                                    stream=None):
    """Returns (dx, dbias, dw).  `workspace` (a CUDA byte tensor of at least
    weighted_bias_bwd_workspace_bytes(rows, n)) is allocated here when not
    given."""
    if in_place:
        dx = x
    elif dx is None:
        dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    if dbias is None:
        dbias = torch.empty_like(bias)
    if dw is None:
        dw = torch.empty(w.shape, dtype=torch.float32, device=x.device)
    _check_cuda(dy, x, dx, bias, dbias)
    rows, two_n, sx = _rows_view(x, "x")
    dyrows, n, sdy = _rows_view(dy, "dy")
    dxrows, dxcols, sdx = _rows_view(dx, "dx")
    if dyrows != rows or 2 * n != two_n or dxrows != rows or dxcols != two_n:
        raise ValueError("shapes must be dy [..., n], x [..., 2n], dx [..., 2n] over the same rows")
    _vector(bias, "bias", two_n, x.dtype)
    _vector(dbias, "dbias", two_n, x.dtype)
    _vector(w, "w", rows, torch.float32)
    _vector(dw, "dw", rows, torch.float32)
    with _on_device(x.device):
        if workspace is None:
            workspace = torch.empty(max(16, weighted_bias_bwd_workspace_bytes(rows, n)),
                                    dtype=torch.uint8, device=x.device)
        st = lib.swiglu_gateup_weighted_bias_bwd(
            dy.data_ptr(), x.data_ptr(), bias.data_ptr(), w.data_ptr(), dx.data_ptr(),
            dbias.data_ptr(), dw.data_ptr(), workspace.data_ptr(), workspace.numel(), rows, n, sdy,
            sx, sdx, _DTYPE[x.dtype], 1 if in_place else 0, _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_weighted_bias_bwd")
    return dx, dbias, dw


def swiglu_fc1_fwd(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor = None,
                   x_out: torch.Tensor = None, return_fc1: bool = False, stream=None):
    """y = silu((x W^T)[..., :n]) * (x W^T)[..., n:] on the tensor cores, with W
    the [2n, K] fc1 weight.  With return_fc1 (or an x_out given) the bf16 fc1
    output is stored too and (y, fc1) is returned."""
    K = x.shape[-1]
    if w.dim() != 2 or w.shape[1] != K or w.shape[0] % 2:
        raise ValueError("w must be [2n, K] with x's K")
    n = w.shape[0] // 2
    M = x.numel() // K if K else 0
    if y is None:
        y = torch.empty((*x.shape[:-1], n), dtype=x.dtype, device=x.device)
    if return_fc1 and x_out is None:
        x_out = torch.empty((*x.shape[:-1], 2 * n), dtype=x.dtype, device=x.device)
    ts = [x, w, y] + ([x_out] if x_out is not None else [])
    _check_cuda(*ts)
    if not all(t.is_contiguous() for t in ts):
        raise ValueError("swiglu_fc1_fwd needs contiguous tensors")
    with _on_device(x.device):
        st = lib.swiglu_fc1_fwd(x.data_ptr(), w.data_ptr(), y.data_ptr(),
                                x_out.data_ptr() if x_out is not None else None, M, n, K,
                                _DTYPE[x.dtype], _stream_handle(x, stream))
    if st != 0:
        raise SwigluError(st, "swiglu_fc1_fwd")
    return (y, x_out) if x_out is not None else y


def fc1_timeout_flag() -> int:
    out = ctypes.c_int(0)
    st = lib.swiglu_fc1_timeout_flag(ctypes.byref(out))
    if st != 0:
        raise SwigluError(st, "swiglu_fc1_timeout_flag")
    return int(out.value)


def host_staging_bytes(chunk_rows: int, n: int, dtype, depth: int) -> int:
    """Device staging bytes swiglu_gateup_fwd_bwd_host needs for this chunking."""
    out = ctypes.c_size_t(0)
    st = lib.swiglu_gateup_fwd_bwd_host_staging_size(int(chunk_rows), int(n), _DTYPE[dtype],
                                                     int(depth), ctypes.byref(out))
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_fwd_bwd_host_staging_size")
    return int(out.value)


def swiglu_gateup_fwd_bwd_host(x_h: torch.Tensor, dy_h: torch.Tensor, y_h: torch.Tensor,
                               dx_h: torch.Tensor, staging: torch.Tensor, chunk_rows: int,
                               depth: int, streams) -> None:
    """y_h = forward(x_h), dx_h = backward(dy_h, x_h) for contiguous 2D host
    tensors (pin them for overlap) through the device staging buffer `staging`
    (a CUDA tensor of at least host_staging_bytes(...) bytes) and the three
    CUDA streams (h2d, compute, d2h); returns once the results are in y_h and
    dx_h."""
    rows, two_n = x_h.shape
    n = two_n // 2
    for t, shape in ((x_h, (rows, 2 * n)), (dy_h, (rows, n)), (y_h, (rows, n)), (dx_h, (rows, 2 * n))):
        if t.device.type != "cpu" or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors x [rows, 2n], "
                             "dy [rows, n], y [rows, n], dx [rows, 2n]")
        if t.dtype != x_h.dtype or t.dtype not in _DTYPE:
            raise ValueError("host buffers must all be float32 or all bfloat16")
    if not staging.is_cuda:
        raise ValueError("staging must be a CUDA tensor")
    h = [int(s.cuda_stream if hasattr(s, "cuda_stream") else s) for s in streams]
    with _on_device(staging.device):
        st = lib.swiglu_gateup_fwd_bwd_host(
            x_h.data_ptr(), dy_h.data_ptr(), y_h.data_ptr(), dx_h.data_ptr(), rows, n,
            _DTYPE[x_h.dtype], staging.data_ptr(), staging.numel() * staging.element_size(),
            int(chunk_rows), int(depth), h[0], h[1], h[2])
    if st != 0:
        raise SwigluError(st, "swiglu_gateup_fwd_bwd_host")


__all__ = ["swiglu_gateup_fwd", "swiglu_gateup_bwd", "swiglu_silu_mul_fwd", "swiglu_silu_mul_bwd",
           "swiglu_gateup_weighted_fwd", "swiglu_gateup_weighted_bwd", "swiglu_gateup_bias_fwd",
           "swiglu_gateup_bias_bwd", "bias_bwd_workspace_bytes", "swiglu_gateup_weighted_bias_fwd",
           "swiglu_gateup_weighted_bias_bwd", "weighted_bias_bwd_workspace_bytes",
           "swiglu_fc1_fwd", "fc1_timeout_flag", "host_staging_bytes",
           "swiglu_gateup_fwd_bwd_host", "status_string", "SwigluError", "lib",
           "SWIGLU_F32", "SWIGLU_BF16", "EXPORTS", "LIB_PATH"]
