"""Forward + backward over buffers that live in host memory.

When the fc1 buffer and the incoming gradient are in (pinned) host memory --
offloaded activations, or a caller that keeps its tensors on the CPU side of
the Grace-Blackwell link -- copying everything in, computing, and copying
everything out leaves the link idle while the kernels run and the GPU idle
while the link works.  ``gateup_fwd_bwd_host`` instead streams row chunks
through a small ring of device buffers on three CUDA streams: the copy-in of
chunk i + 1, the kernels of chunk i and the copy-out of chunk i - 1 run at the
same time, and the two link directions are used together.

Only plumbing lives here: every element is computed by the C-ABI kernels
(``swiglu_gateup_fwd`` / ``swiglu_gateup_bwd``).
"""
from __future__ import annotations

import torch

from . import swiglu_gateup_bwd, swiglu_gateup_fwd


def default_chunk_rows(n: int, elem_bytes: int, target_bytes: int = 64 << 20) -> int:
    """Rows per chunk so one chunk's inputs (x and dy: 3n elements per row) are
    about target_bytes: large enough to run the link at full speed, small
    enough that the first and last copies, which cannot overlap, stay short."""
    return max(1, target_bytes // max(1, 3 * n * elem_bytes))


class HostPipeline:
    """Device staging buffers and streams for ``gateup_fwd_bwd_host``; keep one
    per device and reuse it across calls (it allocates once, on first use).
    ``depth`` chunks are in flight at a time."""

    def __init__(self, device, chunk_rows: int, depth: int = 3):
        self.device = torch.device(device)
        self.chunk_rows = int(chunk_rows)
        self.depth = depth
        self.h2d = torch.cuda.Stream(self.device)
        self.comp = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self._key = None
        self._bufs = None

    def _buffers(self, n: int, dtype):
        key = (n, dtype)
        if self._key != key:
            r = self.chunk_rows
            mk = lambda cols: torch.empty((r, cols), dtype=dtype, device=self.device)  # noqa: E731
            self._bufs = [dict(x=mk(2 * n), dy=mk(n), y=mk(n), dx=mk(2 * n),
                               loaded=torch.cuda.Event(), done=torch.cuda.Event(),
                               drained=torch.cuda.Event())
                          for _ in range(self.depth)]
            self._key = key
        return self._bufs


def gateup_fwd_bwd_host(x_h: torch.Tensor, dy_h: torch.Tensor, y_h: torch.Tensor,
                        dx_h: torch.Tensor, pipe: HostPipeline) -> None:
    """y_h = forward(x_h), dx_h = backward(dy_h, x_h) for 2D host tensors
    x [rows, 2n], dy [rows, n], y [rows, n], dx [rows, 2n] (pin them for
    overlap), chunk by chunk.  Returns once everything has landed in y_h and
    dx_h."""
    rows, two_n = x_h.shape
    n = two_n // 2
    for t, shape in ((x_h, (rows, 2 * n)), (dy_h, (rows, n)), (y_h, (rows, n)), (dx_h, (rows, 2 * n))):
        if t.device.type != "cpu" or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors x [rows, 2n], "
                             "dy [rows, n], y [rows, n], dx [rows, 2n]")
    bufs = pipe._buffers(n, x_h.dtype)
    cr = pipe.chunk_rows
    chunks = [(r0, min(rows, r0 + cr)) for r0 in range(0, rows, cr)]
    for i, (r0, r1) in enumerate(chunks):
        b = bufs[i % pipe.depth]
        m = r1 - r0
        # refill a slot only after its previous results have left for the host
        if i >= pipe.depth:
            pipe.h2d.wait_event(b["drained"])
        with torch.cuda.stream(pipe.h2d):
            b["x"][:m].copy_(x_h[r0:r1], non_blocking=True)
            b["dy"][:m].copy_(dy_h[r0:r1], non_blocking=True)
            b["loaded"].record(pipe.h2d)
        pipe.comp.wait_event(b["loaded"])
        with torch.cuda.stream(pipe.comp):
            swiglu_gateup_fwd(b["x"][:m], b["y"][:m], stream=pipe.comp)
            swiglu_gateup_bwd(b["dy"][:m], b["x"][:m], b["dx"][:m], stream=pipe.comp)
            b["done"].record(pipe.comp)
        pipe.d2h.wait_event(b["done"])
        with torch.cuda.stream(pipe.d2h):
            y_h[r0:r1].copy_(b["y"][:m], non_blocking=True)
            dx_h[r0:r1].copy_(b["dx"][:m], non_blocking=True)
            b["drained"].record(pipe.d2h)
    pipe.d2h.synchronize()
