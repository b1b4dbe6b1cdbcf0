"""Forward + backward over buffers that live in host memory.

``gateup_fwd_bwd_host`` is the torch-side convenience over the C-ABI call
``swiglu_gateup_fwd_bwd_host``: a ``HostPipeline`` holds the device staging
buffer and the three CUDA streams the call needs (allocated once, reused), and
the library streams row chunks through them with copies in, kernels and copies
out overlapped.  Argument marshalling only: the chunking, ordering and every
computed element are the library's.
"""
from __future__ import annotations

import torch

from . import host_staging_bytes, swiglu_gateup_fwd_bwd_host


def default_chunk_rows(n: int, elem_bytes: int, target_bytes: int = 64 << 20) -> int:
    """Rows per chunk so one chunk's inputs (x and dy: 3n elements per row) are
    about target_bytes: large enough to run the link at full speed, small
    enough that the first and last copies, which cannot overlap, stay short."""
    return max(1, target_bytes // max(1, 3 * n * elem_bytes))


class HostPipeline:
    """Device staging memory and streams for ``gateup_fwd_bwd_host``; keep one
    per device and reuse it across calls (the staging buffer is allocated on
    first use and grown only when a wider row needs it).  ``depth`` chunks are
    in flight at a time."""

    def __init__(self, device, chunk_rows: int, depth: int = 3):
        self.device = torch.device(device)
        self.chunk_rows = int(chunk_rows)
        self.depth = depth
        self.h2d = torch.cuda.Stream(self.device)
        self.comp = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self.staging = None

    def staging_for(self, n: int, dtype) -> torch.Tensor:
        need = host_staging_bytes(self.chunk_rows, n, dtype, self.depth)
        if self.staging is None or self.staging.numel() < need:
            self.staging = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.staging


def gateup_fwd_bwd_host(x_h: torch.Tensor, dy_h: torch.Tensor, y_h: torch.Tensor,
                        dx_h: torch.Tensor, pipe: HostPipeline) -> None:
    """y_h = forward(x_h), dx_h = backward(dy_h, x_h) for 2D host tensors
    x [rows, 2n], dy [rows, n], y [rows, n], dx [rows, 2n] (pin them for
    overlap).  Returns once everything has landed in y_h and dx_h."""
    n = x_h.shape[1] // 2
    staging = pipe.staging_for(n, x_h.dtype)
    swiglu_gateup_fwd_bwd_host(x_h, dy_h, y_h, dx_h, staging, pipe.chunk_rows, pipe.depth,
                               (pipe.h2d, pipe.comp, pipe.d2h))
