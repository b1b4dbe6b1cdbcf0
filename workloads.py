"""Seeded synthetic inputs for the fused gate-up SwiGLU workloads.

This module only draws random numbers and lays them out; it holds none of the
SwiGLU arithmetic.  It is the one module that both the CUDA-side tests/bench
and the oracle-side tests import, so that both sides see identical bytes.

Layout (Liger-Kernel Megatron SwiGLU page, §Background): Megatron's
``linear_fc1`` produces one ``[s, b, 2n]`` (or ``[tokens, 2n]``) buffer whose
columns ``[0, n)`` are the gate and ``[n, 2n)`` the up projection.  The
workloads below are the Megatron training shape (S=2048, B=4, bf16) quoted on
that page, its large-FFN variant, a Llama-3-8B-like 2D MLP, a tiny fp32 case
and an odd-width fp32 stress case.

Recipe per workload: a ``torch.Generator`` seeded with the workload's seed
draws, in this order, the gate block ``[rows, n]``, the up block ``[rows, n]``
and ``dy`` ``[rows, n]``, all in fp32; the gate and up blocks are placed side
by side into ``x`` and every tensor is then rounded to the storage dtype (RNE,
torch's fp32->bf16 conversion).  The odd-width workload additionally writes a
fixed set of special gate values at seeded positions (see ``_inject``).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import torch

F32 = "f32"
BF16 = "bf16"
TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}
ELEM_BYTES = {F32: 4, BF16: 2}

# special gate values of the odd-width stress case: zero, tiny, the edge of
# fp32 exp range, and deep saturation on both sides
SPECIAL_GATES = (0.0, 1e-30, -1e-30, 88.0, -88.0, 1e4, -1e4)
SPECIAL_COUNT = 997


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: Tuple[int, ...]  # shape of x; last dim is 2n
    dtype: str
    seed: int
    gate: Tuple[str, float, float]  # ("normal", mean, std) or ("uniform", lo, hi)
    up: Tuple[str, float, float]
    dy: Tuple[str, float, float]
    inject: bool = False
    describe: str = ""

    @property
    def n(self) -> int:
        return self.shape[-1] // 2

    @property
    def rows(self) -> int:
        r = 1
        for d in self.shape[:-1]:
            r *= d
        return r

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    def fwd_bytes(self, rows: Optional[int] = None) -> int:
        """Algorithmic HBM bytes of one forward: read g and u, write y."""
        return 3 * self.n * (self.rows if rows is None else rows) * self.elem_bytes

    def bwd_bytes(self, rows: Optional[int] = None) -> int:
        """Algorithmic HBM bytes of one backward: read dy, g, u; write dg, du."""
        return 5 * self.n * (self.rows if rows is None else rows) * self.elem_bytes


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_f32", (16, 2, 512), F32, 0, ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
                 ("normal", 0.0, 1.0), describe="x [S=16, B=2, 2n=512] fp32, n=256"),
        Workload("megatron_4096_bf16", (2048, 4, 8192), BF16, 1, ("normal", 0.0, 1.0),
                 ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
                 describe="x [S=2048, B=4, 2n=8192] bf16, ffn_local=4096"),
        Workload("large_32768_bf16", (2048, 4, 65536), BF16, 2, ("normal", 0.0, 1.0),
                 ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
                 describe="x [S=2048, B=4, 2n=65536] bf16, ffn_local=32768 (1 GiB input)"),
        Workload("llama_14336_bf16_2d", (8192, 28672), BF16, 3, ("normal", 0.0, 2.0),
                 ("normal", 0.0, 1.0), ("normal", 0.0, 0.5),
                 describe="x [tokens=8192, 2n=28672] bf16, ffn_local=14336"),
        Workload("odd_5503_f32", (1000, 3, 11006), F32, 4, ("normal", 0.0, 8.0),
                 ("uniform", -4.0, 4.0), ("normal", 0.0, 1.0), inject=True,
                 describe="x [S=1000, B=3, 2n=11006] fp32, ffn_local=5503, special gates injected"),
    )
}

# the workload the headline timing is quoted on
HEADLINE = "large_32768_bf16"


def _draw(gen: torch.Generator, spec, shape, device) -> torch.Tensor:
    kind, a, b = spec
    if kind == "normal":
        t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if b != 1.0:
            t.mul_(b)
        if a != 0.0:
            t.add_(a)
        return t
    if kind == "uniform":
        t = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return t.mul_(b - a).add_(a)
    raise ValueError(kind)


def _inject(gate: torch.Tensor, seed: int) -> None:
    """Write each special gate value at SPECIAL_COUNT seeded positions of the
    gate block, and at the last columns of its first and last rows."""
    rows, n = gate.shape
    total = rows * n
    count = min(SPECIAL_COUNT, max(1, total // (4 * len(SPECIAL_GATES))))
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(total, generator=g)[: count * len(SPECIAL_GATES)].to(gate.device)
    flat = gate.view(-1)
    for k, v in enumerate(SPECIAL_GATES):
        flat[perm[k * count:(k + 1) * count]] = v
    # tail columns n-1, n-2, ... of the first and last rows
    for k, v in enumerate(SPECIAL_GATES):
        col = n - 1 - k
        if col >= 0:
            gate[0, col] = v
            gate[rows - 1, col] = v


def make_inputs(w: Workload, device="cpu", rows: Optional[int] = None,
                x_row_stride: Optional[int] = None):
    """Return ``(x, dy)`` for workload ``w`` as 2D ``[rows, 2n]`` / ``[rows, n]``
    views in the workload's storage dtype.

    ``rows`` overrides the row count (a prefix-sized case of the same
    distributions).  ``x_row_stride`` (elements, >= 2n) places x inside a wider
    buffer so that the row stride differs from 2n; the padding holds NaN.
    Generation happens on ``device`` with a generator of that device seeded
    with the workload's seed, so CPU and CUDA draws differ from each other but
    are each reproducible.
    """
    rows = w.rows if rows is None else rows
    n = w.n
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    gate = _draw(gen, w.gate, (rows, n), dev)
    up = _draw(gen, w.up, (rows, n), dev)
    dy = _draw(gen, w.dy, (rows, n), dev)
    if w.inject and rows > 0 and n > 0:
        _inject(gate, w.seed)
    tdt = TORCH_DTYPE[w.dtype]
    sx = 2 * n if x_row_stride is None else x_row_stride
    assert sx >= 2 * n
    buf = torch.full((rows, sx), float("nan"), dtype=tdt, device=dev)
    buf[:, :n] = gate.to(tdt)
    buf[:, n:2 * n] = up.to(tdt)
    del gate, up
    x = buf[:, : 2 * n]
    return x, dy.to(tdt)


def as_3d(t: torch.Tensor, w: Workload) -> torch.Tensor:
    """View a contiguous 2D ``[rows, k]`` tensor with the workload's leading dims."""
    if len(w.shape) == 2:
        return t
    return t.view(*w.shape[:-1], t.shape[-1])
