"""Comparison rules shared by the CUDA parity tests (no SwiGLU arithmetic here).

Tolerances, stated once:
  * fp32: |gpu - oracle| <= max(2e-6 * |oracle|, 1e-7), oracle = the fp64
    result rounded once to fp32;
  * bf16: at most one bf16 step apart, measured on the sign-magnitude ordering
    of the bit patterns (+0 and -0 coincide);
  * NaN must meet NaN (not graded for value).
The in-place and out-of-place backward must agree bit for bit.
"""
import torch

F32_RTOL = 2e-6
F32_ATOL = 1e-7
BF16_ULPS = 1


def bf16_ordered(t: torch.Tensor) -> torch.Tensor:
    b = t.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF
    mag = b & 0x7FFF
    return torch.where(b & 0x8000 != 0, -mag, mag)


def mismatches(gpu: torch.Tensor, ref: torch.Tensor) -> torch.Tensor:
    """Boolean mask of elements outside tolerance (both tensors on the CPU)."""
    assert gpu.shape == ref.shape and gpu.dtype == ref.dtype
    nan_g, nan_r = torch.isnan(gpu), torch.isnan(ref)
    if gpu.dtype == torch.float32:
        g, r = gpu.double(), ref.double()
        tol = torch.clamp(F32_RTOL * r.abs(), min=F32_ATOL)
        bad = (g - r).abs() > tol
        # equal infinities are fine
        bad &= ~(torch.isinf(g) & torch.isinf(r) & (g == r))
    elif gpu.dtype == torch.bfloat16:
        bad = (bf16_ordered(gpu) - bf16_ordered(ref)).abs() > BF16_ULPS
    else:
        raise TypeError(gpu.dtype)
    return (bad & ~(nan_g & nan_r)) | (nan_g ^ nan_r)


def assert_parity(gpu: torch.Tensor, ref: torch.Tensor, what: str = "", extra=None):
    gpu = gpu.cpu()
    bad = mismatches(gpu, ref)
    nbad = int(bad.sum())
    if nbad:
        idx = bad.nonzero()[:8].tolist()
        detail = [(i, float(gpu[tuple(i)]), float(ref[tuple(i)])) for i in idx]
        if extra is not None:
            detail = [(i, g, r, float(extra[tuple(i)])) for (i, g, r) in detail]
        raise AssertionError(f"{what}: {nbad} of {gpu.numel()} elements out of tolerance; "
                             f"first (index, gpu, oracle[, input]): {detail}")


def assert_bitwise(a: torch.Tensor, b: torch.Tensor, what: str = ""):
    assert a.shape == b.shape and a.dtype == b.dtype
    ia = a.contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32)
    neq = int((ia != ib).sum())
    assert neq == 0, f"{what}: {neq} elements differ bitwise"
