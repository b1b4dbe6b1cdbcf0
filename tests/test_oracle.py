"""Pins of the oracle against facts that do not come from the oracle itself.

Every pin is a function ``pin_*(lib)`` so that ``test_planted_mistakes`` can run
the same pins against deliberately broken copies of the oracle (compiled from a
mutated copy of its C source in a temporary directory) and show that each
plausible mistake is caught by at least one pin.

What each pin rests on:
  * closed forms: silu(0) = 0 and silu'(0) = 1/2; saturation silu(g) -> g for
    g >> 0 and silu(g) -> g*exp(g) for g << 0;
  * the stationary point of silu, g0 = -1 - W(1/e) (scipy's Lambert W), where
    silu'(g0) = 0 and silu has its minimum;
  * central finite differences of the oracle's own forward in float64;
  * torch float64 autograd through F.silu(a) * b on the chunked halves -- the
    two-tensor formulation of the same activation (Liger-Kernel Megatron SwiGLU
    page, §Background: gate = columns [0, n), up = columns [n, 2n));
  * brute-force nearest-even rounding over every bf16 value, and torch's own
    fp32 -> bf16 and fp64 -> fp32 conversions.
"""
import math
import os
import shutil
import tempfile

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle

F64 = torch.float64


def _rand(shape, seed, scale=1.0, dtype=F64):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale).to(dtype)


# ---------------------------------------------------------------- helpers ---

def _bf16_bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF


def _bf16_from_bits(bits) -> torch.Tensor:
    b = torch.as_tensor(np.asarray(bits, dtype=np.uint16).view(np.int16))
    return b.view(torch.bfloat16)


def _all_finite_bf16() -> torch.Tensor:
    """Every finite bf16 value, as float64, one per bit pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = _bf16_from_bits(bits).to(F64)
    return v[torch.isfinite(v)]


def _brute_bf16(v: float) -> int:
    """Bits of the nearest bf16 to v, ties to even, by search over all bf16."""
    if math.isnan(v):
        raise ValueError
    vals = _BF16_TABLE_VALS
    bits = _BF16_TABLE_BITS
    a = abs(v)
    i = int(np.searchsorted(vals, a))
    cands = []
    for k in (i - 1, i):
        if 0 <= k < len(vals):
            cands.append((abs(vals[k] - a), bits[k]))
    best = min(c[0] for c in cands)
    ties = [b for d, b in cands if d == best]
    if len(ties) > 1:
        ties = [b for b in ties if (b & 1) == 0]
    out = ties[0]
    if math.copysign(1.0, v) < 0:
        out |= 0x8000
    return out


def _bf16_table():
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint32).astype(np.uint16)  # +0 .. max finite
    vals = _bf16_from_bits(bits).to(F64).numpy()
    # 2^128 stands for +inf (bits 0x7F80, even): overflow rounds there
    vals = np.append(vals, 2.0 ** 128)
    bits = np.append(bits.astype(np.int64), 0x7F80)
    return vals, bits


_BF16_TABLE_VALS, _BF16_TABLE_BITS = _bf16_table()


# ------------------------------------------------------------------- pins ---

def pin_zero_gate(lib):
    """silu(0) = 0, silu'(0) = 1/2: y = 0, d(gate) = dy*u/2, d(up) = 0."""
    rows, n = 4, 5
    x = _rand((rows, 2 * n), 1)
    x[:, :n] = 0.0
    dy = _rand((rows, n), 2)
    y = oracle.fwd(x, lib=lib)
    assert torch.equal(y, torch.zeros_like(y))
    dx = oracle.bwd(dy, x, lib=lib)
    assert torch.allclose(dx[:, :n], 0.5 * dy * x[:, n:], rtol=1e-15, atol=0)
    assert torch.equal(dx[:, n:], torch.zeros_like(dy))


def pin_saturation(lib):
    """|g| > 20: silu(g) -> g (relative gap e^-g) and silu(g) -> g e^g (relative
    gap e^g); silu'(g) -> 1 and -> 0 likewise."""
    n = 6
    gp = torch.tensor([20.5, 25.0, 30.0, 40.0, 100.0, 1e4], dtype=F64)
    gm = -gp
    u = torch.tensor([1.5, -2.0, 0.75, 3.0, -1.0, 0.5], dtype=F64)
    dy = torch.tensor([0.5, 1.25, -2.0, 1.0, 3.0, -0.25], dtype=F64)
    for g in (gp, gm):
        x = torch.cat([g, u]).view(1, 2 * n)
        y = oracle.fwd(x, lib=lib)[0]
        dx = oracle.bwd(dy.view(1, n), x, lib=lib)[0]
        if g[0] > 0:
            assert torch.allclose(y, g * u, rtol=3e-9, atol=0)
            assert torch.allclose(dx[:n], dy * u, rtol=3e-9 * 1e4, atol=0)
            assert torch.allclose(dx[n:], dy * g, rtol=3e-9, atol=0)
        else:
            lim = g * torch.exp(g) * u  # leading term of g*u*e^g/(1+e^g)
            assert torch.allclose(y, lim, rtol=3e-9, atol=1e-300)
            assert torch.all(y.abs() < 1e-7)
            # silu'(g) ~ e^g (1 + g) as g -> -inf
            lim_d = dy * u * torch.exp(g) * (1 + g)
            assert torch.allclose(dx[:n], lim_d, rtol=1e-7, atol=1e-300)
            assert torch.allclose(dx[n:], dy * g * torch.exp(g), rtol=3e-9, atol=1e-300)


def pin_stationary_point(lib):
    """silu'(g) = 0 at g0 = -1 - W(1/e) (from 1 + g + e^g = 0), a minimum."""
    g0 = -1.0 - float(scipy.special.lambertw(1.0 / math.e).real)
    assert abs(g0 + 1.2784645427610738) < 1e-14
    gs = torch.tensor([g0, g0 - 1e-3, g0 + 1e-3], dtype=F64)
    u = torch.ones(3, dtype=F64)
    x = torch.cat([gs, u]).view(1, 6)
    dx = oracle.bwd(torch.ones(1, 3, dtype=F64), x, lib=lib)[0]
    assert abs(float(dx[0])) < 1e-15
    assert float(dx[1]) < 0 < float(dx[2])
    # silu''(g0) = s (1 - s) (2 + g0 (1 - 2 s)), s = sigma(g0): slope of d(gate)
    s = 1.0 / (1.0 + math.exp(-g0))
    curv = s * (1 - s) * (2 + g0 * (1 - 2 * s))
    assert abs((float(dx[2]) - float(dx[1])) / 2e-3 - curv) < 1e-5
    # the minimum value of silu, g0 * sigma(g0) = -W(1/e) - 1 + ... = 1 + g0
    y = oracle.fwd(x, lib=lib)[0]
    assert abs(float(y[0]) - (g0 + 1.0)) < 1e-15


def pin_finite_differences(lib):
    """d(gate), d(up) equal dy times central differences of the forward (fp64)."""
    for seed, (rows, n) in enumerate([(8, 7), (3, 13), (1, 1)]):
        x = _rand((rows, 2 * n), 10 + seed, 3.0)
        dy = _rand((rows, n), 20 + seed)
        dx = oracle.bwd(dy, x, lib=lib)
        num = torch.empty_like(x)
        for c in range(2 * n):
            h = 1e-6 * torch.clamp(x[:, c].abs(), min=1.0)
            xp, xm = x.clone(), x.clone()
            xp[:, c] += h
            xm[:, c] -= h
            yp, ym = oracle.fwd(xp, lib=lib), oracle.fwd(xm, lib=lib)
            j = c % n
            num[:, c] = dy[:, j] * (yp[:, j] - ym[:, j]) / (2 * h)
        assert torch.allclose(dx, num, rtol=1e-6, atol=1e-9), (dx - num).abs().max()


def pin_torch_two_tensor(lib):
    """Forward and backward equal torch float64 autograd of F.silu(a) * b on the
    chunked halves (ragged sizes)."""
    for seed, (rows, n) in enumerate([(37, 61), (5, 1), (2, 300)]):
        x = _rand((rows, 2 * n), 30 + seed, 4.0)
        dy = _rand((rows, n), 40 + seed)
        a, b = [t.clone().requires_grad_(True) for t in x.chunk(2, dim=-1)]
        y_ref = F.silu(a) * b
        y_ref.backward(dy)
        y = oracle.fwd(x, lib=lib)
        dx = oracle.bwd(dy, x, lib=lib)
        assert torch.allclose(y, y_ref.detach(), rtol=1e-13, atol=1e-300)
        assert torch.allclose(dx[:, :n], a.grad, rtol=1e-12, atol=1e-14)
        assert torch.allclose(dx[:, n:], b.grad, rtol=1e-13, atol=1e-300)


def pin_bf16_rounding_brute(lib):
    """Direct fp64 -> bf16 rounding equals nearest-even found by brute force,
    on values built to sit at, next to and between rounding midpoints."""
    rng = np.random.default_rng(5)
    vals = list(rng.standard_normal(300) * 10.0 ** rng.integers(-40, 39, 300))
    fin = _all_finite_bf16().numpy()
    pos = np.unique(np.abs(fin))
    picks = rng.choice(len(pos) - 1, 200, replace=False)
    for i in picks:
        lo, hi = pos[i], pos[i + 1]
        mid = (lo + hi) / 2
        vals += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), -mid, lo + (hi - lo) * 0.3]
    # a midpoint whose fp32 rounding would round it up first (double rounding trap)
    vals += [1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -8 - 2.0 ** -30, 1.0 + 2.0 ** -8]
    # subnormal range, overflow edge, zeros
    mx = float(pos[-1])
    vals += [2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -134, 2.0 ** -135, 3 * 2.0 ** -134,
             mx, mx + 2.0 ** 119, mx + 2.0 ** 119 - 2.0 ** 90, 1e39, -1e39, 0.0, -0.0]
    for v in vals:
        assert oracle.bf16_from_double(v, lib=lib) == _brute_bf16(float(v)), v


def pin_rounding_matches_torch(lib):
    """fp32 outputs are the fp64 results rounded by torch; for inputs whose fp64
    result is an fp32 value, bf16 rounding equals torch's fp32 -> bf16."""
    rows, n = 9, 33
    x = _rand((rows, 2 * n), 50, 3.0)
    dy = _rand((rows, n), 51)
    y64 = oracle.fwd(x, lib=lib)
    dx64 = oracle.bwd(dy, x, lib=lib)
    xf, dyf = x.float(), dy.float()
    y32 = oracle.fwd(xf, lib=lib)
    dx32 = oracle.bwd(dyf, xf, lib=lib)
    y64b = oracle.fwd(xf.double(), lib=lib)
    dx64b = oracle.bwd(dyf.double(), xf.double(), lib=lib)
    assert torch.equal(y32, y64b.float())
    assert torch.equal(dx32, dx64b.float())
    del y64, dx64
    f = _rand((4096,), 52, 100.0).float().double()
    got = [oracle.bf16_from_double(float(v), lib=lib) for v in f]
    ref = _bf16_bits(f.float().to(torch.bfloat16)).tolist()
    assert got == ref


def pin_bf16_all_gates(lib):
    """bf16 forward over every finite bf16 gate value equals torch's float64
    F.silu(g) * u rounded to nearest-even bf16."""
    g = _all_finite_bf16()
    m = g.numel()
    us = [1.0, -0.375, 3.140625]
    x = torch.empty((len(us), 2 * m), dtype=torch.bfloat16)
    for i, u in enumerate(us):
        x[i, :m] = g.to(torch.bfloat16)
        x[i, m:] = u
    y = oracle.fwd(x, lib=lib)
    got = _bf16_bits(y)
    for i, u in enumerate(us):
        ref64 = F.silu(g) * u
        # exact rounding of the fp64 value; checked against brute force above
        ref = torch.tensor([oracle.bf16_from_double(float(v), lib=lib) for v in ref64[::97]])
        assert torch.equal(got[i, ::97], ref)
        # whole sweep: within half a bf16 spacing of the fp64 value
        yv = y[i].to(F64)
        spacing = torch.clamp(yv.abs(), min=2.0 ** -126) * 2.0 ** -7
        assert torch.all((yv - ref64).abs() <= 0.5 * spacing * (1 + 1e-12))


def pin_strided_layouts(lib):
    """Row strides wider than the rows give the same values and leave the
    padding untouched; the in-place backward equals the out-of-place one."""
    rows, n = 6, 10
    x = _rand((rows, 2 * n), 60).float()
    dy = _rand((rows, n), 61).float()
    y = oracle.fwd(x, lib=lib)
    dx = oracle.bwd(dy, x, lib=lib)
    xb = torch.full((rows, 2 * n + 3), float("nan"))
    xb[:, :2 * n] = x
    yb = torch.full((rows, n + 5), -7.0)
    oracle.fwd(xb[:, :2 * n], yb[:, :n], lib=lib)
    assert torch.equal(yb[:, :n], y) and torch.all(yb[:, n:] == -7.0)
    dyb = torch.full((rows, n + 1), float("nan"))
    dyb[:, :n] = dy
    dxb = torch.full((rows, 2 * n + 2), -9.0)
    oracle.bwd(dyb[:, :n], xb[:, :2 * n], dxb[:, :2 * n], lib=lib)
    assert torch.equal(dxb[:, :2 * n], dx) and torch.all(dxb[:, 2 * n:] == -9.0)
    xi = xb.clone()
    oracle.bwd(dyb[:, :n], xi[:, :2 * n], xi[:, :2 * n], lib=lib)
    assert torch.equal(xi[:, :2 * n], dx) and torch.all(torch.isnan(xi[:, 2 * n:]))


def pin_two_tensor_form(lib):
    """The two-tensor entry points equal torch float64 autograd of
    F.silu(a) * b on separately strided buffers, and equal the fused form on
    the halves of one buffer."""
    for seed, (rows, n) in enumerate([(13, 29), (4, 1), (3, 257)]):
        a = _rand((rows, n + 3), 70 + seed, 4.0)[:, :n]
        b = _rand((rows, n + 5), 80 + seed, 2.0)[:, :n]
        dc = _rand((rows, n), 90 + seed)
        at, bt = a.clone().requires_grad_(True), b.clone().requires_grad_(True)
        ref = F.silu(at) * bt
        ref.backward(dc)
        c = oracle.silu_mul_fwd(a, b, torch.empty(rows, n + 4, dtype=F64)[:, :n], lib=lib)
        da, db = oracle.silu_mul_bwd(dc, a, b, torch.empty(rows, n + 2, dtype=F64)[:, :n],
                                     torch.empty(rows, n + 7, dtype=F64)[:, :n], lib=lib)
        assert torch.allclose(c, ref.detach(), rtol=1e-13, atol=1e-300)
        assert torch.allclose(da, at.grad, rtol=1e-12, atol=1e-14)
        assert torch.allclose(db, bt.grad, rtol=1e-13, atol=1e-300)
        x = torch.cat([a, b], dim=1).float()
        dcf = dc.float()
        af, bf = x[:, :n].contiguous(), x[:, n:].contiguous()
        assert torch.equal(oracle.silu_mul_fwd(af, bf, lib=lib), oracle.fwd(x, lib=lib))
        da2, db2 = oracle.silu_mul_bwd(dcf, af, bf, lib=lib)
        assert torch.equal(torch.cat([da2, db2], 1), oracle.bwd(dcf, x, lib=lib))
        # in place over a and b
        ai, bi = af.clone(), bf.clone()
        oracle.silu_mul_bwd(dcf, ai, bi, ai, bi, lib=lib)
        assert torch.equal(ai, da2) and torch.equal(bi, db2)


def pin_weighted(lib):
    """Per-token weights: torch float64 autograd of w[:, None] * F.silu(a) * b
    gives y, the input gradient and dw; w = 1 reduces to the plain form."""
    for seed, (rows, n) in enumerate([(11, 37), (3, 1), (2, 500)]):
        x = _rand((rows, 2 * n), 100 + seed, 3.0)
        dy = _rand((rows, n), 110 + seed)
        w = _rand((rows,), 120 + seed).float()
        a, b = [t.clone().requires_grad_(True) for t in x.chunk(2, dim=-1)]
        wt = w.double().clone().requires_grad_(True)
        ref = wt[:, None] * F.silu(a) * b
        ref.backward(dy)
        y = oracle.weighted_fwd(x, w, lib=lib)
        dx, dw = oracle.weighted_bwd(dy, x, w, lib=lib)
        assert torch.allclose(y, ref.detach(), rtol=1e-13, atol=1e-300)
        assert torch.allclose(dx[:, :n], a.grad, rtol=1e-12, atol=1e-14)
        assert torch.allclose(dx[:, n:], b.grad, rtol=1e-12, atol=1e-300)
        assert torch.allclose(dw.double(), wt.grad, rtol=2e-7, atol=1e-30)
        one = torch.ones(rows)
        assert torch.equal(oracle.weighted_fwd(x, one, lib=lib), oracle.fwd(x, lib=lib))
        assert torch.equal(oracle.weighted_bwd(dy, x, one, lib=lib)[0], oracle.bwd(dy, x, lib=lib))


def pin_bias(lib):
    """Bias: torch float64 autograd of F.silu(a + bias[:n]) * (b + bias[n:])
    gives y, dx and the bias gradient (summed over rows); zero bias reduces to
    the plain form."""
    for seed, (rows, n) in enumerate([(13, 21), (1, 3), (40, 7)]):
        x = _rand((rows, 2 * n), 130 + seed, 3.0)
        dy = _rand((rows, n), 140 + seed)
        bias = _rand((2 * n,), 150 + seed)
        a, b = [t.clone().requires_grad_(True) for t in x.chunk(2, dim=-1)]
        bt = bias.clone().requires_grad_(True)
        ref = F.silu(a + bt[:n]) * (b + bt[n:])
        ref.backward(dy)
        y = oracle.bias_fwd(x, bias, lib=lib)
        dx, db = oracle.bias_bwd(dy, x, bias, lib=lib)
        assert torch.allclose(y, ref.detach(), rtol=1e-12, atol=1e-300)
        assert torch.allclose(dx[:, :n], a.grad, rtol=1e-11, atol=1e-13)
        assert torch.allclose(dx[:, n:], b.grad, rtol=1e-12, atol=1e-300)
        assert torch.allclose(db, bt.grad, rtol=1e-11, atol=1e-13)
        zero = torch.zeros(2 * n, dtype=F64)
        assert torch.equal(oracle.bias_fwd(x, zero, lib=lib), oracle.fwd(x, lib=lib))
        assert torch.equal(oracle.bias_bwd(dy, x, zero, lib=lib)[0], oracle.bwd(dy, x, lib=lib))
        # bf16: dbias is the once-rounded sum of the unrounded gradients
        xb, dyb, bb = x.to(torch.bfloat16), dy.to(torch.bfloat16), bias.to(torch.bfloat16)
        dx64, db64 = oracle.bias_bwd(dyb.double(), xb.double(), bb.double(), lib=lib)
        dxb, dbb = oracle.bias_bwd(dyb, xb, bb, lib=lib)
        assert torch.equal(_bf16_bits(dbb),
                           torch.tensor([oracle.bf16_from_double(float(v), lib=lib) for v in db64]))


def pin_weighted_bias(lib):
    """Weights and bias together: torch float64 autograd of
    w[:, None] * F.silu(a + bias[:n]) * (b + bias[n:]) gives y and the gradients
    of x, bias and w; w = 1 gives the bias-only form, zero bias the
    weighted-only form."""
    for seed, (rows, n) in enumerate([(9, 13), (1, 2), (30, 5)]):
        x = _rand((rows, 2 * n), 190 + seed, 3.0)
        dy = _rand((rows, n), 200 + seed)
        bias = _rand((2 * n,), 210 + seed)
        w = _rand((rows,), 220 + seed).float()
        a, b = [t.clone().requires_grad_(True) for t in x.chunk(2, dim=-1)]
        bt = bias.clone().requires_grad_(True)
        wt = w.double().clone().requires_grad_(True)
        ref = wt[:, None] * F.silu(a + bt[:n]) * (b + bt[n:])
        ref.backward(dy)
        y = oracle.weighted_bias_fwd(x, bias, w, lib=lib)
        dx, db, dw = oracle.weighted_bias_bwd(dy, x, bias, w, lib=lib)
        assert torch.allclose(y, ref.detach(), rtol=1e-12, atol=1e-300)
        assert torch.allclose(dx[:, :n], a.grad, rtol=1e-11, atol=1e-13)
        assert torch.allclose(dx[:, n:], b.grad, rtol=1e-11, atol=1e-300)
        assert torch.allclose(db, bt.grad, rtol=1e-11, atol=1e-13)
        assert torch.allclose(dw.double(), wt.grad, rtol=2e-7, atol=1e-30)
        one, zero = torch.ones(rows), torch.zeros(2 * n, dtype=F64)
        assert torch.equal(oracle.weighted_bias_fwd(x, bias, one, lib=lib), oracle.bias_fwd(x, bias, lib=lib))
        assert torch.equal(oracle.weighted_bias_bwd(dy, x, bias, one, lib=lib)[1],
                           oracle.bias_bwd(dy, x, bias, lib=lib)[1])
        assert torch.equal(oracle.weighted_bias_bwd(dy, x, zero, w, lib=lib)[2],
                           oracle.weighted_bwd(dy, x, w, lib=lib)[1])


def pin_fc1_swiglu(lib):
    """linear_fc1 then the activation: equals torch float64 matmul X @ W.T
    followed by F.silu(gate) * up, and its fc1 output equals that matmul; with
    W = [I; I] (K = n) it reduces to the plain form on x = [X, X]."""
    for seed, (M, n, K) in enumerate([(7, 5, 9), (3, 16, 64), (1, 1, 1)]):
        X = _rand((M, K), 160 + seed)
        Wt = _rand((2 * n, K), 170 + seed, 0.3)
        y, fc1 = oracle.fc1_swiglu_fwd(X, Wt, want_fc1=True, lib=lib)
        ref = X @ Wt.T
        assert torch.allclose(fc1, ref, rtol=1e-12, atol=1e-14)
        assert torch.allclose(y, F.silu(ref[:, :n]) * ref[:, n:], rtol=1e-12, atol=1e-14)
    n = 6
    X = _rand((4, n), 180)
    Wt = torch.cat([torch.eye(n), torch.eye(n)]).double()
    x2 = torch.cat([X, X], 1)
    assert torch.equal(oracle.fc1_swiglu_fwd(X, Wt, lib=lib), oracle.fwd(x2, lib=lib))


PINS = [pin_zero_gate, pin_saturation, pin_stationary_point, pin_finite_differences,
        pin_torch_two_tensor, pin_bf16_rounding_brute, pin_rounding_matches_torch,
        pin_bf16_all_gates, pin_strided_layouts, pin_two_tensor_form, pin_weighted, pin_bias,
        pin_fc1_swiglu, pin_weighted_bias]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# ------------------------------------------------------ planted mistakes ---

# Each mutation is a plausible slip in the oracle's C source: a transposed
# operand, a wrong sign, a dropped term, a wrong index or stride, a wrong
# rounding.  Every one must make at least one pin fail.
MUTATIONS = {
    "gate_up_swapped": ("double g = load_elem(x, r * sx + j, dtype);\n            double u = load_elem(x, r * sx + n + j, dtype);\n            store_elem(y",
                        "double u = load_elem(x, r * sx + j, dtype);\n            double g = load_elem(x, r * sx + n + j, dtype);\n            store_elem(y"),
    "sigmoid_sign": ("exp(-g)", "exp(g)"),
    "dropped_g_term": ("(1.0 + g * (1.0 - s))", "(1.0 + (1.0 - s))"),
    "dgate_without_s": ("*dgate = dy * u * s * (", "*dgate = dy * u * ("),
    "dup_without_g": ("*dup = dy * g * s;", "*dup = dy * s;"),
    "wrong_one_minus": ("(1.0 - s))", "(s - 1.0))"),
    "outputs_swapped": ("store_elem(dx, r * sdx + j, dtype, dg);\n            store_elem(dx, r * sdx + n + j, dtype, du);",
                        "store_elem(dx, r * sdx + j, dtype, du);\n            store_elem(dx, r * sdx + n + j, dtype, dg);"),
    "y_stride_ignored": ("store_elem(y, r * sy + j", "store_elem(y, r * n + j"),
    "x_stride_is_2n": ("double g = load_elem(x, r * sx + j, dtype);\n            double u = load_elem(x, r * sx + n + j, dtype);\n            double dg",
                       "double g = load_elem(x, r * 2 * n + j, dtype);\n            double u = load_elem(x, r * 2 * n + n + j, dtype);\n            double dg"),
    "bf16_truncates": ("nearbyint(a / spacing)", "floor(a / spacing)"),
    "bf16_via_fp32": ("uint16_t h = oracle_bf16_from_double(v);",
                      "uint16_t h = oracle_bf16_from_double((double)(float)v);"),
    "bf16_subnormal_spacing": ("if (k < -126) k = -126;", ""),
    "f32_truncates": ("float f = (float)v; /* IEEE",
                      "float f = (float)v; if (fabs((double)f) > fabs(v)) f = nextafterf(f, 0.0f); /* IEEE"),
    "dy_stride_ignored": ("load_elem(dy, r * sdy + j", "load_elem(dy, r * n + j"),
    "two_tensor_a_b_swapped": ("double g = load_elem(a, r * sa + j, dtype);\n            double u = load_elem(b, r * sb + j, dtype);\n            store_elem(c",
                               "double g = load_elem(b, r * sb + j, dtype);\n            double u = load_elem(a, r * sa + j, dtype);\n            store_elem(c"),
    "two_tensor_db_stride": ("store_elem(db, r * sdb + j", "store_elem(db, r * sda + j"),
    "weighted_dw_without_u": ("acc += d * swiglu_fwd_pair(g, u);", "acc += d * swiglu_fwd_pair(g, 1.0);"),
    "weighted_grad_unscaled": ("swiglu_bwd_pair(d * wr, g, u, &dg, &du);", "swiglu_bwd_pair(d, g, u, &dg, &du);"),
    "bias_halves_swapped": ("double u = load_elem(x, r * sx + n + j, dtype) + load_elem(bias, n + j, dtype);\n            store_elem(y",
                            "double u = load_elem(x, r * sx + n + j, dtype) + load_elem(bias, j, dtype);\n            store_elem(y"),
    "weighted_bias_dw_unshifted": ("sum += d * swiglu_fwd_pair(g, u);\n            swiglu_bwd_pair(d * wr, g, u, &dg, &du);\n            acc[j] += dg;",
                                   "sum += d * swiglu_fwd_pair(g - load_elem(bias, j, dtype), u);\n            swiglu_bwd_pair(d * wr, g, u, &dg, &du);\n            acc[j] += dg;"),
    "fc1_weight_transposed": ("load_elem(W, c * K + k, dtype)", "load_elem(W, k * 2 * n + c, dtype)"),
    "fc1_halves_swapped": ("store_elem(y, m * n + j, dtype, swiglu_fwd_pair(acc[j], acc[n + j]));",
                           "store_elem(y, m * n + j, dtype, swiglu_fwd_pair(acc[n + j], acc[j]));"),
    "dbias_last_row_only": ("            acc[j] += dg;\n            acc[n + j] += du;", "            acc[j] = dg;\n            acc[n + j] = du;"),
}


def _build_mutant(tmpdir, name):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation {name} does not apply"
    msrc = os.path.join(tmpdir, f"{name}.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    out = os.path.join(tmpdir, f"lib{name}.so")
    oracle.compile_library(msrc, out)
    return oracle.load(out)


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes(name, mutant_dir):
    lib = _build_mutant(mutant_dir, name)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
