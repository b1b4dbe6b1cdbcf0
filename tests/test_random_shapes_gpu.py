"""Seeded random shapes through every form, against the oracle.

Each case draws rows, n, the row-stride padding of every tensor, a common
base misalignment and the dtype, so the calls land on every pack width
(32 / 16 / 8 bytes, the row-segment kernels of narrow packs), on one-pass and
persistent grids, and on ragged last packs, segments and column tiles.  Every
output is compared with the oracle element by element (tolerances of
tests/helpers.py; reductions against the summation bound of the bias tests),
in place must equal out of place bit for bit, and the guard bands around
every written buffer must keep their sentinel.
"""
import pytest
import torch

import oracle
from helpers import assert_bitwise, assert_parity

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def _draw_case(i):
    g = torch.Generator().manual_seed(1000 + i)
    pick = lambda seq: seq[int(torch.randint(len(seq), (1,), generator=g))]  # noqa: E731
    dt = pick([torch.bfloat16, torch.float32])
    rows = pick([1, 2, 3, 7, 33, 130, 257])
    n = pick([1, 2, 3, 5, 8, 31, 64, 100, 1000, 1001, 2048, 2050, 4104, 5503])
    pads = [pick([0, 0, 0, 1, 2, 8, 16]) for _ in range(5)]  # x, y, dy, dx, misc
    mis = pick([0, 0, 1, 2, 3])
    return dt, rows, n, pads, mis


def _guarded(rows, cols, pad, mis, dt, fill, guard=40):
    stride = cols + pad
    buf = torch.full((guard + mis + rows * stride + guard,), fill, dtype=dt, device="cuda")
    off = guard + mis
    return buf, buf[off: off + rows * stride].view(rows, stride)[:, :cols]


def _same_guards(buf, view, ref, fill, what):
    view.fill_(fill)
    assert_bitwise(buf, ref, f"{what}: guard bands or padding written")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_every_form(sw, i):
    from test_bias_weighted_gpu import _bias_depth, _wb_dw_depth, assert_reduction

    dt, rows, n, (px, py, pdy, pdx, _), mis = _draw_case(i)
    g = torch.Generator().manual_seed(2000 + i)
    x_c = (torch.randn(rows, 2 * n, generator=g) * 3).to(dt)
    dy_c = torch.randn(rows, n, generator=g).to(dt)
    b_c = (torch.randn(2 * n, generator=g) * 0.5).to(dt)
    w_c = torch.rand(rows, generator=g)
    what = f"case {i}: {dt} rows {rows} n {n} pads {px},{py},{pdy},{pdx} misalign {mis}"

    xb, x = _guarded(rows, 2 * n, px, mis, dt, float("nan"))
    dyb, dy = _guarded(rows, n, pdy, mis, dt, float("nan"))
    yb, y = _guarded(rows, n, py, mis, dt, -5.0)
    dxb, dx = _guarded(rows, 2 * n, pdx, mis, dt, -5.0)
    x.copy_(x_c)
    dy.copy_(dy_c)
    xb0, yb0, dxb0 = xb.clone(), yb.clone(), dxb.clone()
    bias, wts = b_c.cuda(), w_c.cuda()

    # plain forward, backward, in-place backward
    sw.swiglu_gateup_fwd(x, y)
    sw.swiglu_gateup_bwd(dy, x, dx)
    torch.cuda.synchronize()
    assert_parity(y, oracle.fwd(x_c), f"{what} fwd")
    ref_dx = oracle.bwd(dy_c, x_c)
    assert_parity(dx, ref_dx, f"{what} bwd")
    dx_plain = dx.clone()
    _same_guards(yb, y, yb0, -5.0, f"{what} fwd")
    _same_guards(dxb, dx, dxb0, -5.0, f"{what} bwd")
    assert_bitwise(xb, xb0, f"{what}: x changed")

    # two-tensor form on the halves of x (separate operands, same strides)
    c = sw.swiglu_silu_mul_fwd(x[:, :n], x[:, n:])
    da, db_ = sw.swiglu_silu_mul_bwd(dy, x[:, :n], x[:, n:])
    torch.cuda.synchronize()
    assert_parity(c, oracle.fwd(x_c), f"{what} two-tensor fwd")
    assert_bitwise(torch.cat([da, db_], 1), dx_plain, f"{what} two-tensor bwd = fused")

    # bias, weights, both: forward into the guarded y, backward into the guarded dx
    sw.swiglu_gateup_bias_fwd(x, bias, y)
    torch.cuda.synchronize()
    assert_parity(y, oracle.bias_fwd(x_c, b_c), f"{what} bias fwd")
    _same_guards(yb, y, yb0, -5.0, f"{what} bias fwd")
    _, dbias = sw.swiglu_gateup_bias_bwd(dy, x, bias, dx)
    torch.cuda.synchronize()
    assert_parity(dx, oracle.bias_bwd(dy_c, x_c, b_c)[0], f"{what} bias dx")
    dx64, db64 = oracle.bias_bwd(dy_c.double(), x_c.double(), b_c.double())
    assert_reduction(dbias, db64, dx64.abs().sum(0), _bias_depth(rows, n), f"{what} dbias",
                     elem=dt, count=rows)
    _same_guards(dxb, dx, dxb0, -5.0, f"{what} bias bwd")

    sw.swiglu_gateup_weighted_fwd(x, wts, y)
    torch.cuda.synchronize()
    assert_parity(y, oracle.weighted_fwd(x_c, w_c), f"{what} weighted fwd")
    _same_guards(yb, y, yb0, -5.0, f"{what} weighted fwd")
    _, dw = sw.swiglu_gateup_weighted_bwd(dy, x, wts, dx)
    torch.cuda.synchronize()
    assert_parity(dx, oracle.weighted_bwd(dy_c, x_c, w_c)[0], f"{what} weighted dx")
    t = dy_c.double() * oracle.fwd(x_c.double())
    assert_reduction(dw, t.sum(1), t.abs().sum(1), n / 256 + 13, f"{what} weighted dw", elem=dt,
                     count=n)
    _same_guards(dxb, dx, dxb0, -5.0, f"{what} weighted bwd")

    sw.swiglu_gateup_weighted_bias_fwd(x, bias, wts, y)
    torch.cuda.synchronize()
    assert_parity(y, oracle.weighted_bias_fwd(x_c, b_c, w_c), f"{what} weighted bias fwd")
    _same_guards(yb, y, yb0, -5.0, f"{what} weighted bias fwd")
    _, dbw, dww = sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts, dx)
    torch.cuda.synchronize()
    assert_parity(dx, oracle.weighted_bias_bwd(dy_c, x_c, b_c, w_c)[0], f"{what} weighted bias dx")
    dx64, db64, _ = oracle.weighted_bias_bwd(dy_c.double(), x_c.double(), b_c.double(), w_c)
    assert_reduction(dbw, db64, dx64.abs().sum(0), _bias_depth(rows, n, weighted=True),
                     f"{what} weighted bias dbias", elem=dt, count=rows)
    t = dy_c.double() * oracle.bias_fwd(x_c.double(), b_c.double())
    assert_reduction(dww, t.sum(1), t.abs().sum(1), _wb_dw_depth(n), f"{what} weighted bias dw",
                     elem=dt, count=n)
    _same_guards(dxb, dx, dxb0, -5.0, f"{what} weighted bias bwd")

    # in place over the guarded x: the plain backward's bits, and x's padding
    # and guards untouched
    sw.swiglu_gateup_bwd(dy, x, in_place=True)
    torch.cuda.synchronize()
    assert_bitwise(x, dx_plain, f"{what} in place = out of place")
    x.copy_(x_c)
    assert_bitwise(xb, xb0, f"{what}: x guard bands after in place")
