"""Every form, forward and backward, against the oracle for each pack class,
at 2048 rows: enough rows that every row group of the bias tile kernel holds
many of them (the random-shape tests stop at 257 rows).

The widths follow from n and the storage type (fresh, aligned buffers):
  bf16 n = 4100 (n = 4 mod 8)   8-byte packs: bias forms on the cp.async ring
  fp32 n = 2050 (n = 2 mod 4)   8-byte packs: bias forms on 1024-column tiles
  bf16 n = 4098 (n = 2 mod 4)   4-byte packs: row segments of two elements
  bf16 n = 4097 (odd)           2-byte packs: row segments of one element
  fp32 n = 2051 (odd)           4-byte packs: row segments of one element
  bf16 n = 4096                 16-byte packs (the reference point)
Every output is compared with the oracle element by element at the
tolerances of tests/helpers.py; the reductions (dbias, dw) against the
summation bound of the bias tests; and every in-place backward must give the
out-of-place bits.
"""
import pytest
import torch

import oracle
from helpers import assert_parity

pytestmark = pytest.mark.gpu

ROWS = 2048
CASES = [(torch.bfloat16, 4100), (torch.float32, 2050), (torch.bfloat16, 4098),
         (torch.bfloat16, 4097), (torch.float32, 2051), (torch.bfloat16, 4096)]


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def _inputs(dt, n, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(ROWS, 2 * n, generator=g) * 3).to(dt)
    dy = torch.randn(ROWS, n, generator=g).to(dt)
    bias = (torch.randn(2 * n, generator=g) * 0.5).to(dt)
    w = torch.rand(ROWS, generator=g)
    return x, dy, bias, w


@pytest.mark.parametrize("dt,n", CASES, ids=[f"{str(d).split('.')[-1]}-n{n}" for d, n in CASES])
def test_pack_class_every_form(sw, dt, n):
    from test_bias_weighted_gpu import _bias_depth, _wb_dw_depth, assert_reduction

    x_c, dy_c, b_c, w_c = _inputs(dt, n, n)
    x, dy, bias, w = x_c.cuda(), dy_c.cuda(), b_c.cuda(), w_c.cuda()
    what = f"{dt} [{ROWS}, 2 x {n}]"

    # forward, every form
    assert_parity(sw.swiglu_gateup_fwd(x), oracle.fwd(x_c), f"{what} fwd")
    assert_parity(sw.swiglu_gateup_bias_fwd(x, bias), oracle.bias_fwd(x_c, b_c), f"{what} bias fwd")
    assert_parity(sw.swiglu_gateup_weighted_fwd(x, w), oracle.weighted_fwd(x_c, w_c), f"{what} weighted fwd")
    assert_parity(sw.swiglu_gateup_weighted_bias_fwd(x, bias, w), oracle.weighted_bias_fwd(x_c, b_c, w_c),
                  f"{what} weighted bias fwd")

    # plain backward, out of place and in place
    dx = sw.swiglu_gateup_bwd(dy, x)
    assert_parity(dx, oracle.bwd(dy_c, x_c), f"{what} bwd")
    xi = x.clone()
    sw.swiglu_gateup_bwd(dy, xi, in_place=True)
    assert torch.equal(xi, dx), f"{what}: in place differs from out of place"

    x64, dy64, b64 = x_c.double(), dy_c.double(), b_c.double()

    # bias backward: dx elementwise, dbias against the exact column sums
    dxb, db = sw.swiglu_gateup_bias_bwd(dy, x, bias)
    assert_parity(dxb, oracle.bias_bwd(dy_c, x_c, b_c)[0], f"{what} bias dx")
    dx64, db64 = oracle.bias_bwd(dy64, x64, b64)
    assert_reduction(db, db64, dx64.abs().sum(0), _bias_depth(ROWS, n), f"{what} dbias", elem=dt,
                     count=ROWS)

    # per-token weights: dx elementwise, dw against the exact row sums
    dxw, dw = sw.swiglu_gateup_weighted_bwd(dy, x, w)
    assert_parity(dxw, oracle.weighted_bwd(dy_c, x_c, w_c)[0], f"{what} weighted dx")
    t = dy64 * oracle.fwd(x64)
    assert_reduction(dw, t.sum(1), t.abs().sum(1), n / 256 + 13, f"{what} weighted dw", elem=dt, count=n)

    # weights and bias: dx elementwise, dbias and dw against the exact sums
    dxwb, dbw, dww = sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, w)
    assert_parity(dxwb, oracle.weighted_bias_bwd(dy_c, x_c, b_c, w_c)[0], f"{what} weighted bias dx")
    dx64, db64, _ = oracle.weighted_bias_bwd(dy64, x64, b64, w_c)
    assert_reduction(dbw, db64, dx64.abs().sum(0), _bias_depth(ROWS, n, weighted=True),
                     f"{what} weighted bias dbias", elem=dt, count=ROWS)
    t = dy64 * oracle.bias_fwd(x64, b64)
    assert_reduction(dww, t.sum(1), t.abs().sum(1), _wb_dw_depth(n), f"{what} weighted bias dw", elem=dt,
                     count=n)

    # the in-place forms (coherent loads, dx over x) give the out-of-place bits
    for name, call, ref in (
            ("weighted", lambda xi: sw.swiglu_gateup_weighted_bwd(dy, xi, w, in_place=True), (dxw, dw)),
            ("bias", lambda xi: sw.swiglu_gateup_bias_bwd(dy, xi, bias, in_place=True), (dxb, db)),
            ("weighted bias", lambda xi: sw.swiglu_gateup_weighted_bias_bwd(dy, xi, bias, w, in_place=True),
             (dxwb, dbw, dww))):
        xi = x.clone()
        got = call(xi)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"{what}: in-place {name} backward differs from out of place"
        assert torch.equal(xi, ref[0]), f"{what}: in-place {name} dx not written over x"
