"""Per-token-weighted and bias variants vs the oracle, through the C ABI.

Elementwise outputs (y, dx) use the tolerances of tests/helpers.py.  The two
reductions -- dw[r] (a sum over the n columns of a row) and dbias[k] (a sum
over the rows of a column) -- are fp32 sums in a fixed order, so they are held
to the rigorous bound of such a sum: with A = sum |t| over the exact terms and
D the summation depth of the kernel (terms added one after another along the
longest chain),
    |gpu - exact| <= (D + 6) * 2^-24 * A  +  one step of the output type at |exact|.
For dw, D = n / 256 (the columns one thread adds) + 5 (warp shuffle levels) +
8 (warp partials).  For dbias, D = rows per row group + number of groups,
from the same plan the library makes (2048-column tiles, 3 CTAs per SM).
With weights and bias together, dw is summed per 2048-column tile (8 terms per
thread, then the CTA's 5 + 8 levels) and the tiles are added in order:
D = 21 + number of tiles.
"""

import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bitwise, assert_parity

pytestmark = pytest.mark.gpu
U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def _step(dtype, mag: torch.Tensor) -> torch.Tensor:
    """One step of `dtype` at magnitude mag (subnormal steps included)."""
    mant = 7 if dtype == torch.bfloat16 else 23
    return torch.clamp(mag, min=2.0 ** -126) * 2.0 ** -mant


def _term_bound(elem, abs_sum, count):
    """The error the summed terms may carry before the summation: each term is
    one of the kernel's fp32 gradients (or dw terms), computed from inputs of
    dtype `elem`.  fp32: each is held to max(2e-6 |t|, 1e-7) of the exact
    value (the elementwise tolerance), so the terms together to at most
    2e-6 sum|t| + 1e-7 count.  bf16: the hardware exponential and reciprocal
    keep each within 2^-17 relative (the kernels' sigmoid error is below
    3e-6 relative), so 2^-17 sum|t|."""
    if elem == torch.float32:
        return 2e-6 * abs_sum + 1e-7 * count
    if elem == torch.bfloat16:
        return 2.0 ** -17 * abs_sum
    raise TypeError(elem)


def assert_reduction(gpu, exact, abs_sum, depth, what, *, elem, count):
    """A fixed-order fp32 sum of `count` kernel terms against the exact sum of
    the exact terms: the terms' own error (_term_bound) plus the summation's,
    (depth + 6) 2^-24 sum|t| for `depth` chained additions, plus one step of
    the output type."""
    dtype = gpu.dtype
    gpu = gpu.cpu().double()
    bound = (depth + 6) * U32 * abs_sum + _term_bound(elem, abs_sum, count)
    tol = bound + _step(dtype, exact.abs() + bound)
    bad = (gpu - exact).abs() > tol
    nb = int(bad.sum())
    if nb:
        i = bad.nonzero()[:5].flatten().tolist()
        raise AssertionError(f"{what}: {nb} of {gpu.numel()} sums out of bound; first: "
                             f"{[(k, float(gpu[k]), float(exact[k]), float(tol[k])) for k in i]}")


# The tile kernel's launch shapes, (tile columns, CTAs per SM), by pack class:
# packs of 8 or 16 bytes, then packs of at most 4 bytes.  Which one a call takes
# depends on its pointers, so the bounds below take the deeper of the two.
BIAS_SHAPES = [(2048, 2), (1024, 4)]
WEIGHTED_BIAS_SHAPES = [(2048, 3), (1024, 4)]


def _bias_depth(rows, n, weighted=False):
    """Chained additions behind one dbias value: the rows of one row group
    (the tile kernel), then one of 8 contiguous segments of the row groups,
    then the 8 segment sums (the reduce kernel).  The plan fills every SM once
    with the shape's CTAs per SM."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    depth = 0
    for tile, per_sm in WEIGHTED_BIAS_SHAPES if weighted else BIAS_SHAPES:
        tiles = -(-n // tile)
        groups = max(1, min(rows, (sms * per_sm) // tiles))
        rpg = -(-rows // groups)
        groups = -(-rows // rpg)
        depth = max(depth, rpg + -(-groups // 8) + 8)
    return depth


CASES = [("tiny_f32", None), ("megatron_4096_bf16", 300), ("odd_5503_f32", 97),
         ("llama_14336_bf16_2d", 64)]


@pytest.mark.parametrize("name,rows", CASES)
def test_weighted_matches_oracle(sw, name, rows):
    w_ = W.WORKLOADS[name]
    x, dy = W.make_inputs(w_, "cpu", rows=rows)
    r = x.shape[0]
    g = torch.Generator().manual_seed(5)
    wts = torch.rand(r, generator=g)  # routing weights in [0, 1)
    xd, dyd, wd = x.cuda(), dy.cuda(), wts.cuda()
    y = sw.swiglu_gateup_weighted_fwd(xd, wd)
    dx, dw = sw.swiglu_gateup_weighted_bwd(dyd, xd, wd)
    xi = xd.clone()
    dxi, dwi = sw.swiglu_gateup_weighted_bwd(dyd, xi, wd, in_place=True)
    torch.cuda.synchronize()
    assert_parity(y, oracle.weighted_fwd(x, wts), f"{name} weighted fwd")
    rdx, _ = oracle.weighted_bwd(dy, x, wts)
    assert_parity(dx, rdx, f"{name} weighted dx")
    assert_bitwise(xi, dx, "weighted in-place dx")
    assert_bitwise(dwi, dw, "weighted in-place dw")
    # exact dw and |terms| from the fp64 oracle on the same (exactly widened) values
    x64, dy64 = x.double(), dy.double()
    _, dw64 = oracle.weighted_bwd(dy64, x64, wts)  # dw is returned rounded to fp32
    terms = (dy64 * oracle.fwd(x64)).abs().sum(1)
    exact = (dy64 * oracle.fwd(x64)).sum(1)
    assert torch.allclose(dw64.double(), exact, rtol=1e-6, atol=1e-30)
    assert_reduction(dw, exact, terms, w_.n / 256 + 13, f"{name} dw", elem=x.dtype, count=w_.n)


@pytest.mark.parametrize("name,rows", CASES)
def test_bias_matches_oracle(sw, name, rows):
    w_ = W.WORKLOADS[name]
    x, dy = W.make_inputs(w_, "cpu", rows=rows)
    r, n = x.shape[0], w_.n
    g = torch.Generator().manual_seed(6)
    bias = (torch.randn(2 * n, generator=g) * 0.5).to(x.dtype)
    xd, dyd, bd = x.cuda(), dy.cuda(), bias.cuda()
    y = sw.swiglu_gateup_bias_fwd(xd, bd)
    dx, db = sw.swiglu_gateup_bias_bwd(dyd, xd, bd)
    xi = xd.clone()
    dxi, dbi = sw.swiglu_gateup_bias_bwd(dyd, xi, bd, in_place=True)
    torch.cuda.synchronize()
    assert_parity(y, oracle.bias_fwd(x, bias), f"{name} bias fwd")
    rdx, _ = oracle.bias_bwd(dy, x, bias)
    assert_parity(dx, rdx, f"{name} bias dx")
    assert_bitwise(xi, dx, "bias in-place dx")
    assert_bitwise(dbi, db, "bias in-place dbias")
    dx64, db64 = oracle.bias_bwd(dy.double(), x.double(), bias.double())
    assert_reduction(db, db64, dx64.abs().sum(0), _bias_depth(r, n), f"{name} dbias",
                     elem=x.dtype, count=r)


def _wb_dw_depth(n):
    """Chained additions behind one dw value: a thread's tile / 256 columns,
    the 8 warps' sums of a lane, 5 shuffle steps, then the column tiles."""
    return max(tile // 256 + 13 + -(-n // tile) for tile, _ in WEIGHTED_BIAS_SHAPES)


def _check_weighted_bias(dy_c, x_c, bias_c, w_c, y, dx, db, dw, what):
    """y, dx against the oracle elementwise; dbias and dw against the exact sums."""
    rows, n = dy_c.shape
    assert_parity(y, oracle.weighted_bias_fwd(x_c, bias_c, w_c), f"{what} fwd")
    rdx, _, _ = oracle.weighted_bias_bwd(dy_c, x_c, bias_c, w_c)
    assert_parity(dx, rdx, f"{what} dx")
    x64, dy64, b64 = x_c.double(), dy_c.double(), bias_c.double()
    dx64, db64, _ = oracle.weighted_bias_bwd(dy64, x64, b64, w_c)
    assert_reduction(db, db64, dx64.abs().sum(0), _bias_depth(rows, n, weighted=True),
                     f"{what} dbias", elem=x_c.dtype, count=rows)
    t = dy64 * oracle.bias_fwd(x64, b64)
    assert_reduction(dw, t.sum(1), t.abs().sum(1), _wb_dw_depth(n), f"{what} dw", elem=x_c.dtype,
                     count=n)


@pytest.mark.parametrize("name,rows", CASES)
def test_weighted_bias_matches_oracle(sw, name, rows):
    w_ = W.WORKLOADS[name]
    x, dy = W.make_inputs(w_, "cpu", rows=rows)
    r, n = x.shape[0], w_.n
    g = torch.Generator().manual_seed(9)
    bias = (torch.randn(2 * n, generator=g) * 0.5).to(x.dtype)
    wts = torch.rand(r, generator=g)
    xd, dyd, bd, wd = x.cuda(), dy.cuda(), bias.cuda(), wts.cuda()
    y = sw.swiglu_gateup_weighted_bias_fwd(xd, bd, wd)
    dx, db, dw = sw.swiglu_gateup_weighted_bias_bwd(dyd, xd, bd, wd)
    xi = xd.clone()
    dxi, dbi, dwi = sw.swiglu_gateup_weighted_bias_bwd(dyd, xi, bd, wd, in_place=True)
    torch.cuda.synchronize()
    _check_weighted_bias(dy, x, bias, wts, y, dx, db, dw, f"{name} weighted bias")
    assert_bitwise(xi, dx, "weighted bias in-place dx")
    assert_bitwise(dbi, db, "weighted bias in-place dbias")
    assert_bitwise(dwi, dw, "weighted bias in-place dw")
    # the two reductions are deterministic: a second call gives the same bits
    dx2, db2, dw2 = sw.swiglu_gateup_weighted_bias_bwd(dyd, xd, bd, wd)
    torch.cuda.synchronize()
    assert_bitwise(db2, db, "weighted bias dbias, second call")
    assert_bitwise(dw2, dw, "weighted bias dw, second call")
    # with unit weights the combined form is the bias form
    ones = torch.ones(r, device="cuda")
    assert_bitwise(sw.swiglu_gateup_weighted_bias_fwd(xd, bd, ones), sw.swiglu_gateup_bias_fwd(xd, bd),
                   "unit weights fwd")
    dx1, db1, _ = sw.swiglu_gateup_weighted_bias_bwd(dyd, xd, bd, ones)
    dxb, dbb = sw.swiglu_gateup_bias_bwd(dyd, xd, bd)
    torch.cuda.synchronize()
    assert_bitwise(dx1, dxb, "unit weights dx")
    # dbias: the two forms group rows differently (2 or 3 tile CTAs per SM),
    # so their fixed-order sums differ in rounding; each stays within the
    # summation bound of its own order around the exact sum
    dx64, db64 = oracle.bias_bwd(dy.double(), x.double(), bias.double())
    assert_reduction(db1, db64, dx64.abs().sum(0), _bias_depth(r, n, weighted=True),
                     "unit weights dbias (weights + bias form)", elem=x.dtype, count=r)
    assert_reduction(dbb, db64, dx64.abs().sum(0), _bias_depth(r, n), "unit weights dbias (bias form)",
                     elem=x.dtype, count=r)


def test_weighted_bias_full_size(sw):
    """Large-FFN workload at full size: y, dx and dw on sampled rows, dbias on
    sampled columns (the oracle over all 8192 rows of those columns)."""
    w_ = W.WORKLOADS["large_32768_bf16"]
    x, dy = W.make_inputs(w_, "cuda")
    n = w_.n
    g = torch.Generator().manual_seed(10)
    bias = (torch.randn(2 * n, generator=g) * 0.5).to(torch.bfloat16).cuda()
    wts = torch.rand(w_.rows, generator=g).cuda()
    dx, db, dw = sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts)
    y = sw.swiglu_gateup_weighted_bias_fwd(x, bias, wts)
    torch.cuda.synchronize()
    idx = torch.tensor([0, 1, 4097, 8190, 8191], device="cuda")
    xs, dys, ws, bc = x[idx].cpu(), dy[idx].cpu(), wts[idx].cpu(), bias.cpu()
    assert_parity(y[idx], oracle.weighted_bias_fwd(xs, bc, ws), "full weighted bias fwd rows")
    assert_parity(dx[idx], oracle.weighted_bias_bwd(dys, xs, bc, ws)[0], "full weighted bias dx rows")
    t = dys.double() * oracle.bias_fwd(xs.double(), bc.double())
    assert_reduction(dw[idx], t.sum(1), t.abs().sum(1), _wb_dw_depth(n), "full dw rows",
                     elem=x.dtype, count=n)
    cols = torch.tensor(sorted(set([0, 1, 2047, 2048, n - 1] +
                                   torch.randperm(n, generator=g)[:59].tolist())))
    cc = cols.cuda()
    xsub = torch.cat([x[:, cc], x[:, n + cc]], 1).cpu()
    dysub = dy[:, cc].cpu()
    bsub = torch.cat([bias[cc], bias[n + cc]]).cpu()
    dx64, db64, _ = oracle.weighted_bias_bwd(dysub.double(), xsub.double(), bsub.double(), wts.cpu())
    got = torch.cat([db[cc], db[n + cc]])
    assert_reduction(got, db64, dx64.abs().sum(0), _bias_depth(w_.rows, n, weighted=True),
                     "full dbias columns", elem=x.dtype, count=w_.rows)


def test_bias_full_size_columns(sw):
    """Large-FFN workload at full size, the launch configuration of the bench:
    dx on sampled rows, dbias on sampled columns (the oracle over all 8192 rows
    of those columns)."""
    w_ = W.WORKLOADS["large_32768_bf16"]
    x, dy = W.make_inputs(w_, "cuda")
    n = w_.n
    g = torch.Generator().manual_seed(7)
    bias = (torch.randn(2 * n, generator=g) * 0.5).to(torch.bfloat16).cuda()
    dx, db = sw.swiglu_gateup_bias_bwd(dy, x, bias)
    y = sw.swiglu_gateup_bias_fwd(x, bias)
    torch.cuda.synchronize()
    rows_idx = torch.tensor([0, 1, 4097, 8190, 8191], device="cuda")
    xs, dys = x[rows_idx].cpu(), dy[rows_idx].cpu()
    assert_parity(y[rows_idx], oracle.bias_fwd(xs, bias.cpu()), "full bias fwd rows")
    assert_parity(dx[rows_idx], oracle.bias_bwd(dys, xs, bias.cpu())[0], "full bias dx rows")
    cols = torch.tensor(sorted(set([0, 1, 2047, 2048, n - 1] +
                                   torch.randperm(n, generator=g)[:59].tolist())))
    cc = cols.cuda()
    xsub = torch.cat([x[:, cc], x[:, n + cc]], 1).cpu()
    dysub = dy[:, cc].cpu()
    bsub = torch.cat([bias[cc], bias[n + cc]]).cpu()
    dx64, db64 = oracle.bias_bwd(dysub.double(), xsub.double(), bsub.double())
    got = torch.cat([db[cc], db[n + cc]])
    assert_reduction(got, db64, dx64.abs().sum(0), _bias_depth(w_.rows, n), "full dbias columns",
                     elem=x.dtype, count=w_.rows)


def test_weighted_full_size_rows(sw):
    w_ = W.WORKLOADS["large_32768_bf16"]
    x, dy = W.make_inputs(w_, "cuda")
    wts = torch.rand(w_.rows, generator=torch.Generator().manual_seed(8)).cuda()
    y = sw.swiglu_gateup_weighted_fwd(x, wts)
    dx, dw = sw.swiglu_gateup_weighted_bwd(dy, x, wts)
    torch.cuda.synchronize()
    idx = torch.tensor([0, 1, 3000, 8190, 8191], device="cuda")
    xs, dys, ws = x[idx].cpu(), dy[idx].cpu(), wts[idx].cpu()
    assert_parity(y[idx], oracle.weighted_fwd(xs, ws), "full weighted fwd rows")
    assert_parity(dx[idx], oracle.weighted_bwd(dys, xs, ws)[0], "full weighted dx rows")
    t = dys.double() * oracle.fwd(xs.double())
    assert_reduction(dw[idx], t.sum(1), t.abs().sum(1), w_.n / 256 + 13, "full dw rows",
                     elem=x.dtype, count=w_.n)


@pytest.mark.parametrize("rows", [1, 3, 305])
def test_weighted_long_rows_odd_counts(sw, rows):
    """The per-token-weighted kernel takes two rows per pass; rows longer than
    2048 16-byte packs run its unbounded form.  Odd row counts leave a last
    pass with one row.  dx elementwise, dw against the exact row sums."""
    n = 20480  # 2560 packs of 8 bf16
    g = torch.Generator().manual_seed(rows)
    x_c = (torch.randn(rows, 2 * n, generator=g) * 3).to(torch.bfloat16)
    dy_c = torch.randn(rows, n, generator=g).to(torch.bfloat16)
    w_c = torch.rand(rows, generator=g)
    dx, dw = sw.swiglu_gateup_weighted_bwd(dy_c.cuda(), x_c.cuda(), w_c.cuda())
    torch.cuda.synchronize()
    assert_parity(dx, oracle.weighted_bwd(dy_c, x_c, w_c)[0], f"long rows {rows}: weighted dx")
    t = dy_c.double() * oracle.fwd(x_c.double())
    assert_reduction(dw, t.sum(1), t.abs().sum(1), n / 256 + 13, f"long rows {rows}: weighted dw",
                     elem=torch.bfloat16, count=n)


@pytest.mark.parametrize("name", ["megatron_4096_bf16", "llama_14336_bf16_2d"])
def test_bias_forms_full_every_element(sw, name):
    """The ffn-4096 Megatron and the Llama-like workloads at full size (8192
    rows), in the launch configuration the bench times: every element of y and
    dx of the bias, weighted and weights + bias forms against the oracle, and
    every dbias column and dw row against the exact sums."""
    w_ = W.WORKLOADS[name]
    x_c, dy_c = W.make_inputs(w_, "cpu")
    x_c, dy_c = x_c.reshape(-1, 2 * w_.n), dy_c.reshape(-1, w_.n)
    rows, n = x_c.shape[0], w_.n
    g = torch.Generator().manual_seed(12)
    b_c = (torch.randn(2 * n, generator=g) * 0.5).to(torch.bfloat16)
    w_c = torch.rand(rows, generator=g)
    x, dy, bias, wts = x_c.cuda(), dy_c.cuda(), b_c.cuda(), w_c.cuda()
    x64, dy64, b64 = x_c.double(), dy_c.double(), b_c.double()

    assert_parity(sw.swiglu_gateup_bias_fwd(x, bias), oracle.bias_fwd(x_c, b_c), f"{name} bias fwd")
    dx, db = sw.swiglu_gateup_bias_bwd(dy, x, bias)
    assert_parity(dx, oracle.bias_bwd(dy_c, x_c, b_c)[0], f"{name} bias dx")
    dx64, db64 = oracle.bias_bwd(dy64, x64, b64)
    assert_reduction(db, db64, dx64.abs().sum(0), _bias_depth(rows, n), f"{name} dbias",
                     elem=torch.bfloat16, count=rows)

    assert_parity(sw.swiglu_gateup_weighted_fwd(x, wts), oracle.weighted_fwd(x_c, w_c), f"{name} weighted fwd")
    dx, dw = sw.swiglu_gateup_weighted_bwd(dy, x, wts)
    assert_parity(dx, oracle.weighted_bwd(dy_c, x_c, w_c)[0], f"{name} weighted dx")
    t = dy64 * oracle.fwd(x64)
    assert_reduction(dw, t.sum(1), t.abs().sum(1), n / 256 + 13, f"{name} weighted dw",
                     elem=torch.bfloat16, count=n)

    _check_weighted_bias(dy_c, x_c, b_c, w_c, sw.swiglu_gateup_weighted_bias_fwd(x, bias, wts),
                         *sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts), f"{name} weighted bias")


def test_empty_and_workspace_errors(sw):
    n = 64
    bias = torch.randn(2 * n, device="cuda")
    x = torch.empty(0, 2 * n, device="cuda")
    dbias = torch.full((2 * n,), 7.0, device="cuda")
    sw.swiglu_gateup_bias_bwd(torch.empty(0, n, device="cuda"), x, bias, dbias=dbias)
    assert torch.equal(dbias, torch.zeros_like(dbias))  # the sum over no rows
    x = torch.randn(32, 2 * n, device="cuda")
    dy = torch.randn(32, n, device="cuda")
    need = sw.bias_bwd_workspace_bytes(32, n)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(sw.SwigluError) as e:
        sw.swiglu_gateup_bias_bwd(dy, x, bias, workspace=small)
    assert e.value.status == -7
    dw = torch.full((32,), 3.0, device="cuda")
    sw.swiglu_gateup_weighted_bwd(torch.empty(32, 0, device="cuda"), torch.empty(32, 0, device="cuda"),
                                  torch.ones(32, device="cuda"), dw=dw)
    assert torch.equal(dw, torch.zeros_like(dw))
    # weights and bias together: no rows zero dbias, no columns zero dw
    dbias.fill_(7.0)
    sw.swiglu_gateup_weighted_bias_bwd(torch.empty(0, n, device="cuda"),
                                       torch.empty(0, 2 * n, device="cuda"), bias,
                                       torch.empty(0, device="cuda"), dbias=dbias)
    assert torch.equal(dbias, torch.zeros_like(dbias))
    dw.fill_(3.0)
    sw.swiglu_gateup_weighted_bias_bwd(torch.empty(32, 0, device="cuda"),
                                       torch.empty(32, 0, device="cuda"),
                                       torch.empty(0, device="cuda"), torch.ones(32, device="cuda"),
                                       dw=dw)
    assert torch.equal(dw, torch.zeros_like(dw))
    need_wb = sw.weighted_bias_bwd_workspace_bytes(32, n)
    assert need_wb >= need + 32 * 4
    with pytest.raises(sw.SwigluError) as e:
        sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, torch.ones(32, device="cuda"),
                                           workspace=torch.empty(need_wb - 16, dtype=torch.uint8,
                                                                 device="cuda"))
    assert e.value.status == -7


LAYOUTS = [
    # (dtype, rows, n, x_pad, dy_pad, dx_pad, misalign)
    ("bf16", 70, 4100, 0, 0, 0, 0),      # 8-byte packs
    ("bf16", 50, 2050, 2, 2, 6, 0),      # 4-byte packs, padded strides
    ("bf16", 33, 999, 0, 0, 0, 0),       # single elements
    ("bf16", 40, 2048, 0, 0, 0, 1),      # misaligned base pointers
    ("f32", 45, 1026, 0, 0, 0, 0),       # 8-byte packs
    ("f32", 37, 3000, 4, 4, 8, 0),       # 16-byte packs with padding
    ("f32", 21, 5001, 1, 3, 1, 1),       # odd n, odd strides, misaligned
    ("bf16", 600, 40, 0, 0, 0, 0),       # many short rows (row groups, tiles of one)
]


def _guard(rows, cols, pad, mis, dt, fill):
    buf = torch.full((64 + mis + rows * (cols + pad) + 64,), fill, dtype=dt, device="cuda")
    return buf, buf[64 + mis: 64 + mis + rows * (cols + pad)].view(rows, cols + pad)[:, :cols]


@pytest.mark.parametrize("case", LAYOUTS, ids=[f"{c[0]}-r{c[1]}-n{c[2]}-p{c[3]}{c[4]}{c[5]}-m{c[6]}"
                                               for c in LAYOUTS])
def test_bias_and_weighted_layouts(sw, case):
    dts, rows, n, xp, dyp, dxp, mis = case
    dt = torch.float32 if dts == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(rows + n)
    x_c = (torch.randn(rows, 2 * n, generator=g) * 3).to(dt)
    dy_c = torch.randn(rows, n, generator=g).to(dt)
    bias_c = (torch.randn(2 * n, generator=g) * 0.5).to(dt)
    w_c = torch.rand(rows, generator=g)
    xb, x = _guard(rows, 2 * n, xp, mis, dt, float("nan"))
    dyb, dy = _guard(rows, n, dyp, mis, dt, float("nan"))
    dxb, dx = _guard(rows, 2 * n, dxp, mis, dt, -7.0)
    x.copy_(x_c)
    dy.copy_(dy_c)
    dxb0 = dxb.clone()
    bias, wts = bias_c.cuda(), w_c.cuda()
    # bias backward into the guarded dx, and its forward
    _, db = sw.swiglu_gateup_bias_bwd(dy, x, bias, dx)
    y = sw.swiglu_gateup_bias_fwd(x, bias)
    torch.cuda.synchronize()
    rdx, _ = oracle.bias_bwd(dy_c, x_c, bias_c)
    assert_parity(dx, rdx, "bias dx")
    assert_parity(y, oracle.bias_fwd(x_c, bias_c), "bias fwd")
    dx64, db64 = oracle.bias_bwd(dy_c.double(), x_c.double(), bias_c.double())
    assert_reduction(db, db64, dx64.abs().sum(0), _bias_depth(rows, n), "bias dbias", elem=dt,
                     count=rows)
    dx.fill_(-7.0)
    assert torch.equal(dxb.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                       dxb0.view(torch.int16 if dt == torch.bfloat16 else torch.int32)), "guard bands"
    # weighted backward into the same guarded dx, and its forward
    _, dw = sw.swiglu_gateup_weighted_bwd(dy, x, wts, dx)
    yw = sw.swiglu_gateup_weighted_fwd(x, wts)
    torch.cuda.synchronize()
    rdx, _ = oracle.weighted_bwd(dy_c, x_c, w_c)
    assert_parity(dx, rdx, "weighted dx")
    assert_parity(yw, oracle.weighted_fwd(x_c, w_c), "weighted fwd")
    t = dy_c.double() * oracle.fwd(x_c.double())
    assert_reduction(dw, t.sum(1), t.abs().sum(1), n / 256 + 13, "weighted dw", elem=dt, count=n)
    dx.fill_(-7.0)
    assert torch.equal(dxb.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                       dxb0.view(torch.int16 if dt == torch.bfloat16 else torch.int32)), "guard bands"
    # weights and bias together, into the same guarded dx
    _, dbw, dww = sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts, dx)
    ywb = sw.swiglu_gateup_weighted_bias_fwd(x, bias, wts)
    torch.cuda.synchronize()
    _check_weighted_bias(dy_c, x_c, bias_c, w_c, ywb, dx, dbw, dww, "weighted bias")
    dx.fill_(-7.0)
    assert torch.equal(dxb.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                       dxb0.view(torch.int16 if dt == torch.bfloat16 else torch.int32)), "guard bands"
    # the three forward forms into a guarded y with the same padding and
    # misalignment (narrow packs take the row-segment kernel)
    yb, yg = _guard(rows, n, dyp, mis, dt, -7.0)
    yb0 = yb.clone()
    for what, run, ref in (
            ("bias", lambda: sw.swiglu_gateup_bias_fwd(x, bias, yg), oracle.bias_fwd(x_c, bias_c)),
            ("weighted", lambda: sw.swiglu_gateup_weighted_fwd(x, wts, yg), oracle.weighted_fwd(x_c, w_c)),
            ("weighted bias", lambda: sw.swiglu_gateup_weighted_bias_fwd(x, bias, wts, yg),
             oracle.weighted_bias_fwd(x_c, bias_c, w_c))):
        run()
        torch.cuda.synchronize()
        assert_parity(yg, ref, f"{what} fwd into a guarded y")
        yg.fill_(-7.0)
        assert torch.equal(yb.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                           yb0.view(torch.int16 if dt == torch.bfloat16 else torch.int32)), \
            f"{what} fwd guard bands"
