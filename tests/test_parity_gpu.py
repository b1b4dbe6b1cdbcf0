"""CUDA path vs the oracle, element by element, through the C ABI.

Tolerances (tests/helpers.py): fp32 within max(2e-6 relative, 1e-7 absolute) of
the oracle's once-rounded fp64 result; bf16 within one bf16 step; the in-place
backward bit-identical to the out-of-place one.

Sizes: every workload is compared with the oracle on every element at full
size; the large-FFN and Llama-like workloads run in the launch configuration
the bench times, and the oracle works through them in row chunks on several
host threads.  In place must equal out of place bit for bit everywhere.  Smaller ragged
cases cover every pack width (16/8/4/2 bytes and single elements), padded row
strides, misaligned base pointers and guard bands around every buffer.
"""
import os

import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bitwise, assert_parity

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def _run_all(sw, x, dy):
    """fwd, out-of-place bwd, in-place bwd on the GPU; x, dy are 2D device tensors."""
    y = sw.swiglu_gateup_fwd(x)
    dx = sw.swiglu_gateup_bwd(dy, x)
    xi = x.clone()
    sw.swiglu_gateup_bwd(dy, xi, in_place=True)
    torch.cuda.synchronize()
    return y, dx, xi


# ------------------------------------------------------- whole workloads ---

@pytest.mark.parametrize("name", ["tiny_f32", "megatron_4096_bf16", "odd_5503_f32"])
def test_workload_full_compare(sw, name):
    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cpu")
    y, dx, xi = _run_all(sw, x.cuda(), dy.cuda())
    assert_parity(y, oracle.fwd(x), f"{name} fwd", extra=x[:, :w.n])
    ref_dx = oracle.bwd(dy, x)
    assert_parity(dx, ref_dx, f"{name} bwd")
    assert_bitwise(xi, dx, f"{name} in-place vs out-of-place")


def _compare_in_row_chunks(x, dy, outputs, what, chunk_rows=64):
    """Every element of the forward and backward results against the oracle.

    ``outputs`` maps a label to ``(kind, tensor)`` with kind "fwd" (compared
    with ``oracle.fwd``) or "bwd" (``oracle.bwd``).  The host copies are made
    once; rows are then split into chunks that a pool of host threads hands to
    the oracle (ctypes releases the GIL, so the single-threaded oracle runs on
    several cores at once, each chunk by the same plain loop) and compares.
    """
    from concurrent.futures import ThreadPoolExecutor

    rows = x.shape[0]
    xh, dyh = x.cpu(), dy.cpu()
    host = {k: (kind, t.cpu()) for k, (kind, t) in outputs.items()}
    lib = oracle.load()

    def check(r0):
        r1 = min(rows, r0 + chunk_rows)
        xs, dys = xh[r0:r1], dyh[r0:r1]
        ref = {}
        if any(kind == "fwd" for kind, _ in host.values()):
            ref["fwd"] = oracle.fwd(xs, lib=lib)
        if any(kind == "bwd" for kind, _ in host.values()):
            ref["bwd"] = oracle.bwd(dys, xs, lib=lib)
        for label, (kind, t) in host.items():
            assert_parity(t[r0:r1], ref[kind], f"{what} {label} rows [{r0}, {r1})")
        return r1 - r0

    workers = max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as pool:
        done = sum(pool.map(check, range(0, rows, chunk_rows)))
    assert done == rows


@pytest.mark.parametrize("name", ["large_32768_bf16", "llama_14336_bf16_2d"])
def test_workload_full_size_every_element(sw, name):
    """The two largest workloads at full size, in the launch configuration the
    bench times: forward, out-of-place backward and in-place backward compared
    with the oracle on every element (and in place = out of place, bit for
    bit)."""
    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cuda")
    y, dx, xi = _run_all(sw, x, dy)
    assert_bitwise(xi, dx, f"{name} in-place vs out-of-place")
    # a property at full size: finite inputs give finite outputs
    assert bool(torch.isfinite(y).all()) and bool(torch.isfinite(dx).all())
    _compare_in_row_chunks(x, dy, {"fwd": ("fwd", y), "bwd": ("bwd", dx),
                                   "in-place bwd": ("bwd", xi)}, name)


def test_3d_inputs_flatten(sw):
    w = W.WORKLOADS["megatron_4096_bf16"]
    x, dy = W.make_inputs(w, "cuda", rows=64)
    x3 = x.contiguous().view(16, 4, 2 * w.n)
    dy3 = dy.view(16, 4, w.n)
    y3 = sw.swiglu_gateup_fwd(x3)
    dx3 = sw.swiglu_gateup_bwd(dy3, x3)
    assert y3.shape == (16, 4, w.n) and dx3.shape == x3.shape
    assert_bitwise(y3.view(64, w.n), sw.swiglu_gateup_fwd(x), "3D vs 2D fwd")
    assert_bitwise(dx3.view(64, 2 * w.n), sw.swiglu_gateup_bwd(dy, x), "3D vs 2D bwd")


# ------------------------------------------------------ exhaustive sweeps ---

def _bf16_all_patterns():
    b = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    return b.view(torch.bfloat16)


def test_bf16_every_gate_value(sw):
    """All 65536 bf16 gate bit patterns (NaN and inf included) x varied up/dy."""
    gates = _bf16_all_patterns().view(8, 8192)
    n = 8192
    gen = torch.Generator().manual_seed(7)
    for scale in (1.0, 64.0):
        up = (torch.randn(8, n, generator=gen) * scale).to(torch.bfloat16)
        dy = (torch.randn(8, n, generator=gen) * scale).to(torch.bfloat16)
        x = torch.cat([gates, up], dim=1)
        y, dx, xi = _run_all(sw, x.cuda(), dy.cuda())
        assert_parity(y, oracle.fwd(x), "bf16 sweep fwd", extra=gates)
        assert_parity(dx, oracle.bwd(dy, x), "bf16 sweep bwd")
        assert_bitwise(xi, dx, "bf16 sweep in-place")


@pytest.mark.parametrize("lo,hi", [(-1.6, -1.0), (-0.02, 0.02), (8.0, 24.0), (-24.0, -8.0),
                                   (-105.0, -80.0), (80.0, 105.0), (-1e6, 1e6)])
def test_f32_dense_gate_ranges(sw, lo, hi):
    """Dense fp32 gate grids over the ranges where the arithmetic is delicate:
    the root of silu' (-1.28), zero, the sigmoid tails and the ends of the fp32
    exponential's range."""
    m = 1 << 20
    g = torch.linspace(lo, hi, m, dtype=torch.float64).float()
    gen = torch.Generator().manual_seed(11)
    up = torch.rand(m, generator=gen) * 8 - 4
    dy = torch.randn(m, generator=gen) * 3
    n = 4096
    x = torch.cat([g.view(-1, n), up.view(-1, n)], dim=1)
    dy = dy.view(-1, n)
    y, dx, xi = _run_all(sw, x.cuda(), dy.cuda())
    assert_parity(y, oracle.fwd(x), f"f32 [{lo},{hi}] fwd", extra=x[:, :n])
    assert_parity(dx, oracle.bwd(dy, x), f"f32 [{lo},{hi}] bwd")
    assert_bitwise(xi, dx, "f32 sweep in-place")


def _read_golden():
    path = os.path.join(HERE, "golden", "oracle_specials.txt")
    lines = [l for l in open(path).read().splitlines() if l and not l.startswith("#")]
    out = {}
    for head, body in zip(lines[::2], lines[1::2]):
        dt, name, r, c = head.split()
        vals = [int(v, 16) for v in body.split()]
        if dt == "f32":
            t = torch.tensor(vals, dtype=torch.int64).to(torch.int32).view(torch.float32)
        else:
            t = torch.tensor(vals, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
        out[(dt, name)] = t.view(int(r), int(c))
    return out


def test_golden_special_values(sw):
    gold = _read_golden()
    for dt in ("f32", "bf16"):
        x, dy = gold[(dt, "x")], gold[(dt, "dy")]
        y, dx, xi = _run_all(sw, x.cuda(), dy.cuda())
        assert_parity(y, gold[(dt, "y")], f"golden {dt} fwd", extra=x[:, : x.shape[1] // 2])
        assert_parity(dx, gold[(dt, "dx")], f"golden {dt} bwd")
        assert_bitwise(xi, dx, f"golden {dt} in-place")


# ------------------------------------- pack widths, strides, guard bands ---

SENTINEL_F32 = -12345.5
CASES = [
    # (dtype, rows, n, x_pad, y_pad, dy_pad, dx_pad, misalign_elems)
    # pack widths: forward up to 32 bytes, backward up to 16 bytes
    ("bf16", 37, 4096, 0, 0, 0, 0, 0),    # fwd 32-byte, bwd 16-byte packs
    ("bf16", 37, 4104, 0, 0, 0, 0, 0),    # 16-byte packs (n % 16 == 8)
    ("bf16", 37, 4100, 0, 0, 0, 0, 0),    # 8-byte packs (n % 8 == 4)
    ("bf16", 29, 4098, 0, 0, 0, 0, 0),    # 4-byte packs (n % 4 == 2)
    ("bf16", 31, 1001, 0, 0, 0, 0, 0),    # single elements (odd n)
    ("bf16", 23, 2048, 16, 32, 16, 32, 0),  # padded strides keep 32-byte packs
    ("bf16", 23, 2048, 8, 16, 8, 24, 0),  # padding drops the forward to 16 bytes
    ("bf16", 23, 2048, 2, 6, 2, 4, 0),    # padding drops to 4-byte packs
    ("bf16", 19, 2048, 0, 0, 0, 0, 1),    # misaligned base pointers
    ("bf16", 3000, 8, 0, 0, 0, 0, 0),     # many short rows (grid-stride, row carry)
    ("bf16", 5, 1, 0, 0, 0, 0, 0),        # n = 1
    ("f32", 37, 4096, 0, 0, 0, 0, 0),     # fwd 32-byte, bwd 16-byte packs
    ("f32", 37, 4098, 0, 0, 0, 0, 0),     # 8-byte packs
    ("f32", 31, 5503, 0, 0, 0, 0, 0),     # odd n
    ("f32", 23, 1024, 4, 12, 4, 8, 0),    # padded strides, 16-byte packs
    ("f32", 23, 1024, 1, 3, 1, 2, 1),     # odd strides and misaligned pointers
    ("f32", 40000, 3, 0, 0, 0, 0, 0),     # many tiny rows
    ("f32", 1, 70000, 0, 0, 0, 0, 0),     # one long row
]


def _guarded(rows, cols, pad, misalign, dtype, fill, guard=64):
    """A [rows, cols] view with row stride cols + pad, inside a buffer with
    `guard` sentinel elements on both sides; returns (buffer, view, offset)."""
    stride = cols + pad
    total = guard + misalign + rows * stride + guard
    buf = torch.full((total,), fill, dtype=dtype, device="cuda")
    off = guard + misalign
    view = buf[off: off + rows * stride].view(rows, stride)[:, :cols]
    return buf, view


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-r{c[1]}-n{c[2]}-p{c[3]}{c[4]}{c[5]}{c[6]}-m{c[7]}"
                                             for c in CASES])
def test_layouts_and_guard_bands(sw, case):
    dts, rows, n, xp, yp, dyp, dxp, mis = case
    dt = torch.float32 if dts == "f32" else torch.bfloat16
    gen = torch.Generator().manual_seed(rows * 7 + n)
    x_cpu = (torch.randn(rows, 2 * n, generator=gen) * 3).to(dt)
    dy_cpu = torch.randn(rows, n, generator=gen).to(dt)
    xb, x = _guarded(rows, 2 * n, xp, mis, dt, float("nan"))
    dyb, dy = _guarded(rows, n, dyp, mis, dt, float("nan"))
    yb, y = _guarded(rows, n, yp, mis, dt, SENTINEL_F32)
    dxb, dx = _guarded(rows, 2 * n, dxp, mis, dt, SENTINEL_F32)
    x.copy_(x_cpu)
    dy.copy_(dy_cpu)
    xb0, yb0, dxb0 = xb.clone(), yb.clone(), dxb.clone()
    sw.swiglu_gateup_fwd(x, y)
    sw.swiglu_gateup_bwd(dy, x, dx)
    torch.cuda.synchronize()
    assert_parity(y, oracle.fwd(x_cpu), "fwd")
    assert_parity(dx, oracle.bwd(dy_cpu, x_cpu), "bwd")
    assert_bitwise(xb, xb0, "x buffer (read-only) changed")
    # everything outside the written views keeps its sentinel: refill the
    # views and the whole buffers must be back to their initial bits
    y.fill_(SENTINEL_F32)
    assert_bitwise(yb, yb0, "y guard bands / padding")
    dx_after = dx.clone()
    dx.fill_(SENTINEL_F32)
    assert_bitwise(dxb, dxb0, "dx guard bands / padding")
    # in place over the guarded x: same bits as the out-of-place result, and
    # x's padding and guards untouched
    sw.swiglu_gateup_bwd(dy, x, in_place=True)
    torch.cuda.synchronize()
    assert_bitwise(x, dx_after, "in-place vs out-of-place")
    x.copy_(x_cpu)
    assert_bitwise(xb, xb0, "x guard bands / padding after in-place")


# ------------------------------------------------------------ API surface ---

def test_empty_and_errors(sw):
    dt = torch.bfloat16
    x = torch.empty(0, 16, dtype=dt, device="cuda")
    assert sw.swiglu_gateup_fwd(x).shape == (0, 8)
    assert sw.swiglu_gateup_bwd(torch.empty(0, 8, dtype=dt, device="cuda"), x).shape == (0, 16)
    x = torch.randn(4, 16, device="cuda").to(dt)
    # y overlapping x is rejected and nothing is written
    before = x.clone()
    with pytest.raises(sw.SwigluError) as e:
        sw.swiglu_gateup_fwd(x, x[:, :8])
    assert e.value.status == -5
    assert_bitwise(x, before, "rejected call wrote")
    with pytest.raises(sw.SwigluError) as e:
        sw.swiglu_gateup_bwd(x[:, :8].contiguous(), x, x)
    assert e.value.status == -5
    assert sw.lib.swiglu_last_cuda_error() == 0


def test_side_stream(sw):
    w = W.WORKLOADS["megatron_4096_bf16"]
    x, dy = W.make_inputs(w, "cuda", rows=256)
    ref = sw.swiglu_gateup_bwd(dy, x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = sw.swiglu_gateup_fwd(x)
        dx = sw.swiglu_gateup_bwd(dy, x)
    s.synchronize()
    assert_bitwise(dx, ref, "side stream")
    assert_bitwise(y, sw.swiglu_gateup_fwd(x), "side stream fwd")


# ----------------------------------------------------------- maximum sizes ---

def _cols(x, J, n):
    return torch.cat([x[:, J], x[:, n + J]], 1)


def test_maximum_n(sw):
    """n = 2^30 (the largest the ABI accepts), 2 rows of bf16: element offsets
    past 2^31 within a row, and the last packs of each half.  Checked on
    sampled columns (the op is elementwise, so a column subset is a smaller
    problem of its own)."""
    n, rows = 1 << 30, 2
    g = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randn(rows, 2 * n, device="cuda", generator=g, dtype=torch.bfloat16)
    dy = torch.randn(rows, n, device="cuda", generator=g, dtype=torch.bfloat16)
    y = sw.swiglu_gateup_fwd(x)
    dx = sw.swiglu_gateup_bwd(dy, x)
    torch.cuda.synchronize()
    J = torch.cat([torch.arange(0, 64), torch.arange((1 << 29) - 32, (1 << 29) + 32),
                   torch.arange(n - 64, n)]).cuda()
    xs, dys = _cols(x, J, n).cpu(), dy[:, J].cpu()
    assert_parity(y[:, J], oracle.fwd(xs), "max n fwd")
    assert_parity(_cols(dx, J, n), oracle.bwd(dys, xs), "max n bwd")
    del x, dy, y, dx
    torch.cuda.empty_cache()


def test_more_than_2_32_elements(sw):
    """2^20 + 3 rows of n = 4104 (4.3e9 gate/up pairs, 8-byte-aligned packs):
    the flattened (row, pack) index and its carry run past 2^32 in the plain,
    bias and weights + bias kernels.  Checked on sampled rows, and dbias on
    sampled columns over all rows."""
    from test_bias_weighted_gpu import _bias_depth, _wb_dw_depth, assert_reduction

    rows, n = (1 << 20) + 3, 4104
    g = torch.Generator(device="cuda").manual_seed(13)
    x = torch.randn(rows, 2 * n, device="cuda", generator=g, dtype=torch.bfloat16)
    dy = torch.randn(rows, n, device="cuda", generator=g, dtype=torch.bfloat16)
    bias = (torch.randn(2 * n, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    wts = torch.rand(rows, device="cuda", generator=g)
    R = torch.tensor([0, 1, 777, (1 << 19) + 5, rows - 2, rows - 1], device="cuda")
    xs, dys, bc, ws = x[R].cpu(), dy[R].cpu(), bias.cpu(), wts[R].cpu()

    y = sw.swiglu_gateup_fwd(x)
    assert_parity(y[R], oracle.fwd(xs), "2^32 fwd")
    del y
    dx = sw.swiglu_gateup_bwd(dy, x)
    assert_parity(dx[R], oracle.bwd(dys, xs), "2^32 bwd")
    dx, db, dw = sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts, dx=dx)
    torch.cuda.synchronize()
    assert_parity(dx[R], oracle.weighted_bias_bwd(dys, xs, bc, ws)[0], "2^32 weighted bias dx")
    t = dys.double() * oracle.bias_fwd(xs.double(), bc.double())
    assert_reduction(dw[R], t.sum(1), t.abs().sum(1), _wb_dw_depth(n), "2^32 dw rows",
                     elem=torch.bfloat16, count=n)
    J = torch.tensor([0, 1, 2047, 2048, 4095, 4096, n - 1], device="cuda")
    xsub, dysub = _cols(x, J, n).cpu(), dy[:, J].cpu()
    bsub = torch.cat([bias[J], bias[n + J]]).cpu()
    dx64, db64, _ = oracle.weighted_bias_bwd(dysub.double(), xsub.double(), bsub.double(), wts.cpu())
    assert_reduction(torch.cat([db[J], db[n + J]]), db64, dx64.abs().sum(0),
                     _bias_depth(rows, n, weighted=True),
                     "2^32 dbias columns", elem=torch.bfloat16, count=rows)
    del x, dy, dx
    torch.cuda.empty_cache()


def test_concurrent_threads_on_separate_streams(sw):
    """The library keeps only per-device caches (atomics) and no per-call
    state: four host threads calling it at once (ctypes releases the GIL),
    each on its own stream and buffers, get bit-identical results to a single
    thread."""
    import threading

    w = W.WORKLOADS["megatron_4096_bf16"]
    inputs = [W.make_inputs(w, "cuda", rows=128 + 64 * i) for i in range(4)]
    g = torch.Generator(device="cuda").manual_seed(9)
    biases = [(torch.randn(2 * w.n, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
              for _ in range(4)]
    ref = []
    for (x, dy), b in zip(inputs, biases):
        ref.append((sw.swiglu_gateup_fwd(x), sw.swiglu_gateup_bwd(dy, x),
                    sw.swiglu_gateup_bias_bwd(dy, x, b)))
    torch.cuda.synchronize()
    results, errors = [None] * 4, []

    def work(i):
        try:
            x, dy = inputs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(20):
                    y = sw.swiglu_gateup_fwd(x, stream=s)
                    dx = sw.swiglu_gateup_bwd(dy, x, stream=s)
                    dxb, db = sw.swiglu_gateup_bias_bwd(dy, x, biases[i], stream=s)
            s.synchronize()
            results[i] = (y, dx, (dxb, db))
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(4):
        assert_bitwise(results[i][0], ref[i][0], f"thread {i} fwd")
        assert_bitwise(results[i][1], ref[i][1], f"thread {i} bwd")
        assert_bitwise(results[i][2][0], ref[i][2][0], f"thread {i} bias dx")
        assert_bitwise(results[i][2][1], ref[i][2][1], f"thread {i} dbias")
