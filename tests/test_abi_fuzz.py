"""Random calls against an independent statement of the argument contract of
swiglu_gateup_fwd / swiglu_gateup_bwd (the rules written in include/swiglu.h,
restated here in Python): the library must return the status the contract
predicts, in the order the header gives.  Pointers are fake integers that are
never dereferenced: a call the contract accepts goes on to the CUDA runtime,
which on a machine without a GPU fails with SWIGLU_ERR_CUDA.  On a machine with
a GPU such a call would launch a kernel on fake addresses, so the test only
runs where there is none."""
import random

import pytest
import torch

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="valid calls would launch kernels on fake pointers")

OK, NULL, DTYPE, SHAPE, STRIDE, ALIAS, CUDA = 0, -1, -2, -3, -4, -5, -6
MAX_N = 1 << 30


@pytest.fixture(scope="module")
def lib():
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw.lib


def span(p, rows, cols, stride, eb):
    return (p, p + ((rows - 1) * stride + cols) * eb)


def overl(a, b):
    return a[0] < b[1] and b[0] < a[1]


def expect_fwd(x, y, rows, n, sx, sy, dt):
    if dt not in (0, 1):
        return DTYPE
    if rows < 0 or n < 0 or n > MAX_N:
        return SHAPE
    if rows == 0 or n == 0:
        return OK
    if not x or not y:
        return NULL
    if sx < 2 * n or sy < n:
        return STRIDE
    eb = 4 if dt == 0 else 2
    if overl(span(x, rows, 2 * n, sx, eb), span(y, rows, n, sy, eb)):
        return ALIAS
    if x % eb or y % eb:  # every pointer on its element size
        return STRIDE
    return CUDA


def expect_bwd(dy, x, dx, rows, n, sdy, sx, sdx, dt, ip):
    if dt not in (0, 1):
        return DTYPE
    if rows < 0 or n < 0 or n > MAX_N:
        return SHAPE
    if rows == 0 or n == 0:
        return OK
    if ip:
        dx = dx or x
        sdx = sdx or sx
    if not dy or not x or not dx:
        return NULL
    if sdy < n or sx < 2 * n or sdx < 2 * n:
        return STRIDE
    eb = 4 if dt == 0 else 2
    s_dy, s_x, s_dx = span(dy, rows, n, sdy, eb), span(x, rows, 2 * n, sx, eb), span(dx, rows, 2 * n, sdx, eb)
    if ip:
        if dx != x:
            return ALIAS
        if sdx != sx:
            return STRIDE
        if overl(s_dy, s_x):
            return ALIAS
    elif overl(s_dx, s_x) or overl(s_dx, s_dy):
        return ALIAS
    if dy % eb or x % eb or dx % eb:  # every pointer on its element size
        return STRIDE
    return CUDA


ARENA = 1 << 36


def rand_ptr(rng, base):
    """Mostly far-apart arenas, sometimes inside another operand's arena, now
    and then NULL."""
    r = rng.random()
    if r < 0.05:
        return 0
    if r < 0.35:
        return ARENA + 2 * rng.randrange(0, 4096)  # shared arena: overlaps likely
    return base


def rand_shape(rng):
    rows = rng.choice([-1, 0, 1, 2, 3, 7, 64])
    n = rng.choice([-3, 0, 1, 5, 8, 64, 100, MAX_N + 1])
    return rows, n


def rand_stride(rng, need):
    return max(0, need + rng.choice([-2, -1, 0, 0, 0, 1, 8, 64]))


def test_fwd_matches_contract(lib):
    rng = random.Random(1)
    for _ in range(4000):
        rows, n = rand_shape(rng)
        x, y = rand_ptr(rng, 3 * ARENA), rand_ptr(rng, 5 * ARENA)
        sx, sy = rand_stride(rng, 2 * n), rand_stride(rng, n)
        dt = rng.choice([0, 1, 1, 2])
        want = expect_fwd(x, y, rows, n, sx, sy, dt)
        got = lib.swiglu_gateup_fwd(x or None, y or None, rows, n, sx, sy, dt, None)
        assert got == want, (x, y, rows, n, sx, sy, dt)


def test_bwd_matches_contract(lib):
    rng = random.Random(2)
    for _ in range(6000):
        rows, n = rand_shape(rng)
        ip = rng.random() < 0.4
        dy, x = rand_ptr(rng, 3 * ARENA), rand_ptr(rng, 5 * ARENA)
        dx = rng.choice([0, x, x, rand_ptr(rng, 7 * ARENA)]) if ip else rand_ptr(rng, 7 * ARENA)
        sdy, sx = rand_stride(rng, n), rand_stride(rng, 2 * n)
        sdx = rng.choice([0, sx, rand_stride(rng, 2 * n)]) if ip else rand_stride(rng, 2 * n)
        dt = rng.choice([0, 1, 1, 5])
        want = expect_bwd(dy, x, dx, rows, n, sdy, sx, sdx, dt, ip)
        got = lib.swiglu_gateup_bwd(dy or None, x or None, dx or None, rows, n, sdy, sx, sdx, dt,
                                    1 if ip else 0, None)
        assert got == want, (dy, x, dx, rows, n, sdy, sx, sdx, dt, ip)
