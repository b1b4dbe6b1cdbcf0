"""The allocation-free bias backward, through the C ABI.

swiglu_gateup_bias_bwd_noalloc serves callers that cannot give the library any
device memory (engines that plan all memory ahead and forbid allocation
mid-step, plugin hosts that own the allocator, latency-bound paths that cannot
take cudaMalloc's synchronisation): its scratch is a fixed array inside the
library.  Its results must match the workspace entry point's, within the
tolerances the other tests use, and the oracle's (dx element by element, dbias
within the summation bound of the other bias tests), on two calls in a row
(the second call must not see anything the first left in the shared array),
and a problem too large for the fixed array must be refused without touching
the outputs.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""

import pytest
import torch

import oracle
import workloads as W
from helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def _noalloc(sw, dy, x, bias, dx, dbias, in_place=False):
    rows, n = dy.shape
    stream = torch.cuda.current_stream().cuda_stream
    return sw.lib.swiglu_gateup_bias_bwd_noalloc(
        dy.data_ptr(), x.data_ptr(), bias.data_ptr(), dx.data_ptr(), dbias.data_ptr(), rows, n,
        dy.stride(0), x.stride(0), dx.stride(0),
        sw.SWIGLU_BF16 if x.dtype == torch.bfloat16 else sw.SWIGLU_F32, 1 if in_place else 0,
        stream)


def _inputs(name, rows, seed):
    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cuda", rows=rows)
    g = torch.Generator().manual_seed(seed)
    bias = (torch.randn(2 * w.n, generator=g) * 0.5).to(x.dtype).cuda()
    return x.contiguous(), dy, bias


@pytest.mark.parametrize("name,rows", [("megatron_4096_bf16", 1024), ("odd_5503_f32", 300),
                                       ("large_32768_bf16", 512)])
def test_noalloc_matches_workspace_entry_point_twice(sw, name, rows):
    first = _inputs(name, rows, seed=1)
    second = _inputs(name, rows, seed=2)
    second = (second[0] * 3, second[1], -second[2])  # other values, same shapes
    for x, dy, bias in (first, second):
        ref_dx, ref_db = sw.swiglu_gateup_bias_bwd(dy, x, bias)
        dx = torch.full_like(x, float("nan"))
        db = torch.full_like(bias, float("nan"))
        assert _noalloc(sw, dy, x, bias, dx, db) == 0
        torch.cuda.synchronize()
        assert_parity(dx, ref_dx.cpu(), f"{name} no-alloc dx")
        assert_parity(db, ref_db.cpu(), f"{name} no-alloc dbias")
        _against_oracle(dy, x, bias, dx, db, f"{name} no-alloc")
    # the in-place form through the same entry point
    x, dy, bias = first
    ref_dx, ref_db = sw.swiglu_gateup_bias_bwd(dy, x, bias)
    xi = x.clone()
    db = torch.empty_like(bias)
    assert _noalloc(sw, dy, xi, bias, xi, db, in_place=True) == 0
    torch.cuda.synchronize()
    assert_parity(xi, ref_dx.cpu(), f"{name} no-alloc in-place dx")
    assert_parity(db, ref_db.cpu(), f"{name} no-alloc in-place dbias")


def _against_oracle(dy, x, bias, dx, db, what):
    """dx element by element against the oracle's once-rounded value, dbias
    against the exact column sums within the fixed-order fp32 summation bound
    the other bias tests use."""
    from test_bias_weighted_gpu import _bias_depth, assert_reduction

    dy_c, x_c, b_c = dy.cpu(), x.cpu(), bias.cpu()
    rows, n = dy_c.shape
    assert_parity(dx, oracle.bias_bwd(dy_c, x_c, b_c)[0], f"{what} dx vs oracle")
    dx64, db64 = oracle.bias_bwd(dy_c.double(), x_c.double(), b_c.double())
    assert_reduction(db, db64, dx64.abs().sum(0), _bias_depth(rows, n), f"{what} dbias vs oracle",
                     elem=x.dtype, count=rows)


def test_noalloc_refuses_what_does_not_fit(sw):
    # one row of n = 2^22: a single row group already needs 2 * n * 4 = 32 MiB
    n = 1 << 22
    need = sw.bias_bwd_workspace_bytes(1, n)
    limit = 16 << 20
    assert need > limit
    x = torch.zeros(1, 2 * n, dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros(1, n, dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(2 * n, dtype=torch.bfloat16, device="cuda")
    dx = torch.full_like(x, 5.0)
    db = torch.full_like(bias, 5.0)
    assert _noalloc(sw, dy, x, bias, dx, db) == -7
    torch.cuda.synchronize()
    assert bool((dx == 5.0).all()) and bool((db == 5.0).all())
