"""Launch order: the streaming kernels launch early (programmatic dependent
launch) and wait inside for the grid before them in the stream.

A chain in which every call reads what the call before it wrote is run once
with no synchronisation and once with a device synchronisation after every
call; the two must agree bit for bit.  Steps alternate between the library's
kernels and torch kernels (which launch the ordinary way), so a library
kernel that read or wrote before its predecessor completed, or a torch kernel
that ran before a library kernel finished, would show as a difference.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


def _chain(sw, x, dy, bias, w, steps, sync):
    """Each step: y = fwd(x); dy = y / 2 (torch); dx over x in place; x scaled
    back into range (torch); then the bias and weights + bias backward on the
    new x, whose dbias feeds the next step's bias and whose dw the next
    weights."""
    done = torch.cuda.synchronize if sync else (lambda: None)
    out = []
    for _ in range(steps):
        y = sw.swiglu_gateup_fwd(x)
        done()
        dy.copy_(y * 0.5)
        done()
        sw.swiglu_gateup_bwd(dy, x, in_place=True)
        done()
        x.mul_(4.0).clamp_(-6.0, 6.0)
        done()
        dx_b, dbias = sw.swiglu_gateup_bias_bwd(dy, x, bias)
        done()
        bias = (dbias * 1e-3).to(x.dtype)
        done()
        dx_w, dbias_w, dw = sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, w)
        done()
        w = (dw.abs() * 1e-2 + 0.5).contiguous()
        done()
        out += [y, dx_b, dbias, dx_w, dbias_w, dw]
    torch.cuda.synchronize()
    return out + [x, bias, w]


@pytest.mark.parametrize("rows,n", [(8192, 4096), (300, 5000)])
def test_dependent_chain_without_sync_matches_synchronised(sw, rows, n):
    g = torch.Generator(device="cuda").manual_seed(rows + n)
    x0 = (torch.randn(rows, 2 * n, generator=g, device="cuda") * 2).to(torch.bfloat16)
    dy = torch.empty(rows, n, dtype=torch.bfloat16, device="cuda")
    b0 = (torch.randn(2 * n, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    w0 = torch.rand(rows, generator=g, device="cuda")
    free = _chain(sw, x0.clone(), dy.clone(), b0.clone(), w0.clone(), 4, sync=False)
    synced = _chain(sw, x0.clone(), dy.clone(), b0.clone(), w0.clone(), 4, sync=True)
    assert len(free) == len(synced)
    for i, (a, b) in enumerate(zip(free, synced)):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), \
            f"tensor {i} of the chain differs without synchronisation"
