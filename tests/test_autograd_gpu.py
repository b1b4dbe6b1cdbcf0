"""The autograd function and module on the GPU: gradients through autograd
equal the oracle, the in-place backward reuses the fc1 buffer and refuses a
second backward, and the module delegates a bias to its fallback."""
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bitwise, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ag():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300.autograd as ag

    return ag


@pytest.mark.parametrize("name,rows", [("tiny_f32", None), ("megatron_4096_bf16", 96),
                                       ("odd_5503_f32", 40)])
@pytest.mark.parametrize("in_place", [False, True])
def test_autograd_matches_oracle(ag, name, rows, in_place):
    w = W.WORKLOADS[name]
    x_cpu, dy_cpu = W.make_inputs(w, "cpu", rows=rows)
    leaf = x_cpu.cuda().requires_grad_(True)
    x = leaf * 1  # a non-leaf fc1 output, as in Megatron
    y = ag.GateUpSwiGLUFunction.apply(x, in_place)
    assert_parity(y.detach(), oracle.fwd(x_cpu), f"{name} autograd fwd")
    y.backward(dy_cpu.cuda())
    assert_parity(leaf.grad, oracle.bwd(dy_cpu, x_cpu), f"{name} autograd bwd (in_place={in_place})")


def test_3d_module_and_in_place_reuses_buffer(ag):
    w = W.WORKLOADS["megatron_4096_bf16"]
    x_cpu, dy_cpu = W.make_inputs(w, "cpu", rows=64)
    x3 = x_cpu.cuda().view(16, 4, 2 * w.n)
    dy3 = dy_cpu.cuda().view(16, 4, w.n)
    ref = oracle.bwd(dy_cpu, x_cpu)

    leaf = x3.clone().requires_grad_(True)
    x = leaf * 1
    ptr = x.data_ptr()
    v0 = x._version
    y = ag.GateUpSwiGLU(in_place=True)(x)
    assert y.shape == (16, 4, w.n)
    y.backward(dy3)
    # the gradient now lives in the fc1 buffer itself
    assert x.data_ptr() == ptr and x._version > v0
    assert_bitwise(x.detach().view(64, 2 * w.n), leaf.grad.view(64, 2 * w.n), "grad is the buffer")
    assert_parity(leaf.grad.view(64, 2 * w.n), ref, "3D in-place module bwd")


def test_second_backward_after_in_place_raises(ag):
    x_cpu, dy_cpu = W.make_inputs(W.WORKLOADS["tiny_f32"], "cpu")
    for in_place in (False, True):
        leaf = x_cpu.cuda().requires_grad_(True)
        y = ag.GateUpSwiGLUFunction.apply(leaf * 1, in_place)
        y.backward(dy_cpu.cuda(), retain_graph=True)
        if in_place:
            with pytest.raises(RuntimeError, match="in_place=True"):
                y.backward(dy_cpu.cuda())
        else:
            g1 = leaf.grad.clone()
            y.backward(dy_cpu.cuda())
            assert torch.allclose(leaf.grad, 2 * g1)


def test_module_delegates_bias_to_fallback(ag):
    def megatron_like(inter, bias, fp8, off):
        a, b = (inter + bias).chunk(2, -1)
        return torch.nn.functional.silu(a) * b

    m = ag.GateUpSwiGLU(fallback_impl=megatron_like)
    x = torch.randn(8, 32, device="cuda")
    bias = torch.randn(32, device="cuda")
    out = m(x, bias)
    assert torch.allclose(out, megatron_like(x, bias, False, False))
    # without a bias the fused kernels run and agree with the oracle
    assert_parity(m(x), oracle.fwd(x.cpu()), "module fwd")
