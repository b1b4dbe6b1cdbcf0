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


@pytest.mark.parametrize("name,rows", [("tiny_f32", None), ("megatron_4096_bf16", 96),
                                       ("odd_5503_f32", 40)])
@pytest.mark.parametrize("in_place", [False, True])
def test_bias_and_weighted_autograd_match_oracle(ag, name, rows, in_place):
    """Bias, per-token weights, and both, through autograd: every gradient the
    graph asks for (input, bias, weights) against the oracle."""
    w = W.WORKLOADS[name]
    x_cpu, dy_cpu = W.make_inputs(w, "cpu", rows=rows)
    r, n = x_cpu.shape[0], w.n
    g = torch.Generator().manual_seed(21)
    b_cpu = (torch.randn(2 * n, generator=g) * 0.5).to(x_cpu.dtype)
    w_cpu = torch.rand(r, 1, generator=g)  # Megatron's [tokens, 1] routing weights
    dy = dy_cpu.cuda()

    leaf = x_cpu.cuda().requires_grad_(True)
    bias = b_cpu.cuda().requires_grad_(True)
    y = ag.bias_gate_up_swiglu(leaf * 1, bias, in_place)
    assert_parity(y.detach(), oracle.bias_fwd(x_cpu, b_cpu), f"{name} bias fwd")
    y.backward(dy)
    rdx, _ = oracle.bias_bwd(dy_cpu, x_cpu, b_cpu)
    assert_parity(leaf.grad, rdx, f"{name} bias dx")
    import gate_up_swiglu_gb300 as sw

    # the reductions (bounded against the oracle in the variant tests) are
    # deterministic, so autograd must hand back exactly the kernels' sums
    _, db_ref = sw.swiglu_gateup_bias_bwd(dy, x_cpu.cuda(), b_cpu.cuda())
    assert_bitwise(bias.grad, db_ref, f"{name} autograd dbias is the kernel's")

    for with_bias in (False, True):
        leaf = x_cpu.cuda().requires_grad_(True)
        wts = w_cpu.cuda().requires_grad_(True)
        bias = b_cpu.cuda().requires_grad_(True) if with_bias else None
        y = ag.weighted_gate_up_swiglu(leaf * 1, bias, wts, in_place)
        y.backward(dy)
        w32 = w_cpu.view(-1).cuda()
        if with_bias:
            assert_parity(y.detach(), oracle.weighted_bias_fwd(x_cpu, b_cpu, w_cpu.view(-1)),
                          f"{name} weighted bias fwd")
            rdx, _, _ = oracle.weighted_bias_bwd(dy_cpu, x_cpu, b_cpu, w_cpu.view(-1))
            _, db_ref, dw_ref = sw.swiglu_gateup_weighted_bias_bwd(dy, x_cpu.cuda(), b_cpu.cuda(), w32)
            assert_bitwise(bias.grad, db_ref, f"{name} autograd weighted dbias")
        else:
            assert_parity(y.detach(), oracle.weighted_fwd(x_cpu, w_cpu.view(-1)),
                          f"{name} weighted fwd")
            rdx, _ = oracle.weighted_bwd(dy_cpu, x_cpu, w_cpu.view(-1))
            _, dw_ref = sw.swiglu_gateup_weighted_bwd(dy, x_cpu.cuda(), w32)
        assert_parity(leaf.grad, rdx, f"{name} weighted dx (bias={with_bias})")
        assert wts.grad.shape == (r, 1) and wts.grad.dtype == torch.float32
        assert_bitwise(wts.grad.view(-1), dw_ref, f"{name} autograd dw (bias={with_bias})")


def test_module_native_bias_and_weighted_module(ag):
    w = W.WORKLOADS["megatron_4096_bf16"]
    x_cpu, dy_cpu = W.make_inputs(w, "cpu", rows=64)
    n = w.n
    b_cpu = (torch.randn(2 * n, generator=torch.Generator().manual_seed(3)) * 0.5).to(torch.bfloat16)
    x3 = x_cpu.cuda().view(16, 4, 2 * n)
    m = ag.GateUpSwiGLU(native_bias=True)  # no fallback needed
    y = m(x3, b_cpu.cuda())
    assert y.shape == (16, 4, n)
    assert_parity(y.detach().view(64, n), oracle.bias_fwd(x_cpu, b_cpu), "native bias module fwd")
    mw = ag.WeightedGateUpSwiGLU()
    wts = torch.rand(64, 1, generator=torch.Generator().manual_seed(4))
    yw = mw(x3, None, wts.cuda())
    assert_parity(yw.detach().view(64, n), oracle.weighted_fwd(x_cpu, wts.view(-1)),
                  "weighted module fwd")
    with pytest.raises(NotImplementedError):
        mw(x3, None, wts.cuda(), True)


def test_function_forms_match_the_modules(ag):
    w = W.WORKLOADS["megatron_4096_bf16"]
    x_cpu, dy_cpu = W.make_inputs(w, "cpu", rows=64)
    n = w.n
    b_cpu = (torch.randn(2 * n, generator=torch.Generator().manual_seed(5)) * 0.5).to(torch.bfloat16)
    wts = torch.rand(64, 1, generator=torch.Generator().manual_seed(6))
    x3 = x_cpu.cuda().view(16, 4, 2 * n)
    y = ag.bias_swiglu_impl(x3, b_cpu.cuda())
    assert_parity(y.view(64, n), oracle.bias_fwd(x_cpu, b_cpu), "bias_swiglu_impl")
    y0 = ag.bias_swiglu_impl(x3, None)
    assert_parity(y0.view(64, n), oracle.fwd(x_cpu), "bias_swiglu_impl without bias")
    yw = ag.weighted_bias_swiglu_impl(x_cpu.cuda(), b_cpu.cuda(), wts.cuda())
    assert_parity(yw, oracle.weighted_bias_fwd(x_cpu, b_cpu, wts.view(-1)), "weighted_bias_swiglu_impl")
