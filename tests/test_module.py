"""Policy of the Megatron-style module that needs no GPU: unsupported Megatron
features go to the fallback (logged once) or raise, and bad shapes are
rejected before any kernel is called."""
import logging

import pytest
import torch


@pytest.fixture(scope="module")
def mod():
    from conftest import build_library

    build_library()
    from gate_up_swiglu_gb300.autograd import GateUpSwiGLU

    return GateUpSwiGLU


def test_unsupported_features_raise_without_fallback(mod):
    m = mod()
    x = torch.zeros(4, 8)
    with pytest.raises(NotImplementedError, match="bias"):
        m(x, torch.zeros(8))
    with pytest.raises(NotImplementedError, match="fp8_input_store"):
        m(x, None, True, False)
    with pytest.raises(NotImplementedError, match="cpu_offload_input"):
        m(x, None, False, True)


def test_fallback_called_and_logged_once(mod, caplog):
    calls = []

    def fallback(inter, bias, fp8, off):
        calls.append((inter.shape, bias is None, fp8, off))
        return "fallback-result"

    m = mod(fallback_impl=fallback)
    x = torch.zeros(4, 8)
    with caplog.at_level(logging.WARNING):
        assert m(x, torch.zeros(8)) == "fallback-result"
        assert m(x, torch.zeros(8)) == "fallback-result"
        assert m(x, None, True, False) == "fallback-result"
    assert len(calls) == 3
    msgs = [r.getMessage() for r in caplog.records]
    assert sum("bias is not None" in s for s in msgs) == 1
    assert sum("fp8_input_store" in s for s in msgs) == 1


def test_shape_and_dtype_validation(mod):
    m = mod()
    with pytest.raises(ValueError, match="2D"):
        m(torch.zeros(8))
    with pytest.raises(ValueError, match="even"):
        m(torch.zeros(4, 7))
    with pytest.raises(ValueError, match="dtype"):
        m(torch.zeros(4, 8, dtype=torch.float16))


def test_native_bias_skips_the_fallback(mod):
    def fallback(*a):
        raise AssertionError("fallback must not be called with native_bias=True")

    m = mod(fallback_impl=fallback, native_bias=True)
    with pytest.raises(ValueError, match="even"):  # validated, then the kernels would run
        m(torch.zeros(4, 7), torch.zeros(7))


def test_weighted_module_policy(caplog):
    from conftest import build_library

    build_library()
    from gate_up_swiglu_gb300.autograd import WeightedGateUpSwiGLU

    with pytest.raises(NotImplementedError, match="fp8_input_store"):
        WeightedGateUpSwiGLU()(torch.zeros(4, 8), None, torch.ones(4), True)
    calls = []
    m = WeightedGateUpSwiGLU(fallback_impl=lambda *a: calls.append(a) or "fb")
    with caplog.at_level(logging.WARNING):
        assert m(torch.zeros(4, 8), None, torch.ones(4), True) == "fb"
        assert m(torch.zeros(4, 8), None, torch.ones(4), True) == "fb"
    assert len(calls) == 2
    assert sum("fp8_input_store" in r.getMessage() for r in caplog.records) == 1
    with pytest.raises(ValueError, match="even"):
        m(torch.zeros(4, 7), None, torch.ones(4))
    with pytest.raises(ValueError, match="dtype"):
        m(torch.zeros(4, 8, dtype=torch.float16), None, torch.ones(4))


def test_function_forms_policy():
    from conftest import build_library

    build_library()
    from gate_up_swiglu_gb300.autograd import bias_swiglu_impl, weighted_bias_swiglu_impl

    x = torch.zeros(4, 8)
    with pytest.raises(NotImplementedError, match="fp8_input_store"):
        bias_swiglu_impl(x, None, True, False)
    with pytest.raises(NotImplementedError, match="cpu_offload_input"):
        bias_swiglu_impl(x, None, False, True)
    with pytest.raises(NotImplementedError, match="fp8_input_store"):
        weighted_bias_swiglu_impl(x, None, torch.ones(4), True)
    with pytest.raises(ValueError, match="even"):
        bias_swiglu_impl(torch.zeros(4, 7), None)
