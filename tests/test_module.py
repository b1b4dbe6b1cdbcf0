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
