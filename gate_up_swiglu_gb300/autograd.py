"""Autograd function and Megatron-style module over the libswiglu C ABI.

The user-facing layer of the Liger-Kernel Megatron SwiGLU page:
``GateUpSwiGLUFunction`` plays the part of its fused gate-up autograd function
(§What's added) and ``GateUpSwiGLU`` the part of its Megatron module: the
positional signature of Megatron's ``bias_swiglu_impl`` (§How to use, Mode 2),
the opt-in ``in_place`` backward (§Optional in_place=True), the delegation of
unsupported Megatron features to a fallback that is logged once, or an error
when no fallback is given (§Scope), and the guard against a second backward
after an in-place one (§Known issues 1).

All arithmetic runs in the CUDA kernels; this module only decides what to call.
"""
from __future__ import annotations

import logging
import math
from typing import Callable, Optional

import torch

from . import (swiglu_gateup_bias_bwd, swiglu_gateup_bias_fwd, swiglu_gateup_bwd,
               swiglu_gateup_fwd, swiglu_gateup_weighted_bias_bwd,
               swiglu_gateup_weighted_bias_fwd, swiglu_gateup_weighted_bwd,
               swiglu_gateup_weighted_fwd)

log = logging.getLogger(__name__)


def _bump_version(t: torch.Tensor) -> None:
    # the kernel writes through a raw pointer, which autograd cannot see
    inc = getattr(torch.autograd.graph, "increment_version", None)
    if inc is not None:
        inc(t)


class GateUpSwiGLUFunction(torch.autograd.Function):
    """y = silu(x[..., :n]) * x[..., n:] with the fused backward.

    ``in_place=True`` makes the backward write the gradient over the saved fc1
    buffer ``x`` and return that buffer as the input gradient: no extra
    ``[..., 2n]`` allocation, and ``x`` is destroyed.  Running the backward a
    second time over the same graph (``retain_graph=True``) then raises instead
    of silently producing garbage.
    """

    @staticmethod
    def forward(ctx, x: torch.Tensor, in_place: bool = False):
        y = swiglu_gateup_fwd(x)
        ctx.save_for_backward(x)
        ctx.in_place = bool(in_place)
        ctx.already_backward = False
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        # checked before the saved buffer is unpacked: after an in-place backward
        # autograd's own version check would fire with a less specific message
        if ctx.in_place:
            if ctx.already_backward:
                raise RuntimeError(
                    "GateUpSwiGLUFunction: backward already ran with in_place=True, which "
                    "overwrote the saved fc1 buffer; a second backward (retain_graph=True) "
                    "would compute garbage")
            ctx.already_backward = True
        (x,) = ctx.saved_tensors
        dy = dy.contiguous()
        if ctx.in_place:
            dx = swiglu_gateup_bwd(dy, x, in_place=True)
            _bump_version(x)
        else:
            dx = swiglu_gateup_bwd(dy, x)
        return dx, None


def gate_up_swiglu(x: torch.Tensor, in_place: bool = False) -> torch.Tensor:
    return GateUpSwiGLUFunction.apply(x, in_place)


def _guard_second_backward(ctx, name: str) -> None:
    if ctx.in_place:
        if ctx.already_backward:
            raise RuntimeError(f"{name}: backward already ran with in_place=True, which overwrote "
                               "the saved fc1 buffer; a second backward (retain_graph=True) would "
                               "compute garbage")
        ctx.already_backward = True


class BiasGateUpSwiGLUFunction(torch.autograd.Function):
    """y = silu(x[..., :n] + bias[:n]) * (x[..., n:] + bias[n:]) -- Megatron's
    bias_swiglu_impl with a bias -- returning (dx, dbias) from one fused
    backward (the column sums of dbias are a deterministic two-pass reduction
    in the kernels).  ``in_place`` as for GateUpSwiGLUFunction."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, bias: torch.Tensor, in_place: bool = False):
        bias = bias.contiguous()
        y = swiglu_gateup_bias_fwd(x, bias)
        ctx.save_for_backward(x, bias)
        ctx.in_place = bool(in_place)
        ctx.already_backward = False
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        _guard_second_backward(ctx, "BiasGateUpSwiGLUFunction")
        x, bias = ctx.saved_tensors
        dx, dbias = swiglu_gateup_bias_bwd(dy.contiguous(), x, bias, in_place=ctx.in_place)
        if ctx.in_place:
            _bump_version(x)
        return dx, dbias, None


class WeightedGateUpSwiGLUFunction(torch.autograd.Function):
    """y = w[token] * silu(g + bias_g) * (u + bias_u) -- the per-token-scaled
    SwiGLU of MoE routed experts (Megatron's weighted_bias_swiglu_impl) --
    with the bias optional.  ``weights`` holds one routing weight per row
    (shape ``[tokens]`` or ``[tokens, 1]``, any float dtype; the kernels take
    it as fp32).  The backward returns dx, dbias (when there is a bias) and the
    weight gradient in the weights' shape and dtype."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, bias: Optional[torch.Tensor], weights: torch.Tensor,
                in_place: bool = False):
        rows = math.prod(x.shape[:-1])
        if weights.numel() != rows:
            raise ValueError(f"weights must hold one value per row ({rows}), got shape "
                             f"{tuple(weights.shape)}")
        w32 = weights.detach().reshape(-1).to(torch.float32).contiguous()
        if bias is None:
            y = swiglu_gateup_weighted_fwd(x, w32)
        else:
            bias = bias.contiguous()
            y = swiglu_gateup_weighted_bias_fwd(x, bias, w32)
        ctx.save_for_backward(x, bias, w32)
        ctx.has_bias = bias is not None
        ctx.w_shape, ctx.w_dtype = weights.shape, weights.dtype
        ctx.in_place = bool(in_place)
        ctx.already_backward = False
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        _guard_second_backward(ctx, "WeightedGateUpSwiGLUFunction")
        x, bias, w32 = ctx.saved_tensors
        dy = dy.contiguous()
        dbias = None
        if ctx.has_bias:
            dx, dbias, dw = swiglu_gateup_weighted_bias_bwd(dy, x, bias, w32, in_place=ctx.in_place)
        else:
            dx, dw = swiglu_gateup_weighted_bwd(dy, x, w32, in_place=ctx.in_place)
        if ctx.in_place:
            _bump_version(x)
        return dx, dbias, dw.reshape(ctx.w_shape).to(ctx.w_dtype), None


def bias_gate_up_swiglu(x: torch.Tensor, bias: torch.Tensor, in_place: bool = False) -> torch.Tensor:
    return BiasGateUpSwiGLUFunction.apply(x, bias, in_place)


def weighted_gate_up_swiglu(x: torch.Tensor, bias: Optional[torch.Tensor], weights: torch.Tensor,
                            in_place: bool = False) -> torch.Tensor:
    return WeightedGateUpSwiGLUFunction.apply(x, bias, weights, in_place)


class GateUpSwiGLU(torch.nn.Module):
    """Drop-in for Megatron's ``bias_swiglu_impl(intermediate, bias,
    fp8_input_store, cpu_offload_input)``.

    Supported: ``bias=None``, fp32 or bf16, 2D ``[tokens, 2n]`` or 3D
    ``[s, b, 2n]`` CUDA tensors.  A call that needs a feature the kernels do
    not have (fp8 input storage, cpu offload of the input) goes to
    ``fallback_impl`` (logged once per reason); with ``fallback_impl=None`` it
    raises ``NotImplementedError``.  A bias is delegated the same way, as the
    page's module does, unless ``native_bias=True``: then the fused bias
    kernels take it (BiasGateUpSwiGLUFunction).
    """

    def __init__(self, in_place: bool = False,
                 fallback_impl: Optional[Callable] = None, native_bias: bool = False):
        super().__init__()
        self.in_place = in_place
        self.fallback_impl = fallback_impl
        self.native_bias = native_bias
        self._logged = set()

    def _unsupported(self, bias, fp8_input_store, cpu_offload_input) -> Optional[str]:
        if bias is not None and not self.native_bias:
            return "bias is not None"
        if fp8_input_store:
            return "fp8_input_store=True"
        if cpu_offload_input:
            return "cpu_offload_input=True"
        return None

    def forward(self, intermediate: torch.Tensor, bias: Optional[torch.Tensor] = None,
                fp8_input_store: bool = False, cpu_offload_input: bool = False) -> torch.Tensor:
        reason = self._unsupported(bias, fp8_input_store, cpu_offload_input)
        if reason is not None:
            if self.fallback_impl is None:
                raise NotImplementedError(f"GateUpSwiGLU: {reason} is not supported by the fused "
                                          "kernels and no fallback_impl was given")
            if reason not in self._logged:
                self._logged.add(reason)
                log.warning("GateUpSwiGLU: %s; delegating to the fallback implementation", reason)
            return self.fallback_impl(intermediate, bias, fp8_input_store, cpu_offload_input)
        if intermediate.dim() not in (2, 3):
            raise ValueError(f"GateUpSwiGLU: expected a 2D [tokens, 2n] or 3D [s, b, 2n] input, "
                             f"got shape {tuple(intermediate.shape)}")
        if intermediate.shape[-1] % 2:
            raise ValueError("GateUpSwiGLU: the last dimension (2n) must be even")
        if intermediate.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError(f"GateUpSwiGLU: dtype {intermediate.dtype} is not supported "
                             "(float32 or bfloat16)")
        if bias is not None:
            return BiasGateUpSwiGLUFunction.apply(intermediate, bias, self.in_place)
        return GateUpSwiGLUFunction.apply(intermediate, self.in_place)


class WeightedGateUpSwiGLU(torch.nn.Module):
    """Drop-in for Megatron's ``weighted_bias_swiglu_impl(input, bias, weights,
    fp8_input_store)`` of MoE routed experts: y = weights[token] * swiglu, the
    bias optional.  fp8 input storage goes to ``fallback_impl`` (logged once),
    or raises ``NotImplementedError`` without one."""

    def __init__(self, in_place: bool = False, fallback_impl: Optional[Callable] = None):
        super().__init__()
        self.in_place = in_place
        self.fallback_impl = fallback_impl
        self._logged = False

    def forward(self, intermediate: torch.Tensor, bias: Optional[torch.Tensor],
                weights: torch.Tensor, fp8_input_store: bool = False) -> torch.Tensor:
        if fp8_input_store:
            if self.fallback_impl is None:
                raise NotImplementedError("WeightedGateUpSwiGLU: fp8_input_store=True is not "
                                          "supported by the fused kernels and no fallback_impl "
                                          "was given")
            if not self._logged:
                self._logged = True
                log.warning("WeightedGateUpSwiGLU: fp8_input_store=True; delegating to the "
                            "fallback implementation")
            return self.fallback_impl(intermediate, bias, weights, fp8_input_store)
        if intermediate.dim() not in (2, 3) or intermediate.shape[-1] % 2:
            raise ValueError("WeightedGateUpSwiGLU: expected a 2D [tokens, 2n] or 3D [s, b, 2n] "
                             f"input with even last dimension, got {tuple(intermediate.shape)}")
        if intermediate.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError(f"WeightedGateUpSwiGLU: dtype {intermediate.dtype} is not supported "
                             "(float32 or bfloat16)")
        return WeightedGateUpSwiGLUFunction.apply(intermediate, bias, weights, self.in_place)


class Fc1SwiGLUFunction(torch.autograd.Function):
    """linear_fc1 followed by the activation, y = silu((X W^T)[..., :n]) *
    (X W^T)[..., n:], with the activation in the tensor-core GEMM's epilogue.

    The forward stores the bf16 fc1 output for the backward (the buffer the
    Megatron layout keeps); the backward runs the fused activation backward on
    it -- in place when ``in_place`` -- and then the two plain GEMMs
    dX = d(fc1) W and dW = d(fc1)^T X through cuBLAS."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: torch.Tensor, in_place: bool = False):
        from . import swiglu_fc1_fwd

        y, fc1 = swiglu_fc1_fwd(x.contiguous(), weight.contiguous(), return_fc1=True)
        ctx.save_for_backward(x, weight, fc1)
        ctx.in_place = bool(in_place)
        ctx.already_backward = False
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        if ctx.in_place:
            if ctx.already_backward:
                raise RuntimeError("Fc1SwiGLUFunction: backward already ran with in_place=True")
            ctx.already_backward = True
        x, weight, fc1 = ctx.saved_tensors
        dfc1 = swiglu_gateup_bwd(dy.contiguous(), fc1, in_place=ctx.in_place)
        k = x.shape[-1]
        d2 = dfc1.reshape(-1, dfc1.shape[-1])
        dx = (d2 @ weight).reshape(x.shape) if ctx.needs_input_grad[0] else None
        dw = d2.t() @ x.reshape(-1, k) if ctx.needs_input_grad[1] else None
        return dx, dw, None


class Fc1SwiGLU(torch.nn.Module):
    """Megatron's linear_fc1 (bias-free, gate rows then up rows in one
    [2 * ffn_hidden, in_features] weight) fused with the activation."""

    def __init__(self, in_features: int, ffn_hidden: int, in_place: bool = False,
                 device=None, dtype=torch.bfloat16):
        super().__init__()
        self.weight = torch.nn.Parameter(
            torch.empty(2 * ffn_hidden, in_features, device=device, dtype=dtype))
        torch.nn.init.normal_(self.weight, std=in_features ** -0.5)
        self.in_place = in_place

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return Fc1SwiGLUFunction.apply(x, self.weight, self.in_place)


# Function forms with the positional signatures of Megatron's activation
# entry points, for code that calls (or patches in) a function rather than a
# module.  A bias goes to the fused bias kernels; fp8 input storage and cpu
# offload of the input are not supported and raise.
_plain_module = GateUpSwiGLU(native_bias=True)
_weighted_module = WeightedGateUpSwiGLU()


def bias_swiglu_impl(input: torch.Tensor, bias: Optional[torch.Tensor],
                     fp8_input_store: bool = False, cpu_offload_input: bool = False) -> torch.Tensor:
    """silu(input[..., :n] + bias[:n]) * (input[..., n:] + bias[n:]) (bias optional),
    differentiable, on the fused kernels; 2D or 3D input."""
    return _plain_module(input, bias, fp8_input_store, cpu_offload_input)


def weighted_bias_swiglu_impl(input: torch.Tensor, bias: Optional[torch.Tensor],
                              weights: torch.Tensor, fp8_input_store: bool = False) -> torch.Tensor:
    """weights[token] * the SwiGLU above (MoE routed experts), differentiable in
    input, bias and weights."""
    return _weighted_module(input, bias, weights, fp8_input_store)
