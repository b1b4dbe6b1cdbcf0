"""The host-buffer pipeline produces exactly what the device entry points
produce (same kernels, chunk by chunk), for ragged chunking, and matches the
oracle."""
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bitwise, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


@pytest.mark.parametrize("name,rows,chunk", [("megatron_4096_bf16", 1000, 128),
                                             ("odd_5503_f32", 301, 64),
                                             ("tiny_f32", None, 7)])
def test_host_pipeline_equals_device_path(sw, name, rows, chunk):
    from gate_up_swiglu_gb300.host_pipeline import HostPipeline, gateup_fwd_bwd_host

    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cpu", rows=rows)
    x = x.contiguous()
    xh, dyh = x.pin_memory(), dy.pin_memory()
    yh = torch.empty((x.shape[0], w.n), dtype=x.dtype).pin_memory()
    dxh = torch.empty_like(x).pin_memory()
    pipe = HostPipeline("cuda", chunk)
    for _ in range(2):  # the second call reuses the staging buffers
        yh.fill_(float("nan"))
        dxh.fill_(float("nan"))
        gateup_fwd_bwd_host(xh, dyh, yh, dxh, pipe)
        y_ref = sw.swiglu_gateup_fwd(x.cuda())
        dx_ref = sw.swiglu_gateup_bwd(dy.cuda(), x.cuda())
        assert_bitwise(yh, y_ref.cpu(), f"{name} host pipeline y")
        assert_bitwise(dxh, dx_ref.cpu(), f"{name} host pipeline dx")
    assert_parity(yh, oracle.fwd(x), f"{name} host pipeline vs oracle")
