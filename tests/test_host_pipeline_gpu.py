"""The host-buffer pipeline (swiglu_gateup_fwd_bwd_host, through the C ABI)
produces exactly what the device entry points produce -- the same kernels,
chunk by chunk, with the backward in place over the staged input -- for ragged
chunking, one to four slots, and three streams or one; and matches the oracle
on every element."""
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


def _host_inputs(name, rows):
    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cpu", rows=rows)
    x = x.contiguous()
    xh, dyh = x.pin_memory(), dy.pin_memory()
    yh = torch.empty((x.shape[0], w.n), dtype=x.dtype).pin_memory()
    dxh = torch.empty_like(x).pin_memory()
    return w, x, dy, xh, dyh, yh, dxh


@pytest.mark.parametrize("name,rows,chunk,depth", [("megatron_4096_bf16", 1000, 128, 3),
                                                   ("odd_5503_f32", 301, 64, 2),
                                                   ("tiny_f32", None, 7, 4),
                                                   ("megatron_4096_bf16", 257, 1000, 1)])
def test_host_pipeline_equals_device_path(sw, name, rows, chunk, depth):
    from gate_up_swiglu_gb300.host_pipeline import HostPipeline, gateup_fwd_bwd_host

    w, x, dy, xh, dyh, yh, dxh = _host_inputs(name, rows)
    pipe = HostPipeline("cuda", chunk, depth=depth)
    y_ref = sw.swiglu_gateup_fwd(x.cuda()).cpu()
    dx_ref = sw.swiglu_gateup_bwd(dy.cuda(), x.cuda()).cpu()
    for _ in range(2):  # the second call reuses the staging buffer
        yh.fill_(float("nan"))
        dxh.fill_(float("nan"))
        gateup_fwd_bwd_host(xh, dyh, yh, dxh, pipe)
        assert_bitwise(yh, y_ref, f"{name} host pipeline y")
        assert_bitwise(dxh, dx_ref, f"{name} host pipeline dx")
    assert_parity(yh, oracle.fwd(x), f"{name} host pipeline fwd vs oracle")
    assert_parity(dxh, oracle.bwd(dy, x), f"{name} host pipeline bwd vs oracle")
    # the inputs in host memory are untouched
    assert_bitwise(xh, x, f"{name} host x unchanged")


def test_host_pipeline_one_stream_and_rejections(sw):
    """All three roles on one stream (no overlap, same bits); a short staging
    buffer is refused before anything is copied."""
    w, x, dy, xh, dyh, yh, dxh = _host_inputs("odd_5503_f32", 77)
    s = torch.cuda.Stream()
    need = sw.host_staging_bytes(10, w.n, x.dtype, 2)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    sw.swiglu_gateup_fwd_bwd_host(xh, dyh, yh, dxh, staging, 10, 2, (s, s, s))
    assert_parity(yh, oracle.fwd(x), "one-stream fwd")
    assert_parity(dxh, oracle.bwd(dy, x), "one-stream bwd")
    yh.fill_(7.0)
    with pytest.raises(sw.SwigluError) as e:
        sw.swiglu_gateup_fwd_bwd_host(xh, dyh, yh, dxh, staging[: need - 256], 10, 2, (s, s, s))
    assert e.value.status == -7
    assert bool((yh == 7.0).all())


def test_host_pipeline_full_size_large(sw):
    """The bench's end-to-end configuration: the large-FFN workload from pinned
    host memory, 64 MB chunks, three slots; every element against the device
    path's bits."""
    from gate_up_swiglu_gb300.host_pipeline import HostPipeline, default_chunk_rows, gateup_fwd_bwd_host

    w = W.WORKLOADS["large_32768_bf16"]
    x, dy = W.make_inputs(w, "cuda")
    x = x.contiguous()
    y_ref = sw.swiglu_gateup_fwd(x)
    dx_ref = sw.swiglu_gateup_bwd(dy, x)
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    dyh = torch.empty(dy.shape, dtype=dy.dtype, pin_memory=True)
    xh.copy_(x)
    dyh.copy_(dy)
    del x, dy
    yh = torch.empty(y_ref.shape, dtype=y_ref.dtype, pin_memory=True)
    dxh = torch.empty(dx_ref.shape, dtype=dx_ref.dtype, pin_memory=True)
    pipe = HostPipeline("cuda", default_chunk_rows(w.n, w.elem_bytes))
    gateup_fwd_bwd_host(xh, dyh, yh, dxh, pipe)
    assert_bitwise(yh, y_ref.cpu(), "large host pipeline y")
    assert_bitwise(dxh, dx_ref.cpu(), "large host pipeline dx")
