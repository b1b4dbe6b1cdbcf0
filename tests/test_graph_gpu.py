"""The entry points inside a CUDA graph: captured once after an eager warm-up
(which fills the library's per-device caches), replayed, and bit-identical to
eager calls on the same inputs -- including the bias and weights + bias
backward with their workspaces and reduction passes, and the in-place form.
Replaying after the inputs change must give the new results (no value is
baked into the graph)."""
import pytest
import torch

import workloads as W
from helpers import assert_bitwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sw():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    return sw


@pytest.mark.parametrize("name,rows", [("megatron_4096_bf16", 512), ("odd_5503_f32", 64)])
def test_graph_replay_matches_eager(sw, name, rows):
    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cuda", rows=rows)
    x = x.contiguous()
    n = w.n
    g = torch.Generator(device="cuda").manual_seed(3)
    bias = (torch.randn(2 * n, device="cuda", generator=g) * 0.5).to(x.dtype)
    wts = torch.rand(rows, device="cuda", generator=g)
    y, dx, dxb, dxw = (torch.empty(rows, n, dtype=x.dtype, device="cuda"), torch.empty_like(x),
                       torch.empty_like(x), torch.empty_like(x))
    xi = torch.empty_like(x)
    db, db2 = torch.empty_like(bias), torch.empty_like(bias)
    dw = torch.empty_like(wts)
    ws = torch.empty(sw.weighted_bias_bwd_workspace_bytes(rows, n), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty_like(ws)

    def step(s):
        sw.swiglu_gateup_fwd(x, y, stream=s)
        sw.swiglu_gateup_bwd(dy, x, dx, stream=s)
        xi.copy_(x)
        sw.swiglu_gateup_bwd(dy, xi, in_place=True, stream=s)
        sw.swiglu_gateup_bias_bwd(dy, x, bias, dxb, db, ws, stream=s)
        sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts, dxw, db2, dw, ws2, stream=s)

    def snapshot():
        return [t.clone() for t in (y, dx, xi, dxb, db, dxw, db2, dw)]

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = snapshot()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for t in (y, dx, xi, dxb, db, dxw, db2, dw):
        t.fill_(0)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b, what in zip(snapshot(), eager, ("y", "dx", "in-place dx", "bias dx", "dbias",
                                              "weighted bias dx", "weighted dbias", "dw")):
        assert_bitwise(a, b, f"graph replay {what}")

    # new input values, same buffers: the replay recomputes
    x.mul_(-0.5)
    dy.mul_(2)
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    eager2 = snapshot()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(snapshot(), eager2):
        assert_bitwise(a, b, "graph replay after input change")


def test_fc1_graph_replay_matches_eager(sw):
    M, K, n = 512, 1024, 384
    g = torch.Generator(device="cuda").manual_seed(4)
    X = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    Wt = (torch.randn(2 * n, K, device="cuda", generator=g) * K ** -0.5).to(torch.bfloat16)
    y = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
    fc1 = torch.empty(M, 2 * n, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sw.swiglu_fc1_fwd(X, Wt, y, x_out=fc1, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ey, efc1 = y.clone(), fc1.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        sw.swiglu_fc1_fwd(X, Wt, y, x_out=fc1, stream=s)
    y.zero_()
    fc1.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert_bitwise(y, ey, "fc1 graph y")
    assert_bitwise(fc1, efc1, "fc1 graph fc1")
    assert sw.fc1_timeout_flag() == 0
