"""Two-tensor entry points (gate a and up b as separate tensors) vs the oracle,
through the C ABI.  Same tolerances as the fused form (tests/helpers.py)."""
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


def _padded(t, pad, dev="cuda"):
    """t inside a wider row buffer (row stride = cols + pad), NaN padding."""
    rows, cols = t.shape
    buf = torch.full((rows, cols + pad), float("nan"), dtype=t.dtype, device=dev)
    buf[:, :cols] = t.to(dev)
    return buf[:, :cols]


CASES = [("bf16", 37, 4096, (0, 0, 0)), ("bf16", 29, 4100, (0, 8, 0)), ("bf16", 13, 999, (1, 3, 5)),
         ("f32", 37, 2048, (0, 0, 0)), ("f32", 31, 5503, (2, 0, 1)), ("f32", 3000, 5, (0, 0, 0))]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-r{c[1]}-n{c[2]}-p{c[3]}" for c in CASES])
def test_two_tensor_matches_oracle(sw, case):
    dts, rows, n, pads = case
    dt = torch.float32 if dts == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(rows + n)
    a = (torch.randn(rows, n, generator=g) * 4).to(dt)
    b = (torch.randn(rows, n, generator=g) * 2).to(dt)
    dc = torch.randn(rows, n, generator=g).to(dt)
    ad, bd, dcd = _padded(a, pads[0]), _padded(b, pads[1]), _padded(dc, pads[2])
    c = sw.swiglu_silu_mul_fwd(ad, bd)
    da, db = sw.swiglu_silu_mul_bwd(dcd, ad, bd)
    torch.cuda.synchronize()
    assert_parity(c, oracle.silu_mul_fwd(a, b), "two-tensor fwd")
    rda, rdb = oracle.silu_mul_bwd(dc, a, b)
    assert_parity(da, rda, "two-tensor da")
    assert_parity(db, rdb, "two-tensor db")
    # in place over a and b: same bits as out of place
    ai, bi = ad.clone(), bd.clone()
    sw.swiglu_silu_mul_bwd(dcd, ai, bi, in_place=True)
    assert_bitwise(ai, da, "in-place da")
    assert_bitwise(bi, db, "in-place db")
    # only da in place
    ai = ad.clone()
    _, db2 = sw.swiglu_silu_mul_bwd(dcd, ai, bd, da=ai)
    assert_bitwise(ai, da, "da over a") and assert_bitwise(db2, db, "db alongside")


def test_two_tensor_equals_fused_on_halves(sw):
    w = W.WORKLOADS["llama_14336_bf16_2d"]
    x, dy = W.make_inputs(w, "cuda", rows=128)
    a, b = x[:, :w.n].contiguous(), x[:, w.n:].contiguous()
    y = sw.swiglu_gateup_fwd(x)
    dx = sw.swiglu_gateup_bwd(dy, x)
    c = sw.swiglu_silu_mul_fwd(a, b)
    da, db = sw.swiglu_silu_mul_bwd(dy, a, b)
    assert_bitwise(c, y, "fwd")
    assert_bitwise(torch.cat([da, db], 1), dx, "bwd")
    # and the halves as strided views of the fused buffer itself
    c2 = sw.swiglu_silu_mul_fwd(x[:, :w.n], x[:, w.n:])
    assert_bitwise(c2, y, "fwd on views")


def test_two_tensor_full_size_hf_layout(sw):
    """Gate and up as separate [8192, 14336] bf16 tensors (Llama-3-8B-like MLP
    in HuggingFace layout); sampled rows against the oracle."""
    w = W.WORKLOADS["llama_14336_bf16_2d"]
    x, dy = W.make_inputs(w, "cuda")
    a, b = x[:, :w.n].contiguous(), x[:, w.n:].contiguous()
    del x
    c = sw.swiglu_silu_mul_fwd(a, b)
    da, db = sw.swiglu_silu_mul_bwd(dy, a, b)
    torch.cuda.synchronize()
    idx = torch.tensor([0, 1, 4095, 8190, 8191] + list(range(17, 8000, 397)), device="cuda")
    ac, bc, dyc = a[idx].cpu(), b[idx].cpu(), dy[idx].cpu()
    assert_parity(c[idx], oracle.silu_mul_fwd(ac, bc), "hf fwd")
    rda, rdb = oracle.silu_mul_bwd(dyc, ac, bc)
    assert_parity(da[idx], rda, "hf da")
    assert_parity(db[idx], rdb, "hf db")


def test_two_tensor_errors(sw):
    a = torch.randn(4, 8, device="cuda")
    with pytest.raises(sw.SwigluError) as e:
        sw.swiglu_silu_mul_fwd(a, a, a)
    assert e.value.status == -5
    base = torch.randn(4, 9, device="cuda")
    a2 = base[:, :8]
    with pytest.raises(sw.SwigluError) as e:  # da shifted one element over a
        sw.swiglu_silu_mul_bwd(a.clone(), a2, a.clone(), da=base[:, 1:9])
    assert e.value.status == -5
