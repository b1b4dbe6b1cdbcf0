"""The C ABI from a plain C99 program (tests/c_caller/main.c): the header
compiles as C, and on a GPU the program -- linking libswiglu.so and the CUDA
runtime, with device memory it allocates itself -- produces the oracle's
results for the forward, the backward and the in-place backward, and the same
bits again end to end from page-locked host buffers through
swiglu_gateup_fwd_bwd_host."""
import os
import shutil
import subprocess

import pytest
import torch

import oracle
import workloads as W
from helpers import assert_bitwise, assert_parity

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_caller", "main.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _gcc(*args):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    return subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(CUDA, "include"), *args],
                          capture_output=True, text=True)


def test_header_and_caller_compile_as_c99():
    r = _gcc("-fsyntax-only", SRC)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("name,rows", [("tiny_f32", None), ("megatron_4096_bf16", 48),
                                       ("odd_5503_f32", 7)])
def test_c_program_matches_oracle(tmp_path, name, rows):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from conftest import build_library

    build_library()
    import gate_up_swiglu_gb300 as sw

    exe = str(tmp_path / "c_caller")
    libdir = os.path.dirname(sw.LIB_PATH)
    r = _gcc("-O2", SRC, "-o", exe, "-L", libdir, "-lswiglu", "-L", os.path.join(CUDA, "lib64"),
             "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}")
    assert r.returncode == 0, r.stderr
    w = W.WORKLOADS[name]
    x, dy = W.make_inputs(w, "cpu", rows=rows)
    x = x.contiguous()
    nrows, n = x.shape[0], w.n
    dt = 0 if x.dtype == torch.float32 else 1
    raw = lambda t: t.view(torch.int32 if t.element_size() == 4 else torch.int16).numpy().tobytes()  # noqa: E731
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    inp.write_bytes(raw(x) + raw(dy))
    run = subprocess.run([exe, str(dt), str(nrows), str(n), str(inp), str(outp)],
                         capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert f"abi version {sw.lib.swiglu_abi_version()}" in run.stdout
    blob = outp.read_bytes()
    itype = torch.int32 if dt == 0 else torch.int16
    vals = torch.frombuffer(bytearray(blob), dtype=itype).view(x.dtype)
    ny, nx = nrows * n, nrows * 2 * n
    y = vals[:ny].view(nrows, n)
    dx = vals[ny:ny + nx].view(nrows, 2 * n)
    dx_in_place = vals[ny + nx:ny + 2 * nx].view(nrows, 2 * n)
    y_host = vals[ny + 2 * nx:2 * ny + 2 * nx].view(nrows, n)
    dx_host = vals[2 * ny + 2 * nx:].view(nrows, 2 * n)
    assert_parity(y, oracle.fwd(x), f"{name} C caller fwd")
    assert_parity(dx, oracle.bwd(dy, x), f"{name} C caller bwd")
    assert_bitwise(dx_in_place, dx, f"{name} C caller in place")
    assert_bitwise(y_host, y, f"{name} C caller host pipeline y")
    assert_bitwise(dx_host, dx, f"{name} C caller host pipeline dx")
