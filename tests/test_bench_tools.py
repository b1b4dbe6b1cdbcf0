"""The bench's evidence plumbing, on the CPU: recording DRAM traffic from an
ncu CSV log, the code digest that ties it to the kernel sources (comments do
not count), and the ncu-based fractions of 8 TB/s derived from it."""
import csv
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture()
def bench(tmp_path, monkeypatch):
    import bench as b

    monkeypatch.setattr(b, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    return b


def _ncu_csv(path, launches):
    """launches: (kernel name, read, write, duration ns) in ncu's --csv layout."""
    with open(path, "w", newline="") as f:
        f.write("==PROF== Connected to process 1\n")
        w = csv.writer(f)
        w.writerow(["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
                    "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name",
                    "Metric Unit", "Metric Value"])
        for i, (name, rd, wr, ns) in enumerate(launches):
            for metric, unit, v in (("dram__bytes_read.sum", "byte", rd),
                                    ("dram__bytes_write.sum", "byte", wr),
                                    ("gpu__time_duration.sum", "nsecond", ns)):
                w.writerow([str(i), "1", "python", "h", name, "1", "7", "(256, 1, 1)", "(8, 1, 1)", "0",
                            "10.3", "Command line profiler metrics", metric, unit, f"{v:,}"])


def test_record_traffic_and_fractions(bench, tmp_path):
    import workloads as W

    w = W.WORKLOADS["large_32768_bf16"]
    fwd = "void swiglu::swiglu_fwd_kernel<swiglu::BF16, 16, 1, 3, 0, 0>(swiglu::FwdParams)"
    bwd = "void swiglu::swiglu_bwd_kernel<swiglu::BF16, 8, 2, 0, 3, 0>(swiglu::BwdParams)"
    other = "void at::elementwise_kernel<128, 4>(int)"
    p = tmp_path / "dram.csv"
    _ncu_csv(p, [(fwd, 1000, 500, 200000), (bwd, 3000, 2000, 400000), (other, 7, 7, 7),
                 (fwd, 1002, 498, 210000), (bwd, 3000, 2002, 410000)])
    out = bench.record_traffic(str(p), w.name)
    assert out["fwd"]["bytes_per_launch"] == 1500 and out["bwd"]["bytes_per_launch"] == 5001
    assert out["bwd"]["kernel"] == "swiglu_bwd_kernel<BF16, 8, 2, 0, 3, 0>"
    stored = json.load(open(bench.TRAFFIC_FILE))
    assert stored["bwd"]["source_digest"] == bench.source_digest()
    assert bench.stored_traffic("bwd", w.name) == 5001
    assert bench.stored_traffic("bwd", "megatron_4096_bf16") is None  # another workload
    fr = bench.ncu_fractions(w)
    assert fr["fwd_us"] == pytest.approx(205.0) and fr["bwd_us"] == pytest.approx(405.0)
    assert fr["fwd"] == pytest.approx(w.fwd_bytes() / 205e-6 / 8e12, abs=1e-4)
    assert fr["fwdbwd"] == pytest.approx((w.fwd_bytes() + w.bwd_bytes()) / 610e-6 / 8e12, abs=1e-4)


def test_digest_ignores_comments_not_code(bench):
    src = "int f(int a) { // add one\n  return a + 1; /* done */ }\n"
    same = "int f(int a) {\n  return   a + 1;\n}  // other words\n"
    changed = "int f(int a) { return a + 2; }"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(changed)


def test_stale_digest_hides_traffic(bench):
    with open(bench.TRAFFIC_FILE, "w") as f:
        json.dump({"bwd": {"workload": "large_32768_bf16", "bytes_per_launch": 1,
                           "source_digest": "0" * 16}}, f)
    assert bench.stored_traffic("bwd", "large_32768_bf16") is None
