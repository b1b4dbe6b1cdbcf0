"""Bench of the fused gate-up SwiGLU on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline] [--no-extras]
    python bench.py --record-traffic NCU_CSV    # store an ncu DRAM capture

One step = one forward plus one out-of-place backward (the "fwd+bwd" of the
Liger-Kernel Megatron SwiGLU page, §Summary) over the large-FFN bf16 workload
x [S=2048, B=4, 2n=65536] (ffn_local = 32768; 1 GiB input, larger than L2, so
no L2 flush is needed between steps).  Inputs are seeded synthetic tensors
(workloads.py) already resident in HBM when the timed region starts.  Prints
ONE JSON line on rank 0.

The value is milliseconds per step (lower is better).  Alongside: forward-
and backward-only times, in-place backward time, achieved HBM GB/s against the
measured copy bandwidth (and, from the stored ncu capture, against 8 TB/s),
an end-to-end time through host buffers, the oracle timed on the host's cores
on a bounded sample of the same workload, and under "extras" the other rows
(two-tensor, per-token weights, bias, both, the autograd module, an unfused
eager PyTorch composition of the same math, fc1 + SwiGLU on the tensor cores
against cuBLAS) and the other workloads.

Under torchrun (--gpus N > 1) every rank runs the whole workload on its own GPU
(independent replicas: the op has no exchange step), time is the max over
ranks, and the line reports "scaling": "weak".

--impl reference times the oracle (the plain fp64 CPU statement of the op) on
the host's cores instead, each step a bounded row sample of the same workload
scaled to the full workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "SwiGLU gate-up fwd & fwd+bwd ms, HBM GB/s, % of GB300 peak (bf16 S2048 B4)"
CLOCK_WINDOW_S = 0.6  # shortest span of the clock record around the timed steps
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "gate_up_swiglu_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------ setup ---

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Replicas:
    """The ranks of a torchrun launch, or the single process of a plain one.

    The op has no exchange step, so ranks are independent replicas of the
    workload: they meet only to start and stop the clock together and to take
    the slowest rank's time.  `backend` is "nccl" on GPUs ("gloo" in the CPU
    tests of this plumbing)."""

    def __init__(self, backend: str = "nccl", device=None):
        self.world, self.rank, self.local = dist_env()
        self.device = device if device is not None else torch.device("cpu")
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist

            kw = {"device_id": self.device} if backend == "nccl" else {}
            dist.init_process_group(backend=backend, **kw)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float) -> float:
        """The largest of every rank's v (every rank gets it)."""
        if self.dist is None:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    @property
    def reports(self) -> bool:
        """Rank 0 alone prints the JSON line."""
        return self.rank == 0

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# the sources that define the streaming kernels and their launch configuration
STREAMING_SOURCES = ("swiglu_kernels.cuh", "silu_root_poly.h", "swiglu_abi.cu")


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace runs collapsed, so that
    editing a comment does not invalidate stored counters."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest() -> str:
    """Digest of the streaming kernels' code (comments and layout ignored), to
    tell whether stored ncu counters still describe the kernels the bench
    times."""
    h = hashlib.sha256()
    for name in STREAMING_SOURCES:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _stored(kernel_key: str, workload: str):
    try:
        with open(TRAFFIC_FILE) as f:
            e = json.load(f)[kernel_key]
    except (OSError, KeyError, ValueError):
        return None
    if e.get("source_digest") != source_digest() or e.get("workload") != workload:
        return None
    return e


def stored_traffic(kernel_key: str, workload: str):
    e = _stored(kernel_key, workload)
    return None if e is None else e.get("bytes_per_launch")


def ncu_fractions(w) -> dict:
    """Algorithmic bytes over the ncu-measured kernel durations stored with
    the traffic capture (mean over its launches), as fractions of 8000 GB/s:
    the 'as measured by ncu' reading of the HBM target. None when the stored
    capture is for other sources or another workload."""
    f, b = _stored("fwd", w.name), _stored("bwd", w.name)
    if f is None or b is None or not f.get("duration_ns") or not b.get("duration_ns"):
        return None
    tf = statistics.mean(f["duration_ns"]) * 1e-9
    tb = statistics.mean(b["duration_ns"]) * 1e-9
    fb, bb = w.fwd_bytes(), w.bwd_bytes()
    return {"fwd": round(fb / tf / 8e12, 4), "bwd": round(bb / tb / 8e12, 4),
            "fwdbwd": round((fb + bb) / (tf + tb) / 8e12, 4),
            "fwd_us": round(tf * 1e6, 1), "bwd_us": round(tb * 1e6, 1),
            "source": "profiles/traffic.json (gpu__time_duration.sum of the same capture)"}


def record_traffic(csv_path: str, workload: str = W.HEADLINE) -> dict:
    """Write TRAFFIC_FILE from the CSV log of an ncu capture of this bench on
    `workload` with --metrics dram__bytes_read.sum,dram__bytes_write.sum,
    gpu__time_duration.sum (one pass): per-launch DRAM bytes of the forward
    and backward kernels, tied to the digest of the sources they were built
    from."""
    with open(csv_path) as f:
        lines = [ln for ln in f if not ln.startswith("==")]
    rows = list(csv.reader(lines))
    head = rows[0]
    launches = {}
    for row in rows[1:]:
        d = dict(zip(head, row))
        name = d["Kernel Name"]
        key = "fwd" if "swiglu_fwd_kernel" in name else "bwd" if "swiglu_bwd_kernel" in name else None
        if key is None:
            continue
        e = launches.setdefault(key, {}).setdefault(d["ID"], {"name": name})
        e[d["Metric Name"]] = float(d["Metric Value"].replace(",", ""))
    out = {"_note": "dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture "
                    "(1 pass) of the full-size bench workload; bench.py reports it only while "
                    "source_digest matches the streaming kernels' sources."}
    for key, per_id in launches.items():
        L = list(per_id.values())
        rd = [int(x["dram__bytes_read.sum"]) for x in L]
        wr = [int(x["dram__bytes_write.sum"]) for x in L]
        out[key] = {"kernel": L[0]["name"].split("(")[0].replace("void ", "").replace("swiglu::", ""),
                    "workload": workload, "bytes_per_launch": (sum(rd) + sum(wr)) // len(L),
                    "read": rd, "write": wr,
                    "duration_ns": [int(x["gpu__time_duration.sum"]) for x in L],
                    "source_digest": source_digest()}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    return out


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 25 ms in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        sel = str(device_index)
        try:
            uuid = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
            if uuid is not None:
                s = str(uuid)
                sel = s if s.startswith("GPU-") else "GPU-" + s
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "25"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5 and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:  # timed region shorter than the sampling period
            inside = [p for t, p in self.samples if t <= t1][-3:]
            window = "warmup+timed"

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[4 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------- CPU oracle ---

def time_oracle(w: W.Workload, target_s: float):
    """Time the oracle's forward + backward on a row sample sized to about
    `target_s` seconds; return (ms per full-workload step, rows sampled, seconds)."""
    import oracle  # the oracle is only ever timed here, never used for results

    lib = oracle.load()

    def run(rows):
        x, dy = W.make_inputs(w, "cpu", rows=rows)
        t = time.perf_counter()
        oracle.fwd(x, lib=lib)
        oracle.bwd(dy, x, lib=lib)
        return time.perf_counter() - t

    rows = 8
    dt = run(rows)
    per_row = dt / rows
    rows = int(max(8, min(w.rows, target_s / max(per_row, 1e-9))))
    dt = run(rows)
    return dt / rows * w.rows * 1e3, rows, dt


# ------------------------------------------------------------------ arms ---

GB300_L2_BYTES = 129 << 20  # used only when no GPU is visible


def l2_bytes() -> int:
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    return GB300_L2_BYTES


def bench_config(w: W.Workload, world: int, form: str = "plain") -> dict:
    """The workload description both arms print (identical dicts)."""
    step = "fwd + out-of-place bwd" + ("" if form == "plain" else f" ({form} form)")
    return {"workload": w.name, "shape": list(w.shape), "ffn_local": w.n,
            "storage_dtype": w.dtype, "step": step,
            "parallelism": f"independent replicas x{world}" if world > 1 else "one replica",
            "l2": l2_note(w)}


def reference_arm(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    per_step = max(0.05, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    import oracle

    lib = oracle.load()
    x, dy = W.make_inputs(w, "cpu", rows=max(1, min(w.rows, 64)))
    t = time.perf_counter()
    oracle.fwd(x, lib=lib)
    oracle.bwd(dy, x, lib=lib)
    per_row = (time.perf_counter() - t) / x.shape[0]
    rows = int(max(1, min(w.rows, per_step / max(per_row, 1e-9))))
    x, dy = W.make_inputs(w, "cpu", rows=rows)
    for _ in range(args.warmup):
        oracle.fwd(x, lib=lib)
        oracle.bwd(dy, x, lib=lib)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.fwd(x, lib=lib)
        oracle.bwd(dy, x, lib=lib)
        times.append(time.perf_counter() - t)
    sample_ms = statistics.mean(times) * 1e3       # what each timed step ran
    ms = sample_ms / rows * w.rows                  # the full workload, by proportion
    sample = (f"each step runs fwd + bwd on {rows} of {w.rows} rows ({sample_ms:.1f} ms, "
              f"single thread); value scales that to all rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(ms, 3), "unit": "ms",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sample_ms, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, ws),
        "sample_rows_per_step": rows,
        "cpu_baseline": {"value": round(ms, 3), "unit": "ms", "cores": 1, "kind": "oracle",
                         "host_cpus": os.cpu_count(), "sample": sample},
        "e2e": {"value": round(ms, 3), "unit": "ms", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours_arm(args, w):
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libswiglu has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Replicas("nccl", dev)

    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_libswiglu_build", os.path.join(ROOT, "gate_up_swiglu_gb300", "build.py"))
    builder = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(builder)
    builder.build()
    import gate_up_swiglu_gb300 as sw

    barrier, max_over_ranks = ranks.barrier, ranks.max

    x, dy = W.make_inputs(w, dev)
    x = x.contiguous()
    y = torch.empty((w.rows, w.n), dtype=x.dtype, device=dev)
    dx = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    lib = sw.lib
    dt_code = sw.SWIGLU_BF16 if w.dtype == W.BF16 else sw.SWIGLU_F32
    rows, n = w.rows, w.n

    form = args.form
    if form != "plain":
        # the bias ([2n], storage dtype) and per-token weight (fp32) forms of
        # the step, with their reduction workspace allocated once
        gen = torch.Generator().manual_seed(11)
        wts = torch.rand(rows, generator=gen).to(dev)
        bias = (torch.randn(2 * n, generator=gen) * 0.5).to(x.dtype).to(dev)
        dbias = torch.empty_like(bias)
        dwv = torch.empty_like(wts)
        size = (sw.bias_bwd_workspace_bytes if form == "bias"
                else sw.weighted_bias_bwd_workspace_bytes if form == "weighted_bias"
                else (lambda r, c: 0))(rows, n)
        wsp = torch.empty(max(16, size), dtype=torch.uint8, device=dev)

    def fwd():
        if form == "plain":
            st = lib.swiglu_gateup_fwd(x.data_ptr(), y.data_ptr(), rows, n, 2 * n, n, dt_code, sh)
        elif form == "bias":
            st = lib.swiglu_gateup_bias_fwd(x.data_ptr(), bias.data_ptr(), y.data_ptr(), rows, n,
                                            2 * n, n, dt_code, sh)
        elif form == "weighted":
            st = lib.swiglu_gateup_weighted_fwd(x.data_ptr(), wts.data_ptr(), y.data_ptr(), rows, n,
                                                2 * n, n, dt_code, sh)
        else:
            st = lib.swiglu_gateup_weighted_bias_fwd(x.data_ptr(), bias.data_ptr(), wts.data_ptr(),
                                                     y.data_ptr(), rows, n, 2 * n, n, dt_code, sh)
        if st:
            raise sw.SwigluError(st, "fwd")

    def bwd(out, in_place):
        ip = 1 if in_place else 0
        if form == "plain":
            st = lib.swiglu_gateup_bwd(dy.data_ptr(), x.data_ptr(), out.data_ptr(), rows, n, n,
                                       2 * n, 2 * n, dt_code, ip, sh)
        elif form == "bias":
            st = lib.swiglu_gateup_bias_bwd(dy.data_ptr(), x.data_ptr(), bias.data_ptr(),
                                            out.data_ptr(), dbias.data_ptr(), wsp.data_ptr(),
                                            wsp.numel(), rows, n, n, 2 * n, 2 * n, dt_code, ip, sh)
        elif form == "weighted":
            st = lib.swiglu_gateup_weighted_bwd(dy.data_ptr(), x.data_ptr(), wts.data_ptr(),
                                                out.data_ptr(), dwv.data_ptr(), rows, n, n, 2 * n,
                                                2 * n, dt_code, ip, sh)
        else:
            st = lib.swiglu_gateup_weighted_bias_bwd(
                dy.data_ptr(), x.data_ptr(), bias.data_ptr(), wts.data_ptr(), out.data_ptr(),
                dbias.data_ptr(), dwv.data_ptr(), wsp.data_ptr(), wsp.numel(), rows, n, n, 2 * n,
                2 * n, dt_code, ip, sh)
        if st:
            raise sw.SwigluError(st, "bwd")

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd(dx, False)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for k in range(K):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd(dx, False)
        ev[k][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    # one forward launch per step; the bias forms' backward is the tile
    # kernel plus the reduction launch
    launches = K * (2 + (1 if form in ("bias", "weighted_bias") else 0))
    # the timed steps may be shorter than the clock sampler's period: keep the
    # same work running, untimed, until the sampled window spans CLOCK_WINDOW_S
    extra = 0
    while time.time() - t_wall0 < CLOCK_WINDOW_S:
        for _ in range(50):
            fwd()
            bwd(dx, False)
        extra += 50
        torch.cuda.synchronize(dev)
    t_clk1 = time.time()
    fwd_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    bwd_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    ms_step = max_over_ranks(total_ms / K)
    fwd_avg = max_over_ranks(statistics.mean(fwd_ms))
    bwd_avg = max_over_ranks(statistics.mean(bwd_ms))
    clk = clocks.summary(t_wall0, t_clk1)
    clocks.stop()
    if clk is not None:
        clk["window_s"] = round(t_clk1 - t_wall0, 3)
        clk["window_steps"] = f"{K} timed + {extra} untimed steps of the same work"

    # in-place backward: x is restored from a copy between launches, outside
    # the events, so each timed launch sees the forward input
    x_saved = x.clone()
    ip_ms = []
    for k in range(min(K, 50)):
        x.copy_(x_saved)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bwd(x, True)
        b.record(stream)
        b.synchronize()
        ip_ms.append(a.elapsed_time(b))
    x.copy_(x_saved)
    del x_saved
    ip_avg = max_over_ranks(statistics.mean(ip_ms))

    # the end-to-end step runs before the extras: its page-locked host buffers
    # are then allocated early, as a training process holds them for its whole
    # life (allocated after the extras' compilation and GEMM runs they copied
    # about 7 % slower on the same box)
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(sw, w, x, dy, dev, K=min(K, 20), barrier=barrier, reduce=max_over_ranks)

    extras = None if args.no_extras else measure_extras(sw, w, x, dy, dev, stream, reps=min(K, 100))

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        ms, srows, secs = time_oracle(w, target_s=args.cpu_seconds)
        cpu = {"value": round(ms, 3), "unit": "ms", "cores": 1, "kind": "oracle",
               "host_cpus": os.cpu_count(),
               "sample": f"{srows} of {w.rows} rows (fwd + bwd, {secs:.1f} s single thread), "
                         "scaled to the full workload"}

    if not ranks.reports:
        ranks.close()
        return
    peak, peak_src = measured_peaks()
    fb, bb = w.fwd_bytes(), w.bwd_bytes()
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    bwd_gbs = gbs(bb, bwd_avg)
    # stored counters describe the plain form's kernels only
    traffic = stored_traffic("bwd", w.name) if args.form == "plain" else None
    line = {
        "metric": METRIC, "value": round(ms_step, 4), "unit": "ms", "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": bench_config(w, ws, args.form),
        "fwd_ms": round(fwd_avg, 4), "bwd_ms": round(bwd_avg, 4),
        "bwd_in_place_ms": round(ip_avg, 4),
        "fwd_gbs": round(gbs(fb, fwd_avg), 1), "bwd_gbs": round(bwd_gbs, 1),
        "fwdbwd_gbs": round(gbs(fb + bb, fwd_avg + bwd_avg), 1),
        "bwd_in_place_gbs": round(gbs(bb, ip_avg), 1),
        "frac_of_measured_hbm": {"fwd": round(gbs(fb, fwd_avg) / peak, 4),
                                 "fwdbwd": round(gbs(fb + bb, fwd_avg + bwd_avg) / peak, 4),
                                 "peak_gbs": peak, "peak_source": peak_src},
        "frac_of_8000_gbs": {"fwd": round(gbs(fb, fwd_avg) / 8000, 4),
                             "fwdbwd": round(gbs(fb + bb, fwd_avg + bwd_avg) / 8000, 4)},
        "ncu_frac_of_8000_gbs": ncu_fractions(w) if args.form == "plain" else None,
        "roofline": {"bound": "hbm",
                     "kernel": "swiglu_bwd_kernel (out of place)" if args.form == "plain"
                     else "weighted backward (row kernel, dw included)" if args.form == "weighted"
                     else f"{args.form} backward (tile kernel + reductions)",
                     "achieved": round(bwd_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(bwd_gbs / peak, 4), "peak_source": peak_src,
                     "traffic": traffic, "algorithmic_bytes": bb},
        "extras": extras,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    ranks.close()


MIN_TIMED_MS = 5.0  # shortest span of back-to-back launches one figure is averaged over
FC1_ROUNDS = 3


def _event_ms(fn, stream, reps):
    """Mean CUDA-event time of fn() on `stream` over at least `reps` launches
    and at least MIN_TIMED_MS of them (after 3 warm-up calls): short kernels
    get enough launches for a stable mean."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        fn()
    a.record(stream)
    for _ in range(3):
        fn()
    b.record(stream)
    b.synchronize()
    est = max(a.elapsed_time(b) / 3, 1e-3)
    reps = int(min(5000, max(reps, -(-MIN_TIMED_MS // est))))
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def measure_extras(sw, w, x, dy, dev, stream, reps):
    """The other rows on the same workload: the two-tensor entry points on
    separate gate / up tensors (HuggingFace layout), and one forward + backward
    through the autograd module (wrapper overhead over the raw C ABI)."""
    peak, _ = measured_peaks()
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    n = w.n
    a = x[:, :n].contiguous()
    b = x[:, n:].contiguous()
    c = torch.empty_like(a)
    da, db = torch.empty_like(a), torch.empty_like(b)
    f_ms = _event_ms(lambda: sw.swiglu_silu_mul_fwd(a, b, c, stream=stream), stream, reps)
    b_ms = _event_ms(lambda: sw.swiglu_silu_mul_bwd(dy, a, b, da, db, stream=stream), stream, reps)
    del a, b, c, da, db
    from gate_up_swiglu_gb300.autograd import GateUpSwiGLU

    mod = GateUpSwiGLU()
    xs = x.view(*w.shape).detach().requires_grad_(True)
    dys = dy.view(*w.shape[:-1], n)

    def ag_step():
        y = mod(xs)
        torch.autograd.grad(y, xs, dys)

    ag_ms = _event_ms(ag_step, stream, reps)
    del xs

    # the unfused path the fused kernel replaces: the same math composed from
    # eager PyTorch ops on the [rows, 2n] buffer (chunk into halves, silu and
    # multiply; the backward's two formulas, then a cat), in the storage dtype
    def unfused_fwd():
        g_, u_ = x.chunk(2, -1)
        return torch.nn.functional.silu(g_) * u_

    def unfused_bwd():
        g_, u_ = x.chunk(2, -1)
        s_ = torch.sigmoid(g_)
        return torch.cat((dy * u_ * s_ * (1 + g_ * (1 - s_)), dy * g_ * s_), -1)

    with torch.cuda.stream(stream):
        uf_ms = _event_ms(unfused_fwd, stream, max(3, min(reps, 20)))
        ub_ms = _event_ms(unfused_bwd, stream, max(3, min(reps, 20)))

    # the fused kernels timed the same way as the baselines (back-to-back
    # launches of one kind), for like-for-like ratios
    y_same = torch.empty((w.rows, n), dtype=x.dtype, device=dev)
    dx_same = torch.empty_like(x)
    of_ms = _event_ms(lambda: sw.swiglu_gateup_fwd(x, y_same, stream=stream), stream,
                      max(3, min(reps, 20)))
    ob_ms = _event_ms(lambda: sw.swiglu_gateup_bwd(dy, x, dx_same, stream=stream), stream,
                      max(3, min(reps, 20)))
    del y_same, dx_same

    def speedups(f_ms, b_ms):
        return {"fused_fwd_ms": round(of_ms, 4), "fused_bwd_ms": round(ob_ms, 4),
                "fused_speedup_fwd": round(f_ms / of_ms, 3),
                "fused_speedup_fwdbwd": round((f_ms + b_ms) / (of_ms + ob_ms), 3)}

    # the same code compiled by torch.compile (one fused Triton kernel per
    # direction): the closest analogue of a compiler-fused framework path
    compiled = None
    try:
        t_c = time.perf_counter()
        cfwd, cbwd = torch.compile(unfused_fwd), torch.compile(unfused_bwd)
        with torch.cuda.stream(stream):
            cfwd()
            cbwd()
            torch.cuda.synchronize(dev)
            compile_s = time.perf_counter() - t_c
            cf_ms = _event_ms(cfwd, stream, max(3, min(reps, 20)))
            cb_ms = _event_ms(cbwd, stream, max(3, min(reps, 20)))
        compiled = {"fwd_ms": round(cf_ms, 4), "bwd_ms": round(cb_ms, 4),
                    "compile_s": round(compile_s, 1), **speedups(cf_ms, cb_ms)}
    except Exception as e:  # a box without a working compiler stack
        compiled = {"unavailable": f"{type(e).__name__}: {str(e)[:120]}"}

    # per-token weights and bias on the same x / dy
    g = torch.Generator().manual_seed(11)
    wts = torch.rand(w.rows, generator=g).to(dev)
    bias = (torch.randn(2 * n, generator=g) * 0.5).to(x.dtype).to(dev)
    y = torch.empty((w.rows, n), dtype=x.dtype, device=dev)
    dx = torch.empty_like(x)
    dw = torch.empty_like(wts)
    dbias = torch.empty_like(bias)
    ws = torch.empty(max(16, sw.bias_bwd_workspace_bytes(w.rows, n)), dtype=torch.uint8, device=dev)
    wf = _event_ms(lambda: sw.swiglu_gateup_weighted_fwd(x, wts, y, stream=stream), stream, reps)
    wb = _event_ms(lambda: sw.swiglu_gateup_weighted_bwd(dy, x, wts, dx, dw, stream=stream),
                   stream, reps)
    bf = _event_ms(lambda: sw.swiglu_gateup_bias_fwd(x, bias, y, stream=stream), stream, reps)
    bb = _event_ms(lambda: sw.swiglu_gateup_bias_bwd(dy, x, bias, dx, dbias, ws, stream=stream),
                   stream, reps)
    del ws
    wsb = torch.empty(max(16, sw.weighted_bias_bwd_workspace_bytes(w.rows, n)), dtype=torch.uint8,
                      device=dev)
    wbf = _event_ms(lambda: sw.swiglu_gateup_weighted_bias_fwd(x, bias, wts, y, stream=stream),
                    stream, reps)
    wbb = _event_ms(lambda: sw.swiglu_gateup_weighted_bias_bwd(dy, x, bias, wts, dx, dbias, dw, wsb,
                                                               stream=stream), stream, reps)
    del y, dx, dw, dbias

    def row(f_ms, b_ms, extra_note):
        return {"fwd_ms": round(f_ms, 4), "bwd_ms": round(b_ms, 4),
                "fwd_gbs": round(gbs(w.fwd_bytes(), f_ms), 1),
                "bwd_gbs": round(gbs(w.bwd_bytes(), b_ms), 1),
                "fwd_frac_of_measured": round(gbs(w.fwd_bytes(), f_ms) / peak, 4),
                "bwd_frac_of_measured": round(gbs(w.bwd_bytes(), b_ms) / peak, 4),
                "note": extra_note, "reps": reps}

    # the streaming workloads first: the fc1 GEMMs run into the power cap and
    # leave the clocks lowered for a while after
    per_workload = measure_workloads(sw, dev, stream, skip=w.name, reps=max(5, min(reps, 50)))
    fc1 = measure_fc1(sw, dev, stream, reps=max(5, min(reps, 20)))

    return {
        "timing": f"CUDA events over back-to-back launches of one kind: each figure is the mean "
                  f"over at least its 'reps' launches and at least {MIN_TIMED_MS:g} ms of them",
        "unfused_torch_eager": {
            "what": "eager PyTorch ops on the same buffers: fwd chunk + silu * up, bwd chunk + "
                    "the two formulas + cat (intermediates rounded to the storage dtype)",
            "fwd_ms": round(uf_ms, 4), "bwd_ms": round(ub_ms, 4), **speedups(uf_ms, ub_ms)},
        "torch_compile_same_math": compiled,
        "other_workloads": per_workload,
        "fc1_swiglu_tcgen05": fc1,
        "weighted_per_token": row(wf, wb, "fp32 routing weight per row; bwd also returns dw "
                                          "(one CTA per row); GB/s on the plain algorithmic bytes"),
        "bias": row(bf, bb, "[2n] bias; bwd includes the column-sum pass over a workspace and "
                            "the dbias reduction; GB/s on the plain algorithmic bytes"),
        "weighted_bias": row(wbf, wbb, f"[2n] bias and fp32 per-row weights; bwd returns dx, "
                                       f"dbias and dw ({wsb.numel() / 2**20:.1f} MiB workspace); "
                                       "GB/s on the plain algorithmic bytes"),
        "silu_mul_separate_tensors": {
            "layout": "gate and up as two contiguous [rows, n] tensors", "reps": reps,
            "fwd_ms": round(f_ms, 4), "bwd_ms": round(b_ms, 4),
            "fwd_gbs": round(gbs(w.fwd_bytes(), f_ms), 1), "bwd_gbs": round(gbs(w.bwd_bytes(), b_ms), 1),
            "fwd_frac_of_measured": round(gbs(w.fwd_bytes(), f_ms) / peak, 4),
            "bwd_frac_of_measured": round(gbs(w.bwd_bytes(), b_ms) / peak, 4)},
        "autograd_module_fwd_bwd": {
            "what": "GateUpSwiGLU forward + torch.autograd.grad, 3D input, out of place",
            "reps": reps, "ms": round(ag_ms, 4)},
    }


def measure_workloads(sw, dev, stream, skip, reps):
    """Forward, backward and in-place backward on every other workload (the
    tiny fp32 one, the Megatron-shape and Llama-like bf16 ones, the odd-width
    fp32 one), CUDA events per launch, inputs resident in HBM."""
    peak, _ = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for name, wl in W.WORKLOADS.items():
        if name == skip:
            continue
        x, dy = W.make_inputs(wl, dev)
        x = x.contiguous()
        y = torch.empty((wl.rows, wl.n), dtype=x.dtype, device=dev)
        dx = torch.empty_like(x)
        xi = x.clone()
        f = _event_ms(lambda: sw.swiglu_gateup_fwd(x, y, stream=stream), stream, reps)
        b = _event_ms(lambda: sw.swiglu_gateup_bwd(dy, x, dx, stream=stream), stream, reps)
        # the in-place timing overwrites xi each launch; values change, the
        # work and the arithmetic path do not
        bi = _event_ms(lambda: sw.swiglu_gateup_bwd(dy, xi, in_place=True, stream=stream),
                       stream, reps)
        gb = lambda nbytes, ms: nbytes / (ms * 1e-3) / 1e9  # noqa: E731
        unfused = None
        if wl.dtype == W.BF16:
            # the same math as eager PyTorch ops on the same buffers (the
            # unfused path), at this shape too
            def uf():
                g_, u_ = x.chunk(2, -1)
                return torch.nn.functional.silu(g_) * u_

            def ub():
                g_, u_ = x.chunk(2, -1)
                s_ = torch.sigmoid(g_)
                return torch.cat((dy * u_ * s_ * (1 + g_ * (1 - s_)), dy * g_ * s_), -1)

            with torch.cuda.stream(stream):
                uf_ms = _event_ms(uf, stream, max(3, min(reps, 20)))
                ub_ms = _event_ms(ub, stream, max(3, min(reps, 20)))
            unfused = {"fwd_ms": round(uf_ms, 4), "bwd_ms": round(ub_ms, 4),
                       "fused_speedup_fwd": round(uf_ms / f, 3),
                       "fused_speedup_fwdbwd": round((uf_ms + ub_ms) / (f + b), 3)}
        out[name] = {
            "shape": list(wl.shape), "dtype": wl.dtype, "fwd_ms": round(f, 4), "bwd_ms": round(b, 4),
            "bwd_in_place_ms": round(bi, 4), "fwd_gbs": round(gb(wl.fwd_bytes(), f), 1),
            "bwd_gbs": round(gb(wl.bwd_bytes(), b), 1),
            "fwd_frac_of_measured": round(gb(wl.fwd_bytes(), f) / peak, 4),
            "bwd_frac_of_measured": round(gb(wl.bwd_bytes(), b) / peak, 4),
            "l2": "inputs exceed L2" if 3 * wl.n * wl.rows * wl.elem_bytes > l2
                  else "inputs fit in L2 (back-to-back launches: L2-resident)",
            "unfused_torch_eager": unfused}
        del x, dy, y, dx, xi
    return out


def measure_fc1(sw, dev, stream, reps):
    """linear_fc1 + SwiGLU of a Llama-3-8B MLP (X [8192, 4096], W [28672, 4096],
    bf16) on the tensor cores, against cuBLAS (torch.matmul) followed by the
    separate activation kernel."""
    M, K, n = 8192, 4096, 14336
    g = torch.Generator(device=dev).manual_seed(3)
    X = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    Wt = (torch.randn(2 * n, K, generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
    y = torch.empty(M, n, dtype=torch.bfloat16, device=dev)
    fc1 = torch.empty(M, 2 * n, dtype=torch.bfloat16, device=dev)
    flops = 2.0 * M * K * 2 * n

    def two_step():
        torch.matmul(X, Wt.T, out=fc1)
        sw.swiglu_gateup_fwd(fc1, y, stream=stream)

    kinds = {"fused": lambda: sw.swiglu_fc1_fwd(X, Wt, y, stream=stream),
             "gemm_only": lambda: torch.matmul(X, Wt.T, out=fc1),
             "fused_fc1": lambda: sw.swiglu_fc1_fwd(X, Wt, y, fc1, stream=stream),
             "two_step": two_step}
    # these GEMMs run at the power limit, where the clock drifts with the
    # heat of what ran before: FC1_ROUNDS rounds in rotating order, and the
    # median of each kind
    order = list(kinds)
    rounds = {k: [] for k in kinds}
    for r in range(FC1_ROUNDS):
        for k in order[r % len(order):] + order[:r % len(order)]:
            rounds[k].append(_event_ms(kinds[k], stream, reps))
    fused, gemm_only, fused_fc1, cublas = (statistics.median(rounds[k]) for k in kinds)
    peak, peak_src = None, "measured"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        peak, peak_src = 1900.0, "fallback"
    tf = lambda ms: flops / (ms * 1e-3) / 1e12  # noqa: E731
    return {"shape": "X [8192, 4096] x W [28672, 4096] bf16 -> y [8192, 14336]", "reps": reps,
            "fused_ms": round(fused, 4), "fused_tflops": round(tf(fused), 1),
            "fused_frac_of_measured_bf16": round(tf(fused) / peak, 4),
            "fused_with_fc1_out_ms": round(fused_fc1, 4),
            "cublas_gemm_plus_swiglu_ms": round(cublas, 4),
            "cublas_gemm_only_ms": round(gemm_only, 4),
            "cublas_gemm_tflops": round(tf(gemm_only), 1), "peak_bf16_tflops": peak,
            "peak_source": peak_src,
            "timing": f"median of {FC1_ROUNDS} rounds in rotating order",
            "rounds_ms": {k: [round(v, 4) for v in vals] for k, vals in rounds.items()}}


def l2_note(w: W.Workload) -> str:
    l2 = l2_bytes()
    inputs = (3 * w.n * w.rows) * w.elem_bytes  # x and dy
    if inputs > l2:
        return (f"no flush: inputs {inputs / 2**20:.0f} MiB > L2 {l2 / 2**20:.0f} MiB; "
                f"every step streams {(w.fwd_bytes() + w.bwd_bytes()) / 1e9:.2f} GB")
    return f"inputs {inputs / 2**20:.0f} MiB fit in L2 {l2 / 2**20:.0f} MiB: L2-resident timing"


def link_rates(dev, h_ins, h_outs) -> dict:
    """Host link rates of the given page-locked buffers, same run: every h_in
    copied to the device alone, the device copied into every h_out alone, then
    both directions at once on two streams (GB/s each way, best of 3).  The
    rates depend on where the buffers land in host memory (149-170 GB/s duplex
    on one box across buffer sets), so they are measured on the very buffers
    the end-to-end step uses, all of them."""
    def flat(ts):
        return [t.view(-1).view(torch.uint8) for t in ts]

    srcs, dsts = flat(h_ins), flat(h_outs)
    b_in, b_out = sum(t.numel() for t in srcs), sum(t.numel() for t in dsts)
    d_in = [torch.empty(t.numel(), dtype=torch.uint8, device=dev) for t in srcs]
    d_out = [torch.empty(t.numel(), dtype=torch.uint8, device=dev) for t in dsts]
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def best(fn):
        ts = []
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            ts.append(time.perf_counter() - t)
        return min(ts)

    def copy_in():
        for d, h in zip(d_in, srcs):
            d.copy_(h, non_blocking=True)

    def copy_out():
        for h, d in zip(dsts, d_out):
            h.copy_(d, non_blocking=True)

    def both():
        with torch.cuda.stream(s1):
            copy_in()
        with torch.cuda.stream(s2):
            copy_out()

    t_in, t_out, t_both = best(copy_in), best(copy_out), best(both)
    # both at once: each direction's rate over the time both took
    return {"h2d_gbs": round(b_in / t_in / 1e9, 1), "d2h_gbs": round(b_out / t_out / 1e9, 1),
            "duplex_each_way_gbs": round(max(b_in, b_out) / t_both / 1e9, 1),
            "h2d_bytes": b_in, "d2h_bytes": b_out,
            "how": "the step's own pinned buffers (x, dy in; y, dx out), host clock, best of 3"}


def end_to_end(sw, w, x_dev, dy_dev, dev, K, barrier, reduce):
    """The same step from host memory, through the C-ABI call
    swiglu_gateup_fwd_bwd_host: the inputs are copied in from pinned host
    memory and the results copied back, chunk by chunk with copies and kernels
    overlapped, all inside the timed region (host clock around whole calls,
    each of which returns once its results are in host memory).  The staging
    buffer and streams are set up once, before the timed region."""
    from gate_up_swiglu_gb300.host_pipeline import HostPipeline, default_chunk_rows

    xh = torch.empty(x_dev.shape, dtype=x_dev.dtype, pin_memory=True)
    dyh = torch.empty(dy_dev.shape, dtype=dy_dev.dtype, pin_memory=True)
    xh.copy_(x_dev)
    dyh.copy_(dy_dev)
    yh = torch.empty((w.rows, w.n), dtype=x_dev.dtype, pin_memory=True)
    dxh = torch.empty(x_dev.shape, dtype=x_dev.dtype, pin_memory=True)
    pipe = HostPipeline(dev, default_chunk_rows(w.n, w.elem_bytes))
    staging = pipe.staging_for(w.n, x_dev.dtype)
    streams = (pipe.h2d, pipe.comp, pipe.d2h)

    def step():
        sw.swiglu_gateup_fwd_bwd_host(xh, dyh, yh, dxh, staging, pipe.chunk_rows, pipe.depth,
                                      streams)

    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    barrier()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    torch.cuda.synchronize(dev)
    barrier()
    ms = reduce((time.perf_counter() - t0) * 1e3 / K)
    h2d = xh.numel() * xh.element_size() + dyh.numel() * dyh.element_size()
    d2h = yh.numel() * yh.element_size() + dxh.numel() * dxh.element_size()
    del staging
    link = link_rates(dev, (xh, dyh), (yh, dxh))
    del xh, dyh, yh, dxh
    # the floor set by the link: the larger direction at the measured duplex rate
    floor_ms = max(h2d, d2h) / (link["duplex_each_way_gbs"] * 1e9) * 1e3
    return {"value": round(ms, 3), "unit": "ms", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "how": f"C ABI swiglu_gateup_fwd_bwd_host, {pipe.chunk_rows}-row chunks, "
                   f"{pipe.depth} staging slots, 3 streams",
            "host_link": link, "link_floor_ms": round(floor_ms, 3),
            "frac_of_link_floor": round(floor_ms / ms, 4)}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.HEADLINE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="time the step alone (the command the kernel profiles are taken on)")
    ap.add_argument("--form", choices=["plain", "bias", "weighted", "weighted_bias"], default="plain",
                    help="the entry points of the timed step: plain (the headline), or the bias / "
                         "per-token weights / per-token weights + bias forms")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="write profiles/traffic.json from an ncu CSV log of this bench and exit")
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    if args.record_traffic:
        out = record_traffic(args.record_traffic, w.name)
        print(json.dumps({k: v["bytes_per_launch"] for k, v in out.items() if k != "_note"}))
        return
    if args.impl == "reference":
        if args.form != "plain":
            raise SystemExit("--impl reference times the plain form only")
        reference_arm(args, w)
    else:
        ours_arm(args, w)


if __name__ == "__main__":
    main()
