"""Write ``oracle_specials.txt``: oracle outputs on a grid of special gate values.

Calls only the oracle.  The page prints no worked numeric example, so this
fixture is an oracle regression record (it fails if the oracle's arithmetic
drifts) and a fixed table the CUDA tests compare against.  The gate values are
the ones the method treats specially: zero, tiny, the ends of the fp32 exp
range, deep saturation, and the fp32 values around silu's stationary point
g0 = -1 - W(1/e).

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

GATES = [0.0, -0.0, 1e-30, -1e-30, 1.0, -1.0, 0.5, -0.5, 2.0, -2.0, 8.0, -8.0, 20.0, -20.0,
         30.0, -30.0, 87.0, -87.0, 88.0, -88.0, 89.0, -89.0, 100.0, -100.0, 1e4, -1e4,
         -1.25, -1.3, -1.2734375, -1.28125]
# fp32 neighbours of g0 = -1.2784645427610738 (0, 1, 2, 16 and 256 spacings away)
_g0 = np.float32(-1.2784645427610738)
for _k in (1, 2, 16, 256):
    GATES += [float(_g0 + np.float32(_k) * np.spacing(_g0)), float(_g0 - np.float32(_k) * np.spacing(_g0))]
GATES.append(float(_g0))
UPS = [1.0, -2.5, 0.0078125]
DYS = [1.0, -0.75]


def table(dtype):
    rows = []
    for u in UPS:
        for d in DYS:
            rows.append((u, d))
    n = len(GATES)
    x = torch.empty((len(rows), 2 * n), dtype=torch.float32)
    dy = torch.empty((len(rows), n), dtype=torch.float32)
    for i, (u, d) in enumerate(rows):
        x[i, :n] = torch.tensor(GATES)
        x[i, n:] = u
        dy[i, :] = d
    x, dy = x.to(dtype), dy.to(dtype)
    return x, dy, oracle.fwd(x), oracle.bwd(dy, x)


def bits(t):
    if t.dtype == torch.float32:
        return ["%08x" % (v & 0xFFFFFFFF) for v in t.view(torch.int32).flatten().tolist()]
    return ["%04x" % (v & 0xFFFF) for v in t.view(torch.int16).flatten().tolist()]


def render():
    lines = ["# oracle outputs on special gate values; written by make_golden.py (oracle only)",
             "# format: <dtype> <tensor> <rows> <cols> then hex bit patterns, row-major"]
    for name, dt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        x, dy, y, dx = table(dt)
        for tname, t in (("x", x), ("dy", dy), ("y", y), ("dx", dx)):
            lines.append(f"{name} {tname} {t.shape[0]} {t.shape[1]}")
            lines.append(" ".join(bits(t)))
    return "\n".join(lines) + "\n"


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_specials.txt"), "w") as f:
        f.write(render())
    print("wrote oracle_specials.txt")
