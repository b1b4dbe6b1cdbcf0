"""The oracle still reproduces its stored table of special gate values.

``tests/golden/oracle_specials.txt`` was written by ``tests/golden/make_golden.py``
from the oracle alone; the page prints no worked example, so this is a drift
guard on the oracle (and the table the CUDA tests also read).
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracle_reproduces_golden():
    with open(os.path.join(HERE, "golden", "oracle_specials.txt")) as f:
        stored = f.read()
    assert make_golden.render() == stored
