import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, runs for tens of seconds")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a golden fixture: '# comments', then 'key v1 v2 ...' lines.  Repeated 'name'
    lines start a new record; returns a list of dicts (or one dict when there is no 'name')."""
    recs, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "name":
                if cur:
                    recs.append(cur)
                cur = {"name": vals[0]}
                continue
            cur[key] = vals
    if cur:
        recs.append(cur)
    return recs


def read_table(name):
    """Parse a two-column 'code value' golden table into a list of (int code, float value)."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                c, v = line.split()
                out.append((int(c, 16), float(v)))
    return out
