"""Reader for the hand-worked block fixtures in tests/golden/ (format described
in tests/golden/README.txt)."""
import glob
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TYPES = {"Q8_0": (8, 32, 34), "Q2_K": (10, 256, 84), "Q4_K": (12, 256, 144), "Q5_K": (13, 256, 176),
         "Q6_K": (14, 256, 210)}


def load(path):
    qtype = None
    block = None
    values = None
    for raw in open(path):
        line = raw.split("#", 1)[0].split()
        if not line:
            continue
        op, args = line[0], line[1:]
        if op == "type":
            qtype, qk, bb = TYPES[args[0]]
            block = np.zeros(bb, np.uint8)
            values = [None] * qk
        elif op == "bytes":
            off, cnt, val = int(args[0]), int(args[1]), int(args[2], 16)
            block[off:off + cnt] = val
        elif op == "byte":
            off = int(args[0])
            for i, h in enumerate(args[1:]):
                block[off + i] = int(h, 16)
        elif op == "fill":
            first, cnt, val = int(args[0]), int(args[1]), float(args[2])
            for v in range(first, first + cnt):
                values[v] = val
        elif op == "list":
            first = int(args[0])
            for i, x in enumerate(args[1:]):
                values[first + i] = float(x)
        else:
            raise ValueError("%s: unknown directive %r" % (path, op))
    if any(v is None for v in values):
        raise ValueError("%s: not every value is listed" % path)
    return qtype, block, np.array(values, np.float64)


def all_fixtures():
    return sorted(glob.glob(os.path.join(GOLDEN, "*.txt")))


def fixtures():
    return [p for p in all_fixtures() if not p.endswith("README.txt")]
