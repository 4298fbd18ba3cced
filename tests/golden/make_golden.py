"""Writes tests/golden/oracle_snapshot.txt from the CPU oracle alone.

The pages ("UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract) print no worked example of the encoding, so there are no page
values to store; this file freezes what the pinned oracle computes on the
tiny configuration (two seeded 256 x 256 BF16 operands with 1 % outliers),
so that any later change to the oracle's arithmetic shows up as a changed
fixture, and so that the GPU tests can compare with stored values without
running the oracle.

Each line: case name, then key=value fields.  Byte arrays are given by their
SHA-256 (first 16 hex digits); T and the GEMM checksums as exact hex floats.

    python tests/golden/make_golden.py        # rewrites the fixture
"""
import hashlib
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from fp4_block_scaled_bf16_gb300 import workloads  # noqa: E402

OUT = os.path.join(HERE, "oracle_snapshot.txt")


def h(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()[:16]


def cases():
    """(name, operand, axis, rnd, fmt, seed) of every stored quantisation."""
    a, b = workloads.tiny_operands(seed=0)
    for opname, x in (("A", a), ("B", b)):
        for fmt in (oracle.UE5M3, oracle.UE4M3):
            for axis in (oracle.ROW, oracle.COL):
                for rnd, seed in ((oracle.RNE, 0), (oracle.SR, 7)):
                    yield f"{opname}_fmt{fmt}_axis{axis}_rnd{rnd}", x, axis, rnd, fmt, seed


def snapshot():
    lines = []
    for name, x, axis, rnd, fmt, seed in cases():
        T = oracle.tensor_scale(oracle.amax(x)[0], fmt)
        p, s, st = oracle.quantize(x, axis, T, fmt, rnd, seed)
        lines.append(f"quantize {name} T={float(T).hex()} payload={h(p)} scales={h(s)} "
                     f"stats={','.join(str(int(v)) for v in st)}")
    a, b = workloads.tiny_operands(seed=0)
    for fmt in (oracle.UE5M3, oracle.UE4M3):
        TA = oracle.tensor_scale(oracle.amax(a)[0], fmt)
        TB = oracle.tensor_scale(oracle.amax(b)[0], fmt)
        pa, sa, _ = oracle.quantize(a, oracle.ROW, TA, fmt)
        pb, sb, _ = oracle.quantize(b, oracle.ROW, TB, fmt)
        R = oracle.gemm(pa, sa, TA, pb, sb, TB, fmt)
        lines.append(f"gemm tiny_fmt{fmt} sum={float(R.sum()).hex()} absmax={float(np.abs(R).max()).hex()} "
                     f"r00={float(R[0, 0]).hex()} r_last={float(R[-1, -1]).hex()}")
    return lines


def parse(path=OUT):
    out = {}
    with open(path) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            kind, name, *fields = line.split()
            out[(kind, name)] = dict(fv.split("=", 1) for fv in fields)
    return out


if __name__ == "__main__":
    with open(OUT, "w") as f:
        f.write("# written by tests/golden/make_golden.py from the CPU oracle only; "
                "tiny configuration (workloads.tiny_operands(seed=0)), current tensor scale, "
                "SR seed 7\n")
        for line in snapshot():
            f.write(line + "\n")
    print(OUT)
