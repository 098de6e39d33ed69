"""Writes tests/golden/oracle_tiny.txt: regression values of the float64 oracle.

Calls only ``oracle`` and the seeded generators of ``workloads``. The pages
print no worked example of the update, so these values pin later changes of
the oracle against its present, independently pinned state (see
tests/test_oracle_pins.py); they are not a pin against the pages.
Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as wl  # noqa: E402


def main():
    N, c_z, c_h = 6, 4, 3
    z = wl.make_z(N, c_z, 123, "bf16")
    m = wl.make_mask(N, "full")
    m[4] = 0
    W = wl.make_weights(c_z, c_h, 124, ln_random=True)
    lines = [f"# oracle regression: N={N} c_z={c_z} c_h={c_h} z seed 123 (bf16), weights seed 124 "
             f"(ln_random), token 4 masked; columns: direction i j channel value"]
    for d in ("outgoing", "incoming"):
        out = oracle.full(z, m, W, d)
        for i in range(N):
            for j in range(N):
                for c in range(c_z):
                    lines.append(f"{d} {i} {j} {c} {out[i, j, c]:.17e}")
    with open(os.path.join(HERE, "oracle_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
