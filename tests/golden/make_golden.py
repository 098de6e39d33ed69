"""Writes tests/golden/oracle_tiny.txt, oracle_backward_tiny.txt and oracle_attention_tiny.txt:
regression values of the float64 oracles (the update, its gradient, triangle attention).

Calls only ``oracle`` and the seeded generators of ``workloads``. The pages
print no worked example of these operations, so the values pin later changes
of the oracles against their present, independently pinned state (see
tests/test_oracle_pins.py, test_oracle_backward.py, test_oracle_attention.py);
they are not a pin against the pages.
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

    # the gradient of sum(dout * update): dz and every parameter, both directions
    dout = wl.make_z(N, c_z, 125, "bf16")
    lines = [f"# backward oracle regression: the update's inputs above, cotangent seed 125 (bf16); "
             f"columns: direction tensor flat-index value"]
    for d in ("outgoing", "incoming"):
        g = oracle.full_backward(z, m, W, d, dout)
        for name in ("z",) + oracle.WEIGHT_NAMES:
            for k, v in enumerate(np.asarray(g[name]).ravel()):
                lines.append(f"{d} {name} {k} {v:.17e}")
    with open(os.path.join(HERE, "oracle_backward_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")

    # triangle attention, both nodes: N = 5, c_z = 6, two heads of 3
    import oracle.triangle_attention as TA
    Na, cza, H, c = 5, 6, 2, 3
    za = wl.make_z(Na, cza, 126, "bf16")
    ma = wl.make_mask(Na, "full")
    ma[1] = 0
    rng = np.random.default_rng(127)
    Wa = {k: rng.standard_normal(sh) / np.sqrt(sh[-1]) for k, sh in TA.weight_shapes(cza, H, c).items()}
    Wa["ln_gamma"] = 1.0 + 0.3 * rng.standard_normal(cza)
    Wa["ln_beta"] = 0.3 * rng.standard_normal(cza)
    lines = [f"# triangle attention oracle regression: N={Na} c_z={cza} H={H} c={c}, z seed 126 (bf16), "
             f"weights from default_rng(127) in weight_shapes order, token 1 masked; columns: node i j channel value"]
    for node in TA.NODES:
        out = TA.full(za, ma, Wa, node, H, c)
        for i in range(Na):
            for j in range(Na):
                for ch in range(cza):
                    lines.append(f"{node} {i} {j} {ch} {out[i, j, ch]:.17e}")
    with open(os.path.join(HERE, "oracle_attention_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
