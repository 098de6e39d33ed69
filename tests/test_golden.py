"""Golden fixtures: the sizes the pages print, and the oracle's regression values."""
import os

import numpy as np

import oracle
import workloads as wl

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_sizes():
    out = {}
    with open(os.path.join(HERE, "page_sizes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                out[k] = int(v)
    return out


def test_workload_sizes_match_pages():
    s = _read_sizes()
    W = wl.WORKLOADS
    assert W["crop768"].N == s["crop_tokens"]
    assert W["complex3605"].N == s["complex_tokens"]
    assert len(W["complex3605"].chains) == s["complex_chains"]
    assert sum(W["complex3605"].chains) == s["complex_tokens"]
    assert W["ppi6500"].N == s["ppi_tokens"]
    assert W["n10000"].N == s["large_tokens"]
    assert W["n10000"].N ** 2 == s["large_pairs"]


def test_oracle_regression_values():
    N, c_z, c_h = 6, 4, 3
    z = wl.make_z(N, c_z, 123, "bf16")
    m = wl.make_mask(N, "full")
    m[4] = 0
    W = wl.make_weights(c_z, c_h, 124, ln_random=True)
    outs = {d: oracle.full(z, m, W, d) for d in ("outgoing", "incoming")}
    n = 0
    with open(os.path.join(HERE, "oracle_tiny.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            d, i, j, c, v = line.split()
            assert abs(outs[d][int(i), int(j), int(c)] - float(v)) <= 1e-13 * max(1.0, abs(float(v)))
            n += 1
    assert n == 2 * N * N * c_z


def test_backward_oracle_regression_values():
    N, c_z, c_h = 6, 4, 3
    z = wl.make_z(N, c_z, 123, "bf16")
    m = wl.make_mask(N, "full")
    m[4] = 0
    W = wl.make_weights(c_z, c_h, 124, ln_random=True)
    dout = wl.make_z(N, c_z, 125, "bf16")
    grads = {d: oracle.full_backward(z, m, W, d, dout) for d in ("outgoing", "incoming")}
    n = 0
    with open(os.path.join(HERE, "oracle_backward_tiny.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            d, name, k, v = line.split()
            got = np.asarray(grads[d][name]).ravel()[int(k)]
            assert abs(got - float(v)) <= 1e-12 * max(1.0, abs(float(v))), (d, name, k)
            n += 1
    per_direction = N * N * c_z + sum(int(np.prod(np.shape(W[k]))) for k in oracle.WEIGHT_NAMES)
    assert n == 2 * per_direction


def test_attention_oracle_regression_values():
    import oracle.triangle_attention as TA
    Na, cza, H, c = 5, 6, 2, 3
    za = wl.make_z(Na, cza, 126, "bf16")
    ma = wl.make_mask(Na, "full")
    ma[1] = 0
    rng = np.random.default_rng(127)
    Wa = {k: rng.standard_normal(sh) / np.sqrt(sh[-1]) for k, sh in TA.weight_shapes(cza, H, c).items()}
    Wa["ln_gamma"] = 1.0 + 0.3 * rng.standard_normal(cza)
    Wa["ln_beta"] = 0.3 * rng.standard_normal(cza)
    outs = {node: TA.full(za, ma, Wa, node, H, c) for node in TA.NODES}
    n = 0
    with open(os.path.join(HERE, "oracle_attention_tiny.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            node, i, j, ch, v = line.split()
            assert abs(outs[node][int(i), int(j), int(ch)] - float(v)) <= 1e-13 * max(1.0, abs(float(v)))
            n += 1
    assert n == 2 * Na * Na * cza
