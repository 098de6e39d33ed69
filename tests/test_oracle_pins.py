"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a swapped index, a transposed operand, the mask applied at the
wrong index) fails at least one of them:

* brute force: scalar loops written from the definition, tiny N;
* library routines: LayerNorm against torch.nn.functional.layer_norm, the
  logistic function against scipy.special.expit, bf16 rounding against
  torch's float32 -> bfloat16 conversion;
* invariants: permutation equivariance, the swap-transpose identity linking
  the two directions, masked-token invariants, trailing padding;
* closed forms: constant z, and the linear special case that reduces the
  contraction to one matrix product per channel.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import workloads as wl

DIRS = ("outgoing", "incoming")


def _inputs(N, c_z, c_h, seed=0, mask="scatter", ln_random=True, dtype="f32"):
    z = wl.make_z(N, c_z, seed, dtype)
    m = wl.make_mask(N, mask, seed=seed + 11)
    W = wl.make_weights(c_z, c_h, seed + 1, ln_random=ln_random)
    return wl.as_f64(z), m.astype(np.float64), W


# --------------------------------------------------------------------------- brute force

def _brute_force(z, m, W, direction):
    """Scalar loops straight from the definition (no numpy algebra)."""
    N = z.shape[0]
    c_z = z.shape[2]
    c_h = W["w_a"].shape[0]
    Wl = {k: np.asarray(v, np.float64).tolist() for k, v in W.items()}

    def ln(v, g, b):
        mu = sum(v) / len(v)
        var = sum((t - mu) ** 2 for t in v) / len(v)
        return [(v[q] - mu) / math.sqrt(var + 1e-5) * g[q] + b[q] for q in range(len(v))]

    def matvec(Wm, v):
        return [sum(Wm[o][q] * v[q] for q in range(len(v))) for o in range(len(Wm))]

    def sig(t):
        return 1.0 / (1.0 + math.exp(-t))

    zl = z.tolist()
    zh = [[ln(zl[i][j], Wl["ln_in_gamma"], Wl["ln_in_beta"]) for j in range(N)] for i in range(N)]
    a = [[[0.0] * c_h for _ in range(N)] for _ in range(N)]
    b = [[[0.0] * c_h for _ in range(N)] for _ in range(N)]
    for i in range(N):
        for k in range(N):
            ga = matvec(Wl["w_ga"], zh[i][k]); pa = matvec(Wl["w_a"], zh[i][k])
            gb = matvec(Wl["w_gb"], zh[i][k]); pb = matvec(Wl["w_b"], zh[i][k])
            for c in range(c_h):
                a[i][k][c] = sig(ga[c]) * pa[c] * m[i] * m[k]
                b[i][k][c] = sig(gb[c]) * pb[c] * m[i] * m[k]
    out = np.zeros((N, N, c_z))
    for i in range(N):
        for j in range(N):
            x = [0.0] * c_h
            for c in range(c_h):
                s = 0.0
                for k in range(N):
                    if direction == "outgoing":
                        s += a[i][k][c] * b[j][k][c]
                    else:
                        s += a[k][i][c] * b[k][j][c]
                x[c] = s
            y = matvec(Wl["w_o"], ln(x, Wl["ln_out_gamma"], Wl["ln_out_beta"]))
            g = matvec(Wl["w_g"], zh[i][j])
            for o in range(c_z):
                out[i, j, o] = sig(g[o]) * y[o]
    return out


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("shape", [(5, 3, 2), (6, 4, 5), (4, 2, 3)])
def test_brute_force_tiny(direction, shape):
    N, c_z, c_h = shape
    z, m, W = _inputs(N, c_z, c_h, seed=N + c_z, mask="scatter")
    m[1] = 0.0                                           # at least one masked token
    ref = _brute_force(z, m, W, direction)
    got = oracle.full(z, m, W, direction)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


# --------------------------------------------------------------------------- library routines

def test_layer_norm_matches_torch():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((7, 9, 33)) * 3 + 1.5
    g = rng.standard_normal(33)
    b = rng.standard_normal(33)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(v), (33,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.max(np.abs(oracle.layer_norm(v, g, b) - ref)) < 1e-12


def test_sigmoid_matches_scipy():
    v = np.concatenate([np.linspace(-700, 700, 30001), [0.0, -0.0, 1e-300, -1e-300]])
    ref = expit(v)
    got = oracle.sigmoid(v)
    assert np.all(np.abs(got - ref) <= 1e-15 * ref + 1e-320)


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(9)
    f = np.concatenate([(rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32),
                        np.float32([1.0, -1.0, 0.0, 3.0, 1.00390625, 1.01171875])]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6)
    assert oracle.round_to_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert oracle.round_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def test_half_ulp_bf16():
    v = np.array([1.0, 1.5, 2.0, 3.99, 0.75, -6.0])
    assert np.allclose(oracle.half_ulp_bf16(v), [2 ** -8, 2 ** -8, 2 ** -7, 2 ** -7, 2 ** -9, 2 ** -6])


# --------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("direction", DIRS)
def test_permutation_equivariance(direction):
    N = 13
    z, m, W = _inputs(N, 6, 5, seed=3)
    perm = np.random.default_rng(4).permutation(N)
    out = oracle.full(z, m, W, direction)
    out_p = oracle.full(z[np.ix_(perm, perm)], m[perm], W, direction)
    assert np.max(np.abs(out_p - out[np.ix_(perm, perm)])) < 1e-12


def _swap_ab(W):
    W2 = dict(W)
    W2["w_a"], W2["w_b"] = W["w_b"], W["w_a"]
    W2["w_ga"], W2["w_gb"] = W["w_gb"], W["w_ga"]
    return W2


def test_swap_transpose_identity():
    """incoming(z; W) == T(outgoing(T(z); W with (W_a, W_ga) <-> (W_b, W_gb))).

    Outgoing on the transposed grid sums a'_jk b'_ik = a_kj b_ki over k, which is
    the incoming x_ji with the roles of a and b exchanged.
    """
    z, m, W = _inputs(11, 5, 4, seed=8)
    zt = np.swapaxes(z, 0, 1)
    inc = oracle.full(z, m, W, "incoming")
    via_out = np.swapaxes(oracle.full(zt, m, _swap_ab(W), "outgoing"), 0, 1)
    assert np.max(np.abs(inc - via_out)) < 1e-12
    # the plain identity holds when a and b share their weights
    Ws = dict(W)
    Ws["w_b"], Ws["w_gb"] = W["w_a"], W["w_ga"]
    inc = oracle.full(z, m, Ws, "incoming")
    via_out = np.swapaxes(oracle.full(zt, m, Ws, "outgoing"), 0, 1)
    assert np.max(np.abs(inc - via_out)) < 1e-12
    # and it is not vacuous: with distinct weights the plain identity fails
    plain = np.swapaxes(oracle.full(zt, m, W, "outgoing"), 0, 1)
    assert np.max(np.abs(oracle.full(z, m, W, "incoming") - plain)) > 1e-3


@pytest.mark.parametrize("direction", DIRS)
def test_masked_tokens(direction):
    N = 12
    z, m, W = _inputs(N, 6, 5, seed=21, mask="full")
    m[[2, 7, 11]] = 0.0
    W["ln_out_beta"] = np.zeros_like(W["ln_out_beta"])
    out = oracle.full(z, m, W, direction)
    masked = m == 0
    # x_ij = 0 for a masked i or j, so out = sigmoid(W_g zh) * W_o beta_out = 0 here
    assert np.all(out[masked, :, :] == 0.0) and np.all(out[:, masked, :] == 0.0)
    # with a non-zero beta_out the masked entries equal the closed form
    W2 = dict(W)
    W2["ln_out_beta"] = np.linspace(-1, 1, 5).astype(np.float32)
    out2 = oracle.full(z, m, W2, direction)
    zh = oracle.layer_norm(z, W["ln_in_gamma"], W["ln_in_beta"])
    expect = expit(zh @ np.asarray(W["w_g"], np.float64).T) * (np.asarray(W2["w_o"], np.float64)
                                                              @ np.asarray(W2["ln_out_beta"], np.float64))
    assert np.max(np.abs(out2[masked] - expect[masked])) < 1e-12
    assert np.max(np.abs(out2[:, masked] - expect[:, masked])) < 1e-12
    # perturbing z on masked rows and columns changes no unmasked entry
    z2 = z.copy()
    rng = np.random.default_rng(1)
    z2[masked, :, :] += rng.standard_normal(z2[masked].shape) * 5
    z2[:, masked, :] += rng.standard_normal(z2[:, masked].shape) * 5
    out3 = oracle.full(z2, m, W, direction)
    keep = ~masked
    assert np.max(np.abs(out3[np.ix_(keep, keep)] - out[np.ix_(keep, keep)])) < 1e-12


@pytest.mark.parametrize("direction", DIRS)
def test_trailing_padding(direction):
    """Padding tokens appended at the end leave the leading block equal to the unpadded problem."""
    n, pad = 9, 4
    z, _, W = _inputs(n + pad, 6, 5, seed=31, mask="full")
    m = np.ones(n + pad)
    m[n:] = 0
    padded = oracle.full(z, m, W, direction)
    small = oracle.full(z[:n, :n], np.ones(n), W, direction)
    assert np.max(np.abs(padded[:n, :n] - small)) < 1e-12


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("direction", DIRS)
def test_constant_z_closed_form(direction):
    """z_ij = v everywhere, full mask: x_ij = N * alpha * beta for both directions, where
    alpha = sigmoid(W_ga vh) * (W_a vh), beta = sigmoid(W_gb vh) * (W_b vh), vh = LN(v)."""
    N, c_z, c_h = 7, 4, 3
    W = wl.make_weights(c_z, c_h, 4, ln_random=True)
    Wd = {k: np.asarray(v, np.float64) for k, v in W.items()}
    v = np.array([0.3, -1.2, 2.0, 0.7])
    z = np.broadcast_to(v, (N, N, c_z)).copy()
    mu = v.mean()
    sd = math.sqrt(((v - mu) ** 2).mean() + 1e-5)
    vh = (v - mu) / sd * Wd["ln_in_gamma"] + Wd["ln_in_beta"]
    sig = lambda t: 1 / (1 + np.exp(-t))          # noqa: E731
    alpha = sig(Wd["w_ga"] @ vh) * (Wd["w_a"] @ vh)
    beta = sig(Wd["w_gb"] @ vh) * (Wd["w_b"] @ vh)
    x = N * alpha * beta
    xm = x.mean()
    xs = math.sqrt(((x - xm) ** 2).mean() + 1e-5)
    y = Wd["w_o"] @ ((x - xm) / xs * Wd["ln_out_gamma"] + Wd["ln_out_beta"])
    expect = sig(Wd["w_g"] @ vh) * y
    out = oracle.full(z, np.ones(N), W, direction)
    assert np.max(np.abs(out - expect)) < 1e-12


@pytest.mark.parametrize("direction", DIRS)
def test_linear_special_case(direction):
    """W_ga = W_gb = 0 (sigmoid = 1/2) and W_a = W_b = I: x_c = Zh_c Zh_c^T / 4 (outgoing)
    or Zh_c^T Zh_c / 4 (incoming), one plain matrix product per channel."""
    N, c = 10, 4
    z, _, W = _inputs(N, c, c, seed=41, mask="full")
    W["w_ga"] = np.zeros((c, c), np.float32)
    W["w_gb"] = np.zeros((c, c), np.float32)
    W["w_a"] = np.eye(c, dtype=np.float32)
    W["w_b"] = np.eye(c, dtype=np.float32)
    zh, a, b, x = oracle.intermediates(z, np.ones(N), W, direction)
    for ch in range(c):
        Z = zh[:, :, ch]
        ref = Z @ Z.T / 4 if direction == "outgoing" else Z.T @ Z / 4
        assert np.max(np.abs(x[:, :, ch] - ref)) < 1e-12
    # the two directions differ on a non-symmetric z
    _, _, _, x_other = oracle.intermediates(z, np.ones(N), W,
                                            "incoming" if direction == "outgoing" else "outgoing")
    assert np.max(np.abs(x - x_other)) > 1e-3


# --------------------------------------------------------------------------- modes and storage

@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("storage", ["exact", "bf16"])
def test_sampled_equals_full(direction, storage):
    N = 37
    z = wl.make_z(N, 8, 5, "bf16")
    m = wl.make_mask(N, "scatter", 6)
    W = wl.make_weights(8, 6, 7, ln_random=True)
    full = oracle.full(z, m, W, direction, storage)
    rows = np.array([0, 3, 17, 36])
    cols = np.array([1, 2, 35, 36, 20])
    s = oracle.sampled(z, m, W, direction, rows, cols, storage)
    assert np.max(np.abs(s - full[np.ix_(rows, cols)])) < 1e-12


def test_bf16_storage_rounds_a_and_b():
    N = 9
    z, m, W = _inputs(N, 6, 5, seed=51)
    _, a, b, _ = oracle.intermediates(z, m, W, "outgoing", "exact")
    _, a16, b16, _ = oracle.intermediates(z, m, W, "outgoing", "bf16")
    for e, r in ((a, a16), (b, b16)):
        assert np.array_equal(r, oracle.round_to_bf16(r))                # bf16-representable
        assert np.all(np.abs(r - e) <= oracle.half_ulp_bf16(e) * (1 + 1e-12))
        assert np.any(r != e)


def test_errors_metric():
    ref = np.array([1.0, -1.0, 3.0, -3.0])
    got = ref + np.array([0.0, 0.01, 0.0, -0.02])
    e = oracle.errors(got, ref)
    rms = math.sqrt(5.0)
    assert abs(e["max_rel"] - 0.02 / rms) < 1e-15
    assert abs(e["rms_rel"] - math.sqrt((0.01 ** 2 + 0.02 ** 2) / 4) / rms) < 1e-15
    # bf16 output: an error within half a bf16 spacing of the reference is not excess
    e2 = oracle.errors(ref + np.array([2 ** -9, 0, 2 ** -7 + 0.001, 0]), ref, "bf16")
    assert e2["excess"] == pytest.approx(0.001 / rms, rel=1e-9)
