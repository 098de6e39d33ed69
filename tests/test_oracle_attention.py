"""Pins of the float64 triangle-attention oracle against facts that do not come from it.

* brute force: scalar loops for both nodes, the ending node written with its own indices
  (q_ij . k_kj + b_ki), not as a transpose of the starting node;
* library: the per-row attention against torch's scaled_dot_product_attention in float64;
* closed form: with W_q = 0 and W_b = 0 every valid key has the same weight;
* invariants: permutation equivariance, masked tokens, rows without a valid key;
* planted mistakes in the oracle are caught by the brute force.
"""
import math

import numpy as np
import pytest
import torch

import oracle.triangle_attention as TA
import workloads as wl

NODES = TA.NODES


def _weights(c_z, H, c, seed, ln_random=True):
    rng = np.random.default_rng(seed)
    W = {k: rng.standard_normal(s) / math.sqrt(s[-1]) for k, s in TA.weight_shapes(c_z, H, c).items()}
    if ln_random:
        W["ln_gamma"] = 1.0 + 0.3 * rng.standard_normal(c_z)
        W["ln_beta"] = 0.3 * rng.standard_normal(c_z)
    else:
        W["ln_gamma"], W["ln_beta"] = np.ones(c_z), np.zeros(c_z)
    return W


def _inputs(N, c_z, H, c, seed=0):
    z = np.random.default_rng(seed).standard_normal((N, N, c_z))
    m = wl.make_mask(N, "scatter", seed + 3).astype(np.float64)
    return z, m, _weights(c_z, H, c, seed + 1)


def _brute(z, m, W, node, H, c):
    N, c_z = z.shape[0], z.shape[2]
    Wl = {k: np.asarray(v, np.float64).tolist() for k, v in W.items()}

    def ln(x):
        mu = sum(x) / len(x)
        var = sum((t - mu) ** 2 for t in x) / len(x)
        return [(x[q] - mu) / math.sqrt(var + 1e-5) * Wl["ln_gamma"][q] + Wl["ln_beta"][q] for q in range(len(x))]

    def mv(M, x):
        return [sum(M[o][q] * x[q] for q in range(len(x))) for o in range(len(M))]

    zh = [[ln(z[i, j].tolist()) for j in range(N)] for i in range(N)]
    proj = {n: [[mv(Wl[n], zh[i][j]) for j in range(N)] for i in range(N)] for n in ("w_q", "w_k", "w_v", "w_b", "w_g")}
    out = np.zeros((N, N, c_z))
    for i in range(N):
        for j in range(N):
            o = []
            for h in range(H):
                q = proj["w_q"][i][j][h * c:(h + 1) * c]
                logits, vals = [], []
                for k in range(N):
                    if node == "starting":
                        if m[i] * m[k] == 0:
                            continue
                        kk = proj["w_k"][i][k][h * c:(h + 1) * c]
                        vv = proj["w_v"][i][k][h * c:(h + 1) * c]
                        bias = proj["w_b"][j][k][h]
                    else:
                        if m[k] * m[j] == 0:
                            continue
                        kk = proj["w_k"][k][j][h * c:(h + 1) * c]
                        vv = proj["w_v"][k][j][h * c:(h + 1) * c]
                        bias = proj["w_b"][k][i][h]
                    logits.append(sum(q[t] * kk[t] for t in range(c)) / math.sqrt(c) + bias)
                    vals.append(vv)
                acc = [0.0] * c
                if logits:
                    mx = max(logits)
                    ws = [math.exp(s - mx) for s in logits]
                    tot = sum(ws)
                    for wgt, vv in zip(ws, vals):
                        for t in range(c):
                            acc[t] += wgt / tot * vv[t]
                gate = [1.0 / (1.0 + math.exp(-t)) for t in proj["w_g"][i][j][h * c:(h + 1) * c]]
                o += [gate[t] * acc[t] for t in range(c)]
            out[i, j] = mv(Wl["w_o"], o)
    return out


@pytest.mark.parametrize("node", NODES)
@pytest.mark.parametrize("shape", [(5, 4, 2, 3), (6, 6, 3, 2), (4, 3, 1, 4)])
def test_brute_force(node, shape):
    N, c_z, H, c = shape
    z, m, W = _inputs(N, c_z, H, c, seed=N * 7 + H)
    m[1] = 0.0
    ref = _brute(z, m, W, node, H, c)
    got = TA.full(z, m, W, node, H, c)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_attention_rows_match_torch_sdpa():
    rng = np.random.default_rng(3)
    N, H, c = 9, 3, 5
    q, k, v = (rng.standard_normal((N, N, H, c)) for _ in range(3))
    bias = rng.standard_normal((H, N, N))
    valid = np.ones((N, N), bool)
    valid[:, 4] = False
    got = TA.attention_rows(q, k, v, bias, valid)
    for i in range(N):
        for h in range(H):
            add = torch.tensor(bias[h]).clone()
            add[:, ~torch.tensor(valid[i])] = -math.inf
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[i, :, h])[None], torch.tensor(k[i, :, h])[None], torch.tensor(v[i, :, h])[None],
                attn_mask=add[None])[0].numpy()
            assert np.max(np.abs(got[i, :, h] - ref)) < 1e-12


@pytest.mark.parametrize("node", NODES)
def test_uniform_weights_when_logits_are_constant(node):
    """W_q = 0 and W_b = 0: every valid key weighs the same, o = g * mean of the valid v."""
    N, c_z, H, c = 7, 6, 2, 3
    z, m, W = _inputs(N, c_z, H, c, seed=5)
    m[2] = 0.0
    W["w_q"] = np.zeros_like(W["w_q"])
    W["w_b"] = np.zeros_like(W["w_b"])
    zz = z if node == "starting" else np.swapaxes(z, 0, 1)
    zh = (zz - zz.mean(-1, keepdims=True)) / np.sqrt(zz.var(-1, keepdims=True) + 1e-5) * W["ln_gamma"] + W["ln_beta"]
    v = (zh @ W["w_v"].T).reshape(N, N, H, c)
    g = 1.0 / (1.0 + np.exp(-(zh @ W["w_g"].T))).reshape(N, N, H, c)
    o = np.zeros((N, N, H, c))
    for i in range(N):
        ks = [k for k in range(N) if m[i] * m[k] != 0]
        if ks:
            o[i] = g[i] * v[i, ks].mean(axis=0)[None]
    ref = o.reshape(N, N, H * c) @ W["w_o"].T
    if node == "ending":
        ref = np.swapaxes(ref, 0, 1)
    assert np.max(np.abs(TA.full(z, m, W, node, H, c) - ref)) < 1e-12


@pytest.mark.parametrize("node", NODES)
def test_permutation_equivariance(node):
    N, c_z, H, c = 8, 5, 2, 3
    z, m, W = _inputs(N, c_z, H, c, seed=9)
    perm = np.random.default_rng(4).permutation(N)
    out = TA.full(z, m, W, node, H, c)
    out_p = TA.full(z[np.ix_(perm, perm)], m[perm], W, node, H, c)
    assert np.max(np.abs(out_p - out[np.ix_(perm, perm)])) < 1e-12


@pytest.mark.parametrize("node", NODES)
def test_masked_tokens(node):
    """Unmasked outputs ignore z at masked tokens' rows and columns; rows (starting) or columns (ending)
    of a masked token have no valid key and give 0."""
    N, c_z, H, c = 8, 5, 2, 3
    z, m, W = _inputs(N, c_z, H, c, seed=11)
    m[:] = 1.0
    m[[2, 5]] = 0.0
    out = TA.full(z, m, W, node, H, c)
    z2 = z.copy()
    z2[[2, 5], :, :] += 3.0 * np.random.default_rng(1).standard_normal((2, N, c_z))
    z2[:, [2, 5], :] -= 2.0
    out2 = TA.full(z2, m, W, node, H, c)
    live = np.flatnonzero(m)
    assert np.max(np.abs(out2[np.ix_(live, live)] - out[np.ix_(live, live)])) < 1e-12
    dead = np.flatnonzero(m == 0)
    if node == "starting":
        assert np.all(out[dead, :, :] == 0.0)
    else:
        assert np.all(out[:, dead, :] == 0.0)


@pytest.mark.parametrize("node", NODES)
def test_sampled_lines_equal_full(node):
    N, c_z, H, c = 11, 6, 2, 3
    z, m, W = _inputs(N, c_z, H, c, seed=13)
    m[4] = 0.0
    full = TA.full(z, m, W, node, H, c)
    lines = [0, 4, 10]
    got = TA.sampled(z, m, W, node, lines, H, c)
    ref = full[lines] if node == "starting" else np.swapaxes(full[:, lines], 0, 1)
    assert np.max(np.abs(got - ref)) < 1e-12


# --------------------------------------------------------------------------- planted mistakes

def _rows_no_scale(q, k, v, bias, key_valid):
    return TA.__dict__["_orig_rows"](q * math.sqrt(q.shape[-1]), k, v, bias, key_valid)


def _rows_bias_transposed(q, k, v, bias, key_valid):
    return TA.__dict__["_orig_rows"](q, k, v, np.swapaxes(bias, 1, 2), key_valid)


def _rows_mask_on_queries(q, k, v, bias, key_valid):
    o = TA.__dict__["_orig_rows"](q, k, v, bias, np.ones_like(key_valid))
    return o * key_valid[:, :, None, None]


def _rows_softmax_over_queries(q, k, v, bias, key_valid):
    c = q.shape[-1]
    s = np.einsum("ijhc,ikhc->ihjk", q, k) / np.sqrt(c) + bias[None]
    s = np.where(key_valid[:, None, None, :], s, -np.inf)
    with np.errstate(invalid="ignore"):
        e = np.exp(s - np.max(s, axis=-2, keepdims=True))
        a = e / e.sum(axis=-2, keepdims=True)
    return np.einsum("ihjk,ikhc->ijhc", np.nan_to_num(a), v)


MUTATIONS = {"no_scale": _rows_no_scale, "bias_transposed": _rows_bias_transposed,
             "mask_on_queries": _rows_mask_on_queries, "softmax_over_queries": _rows_softmax_over_queries}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_brute_force_catches_planted_mistake(monkeypatch, name):
    N, c_z, H, c = 5, 4, 2, 3
    z, m, W = _inputs(N, c_z, H, c, seed=21)
    m[3] = 0.0
    refs = {n: _brute(z, m, W, n, H, c) for n in NODES}
    for n in NODES:
        assert np.max(np.abs(TA.full(z, m, W, n, H, c) - refs[n])) < 1e-12
    monkeypatch.setitem(TA.__dict__, "_orig_rows", TA.attention_rows)
    monkeypatch.setattr(TA, "attention_rows", MUTATIONS[name])
    worst = max(float(np.max(np.abs(TA.full(z, m, W, n, H, c) - refs[n]))) for n in NODES)
    assert worst > 1e-6, f"planted mistake {name} went unnoticed"
