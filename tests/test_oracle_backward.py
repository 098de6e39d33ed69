"""Pins of the float64 backward oracle against facts that do not come from it.

* central finite differences of the forward oracle (itself pinned by brute
  force) for every element of z and of every weight, both directions, with a
  masked token and random LayerNorm affines;
* torch float64 autograd of a forward written here with torch operations;
* exact zeros: with beta_out = 0 no gradient reaches z at a masked token's row
  or column;
* the swap-transpose identity of the two directions, carried to gradients;
* planted mistakes in the backward steps are caught by the finite differences.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.trimul_backward as TB
from tests.test_oracle_pins import _inputs, _swap_ab

DIRS = ("outgoing", "incoming")


def _loss(z, m, W, direction, dout):
    return float(np.sum(oracle.full(z, m, W, direction) * dout))


def _finite_differences(z, m, W, direction, dout, h=1e-6):
    """Central differences of sum(dout * update) for every element of z and of each weight."""
    fd = {"z": np.zeros_like(z)}
    it = np.nditer(z, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        zp, zm = z.copy(), z.copy()
        zp[idx] += h
        zm[idx] -= h
        fd["z"][idx] = (_loss(zp, m, W, direction, dout) - _loss(zm, m, W, direction, dout)) / (2 * h)
    for name in oracle.WEIGHT_NAMES:
        w = np.asarray(W[name], np.float64)
        g = np.zeros_like(w)
        for idx in np.ndindex(*w.shape):
            Wp, Wm = dict(W), dict(W)
            wp, wm = w.copy(), w.copy()
            wp[idx] += h
            wm[idx] -= h
            Wp[name], Wm[name] = wp, wm
            g[idx] = (_loss(z, m, Wp, direction, dout) - _loss(z, m, Wm, direction, dout)) / (2 * h)
        fd[name] = g
    return fd


def _case(N=5, c_z=4, c_h=3, seed=23):
    z, m, W = _inputs(N, c_z, c_h, seed=seed, mask="scatter")
    m[1] = 0.0
    W = {k: np.asarray(v, np.float64) for k, v in W.items()}
    dout = np.random.default_rng(seed + 5).standard_normal((N, N, c_z))
    return z, m, W, dout


def _worst(got, ref):
    """Largest deviation over all gradients, each relative to its own largest magnitude."""
    return max(float(np.max(np.abs(got[k] - ref[k])) / max(np.max(np.abs(ref[k])), 1e-30)) for k in ref)


@pytest.mark.parametrize("direction", DIRS)
def test_backward_matches_finite_differences(direction):
    z, m, W, dout = _case()
    an = oracle.full_backward(z, m, W, direction, dout)
    fd = _finite_differences(z, m, W, direction, dout)
    for k in fd:
        assert an[k].shape == fd[k].shape, k
    # central differences with h = 1e-6 in float64: truncation ~h^2, cancellation ~1e-16/h
    assert _worst(an, fd) < 1e-6


def _torch_forward(z, m, W, direction):
    """The update written with torch float64 operations, for autograd."""
    def ln(v, g, b):
        mu = v.mean(-1, keepdim=True)
        var = ((v - mu) ** 2).mean(-1, keepdim=True)
        return (v - mu) / torch.sqrt(var + 1e-5) * g + b

    zh = ln(z, W["ln_in_gamma"], W["ln_in_beta"])
    M = (m[:, None] * m[None, :])[..., None]
    a = torch.sigmoid(zh @ W["w_ga"].T) * (zh @ W["w_a"].T) * M
    b = torch.sigmoid(zh @ W["w_gb"].T) * (zh @ W["w_b"].T) * M
    if direction == "outgoing":
        x = torch.einsum("ikc,jkc->ijc", a, b)
    else:
        x = torch.einsum("kic,kjc->ijc", a, b)
    return torch.sigmoid(zh @ W["w_g"].T) * (ln(x, W["ln_out_gamma"], W["ln_out_beta"]) @ W["w_o"].T)


@pytest.mark.parametrize("direction", DIRS)
def test_backward_matches_torch_autograd(direction):
    z, m, W, dout = _case(N=9, c_z=6, c_h=5, seed=31)
    zt = torch.tensor(z, requires_grad=True)
    Wt = {k: torch.tensor(v, requires_grad=True) for k, v in W.items()}
    out = _torch_forward(zt, torch.tensor(m), Wt, direction)
    (out * torch.tensor(dout)).sum().backward()
    ref = {"z": zt.grad.numpy()}
    ref.update({k: Wt[k].grad.numpy() for k in oracle.WEIGHT_NAMES})
    assert _worst(oracle.full_backward(z, m, W, direction, dout), ref) < 1e-12


@pytest.mark.parametrize("direction", DIRS)
def test_masked_tokens_get_no_gradient(direction):
    """With beta_out = 0 a masked token's row and column of out are 0 whatever z holds there, and z
    there feeds nothing else (a and b are masked at those pairs): its gradient is exactly 0."""
    z, m, W, dout = _case(N=7, c_z=4, c_h=3, seed=41)
    m[4] = 0.0
    W["ln_out_beta"] = np.zeros_like(W["ln_out_beta"])
    g = oracle.full_backward(z, m, W, direction, dout)
    for t in np.flatnonzero(m == 0):
        assert np.all(g["z"][t, :, :] == 0.0) and np.all(g["z"][:, t, :] == 0.0)
    live = np.flatnonzero(m)
    assert np.all(np.abs(g["z"][np.ix_(live, live)]).max(axis=-1) > 0)


def test_swap_transpose_identity_of_the_gradient():
    """incoming(z; W) = T(outgoing(T(z); W_swap)) makes the gradient of sum(dout * incoming) at z the
    transpose of the outgoing gradient at T(z) for the cotangent T(dout), with the a and b weight
    gradients exchanged."""
    z, m, W, dout = _case(N=8, c_z=5, c_h=4, seed=53)
    gin = oracle.full_backward(z, m, W, "incoming", dout)
    gout = oracle.full_backward(np.swapaxes(z, 0, 1), m, _swap_ab(W), "outgoing", np.swapaxes(dout, 0, 1))
    gout["z"] = np.swapaxes(gout["z"], 0, 1)
    gout = _swap_ab(gout)
    assert _worst(gin, gout) < 1e-12


def test_bf16_storage_differs_only_by_the_rounding_of_a_and_b():
    z, m, W, dout = _case(N=10, c_z=6, c_h=5, seed=61)
    ex = oracle.full_backward(z, m, W, "outgoing", dout)
    bf = oracle.full_backward(z, m, W, "outgoing", dout, storage="bf16")
    assert 0 < _worst(bf, ex) < 3e-2


# --------------------------------------------------------------------------- planted mistakes

def _ln_bwd_drops_projection(v, gamma, dout, eps=oracle.LN_EPS):
    dv, dg, db = TB.__dict__["_orig_ln_bwd"](v, gamma, dout, eps)
    v = np.asarray(v, np.float64)
    mu = v.mean(-1, keepdims=True)
    r = 1.0 / np.sqrt(((v - mu) ** 2).mean(-1, keepdims=True) + eps)
    n = (v - mu) * r
    dn = dout * gamma
    return dv + r * n * (dn * n).mean(-1, keepdims=True), dg, db


def _contract_bwd_swapped(dx, a, b, direction):
    da, db = TB.__dict__["_orig_contract_bwd"](dx, a, b, direction)
    return db, da


def _contract_bwd_untransposed(dx, a, b, direction):
    dX = np.moveaxis(dx, -1, 0)
    A = np.moveaxis(a, -1, 0)
    B = np.moveaxis(b, -1, 0)
    dA = np.matmul(dX, B)
    dB = np.matmul(dX, A)
    return np.moveaxis(dA, 0, -1), np.moveaxis(dB, 0, -1)


def _proj_bwd_no_mask(da, zh, pair_mask, w_gate, w_val):
    return TB.__dict__["_orig_proj_bwd"](da, zh, np.ones_like(pair_mask), w_gate, w_val)


def _proj_bwd_gate_sign(da, zh, pair_mask, w_gate, w_val):
    dzh, dwg, dwv = TB.__dict__["_orig_proj_bwd"](da, zh, pair_mask, w_gate, w_val)
    s = oracle.sigmoid(zh @ w_gate.T)
    dga = da * (zh @ w_val.T) * pair_mask[..., None] * s * (1 - s)
    return dzh - 2 * dga @ w_gate, -dwg, dwv


def _out_bwd_gate_on_dy(dout, x, zh, W):
    dx, dzh, grads = TB.__dict__["_orig_out_bwd"](dout, x, zh, W)
    return dx, dzh * 0.5, grads


BWD_MUTATIONS = {
    "ln_backward_drops_projection": ("layer_norm_backward", _ln_bwd_drops_projection),
    "contract_backward_swapped": ("contract_backward", _contract_bwd_swapped),
    "contract_backward_untransposed": ("contract_backward", _contract_bwd_untransposed),
    "projection_backward_no_mask": ("gated_projection_backward", _proj_bwd_no_mask),
    "projection_backward_gate_sign": ("gated_projection_backward", _proj_bwd_gate_sign),
    "output_backward_halves_gate_term": ("output_backward", _out_bwd_gate_on_dy),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTATIONS))
def test_finite_differences_catch_planted_backward_mistake(monkeypatch, name):
    z, m, W, dout = _case(N=4, c_z=3, c_h=2, seed=71)
    fd = {d: _finite_differences(z, m, W, d, dout) for d in DIRS}
    for d in DIRS:
        assert _worst(oracle.full_backward(z, m, W, d, dout), fd[d]) < 1e-6
    monkeypatch.setitem(TB.__dict__, "_orig_ln_bwd", TB.layer_norm_backward)
    monkeypatch.setitem(TB.__dict__, "_orig_contract_bwd", TB.contract_backward)
    monkeypatch.setitem(TB.__dict__, "_orig_proj_bwd", TB.gated_projection_backward)
    monkeypatch.setitem(TB.__dict__, "_orig_out_bwd", TB.output_backward)
    fn_name, bad = BWD_MUTATIONS[name]
    monkeypatch.setattr(TB, fn_name, bad)
    worst = max(_worst(oracle.full_backward(z, m, W, d, dout), fd[d]) for d in DIRS)
    assert worst > 1e-4, f"planted mistake {name} went unnoticed"
