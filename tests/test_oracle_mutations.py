"""Planted mistakes in the oracle must be caught by its pins.

Each case patches one step of the float64 oracle with a plausible slip (on the
CPU, inside this test only) and checks that the brute-force pin and the
invariant pins tell the patched oracle apart from the definition.
"""
import numpy as np
import pytest

import oracle
import oracle.trimul as T
from tests.test_oracle_pins import _brute_force, _inputs, _swap_ab


def _ln_unbiased(v, gamma, beta, eps=T.LN_EPS):
    v = np.asarray(v, np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    var = v.var(axis=-1, ddof=1, keepdims=True)
    return (v - mu) / np.sqrt(var + eps) * gamma + beta


def _ln_no_affine_beta(v, gamma, beta, eps=T.LN_EPS):
    v = np.asarray(v, np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)
    return (v - mu) / np.sqrt(var + eps) * gamma


def _sigmoid_sign(v):
    return 1.0 / (1.0 + np.exp(np.clip(v, -700, 700)))


def _contract_transposed_b(a, b, direction):
    A = np.moveaxis(a, -1, 0)
    B = np.moveaxis(b, -1, 0)
    X = np.matmul(A, B) if direction == "outgoing" else np.matmul(np.swapaxes(A, 1, 2), np.swapaxes(B, 1, 2))
    return np.moveaxis(X, 0, -1)


def _contract_swapped_direction(a, b, direction):
    return T.__dict__["_orig_contract"](a, b, "incoming" if direction == "outgoing" else "outgoing")


def _projection_no_mask(zh, pair_mask, w_gate, w_val, storage="exact"):
    return T.sigmoid(zh @ w_gate.T) * (zh @ w_val.T)


def _projection_row_mask_only(zh, pair_mask, w_gate, w_val, storage="exact"):
    row = pair_mask.max(axis=1)              # m_i instead of m_i m_k
    return T.sigmoid(zh @ w_gate.T) * (zh @ w_val.T) * row[:, None, None]


def _projection_ungated(zh, pair_mask, w_gate, w_val, storage="exact"):
    return (zh @ w_val.T) * pair_mask[..., None]


def _output_gate_transposed(x, zh, W):
    g = T.sigmoid(zh @ W["w_g"])
    return g * (T.layer_norm(x, W["ln_out_gamma"], W["ln_out_beta"]) @ W["w_o"].T)


def _output_no_norm(x, zh, W):
    return T.sigmoid(zh @ W["w_g"].T) * (x @ W["w_o"].T)


MUTATIONS = {
    "layer_norm_unbiased": ("layer_norm", _ln_unbiased),
    "layer_norm_drops_beta": ("layer_norm", _ln_no_affine_beta),
    "sigmoid_sign": ("sigmoid", _sigmoid_sign),
    "contract_transposed_b": ("contract", _contract_transposed_b),
    "contract_swapped_direction": ("contract", _contract_swapped_direction),
    "projection_no_mask": ("gated_projection", _projection_no_mask),
    "projection_row_mask_only": ("gated_projection", _projection_row_mask_only),
    "projection_ungated": ("gated_projection", _projection_ungated),
    "output_gate_transposed": ("output", _output_gate_transposed),
    "output_no_norm": ("output", _output_no_norm),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(monkeypatch, name):
    fn_name, bad = MUTATIONS[name]
    z, m, W = _inputs(5, 4, 3, seed=17, mask="scatter")
    m[0] = 0.0
    refs = {d: _brute_force(z, m, W, d) for d in ("outgoing", "incoming")}
    # the unpatched oracle agrees with the brute force ...
    for d, ref in refs.items():
        assert np.max(np.abs(oracle.full(z, m, W, d) - ref)) < 1e-12
    monkeypatch.setitem(T.__dict__, "_orig_contract", T.contract)
    monkeypatch.setattr(T, fn_name, bad)
    # ... and the patched one does not, in at least one direction
    worst = max(float(np.max(np.abs(oracle.full(z, m, W, d) - ref))) for d, ref in refs.items())
    assert worst > 1e-6, f"planted mistake {name} went unnoticed"


def test_swap_identity_catches_swapped_direction(monkeypatch):
    """An oracle with the two directions exchanged also breaks the swap-transpose identity
    against the brute force, not only the brute-force comparison."""
    z, m, W = _inputs(6, 4, 3, seed=19)
    ref_in = _brute_force(z, m, W, "incoming")
    monkeypatch.setitem(T.__dict__, "_orig_contract", T.contract)
    monkeypatch.setattr(T, "contract", _contract_swapped_direction)
    via = np.swapaxes(oracle.full(np.swapaxes(z, 0, 1), m, _swap_ab(W), "outgoing"), 0, 1)
    assert np.max(np.abs(via - ref_in)) > 1e-6
