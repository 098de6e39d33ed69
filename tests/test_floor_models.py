"""The storage models logged beside the GPU paths' errors are the oracles' arithmetic plus rounding.

tests/backward_storage_model.py and tests/attention_storage_model.py round values where the paths store
them. With that rounding replaced by the identity each model must reproduce its float64 oracle
exactly; a slip in a model (a dropped term, a wrong index) would otherwise misreport what the storage
costs. With the rounding in place the models must differ from the oracles by an amount the size of
that rounding.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.triangle_attention as TA
import workloads as wl
from tests import attention_storage_model as AF
from tests import backward_storage_model as BF


def _small_attention_case(N=9, seed=3):
    rng = np.random.default_rng(seed)
    W = {k: rng.standard_normal(s) / math.sqrt(s[-1]) for k, s in TA.weight_shapes(128, 4, 32).items()}
    W["ln_gamma"] = 1.0 + 0.3 * rng.standard_normal(128)
    W["ln_beta"] = 0.3 * rng.standard_normal(128)
    z = rng.standard_normal((N, N, 128))
    m = np.ones(N)
    m[2] = 0.0
    return z, m, W


@pytest.mark.parametrize("node", TA.NODES)
def test_attention_model_without_rounding_is_the_oracle(monkeypatch, node):
    z, m, W = _small_attention_case()
    monkeypatch.setattr(AF, "rh", lambda v: np.asarray(v, np.float64))
    monkeypatch.setattr(AF, "rb", lambda v: np.asarray(v, np.float64))
    ref = TA.full(z, m, W, node)
    assert np.max(np.abs(AF.emulated(z, m, W, node) - ref)) < 1e-10
    lines = [0, 2, 8]
    bias = TA.pair_bias(z if node == "starting" else np.swapaxes(z, 0, 1), W)
    got = AF.emulated_lines(z, m, W, node, lines, bias)
    want = ref[lines] if node == "starting" else np.swapaxes(ref[:, lines], 0, 1)
    assert np.max(np.abs(got - want)) < 1e-10


@pytest.mark.parametrize("node", TA.NODES)
def test_attention_model_rounding_is_fp16_sized(monkeypatch, node):
    z, m, W = _small_attention_case()
    ref = TA.full(z, m, W, node)
    rms = np.sqrt(np.mean(ref ** 2))
    # the fp16 intermediates alone (result unrounded): errors of order 2^-11
    monkeypatch.setattr(AF, "rb", lambda v: np.asarray(v, np.float64))
    d = np.max(np.abs(AF.emulated(z, m, W, node) - ref)) / rms
    assert 1e-5 < d < 5e-3
    # fp16 rounding pinned against numpy's own half-precision conversion of exactly representable and
    # halfway values
    assert AF.rh(1.0 + 2.0 ** -11) == 1.0 and AF.rh(1.0 + 3 * 2.0 ** -11) == 1.0 + 2.0 ** -9
    assert AF.rh(65504.0) == 65504.0 and AF.rh(2.0 ** -24) == 2.0 ** -24


def test_backward_model_without_rounding_is_the_oracle(monkeypatch):
    N = 10
    W = wl.make_weights(128, 128, 4, ln_random=True)
    z = wl.as_f64(wl.make_z(N, 128, 5, "bf16"))
    m = wl.make_mask(N, "scatter", 6)
    dout = wl.as_f64(wl.make_z(N, 128, 7, "bf16"))
    ref = oracle.full_backward(z, m, W, "outgoing", dout, storage="bf16")
    monkeypatch.setattr(BF, "rh", lambda v: np.asarray(v, np.float64))
    monkeypatch.setattr(BF, "rb", lambda v: np.asarray(v, np.float64))
    got = BF.emulated_backward(z, m, W, "outgoing", dout)
    for k in ref:
        scale = max(np.max(np.abs(ref[k])), 1e-30)
        assert np.max(np.abs(got[k] - ref[k])) / scale < 1e-10, k


def test_backward_model_rounding_is_fp16_sized(monkeypatch):
    N = 10
    W = wl.make_weights(128, 128, 4, ln_random=True)
    z = wl.as_f64(wl.make_z(N, 128, 5, "bf16"))
    m = wl.make_mask(N, "scatter", 6)
    dout = wl.as_f64(wl.make_z(N, 128, 7, "bf16"))
    ref = oracle.full_backward(z, m, W, "outgoing", dout, storage="bf16")
    monkeypatch.setattr(BF, "rb", lambda v: np.asarray(v, np.float64))   # dz unrounded: fp16 operands alone
    got = BF.emulated_backward(z, m, W, "outgoing", dout)
    worst = max(np.max(np.abs(got[k] - ref[k])) / np.sqrt(np.mean(ref[k] ** 2)) for k in ref)
    assert 1e-5 < worst < 1e-2
