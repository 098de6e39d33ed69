"""Triangle attention through the C ABI (tm_attn_forward) against the float64 oracle.

The gates are fixed numbers against the exact float64 oracle, the bf16 tolerance of the update read
the same way (tests/gpu_util.py): the result is stored as bf16, so the half-ulp rounding of each
output element is not counted, and the error beyond it must stay within BF16_TOL of rms(ref)
("excess"); rms|delta|/rms(ref) within BF16_TOL; the literal max|delta|/rms(ref) within
BF16_LITERAL_BOUND. The path keeps every intermediate in fp16 (zh, the weights, q, k, v, g, the
pair bias, the softmax weights P and the gated output o); tests/attention_storage_model.py, which
applies exactly those roundings to the oracle's arithmetic, is logged beside the path's error as a
diagnostic only (it predicts excess ~5e-3 and rms ~2e-3 for these cases).
"""
import json
import os

import numpy as np
import pytest

import oracle
import oracle.triangle_attention as TA
import workloads as wl
from tests.attention_storage_model import attention_weights, floor as model_error
from tests.gpu_util import BF16_LITERAL_BOUND, BF16_TOL, mask_to_device, to_f64, z_to_device

pytestmark = pytest.mark.gpu


def gate(got, ref):
    """The attention's parity gates; returns the metrics."""
    e = oracle.errors(got, ref, "bf16")
    assert np.all(np.isfinite(got))
    assert e["excess"] <= BF16_TOL, e
    assert e["rms_rel"] <= BF16_TOL, e
    assert e["max_rel"] <= BF16_LITERAL_BOUND, e
    return e


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build, tm
    build.build()
    W = attention_weights()
    mod = tm.TriangleAttention(W)
    yield torch, tm, mod, W
    mod.close()


@pytest.mark.parametrize("node", TA.NODES)
@pytest.mark.parametrize("N,mask", [(64, "scatter"), (129, "last10pct"), (200, "scatter")])
def test_attention_bf16(env, node, N, mask):
    torch, tm, mod, W = env
    z_np = wl.make_z(N, 128, 31 + N, "bf16")
    m_np = wl.make_mask(N, mask, 12)
    out = mod(z_to_device(z_np), mask_to_device(m_np), node)
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    got = to_f64(out)
    ref = TA.full(wl.as_f64(z_np), m_np, W, node)
    fl, fl_rms = model_error(N, mask, node, 31 + N, rms=True)
    e = oracle.errors(got, ref, "bf16")
    log = os.environ.get("TM_METRICS_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": f"attn_{node}_N{N}_{mask}", "max_rel": e["max_rel"], "excess": e["excess"],
                                "rms_rel": e["rms_rel"], "model_max_rel": fl, "model_rms_rel": fl_rms}) + "\n")
    gate(got, ref)
    # rows (starting) or columns (ending) of masked tokens have no valid key: exactly 0
    dead = np.flatnonzero(m_np == 0)
    if dead.size:
        assert np.all((got[dead] if node == "starting" else got[:, dead]) == 0.0)


def test_attention_is_deterministic_and_checks_arguments(env):
    torch, tm, mod, W = env
    N = 150
    z = z_to_device(wl.make_z(N, 128, 5, "bf16"))
    a = mod(z, None, "ending")
    b = mod(z, None, "ending")
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    with pytest.raises(tm.TmError):
        mod(z, None, "starting", out=z)                 # out over z
    with pytest.raises(tm.TmError):
        tm.tm_attn_forward(mod.ctx, z.float(), None, "starting", torch.empty_like(z.float()))   # float32
    upd = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    try:
        with pytest.raises(tm.TmError):                 # an update ctx is not an attention ctx
            tm.tm_attn_forward(upd.ctx, z, None, "starting", torch.empty_like(z))
        with pytest.raises(tm.TmError):
            tm.tm_forward(mod.ctx, z, None, "outgoing", torch.empty_like(z))
    finally:
        upd.close()


def test_attention_refuses_a_workspace_over_the_limit(env):
    torch, tm, mod, W = env
    z = z_to_device(wl.make_z(200, 128, 3, "bf16"))
    launches = tm.tm_launch_count(mod.ctx)
    with pytest.raises(tm.TmError) as err:
        tm.tm_attn_forward(mod.ctx, z, None, "starting", torch.empty_like(z), workspace_limit=1 << 20)
    assert err.value.status == tm.TM_ERR_OOM
    assert tm.tm_launch_count(mod.ctx) == launches
    mod(z, None, "starting")
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK


@pytest.mark.parametrize("name", ["w_q", "w_k", "w_b"])
def test_attention_refuses_logit_weights_that_could_overflow_fp16(env, name):
    """q, k and the pair bias enter the logits unscaled: weights whose bound on them reaches 2^15 are
    refused at creation."""
    torch, tm, mod, W = env
    big = dict(W)
    big[name] = W[name] * 1e5
    with pytest.raises(tm.TmError) as err:
        tm.TriangleAttention(big)
    assert err.value.status == tm.TM_ERR_UNSUPPORTED


@pytest.mark.parametrize("gain", [1e5, 2.0 ** -20])
def test_attention_scales_v_and_the_weight_images(env, gain):
    """v (and o) are stored times a power of two set by the bound on |v|, and every weight image by its
    own: very large or very small W_v and W_o (the output is linear in each, so the problem's conditioning
    does not change; a scaled W_g would turn the gate into a step function) meet the same gates."""
    torch, tm, mod, W = env
    scaled = dict(W)
    for k in ("w_v", "w_o"):
        scaled[k] = W[k] * gain
    att = tm.TriangleAttention(scaled)
    try:
        N = 40
        z_np = wl.make_z(N, 128, 9, "bf16")
        got = to_f64(att(z_to_device(z_np), None, "starting"))
        gate(got, TA.full(wl.as_f64(z_np), np.ones(N), scaled, "starting"))
    finally:
        att.close()


def test_ex2_probe_rate_is_plausible(env):
    """The special-function pipe probe (the attention roofline's peak) returns a rate between a quarter of
    the nominal unit count (16 per clock per SM at the maximum clock) and two and a half times it."""
    _, tm, _, _ = env
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    try:
        launches = tm.tm_launch_count(mod.ctx)
        rate = tm.tm_probe_ex2_rate(mod.ctx)
        assert tm.tm_launch_count(mod.ctx) == launches + 2
        nominal = 16 * 148 * 2032e6
        assert 0.25 * nominal < rate < 2.5 * nominal, rate
    finally:
        mod.close()
