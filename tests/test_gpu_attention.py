"""Triangle attention through the C ABI (tm_attn_forward) against the float64 oracle.

Metric: max|got - ref| / rms(ref) over the whole grid, ref the exact float64 oracle. The bf16 path
stores zh, the weights, q, k, v, g, the pair bias, the softmax weights P, the gated output o and the
result in bf16; tests/bf16_attention_floor.py applies exactly those roundings to the oracle's
arithmetic and gives the error they alone cause (0.040-0.056 of rms for these cases). The path must
stay within FLOOR_FACTOR times that floor (plus FLOOR_SLACK) and within ABS_TOL, about twice the
largest floor; its rms error must stay within FLOOR_FACTOR times the model's rms error.
"""
import json
import os

import numpy as np
import pytest

import oracle.triangle_attention as TA
import workloads as wl
from tests.bf16_attention_floor import attention_weights, floor as attn_floor
from tests.gpu_util import mask_to_device, to_f64, z_to_device

pytestmark = pytest.mark.gpu

FLOOR_FACTOR = 1.5
FLOOR_SLACK = 3e-3
ABS_TOL = 0.12


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
    rms_ref = np.sqrt(np.mean(ref ** 2))
    err = float(np.max(np.abs(got - ref)) / rms_ref)
    err_rms = float(np.sqrt(np.mean((got - ref) ** 2)) / rms_ref)
    fl, fl_rms = attn_floor(N, mask, node, 31 + N, rms=True)
    log = os.environ.get("TM_METRICS_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": f"attn_{node}_N{N}_{mask}", "max_rel": err, "floor": fl,
                                "rms_rel": err_rms, "floor_rms": fl_rms}) + "\n")
    assert np.all(np.isfinite(got))
    assert err <= ABS_TOL, (err, fl)
    assert err <= FLOOR_FACTOR * fl + FLOOR_SLACK, (err, fl)
    assert err_rms <= FLOOR_FACTOR * fl_rms + 1e-4, (err_rms, fl_rms)
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
