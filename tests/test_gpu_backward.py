"""The backward pass through the C ABI (tm_backward) against the float64 oracle of the gradient.

The metric of each gradient (dz and every parameter) is max|got - ref| / rms(ref) over all of its
values, with ref the oracle's gradient for the same inputs and cotangent. Bounds:
  * float32 path: F32_GRAD_TOL. Its arithmetic is the forward's (max_rel ~2e-6) followed by the
    chain rule in float32 and sums over the N^2 pairs for the parameters; a float32 sum of P terms
    errs by about sqrt(P) u sum|terms| (u = 2^-24) with independent rounding errors, 3e-6 at
    P = 2304, and at most P u = 1.4e-4 in the worst case. Measured: <= 9.1e-6 on every gradient;
    the bound takes five times that;
  * bf16 path: fixed gates against the oracle's gradient of the update as the bf16 path defines it
    (a and b stored as bf16; storage="bf16"), the bf16 tolerance of the update read the same way
    (tests/gpu_util.py): every parameter gradient (float32) within BF16_TOL in max|delta|/rms, dz
    (stored as bf16) within BF16_TOL beyond its own bf16 rounding ("excess"), and every gradient
    within BF16_TOL in rms|delta|/rms. The path's tensor-core operands are fp16;
    tests/backward_storage_model.py applies those roundings to the oracle's chain rule and is logged
    beside the path's error as a diagnostic (it predicts <= 5e-3 for these cases).
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.backward_storage_model import floor as storage_model_error
from tests.gpu_util import BF16_TOL, mask_to_device, to_f64, z_to_device

pytestmark = pytest.mark.gpu

F32_GRAD_TOL = 5e-5


@pytest.fixture(scope="module")
def torch_tm():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build, tm
    build.build()
    return torch, tm


def _metrics(got, ref):
    out = {}
    for k, r in ref.items():
        g = got[k]
        rms = float(np.sqrt(np.mean(r * r))) or 1.0
        out[k] = float(np.max(np.abs(g - r)) / rms)
    return out


def _log(name, metrics):
    log = os.environ.get("TM_METRICS_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": name, **metrics}) + "\n")


def _run(torch, tm, W, c_z, c_h, z_np, m_np, dout_np, direction, dtype):
    mod = tm.TriMul(c_z, c_h, W)
    try:
        z = z_to_device(z_np)
        dout = z_to_device(dout_np)
        m = mask_to_device(m_np) if m_np is not None else None
        dz, grads = mod.backward(z, dout, m, direction)
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
        got = {"z": to_f64(dz)}
        got.update({k: v.double().cpu().numpy() for k, v in grads.items()})
        return got
    finally:
        mod.close()


def _dout(N, c, seed, dtype):
    d = np.random.default_rng(seed).standard_normal((N, N, c)).astype(np.float32)
    return wl.f32_to_bf16_bits(d) if dtype == "bf16" else d


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
def test_backward_f32_tiny48(torch_tm, direction):
    torch, tm = torch_tm
    w = wl.WORKLOADS["tiny48"]
    W = wl.make_weights(w.c_z, w.c_h, w.seed_w, ln_random=True)
    z = wl.make_z(w.N, w.c_z, w.seed_z, "f32")
    m = wl.make_mask(w.N, w.mask)
    dout = _dout(w.N, w.c_z, 5, "f32")
    got = _run(torch, tm, W, w.c_z, w.c_h, z, m, dout, direction, "f32")
    ref = oracle.full_backward(wl.as_f64(z), m, W, direction, dout.astype(np.float64))
    met = _metrics(got, ref)
    _log(f"f32_tiny48_{direction}", met)
    assert max(met.values()) <= F32_GRAD_TOL, met


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
def test_backward_f32_c128_ragged(torch_tm, direction):
    torch, tm = torch_tm
    N = 37
    W = wl.make_weights(128, 128, 3, ln_random=True)
    z = wl.make_z(N, 128, 7, "f32")
    m = wl.make_mask(N, "scatter", 8)
    dout = _dout(N, 128, 9, "f32")
    got = _run(torch, tm, W, 128, 128, z, m, dout, direction, "f32")
    ref = oracle.full_backward(wl.as_f64(z), m, W, direction, dout.astype(np.float64))
    met = _metrics(got, ref)
    _log(f"f32_c128_N37_{direction}", met)
    assert max(met.values()) <= F32_GRAD_TOL, met


def test_backward_in_place_and_without_parameter_gradients(torch_tm):
    torch, tm = torch_tm
    N, c = 20, 12
    W = wl.make_weights(c, 9, 4, ln_random=True)
    mod = tm.TriMul(c, 9, W)
    try:
        z = z_to_device(wl.make_z(N, c, 1, "f32"))
        dout = z_to_device(_dout(N, c, 2, "f32"))
        dz, _ = mod.backward(z, dout, None, "incoming")
        inplace = dout.clone()
        tm.tm_backward(mod.ctx, z, None, "incoming", inplace, inplace, None)
        torch.cuda.synchronize()
        assert torch.equal(inplace, dz)
        with pytest.raises(tm.TmError):
            tm.tm_backward(mod.ctx, z, None, "incoming", dout, z, None)      # dz over z
    finally:
        mod.close()


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
@pytest.mark.parametrize("N,mask", [(64, "scatter"), (129, "last10pct"), (200, "scatter")])
def test_backward_bf16(torch_tm, direction, N, mask):
    """Tiles of 128 pairs across row ends, a ragged last tile, masked tokens, random LayerNorm affines."""
    torch, tm = torch_tm
    W = wl.make_weights(128, 128, 1, ln_random=True)
    z = wl.make_z(N, 128, 11 + N, "bf16")
    m = wl.make_mask(N, mask, 12)
    dout = _dout(N, 128, 13 + N, "bf16")
    got = _run(torch, tm, W, 128, 128, z, m, dout, direction, "bf16")
    ref = oracle.full_backward(wl.as_f64(z), m, W, direction, wl.as_f64(dout), storage="bf16")
    met = bf16_gate(got, ref)
    fl = storage_model_error(N, mask, direction, 11 + N, 13 + N)
    _log(f"bf16_N{N}_{mask}_{direction}", {**met, **{"model_" + k: v for k, v in fl.items()}})


def bf16_gate(got, ref):
    """The bf16 backward's gates; returns the metrics (per gradient: excess for dz, max_rel for the
    float32 parameter gradients, and rms_rel)."""
    met = {}
    for k, r in ref.items():
        assert np.all(np.isfinite(got[k])), k
        e = oracle.errors(got[k], r, "bf16" if k == "z" else None)
        met[k] = e["excess"]
        met[k + "_rms"] = e["rms_rel"]
        assert e["excess"] <= BF16_TOL, (k, e)
        assert e["rms_rel"] <= BF16_TOL, (k, e)
    return met


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
def test_backward_bf16_block_streamed(torch_tm, direction):
    """The block-streamed schedule (blocks of 128 over N = 300: three block rows, the last 44 wide):
    dz bit for bit the whole-grid schedule's (the same per-pair arithmetic, the same order over k in
    every contraction), the parameter gradients within float32 reordering of their sums over pairs
    (the CTAs' shares of the pairs differ), and the oracle's gates."""
    torch, tm = torch_tm
    N = 300
    W = wl.make_weights(128, 128, 3, ln_random=True)
    z_np = wl.make_z(N, 128, 21, "bf16")
    m_np = wl.make_mask(N, "scatter", 22)
    dout_np = _dout(N, 128, 23, "bf16")
    mod = tm.TriMul(128, 128, W)
    try:
        z = z_to_device(z_np)
        dout = z_to_device(dout_np)
        m = mask_to_device(m_np)
        dz_w, g_w = mod.backward(z, dout, m, direction)
        dz_b, g_b = mod.backward(z, dout, m, direction, block=128)
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
        assert torch.equal(dz_b, dz_w)
        for k in g_w:
            d = (g_b[k] - g_w[k]).abs().max().item()
            assert d <= 1e-5 * g_w[k].abs().max().item(), (k, d)
        got = {"z": to_f64(dz_b)}
        got.update({k: v.double().cpu().numpy() for k, v in g_b.items()})
    finally:
        mod.close()
    ref = oracle.full_backward(wl.as_f64(z_np), m_np, W, direction, wl.as_f64(dout_np), storage="bf16")
    met = bf16_gate(got, ref)
    _log(f"bf16_N{N}_block128_{direction}", met)


def test_backward_block_edge_is_checked(torch_tm):
    """A block edge below 128 or off the 8-element grid is refused before any launch."""
    torch, tm = torch_tm
    N = 300
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    try:
        z = z_to_device(wl.make_z(N, 128, 1, "bf16"))
        dout = z_to_device(_dout(N, 128, 2, "bf16"))
        dz = torch.empty_like(z)
        launches = tm.tm_launch_count(mod.ctx)
        for bad in (64, 100):
            with pytest.raises(tm.TmError) as err:
                tm.tm_backward(mod.ctx, z, None, "outgoing", dout, dz, None, block=bad)
            assert err.value.status == tm.TM_ERR_INVALID
        assert tm.tm_launch_count(mod.ctx) == launches
    finally:
        mod.close()


def test_backward_bf16_is_deterministic_and_in_place(torch_tm):
    torch, tm = torch_tm
    N = 150
    W = wl.make_weights(128, 128, 2, ln_random=True)
    mod = tm.TriMul(128, 128, W)
    try:
        z = z_to_device(wl.make_z(N, 128, 3, "bf16"))
        dout = z_to_device(_dout(N, 128, 4, "bf16"))
        dz1, g1 = mod.backward(z, dout, None, "outgoing")
        dz2, g2 = mod.backward(z, dout, None, "outgoing")
        inplace = dout.clone()
        tm.tm_backward(mod.ctx, z, None, "outgoing", inplace, inplace, None)
        torch.cuda.synchronize()
        assert torch.equal(dz1, dz2) and torch.equal(inplace, dz1)
        for k in g1:
            assert torch.equal(g1[k], g2[k]), k
    finally:
        mod.close()


def test_backward_refuses_a_workspace_over_the_limit(torch_tm):
    """Beyond tm_options.workspace_limit the backward returns TM_ERR_OOM before any launch, and the ctx
    keeps working."""
    torch, tm = torch_tm
    N = 200
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    try:
        z = z_to_device(wl.make_z(N, 128, 1, "bf16"))
        dout = z_to_device(_dout(N, 128, 2, "bf16"))
        dz = torch.empty_like(z)
        launches = tm.tm_launch_count(mod.ctx)
        with pytest.raises(tm.TmError) as err:
            tm.tm_backward(mod.ctx, z, None, "outgoing", dout, dz, None, workspace_limit=1 << 20)
        assert err.value.status == tm.TM_ERR_OOM
        assert tm.tm_launch_count(mod.ctx) == launches
        tm.tm_backward(mod.ctx, z, None, "outgoing", dout, dz, None)
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    finally:
        mod.close()
