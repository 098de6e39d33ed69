"""The residual form of the update and the two-update Pairformer step, through the C ABI.

tm_options.residual = 1 makes the update write out = z + update (the residual connection around the
layer in a Pairformer block); out may be z itself. tm_pair_update runs z <- z + outgoing(z) and then
z <- z + incoming(z) in place. Checked here:
  * the residual result equals the plain result added to z in the output dtype (bf16: one rounding of
    the float sum; float32: the float sum), in place and into a separate buffer;
  * tm_pair_update equals the two residual calls made one after the other, bit for bit;
  * each of its two updates meets the bf16 gates against the float64 oracle run on the GPU's own input
    of that update (so the checks do not compound);
  * the step captured into a CUDA graph and replayed gives the same z as the eager call.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_util import BF16_TOL, mask_to_device, to_f64, z_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build, tm
    build.build()
    W = wl.make_weights(128, 128, 1, ln_random=True)
    mod = tm.TriMul(128, 128, W)
    yield torch, tm, mod, W
    mod.close()


def _bf16_bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
@pytest.mark.parametrize("N,mask", [(129, "scatter"), (300, "last10pct")])
def test_residual_bf16_is_plain_plus_z(env, direction, N, mask):
    torch, tm, mod, _ = env
    z = z_to_device(wl.make_z(N, 128, 81 + N, "bf16"))
    m = mask_to_device(wl.make_mask(N, mask, 82))
    plain = mod(z, m, direction)
    want = (z.float() + plain.float()).to(torch.bfloat16)
    sep = torch.empty_like(z)
    tm.tm_forward_ex(mod.ctx, z, m, direction, sep, residual=True)
    inplace = z.clone()
    tm.tm_forward_ex(mod.ctx, inplace, m, direction, inplace, residual=True)
    torch.cuda.synchronize()
    assert torch.equal(sep, want)
    assert torch.equal(inplace, want)
    assert not torch.equal(inplace, z)


def test_residual_f32_is_plain_plus_z(env):
    torch, tm, _, _ = env
    w = wl.WORKLOADS["tiny48"]
    W = wl.make_weights(w.c_z, w.c_h, w.seed_w)
    mod = tm.TriMul(w.c_z, w.c_h, W)
    z = torch.from_numpy(wl.make_z(w.N, w.c_z, w.seed_z, "f32")).cuda()
    m = mask_to_device(wl.make_mask(w.N, w.mask))
    for d in ("outgoing", "incoming"):
        plain = mod(z, m, d)
        inplace = z.clone()
        tm.tm_forward_ex(mod.ctx, inplace, m, d, inplace, residual=True)
        torch.cuda.synchronize()
        assert torch.equal(inplace, z + plain)
    mod.close()


def test_residual_rejects_partial_overlap(env):
    torch, tm, mod, _ = env
    N = 64
    buf = torch.zeros(2 * N * N * 128, dtype=torch.bfloat16, device="cuda")
    z = buf[: N * N * 128].view(N, N, 128)
    out = buf[128: 128 + N * N * 128].view(N, N, 128)
    with pytest.raises(tm.TmError):
        tm.tm_forward_ex(mod.ctx, z, None, "outgoing", out, residual=True)


def test_pair_update_is_two_residual_updates_and_meets_the_gates(env):
    torch, tm, mod, W = env
    N = 200
    z0 = z_to_device(wl.make_z(N, 128, 91, "bf16"))
    m_np = wl.make_mask(N, "last10pct", 92)
    m = mask_to_device(m_np)
    step = z0.clone()
    tm.tm_pair_update(mod.ctx, step, m)
    z1 = z0.clone()
    tm.tm_forward_ex(mod.ctx, z1, m, "outgoing", z1, residual=True)
    z2 = z1.clone()
    tm.tm_forward_ex(mod.ctx, z2, m, "incoming", z2, residual=True)
    torch.cuda.synchronize()
    assert torch.equal(step, z2)
    # each update against the oracle on the GPU's own input. The stored result is rounded twice, as a
    # bf16 residual add is: the update to bf16, then the sum; half a bf16 step of each is not counted
    # (the excess of the plain update's gate, with the sum's own rounding added)
    for zin, zout, d in ((z0, z1, "outgoing"), (z1, z2, "incoming")):
        zin_np = _bf16_bits(zin)
        ref_upd = oracle.full(zin_np, m_np, W, d, storage="bf16")
        ref = wl.as_f64(zin_np) + ref_upd
        got = to_f64(zout)
        ulp = oracle.half_ulp_bf16(ref) + oracle.half_ulp_bf16(ref_upd)
        rms = np.sqrt(np.mean(ref_upd ** 2))
        excess = np.max(np.maximum(np.abs(got - ref) - ulp, 0.0)) / rms
        assert excess <= BF16_TOL, excess


def test_pair_update_replays_from_a_cuda_graph(env):
    torch, tm, mod, _ = env
    N = 160
    z0 = z_to_device(wl.make_z(N, 128, 101, "bf16"))
    m = mask_to_device(wl.make_mask(N, "scatter", 102))
    eager = z0.clone()
    tm.tm_pair_update(mod.ctx, eager, m)        # also sizes the workspace before the capture
    torch.cuda.synchronize()
    zg = z0.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            tm.tm_pair_update(mod.ctx, zg, m, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    zg.copy_(z0)
    g.replay()
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    assert torch.equal(zg, eager)
    zg.copy_(z0)                                # a second replay from the same start
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(zg, eager)
