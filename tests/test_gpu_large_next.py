"""The backward pass and triangle attention at the four-chain complex's size (N = 3605, c = 128, bf16,
full mask), in the launch configuration the benchmark times.

* triangle attention: whole output lines (rows of the starting node, columns of the ending node) against
  the float64 oracle's sampled lines, with the fixed gates of tests/test_gpu_attention.py;
* backward: the gradient is linear in the cotangent and every stored rounding commutes with a factor
  of two, so tm_backward(2 dout) must equal 2 tm_backward(dout) bit for bit, for dz and every parameter;
  all values finite. The same at N = 10000, where the backward runs block-streamed with a workspace
  under 120 GB.
"""
import numpy as np
import pytest

import oracle.triangle_attention as TA
import workloads as wl
from tests.attention_storage_model import attention_weights
from tests.gpu_util import mask_to_device, to_f64, z_to_device
from tests.test_gpu_attention import gate

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N = 3605
LINES = [0, 1800, 3604]


@pytest.fixture(scope="module")
def big():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build, tm
    build.build()
    w = wl.WORKLOADS["complex3605"]
    z_np = wl.make_z(w.N, w.c_z, w.seed_z, "bf16")
    m_np = wl.make_mask(w.N, w.mask)
    return torch, tm, z_np, m_np


@pytest.mark.parametrize("node", TA.NODES)
def test_attention_complex3605_sampled_lines(big, node):
    torch, tm, z_np, m_np = big
    W = attention_weights()
    mod = tm.TriangleAttention(W)
    try:
        z = z_to_device(z_np)
        out = mod(z, mask_to_device(m_np), node)
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
        idx = torch.tensor(LINES, device="cuda")
        got = to_f64(out.index_select(0, idx) if node == "starting" else out.index_select(1, idx).transpose(0, 1))
        del z, out
    finally:
        mod.close()
    bias = TA.pair_bias(z_np if node == "starting" else np.swapaxes(z_np, 0, 1), W)
    ref = TA.sampled(z_np, m_np, W, node, LINES, bias=bias)
    gate(got, ref)


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
def test_backward_complex3605_is_linear_in_the_cotangent(big, direction):
    torch, tm, z_np, m_np = big
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    try:
        z = z_to_device(z_np)
        gen = torch.Generator(device="cuda").manual_seed(7)
        dout = torch.randn(z.shape, device="cuda", generator=gen).to(torch.bfloat16)
        dz1, g1 = mod.backward(z, dout, None, direction)
        dz2, g2 = mod.backward(z, dout * 2, None, direction)
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
        assert torch.isfinite(dz1.float()).all()
        assert torch.equal(dz2, dz1 * 2)
        for k in g1:
            assert torch.isfinite(g1[k]).all(), k
            assert torch.equal(g2[k], g1[k] * 2), k
    finally:
        mod.close()


def test_backward_n10000_block_streamed(big):
    """N = 10000 (10^8 pairs): the automatic schedule streams blocks; its workspace stays under 120 GB.
    2 dout (in place, dz over it) gives 2 dz bit for bit; everything finite, dz not zero."""
    torch, tm, _, _ = big
    N = 10000
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    try:
        gen = torch.Generator(device="cuda").manual_seed(11)
        z = torch.empty((N, N, 128), device="cuda", dtype=torch.bfloat16)
        dout = torch.empty_like(z)
        for t in (z, dout):                            # row slabs: no float32 copy of the whole grid
            for r0 in range(0, N, 500):
                t[r0:r0 + 500] = torch.randn((min(500, N - r0), N, 128), device="cuda", generator=gen)
        torch.cuda.empty_cache()
        dz1, g1 = mod.backward(z, dout, None, "outgoing")
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
        assert tm.tm_workspace_bytes(mod.ctx) < 120e9, tm.tm_workspace_bytes(mod.ctx)
        dout.mul_(2)                                   # exact in bf16
        _, g2 = mod.backward(z, dout, None, "outgoing", dz=dout)
        torch.cuda.synchronize()
        assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
        del z
        nonzero = False
        for r0 in range(0, N, 500):                    # row slabs: no full-size temporaries
            a = dz1[r0:r0 + 500]
            assert torch.isfinite(a.float()).all()
            assert torch.equal(dout[r0:r0 + 500], a * 2), r0
            nonzero = nonzero or bool((a != 0).any())
        assert nonzero
        for k in g1:
            assert torch.isfinite(g1[k]).all(), k
            assert torch.equal(g2[k], g1[k] * 2), k
    finally:
        mod.close()
