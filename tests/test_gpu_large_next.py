"""The backward pass and triangle attention at the four-chain complex's size (N = 3605, c = 128, bf16,
full mask), in the launch configuration the benchmark times.

* triangle attention: whole output lines (rows of the starting node, columns of the ending node) against
  the float64 oracle's sampled lines, with the fixed gates of tests/test_gpu_attention.py;
* backward: the gradient is linear in the cotangent and every stored rounding commutes with a factor
  of two, so tm_backward(2 dout) must equal 2 tm_backward(dout) bit for bit, for dz and every parameter;
  all values finite.
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
