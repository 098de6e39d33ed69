"""tm_forward_host: the update on host buffers, with its copies overlapped (z in on one copy stream, out
back in strips of 512 rows on another, the next call's copy in beside the last call's copy back).

The device part runs the same kernels on the same values as tm_forward, strip by strip (the contraction's
arithmetic for an output element does not depend on the block it is computed in), so the host result
must equal tm_forward's bit for bit -- for one strip and several, back-to-back calls, and a chain in which
one call's output buffer is the next call's input.
"""
import numpy as np
import pytest

import workloads as wl
from tests.gpu_util import mask_to_device, z_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build, tm
    build.build()
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    yield torch, tm, mod
    mod.close()


def _host(torch, z_np):
    return torch.from_numpy(np.ascontiguousarray(z_np).view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("N,mask", [(77, "scatter"), (600, "last10pct"), (1100, "full")])
def test_host_buffers_give_the_device_result(env, N, mask):
    torch, tm, mod = env
    z_np = wl.make_z(N, 128, 81 + N, "bf16")
    m_np = wl.make_mask(N, mask, 82)
    zh = _host(torch, z_np)
    mh = torch.from_numpy(m_np).pin_memory()
    outs = {d: torch.empty_like(zh).pin_memory() for d in ("outgoing", "incoming")}
    for d in ("outgoing", "incoming"):          # back to back: the second copy in beside the first copy back
        tm.tm_forward_host(mod.ctx, zh, mh, d, outs[d])
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    z, m = z_to_device(z_np), mask_to_device(m_np)
    for d in ("outgoing", "incoming"):
        ref = mod(z, m, d).cpu()
        assert torch.equal(outs[d], ref), d


def test_host_chain_reads_the_previous_output(env):
    """out_host of one call as z_host of the next: the second copy in waits for the first copy back."""
    torch, tm, mod = env
    N = 700
    z_np = wl.make_z(N, 128, 91, "bf16")
    zh = _host(torch, z_np)
    mid = torch.empty_like(zh).pin_memory()
    out = torch.empty_like(zh).pin_memory()
    tm.tm_forward_host(mod.ctx, zh, None, "outgoing", mid)
    tm.tm_forward_host(mod.ctx, mid, None, "incoming", out)
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    first = mod(z_to_device(z_np), None, "outgoing")
    ref = mod(first, None, "incoming").cpu()
    assert torch.equal(mid, first.cpu())
    assert torch.equal(out, ref)
