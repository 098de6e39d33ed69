"""The allocation-free forward entry point, through the C ABI.

tm_forward_noalloc serves callers that may not allocate device memory (their
device memory belongs to another allocator or to a fixed budget, or they must
not pay an allocation's host-side stall): its scratch is a static array inside
libtm. These checks compare it with tm_forward, the entry point that allocates
its workspace, bit for bit, on two calls in a row with different inputs (the
second call sees the first call's leftovers in the shared array), and check
that it allocates nothing and refuses grids beyond its 128-token limit.

Kept in a file of its own that pytest collects last.
"""
import pytest

import workloads as wl
from tests.gpu_util import mask_to_device, z_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build, tm
    build.build()
    mod = tm.TriMul(128, 128, wl.make_weights(128, 128, 1))
    yield torch, tm, mod
    mod.close()


def test_noalloc_matches_forward_on_two_calls_in_a_row(setup):
    torch, tm, mod = setup
    cases = [(128, "outgoing", "last10pct", 51), (77, "incoming", "scatter", 52)]
    ws_before = tm.tm_workspace_bytes(mod.ctx)
    outs = []
    for N, direction, mask, seed in cases:
        z = z_to_device(wl.make_z(N, 128, seed, "bf16"))
        m = mask_to_device(wl.make_mask(N, mask, seed))
        out = torch.full_like(z, float("nan"))
        tm.tm_forward_noalloc(mod.ctx, z, m, direction, out)
        outs.append((z, m, direction, out))
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    assert tm.tm_workspace_bytes(mod.ctx) == ws_before      # no workspace was allocated for these calls
    for z, m, direction, out in outs:
        ref = tm.tm_forward(mod.ctx, z, m, direction, torch.empty_like(z))
        # the same kernels on the same values (x kept as fp16 with the same exponent): bit for bit,
        # so leftovers of the first call in the shared array would show in the second
        assert torch.equal(out, ref), direction
        assert torch.isfinite(out.float()).all()


def test_noalloc_repeat_is_deterministic(setup):
    torch, tm, mod = setup
    N = 96
    z = z_to_device(wl.make_z(N, 128, 53, "bf16"))
    first = tm.tm_forward_noalloc(mod.ctx, z, None, "outgoing", torch.empty_like(z)).clone()
    second = tm.tm_forward_noalloc(mod.ctx, z, None, "outgoing", torch.empty_like(z))
    assert torch.equal(first, second)


def test_noalloc_rejects_grids_beyond_its_limit(setup):
    torch, tm, mod = setup
    z = z_to_device(wl.make_z(129, 128, 54, "bf16"))
    with pytest.raises(tm.TmError) as e:
        tm.tm_forward_noalloc(mod.ctx, z, None, "outgoing", torch.empty_like(z))
    assert e.value.status == tm.TM_ERR_UNSUPPORTED
    assert "N <= 128" in str(e.value)
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
