"""The 2D block split of the update (pair_representation_boltz_b300/ring2d.py) on one GPU: every rank of a
2 x 2 and of a 3 x 3 mesh runs in this process (LocalMeshDriver moves the blocks between them), each
through libtm's block kernels (tm_project_block with its row and column masks, tm_contract_block adding
the k-block products into float32 x, tm_finish_ex). The assembled output must meet the bf16 gates of the
whole-grid update against the float64 oracle; padding tokens are masked and dropped.
"""
import numpy as np
import pytest

import workloads as wl
from pair_representation_boltz_b300 import ring2d as R
from tests.gpu_util import check_bf16, to_f64

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


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
@pytest.mark.parametrize("world,N,mask", [(4, 200, "scatter"), (9, 150, "last10pct")])
def test_split_update_meets_the_gates(env, direction, world, N, mask):
    torch, tm, mod, W = env
    layout = R.MeshLayout.make(world, N)
    z_np = wl.make_z(N, 128, 71 + N, "bf16")
    m_np = wl.make_mask(N, mask, 72)
    n = layout.padded
    zp = np.zeros((n, n, 128), np.uint16)
    zp[:N, :N] = z_np
    mp_ = np.zeros(n, np.float32)
    mp_[:N] = m_np
    z = torch.from_numpy(zp.view(np.int16)).view(torch.bfloat16).cuda()
    m = torch.from_numpy(mp_).cuda()
    outs, programs = {}, []
    for rank in range(world):
        p, q = layout.coords(rank)
        I, J = layout.tokens(p), layout.tokens(q)
        zb = z[I.start:I.stop, J.start:J.stop].contiguous()
        outs[rank] = torch.full_like(zb, float("nan"))
        programs.append(R.forward_2d(mod.ctx, layout, rank, zb, m[I.start:I.stop].contiguous(),
                                     m[J.start:J.stop].contiguous(), direction, outs[rank]))
    R.LocalMeshDriver().run(programs)
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    full = torch.empty_like(z)
    for rank in range(world):
        p, q = layout.coords(rank)
        I, J = layout.tokens(p), layout.tokens(q)
        full[I.start:I.stop, J.start:J.stop] = outs[rank]
    got = to_f64(full[:N, :N])
    check_bf16(got, z_np, m_np, W, direction)


def test_accumulating_contraction_adds_into_x(env):
    """tm_contract_block with accumulate = 1 adds the product to what x holds."""
    torch, tm, mod, W = env
    B = 72
    ld = 128
    gen = torch.Generator(device="cuda").manual_seed(3)
    a = torch.randn((128, B, ld), device="cuda", generator=gen).to(torch.bfloat16)
    b = torch.randn((128, B, ld), device="cuda", generator=gen).to(torch.bfloat16)
    ldx = 96
    x = torch.empty((128, B, ldx), device="cuda")
    tm.tm_contract_block(mod.ctx, a, b, B, ld, "outgoing", x, ldx, accumulate=False)
    once = x.clone()
    tm.tm_contract_block(mod.ctx, a, b, B, ld, "outgoing", x, ldx, accumulate=True)
    torch.cuda.synchronize()
    ref = torch.matmul(a[:, :, :B].double(), b[:, :, :B].double().transpose(1, 2))
    assert torch.allclose(once[:, :, :B].double(), ref, rtol=1e-5, atol=1e-3)
    assert torch.equal(x[:, :, :B], once[:, :, :B] * 2)
