"""The 2D block split of the update over a square mesh (pair_representation_boltz_b300/ring2d.py), on CPU.

The schedule (transpose exchange, Cannon skew, r ring steps) is checked two ways, for both directions:
  * with tagged blocks: every block carries (operand, row block, column block) of its origin, and each
    step's resident pair must be exactly the pair the block product needs, over every k block once;
  * with numbers: each rank's accumulated block product must equal the full per-channel contraction of
    the assembled global operands (float64, up to rounding).
Once with every rank of a 2 x 2 and a 3 x 3 mesh in one process (LocalMeshDriver), and once with four
gloo processes over 127.0.0.1 exchanging the blocks through torch.distributed (DistDriver).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from pair_representation_boltz_b300 import ring2d as R

C = 3           # channels of the numeric check


def _tag_block(kind, i, k):
    return torch.tensor([kind, i, k], dtype=torch.int64)


def _tagged_program(layout, rank, direction, seen):
    p, q = layout.coords(rank)
    a_loc, b_loc = _tag_block(0, p, q), _tag_block(1, p, q)

    def compute(row, col, k):
        seen.append((tuple(row.tolist()), tuple(col.tolist()), k))
    return R.rank_program(layout, rank, direction, a_loc, b_loc, compute, torch.empty_like)


def _check_tags(layout, rank, direction, seen):
    p, q = layout.coords(rank)
    assert sorted(k for _, _, k in seen) == list(range(layout.r)), seen
    for row, col, k in seen:
        if direction == "outgoing":     # x[I_p, J_q] += a[I_p, K_k] b[J_q, K_k]^T
            assert row == (0, p, k) and col == (1, q, k), (rank, row, col, k)
        else:                           # x[I_p, J_q] += a[K_k, I_p]^T b[K_k, J_q]
            assert row == (0, k, p) and col == (1, k, q), (rank, row, col, k)


def _global_operands(layout, seed=3):
    n = layout.padded
    rng = np.random.default_rng(seed)
    return rng.standard_normal((C, n, n)), rng.standard_normal((C, n, n))


def _numeric_program(layout, rank, direction, A, Bm, out):
    p, q = layout.coords(rank)
    I, K = layout.tokens(p), layout.tokens(q)
    a_loc = torch.from_numpy(np.ascontiguousarray(A[:, I.start:I.stop, K.start:K.stop]))
    b_loc = torch.from_numpy(np.ascontiguousarray(Bm[:, I.start:I.stop, K.start:K.stop]))
    x = torch.zeros((C, layout.B, layout.B), dtype=torch.float64)

    def compute(row, col, k):
        if direction == "outgoing":
            x.add_(torch.matmul(row, col.transpose(1, 2)))
        else:
            x.add_(torch.matmul(row.transpose(1, 2), col))
    out[rank] = x
    return R.rank_program(layout, rank, direction, a_loc, b_loc, compute, torch.empty_like)


def _check_numbers(layout, rank, direction, A, Bm, x):
    p, q = layout.coords(rank)
    I, J = layout.tokens(p), layout.tokens(q)
    full = np.matmul(A, np.swapaxes(Bm, 1, 2)) if direction == "outgoing" else np.matmul(np.swapaxes(A, 1, 2), Bm)
    np.testing.assert_allclose(x.numpy(), full[:, I.start:I.stop, J.start:J.stop], rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("direction", ("outgoing", "incoming"))
@pytest.mark.parametrize("world,N", [(1, 5), (4, 10), (9, 20)])
def test_local_mesh_schedule(direction, world, N):
    layout = R.MeshLayout.make(world, N, align=1)
    seen = [[] for _ in range(world)]
    R.LocalMeshDriver().run([_tagged_program(layout, k, direction, seen[k]) for k in range(world)])
    for k in range(world):
        _check_tags(layout, k, direction, seen[k])
    A, Bm = _global_operands(layout)
    out = {}
    R.LocalMeshDriver().run([_numeric_program(layout, k, direction, A, Bm, out) for k in range(world)])
    for k in range(world):
        _check_numbers(layout, k, direction, A, Bm, out[k])


def test_layout_pads_to_a_square_mesh_of_aligned_blocks():
    lay = R.MeshLayout.make(4, 3605)
    assert lay.r == 2 and lay.B % 8 == 0 and lay.padded >= 3605 and lay.B * (lay.r - 1) < 3605
    assert [lay.coords(k) for k in range(4)] == [(0, 0), (0, 1), (1, 0), (1, 1)]
    with pytest.raises(ValueError):
        R.MeshLayout.make(8, 100)           # not a square


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_rank(rank, world, port, result):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        layout = R.MeshLayout.make(world, 14, align=1)
        for direction in ("outgoing", "incoming"):
            seen = []
            R.DistDriver().run(_tagged_program(layout, rank, direction, seen))
            _check_tags(layout, rank, direction, seen)
            A, Bm = _global_operands(layout)
            out = {}
            R.DistDriver().run(_numeric_program(layout, rank, direction, A, Bm, out))
            _check_numbers(layout, rank, direction, A, Bm, out[rank])
        result[rank] = "ok"
    except Exception as e:          # reported by the parent
        result[rank] = repr(e)
    finally:
        dist.destroy_process_group()


def test_four_gloo_ranks_exchange_the_blocks_each_product_needs():
    world, port = 4, _free_port()
    with mp.Manager() as m:
        result = m.dict()
        mp.spawn(_gloo_rank, args=(world, port, result), nprocs=world, join=True)
        assert dict(result) == {k: "ok" for k in range(world)}, dict(result)
