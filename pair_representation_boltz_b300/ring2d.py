"""2D block split of the triangle multiplicative update over a square mesh of ranks.

The pages shard the N x N pair representation into a grid of blocks, one per GPU, so that each device
holds O(N^2 / P) of it ("2D tiling da pair representation" on the BioNeMo page "NVIDIA BioNeMo escala
modelagem biomolecular com context parallelism e quebra barreira de memória da GPU"), on a square mesh
whose rows and columns are rings along which blocks circulate while each device computes its local
update ("Sobreposição de computação e comunicação"; the code-sample section builds the mesh with
cp = (sqrt(P), sqrt(P))). They give no schedule; this module is one, written for the update's
contraction:

Layout. P = r * r ranks; rank p * r + q holds the block (p, q): tokens I_p x J_q, where the token axis
is cut into r blocks of B tokens each (N padded up to r * B with masked tokens, which contribute
nothing). The same cut indexes the contraction's k.

Contraction of output block (p, q), per channel:
    outgoing  x[I_p, J_q] = sum_t a[I_p, K_t] b[J_q, K_t]^T
    incoming  x[I_p, J_q] = sum_t a[K_t, I_p]^T b[K_t, J_q]
Each rank projects its own z block into a_loc = a[I_p, K_q] and b_loc = b[I_p, K_q]. Call R(p, t) the
row-side operand of k-block t for mesh row p and C(t, q) the column-side one for mesh column q:
outgoing R(p, t) = a[I_p, K_t] (rank (p, t)'s own a) and C(t, q) = b[J_q, K_t] (rank (q, t)'s b);
incoming R(p, t) = a[K_t, I_p] (rank (t, p)'s a) and C(t, q) = b[K_t, J_q] (rank (t, q)'s b). One
transpose exchange -- of b for outgoing, of a for incoming, between ranks (p, q) and (q, p) -- puts
R(p, t) on rank (p, t) and C(t, q) on rank (t, q); the block product over the mesh is then
x(p, q) = sum_t R(p, t) C(t, q), which Cannon's algorithm streams with one block of each operand
resident per rank: a skew (row p shifted left by p, column q up by q) gives rank (p, q) the pair of
k-block (p + q) mod r, and each of r steps contracts the resident pair while the next pair arrives
over the row ring (R, from the right neighbour) and the column ring (C, from the one below).

The schedule is a generator per rank that yields its point-to-point exchanges; a driver carries them
out. DistDriver uses torch.distributed (NCCL on GPUs, gloo on CPUs) with one process per rank;
LocalMeshDriver runs every rank of a mesh in one process, in lockstep, moving the blocks itself (the
ranks' work is then serial). `forward_2d` runs the whole update of one rank's block through libtm.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class MeshLayout:
    """A square mesh of r x r ranks over a grid of N tokens cut into r blocks of B tokens."""
    r: int
    N: int
    B: int

    @staticmethod
    def make(world_size: int, N: int, align: int = 8) -> "MeshLayout":
        r = math.isqrt(world_size)
        if r * r != world_size:
            raise ValueError(f"the mesh must be square: world size {world_size} is not a square")
        if N < 1:
            raise ValueError("N must be positive")
        B = -(-N // r)
        B = -(-B // align) * align          # block origins on the 16-byte grid of the kernels' copies
        return MeshLayout(r, N, B)

    @property
    def world(self) -> int:
        return self.r * self.r

    @property
    def padded(self) -> int:
        return self.r * self.B

    def coords(self, rank: int) -> tuple[int, int]:
        return divmod(rank, self.r)

    def rank_of(self, p: int, q: int) -> int:
        return (p % self.r) * self.r + (q % self.r)

    def tokens(self, t: int) -> range:
        """The padded token indices of block t."""
        return range(t * self.B, (t + 1) * self.B)


@dataclass
class Start:
    """Post point-to-point transfers: sends [(dst rank, tensor)], receives [(src rank, buffer)]. The
    tensors of both lists must not be touched until the matching Wait."""
    sends: list
    recvs: list


@dataclass
class Wait:
    """Complete the transfers of the last Start."""


def _exchange(send_to, recv_from, tensor, buffer):
    """A Start + Wait pair that sends `tensor` and receives into `buffer`. Every rank issues the same
    sequence of requests (a rank may send to itself: the drivers copy such blocks locally)."""
    yield Start([(send_to, tensor)], [(recv_from, buffer)])
    yield Wait()


def rank_program(layout: MeshLayout, rank: int, direction: str, a_loc, b_loc, compute, new_like):
    """The schedule of one rank (a generator of Start / Wait requests).

    a_loc, b_loc: this rank's projected blocks. compute(row, col, t) contracts one resident pair of
    k-block t into the rank's output block. new_like(t) returns an empty buffer shaped like t.
    """
    if direction not in ("outgoing", "incoming"):
        raise ValueError(f"unknown direction {direction!r}")
    r = layout.r
    p, q = layout.coords(rank)
    mirror = layout.rank_of(q, p)
    # transpose exchange: outgoing's column operand is the mirror rank's b, incoming's row operand the
    # mirror rank's a
    if direction == "outgoing":
        row = a_loc
        col = new_like(b_loc)
        yield from _exchange(mirror, mirror, b_loc, col)
    else:
        col = b_loc
        row = new_like(a_loc)
        yield from _exchange(mirror, mirror, a_loc, row)
    # skew: rank (p, q) takes R(p, q + p) and C(p + q, q)
    row2, col2 = new_like(row), new_like(col)
    yield Start([(layout.rank_of(p, q - p), row), (layout.rank_of(p - q, q), col)],
                [(layout.rank_of(p, q + p), row2), (layout.rank_of(p + q, q), col2)])
    yield Wait()
    row, col = row2, col2
    # r steps: contract the resident pair while the next one moves along the row and column rings
    nrow, ncol = new_like(row), new_like(col)
    for s in range(r):
        k = (p + q + s) % r
        last = s == r - 1
        if not last:
            yield Start([(layout.rank_of(p, q - 1), row), (layout.rank_of(p - 1, q), col)],
                        [(layout.rank_of(p, q + 1), nrow), (layout.rank_of(p + 1, q), ncol)])
        compute(row, col, k)
        if not last:
            yield Wait()
            row, nrow = nrow, row
            col, ncol = ncol, col


class DistDriver:
    """Carries out one rank's requests with torch.distributed point-to-point calls (one process per
    rank; the default process group must be initialised)."""

    def __init__(self, group=None):
        self.group = group
        self.pending = []

    def run(self, program) -> None:
        import torch.distributed as dist
        me = dist.get_rank(self.group)
        for req in program:
            if isinstance(req, Start):
                # blocks a rank sends to itself are copied here, in order; the rest go point to point
                own = [t for peer, t in req.sends if peer == me]
                for peer, buf in req.recvs:
                    if peer == me:
                        buf.copy_(own.pop(0))
                ops = [dist.P2POp(dist.isend, t, peer, self.group) for peer, t in req.sends if peer != me]
                ops += [dist.P2POp(dist.irecv, t, peer, self.group) for peer, t in req.recvs if peer != me]
                self.pending = dist.batch_isend_irecv(ops) if ops else []
            elif isinstance(req, Wait):
                for w in self.pending:
                    w.wait()
                self.pending = []
            else:
                raise TypeError(f"unknown request {req!r}")


class LocalMeshDriver:
    """Runs the programs of all ranks of a mesh in one process, in lockstep: every rank must issue the
    same kind of request at the same time (the schedule is SPMD); a Start moves every rank's blocks to
    their receivers at once."""

    def run(self, programs: list) -> None:
        live = list(programs)
        reqs = [next(g, None) for g in live]
        while any(r is not None for r in reqs):
            kinds = {type(r) for r in reqs}
            if len(kinds) != 1 or None in reqs:
                raise RuntimeError("the ranks' schedules diverged")
            if isinstance(reqs[0], Start):
                inbox = {}
                for src, req in enumerate(reqs):
                    for dst, t in req.sends:
                        inbox.setdefault((src, dst), []).append(t)
                for dst, req in enumerate(reqs):
                    for src, buf in req.recvs:
                        buf.copy_(inbox[(src, dst)].pop(0))
            reqs = [next(g, None) for g in live]


def forward_2d(ctx, layout: MeshLayout, rank: int, z_blk, mask_rows, mask_cols, direction: str, out_blk,
               stream=None):
    """The update of one rank's output block (GPU, through libtm): returns the rank's program, to be run
    by a driver together with the other ranks'.

    z_blk: bf16 [B][B][128], this rank's block of the (padded) pair representation; mask_rows /
    mask_cols: float32 [B] token masks of its row and column blocks (padding tokens 0); out_blk: bf16
    [B][B][128]. a and b are projected from the local block, the contraction accumulates the r k-block
    products into a float32 x block (the first product writes it, the others add into it with TMA
    reduce-adds), and the finish kernel reads x and the local z.
    """
    import torch

    from . import tm
    B = layout.B
    ld = -(-B // 64) * 64
    dev = z_blk.device
    a = torch.empty((128, B, ld), dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    zstat = torch.empty((B, B, 2), dtype=torch.float32, device=dev)
    ldx = -(-B // 32) * 32
    x = torch.empty((128, B, ldx), dtype=torch.float32, device=dev)
    tm.tm_project_block(ctx, z_blk, mask_rows, mask_cols, a, b, ld, zstat, stream)
    done = [0]

    def compute(row, col, k):
        tm.tm_contract_block(ctx, row, col, B, ld, direction, x, ldx, accumulate=done[0] > 0, stream=stream)
        done[0] += 1

    def program():
        yield from rank_program(layout, rank, direction, a, b, compute, torch.empty_like)
        tm.tm_finish_ex(ctx, x, ldx, z_blk, 0, 0, B, B, out_blk, "fp32", zstat, stream)

    return program()
