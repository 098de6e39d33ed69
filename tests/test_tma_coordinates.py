"""Host-side check of the TMA box coordinates the kernels issue (no GPU needed).

A tiled TMA copy must start at an inner-axis coordinate whose byte offset is a
multiple of 16 (8 elements for bf16/fp16, 4 for fp32). This test replays the
coordinate arithmetic of the projection, contraction and finish kernels for
every workload and block schedule the tests and the benchmark use, including
unaligned block origins, and asserts that rule for each box; the same for the
triangle-attention kernel's copies (with the bytes each barrier expects), and
the alignment and bounds of the backward kernels' L2 prefetch ranges.
"""
import itertools

import pytest

BM, BN, BK = 256, 256, 64          # contraction tile of a CTA pair: each CTA stages 128 rows of A and of B
HM, HN = BM // 2, BN // 2
PROJ_J = 128                       # projection tile (pairs)
FIN_J = 128                        # finish tile (pairs)


def contraction_boxes(N, i0, j0, bi, bj, incoming):
    """Yield (tensor, inner coordinate, element bytes) for every box of one contraction launch."""
    i_base, j_base = i0 & ~7, j0 & ~7
    tiles_i = (i0 + bi - i_base + BM - 1) // BM
    tiles_j = (j0 + bj - j_base + BN - 1) // BN
    kb_n = (N + BK - 1) // BK
    for ti in range(tiles_i):
        for tj in range(tiles_j):
            rest = j0 + bj - j_base - (tiles_j - 1) * BN
            ntile = (rest + 15) // 16 * 16 if tj == tiles_j - 1 else BN
            for rank in (0, 1):
                ia, jb = i_base + ti * BM + rank * HM, j_base + tj * BN + rank * (ntile // 2)
                for kb in range(kb_n):
                    if not incoming:
                        yield ("a", kb * BK, 2)
                        yield ("b", kb * BK, 2)
                    else:
                        for h in range(HM // 64):
                            yield ("a", ia + 64 * h, 2)
                        for h in range(HN // 64):
                            yield ("b", jb + 64 * h, 2)


def contraction_store_boxes(N, i0, j0, bi, bj):
    """TMA stores of x (float32) when the block origin is on the 8-element grid; else direct stores."""
    if i0 % 8 or j0 % 8:
        return
    tiles_i = (bi + BM - 1) // BM
    tiles_j = (bj + BN - 1) // BN
    for ti in range(tiles_i):
        for tj in range(tiles_j):
            for rank in (0, 1):
                for q in range(4):
                    for ch in range(BN // 32):
                        row0, col0 = ti * BM + rank * HM + 32 * q, tj * BN + 32 * ch
                        if row0 < bi and col0 < bj:
                            yield ("x-store", col0, 4, row0)
                    for ch in range(BN // 64):        # fp16 x: 64-column boxes
                        row0, col0 = ti * BM + rank * HM + 32 * q, tj * BN + 64 * ch
                        if row0 < bi and col0 < bj:
                            yield ("x16-store", col0, 2, row0)


def projection_boxes(N):
    for kc in (0, 1):
        yield ("z", kc * 64, 2)
    for kc in (0, 1):
        yield ("w", kc * 64, 2)
    # stores of a / b: 64 pairs x 32 channels per box, two pair-boxes x four channel quadrants per tile
    tiles_per_row = (N + PROJ_J - 1) // PROJ_J
    for jt in range(tiles_per_row):
        for pb in range(0, PROJ_J, 64):
            x = jt * PROJ_J + pb
            if x < N:
                yield ("ab-store", x, 2)


def finish_boxes(N, i0, j0, bi, bj):
    for jt in range((bj + FIN_J - 1) // FIN_J):
        yield ("x", jt * FIN_J, 4)
        yield ("x16", jt * FIN_J, 2)          # fp16 x: two 64-pair boxes per tile
        yield ("x16", jt * FIN_J + 64, 2)
        # out: one 32-pair x 64-channel store per epilogue warp, on a map based at the block origin
        for q in range(4):
            if jt * FIN_J + 32 * q < bj:
                for h in (0, 1):
                    yield ("out-store", 64 * h, 2)
    for kc in (0, 1):
        yield ("z", kc * 64, 2)
        yield ("w_o", kc * 64, 2)
        yield ("w_g", kc * 64, 2)


def schedule(N, B):
    for i0 in range(0, N, B):
        for j0 in range(0, N, B):
            yield i0, j0, min(B, N - i0), min(B, N - j0)


CASES = [(1, 1), (7, 7), (129, 129), (300, 300), (300, 128), (300, 100), (300, 257), (768, 768),
         (3605, 3605), (6500, 6500), (10000, 2500), (10000, 2504), (45, 16)]


@pytest.mark.parametrize("N,B", CASES)
def test_inner_coordinates_are_16_byte_aligned(N, B):
    for incoming in (False, True):
        for (i0, j0, bi, bj) in schedule(N, B):
            if N > 3000 and (i0, j0) != (0, 0) and (i0, j0) != (B, B):
                continue                      # the arithmetic is the same for every interior block
            for name, x, esz in itertools.chain(contraction_boxes(N, i0, j0, bi, bj, incoming),
                                                finish_boxes(N, i0, j0, bi, bj)):
                assert x >= 0 and (x * esz) % 16 == 0, (N, B, incoming, (i0, j0), name, x)
    for name, x, esz in projection_boxes(N):
        assert (x * esz) % 16 == 0
    for (i0, j0, bi, bj) in list(schedule(N, B))[:2]:
        for name, x, esz, y in contraction_store_boxes(N, i0, j0, bi, bj):
            # a store box starts at a non-negative, 16-byte-aligned coordinate inside the block
            assert x >= 0 and y >= 0 and (x * esz) % 16 == 0 and x < bj and y < bi


def test_unaligned_block_origins_are_covered():
    """Block origins that are not multiples of 8 still yield aligned boxes, and the tiles cover the block."""
    for (N, i0, j0, bi, bj) in [(129, 3, 43, 121, 85), (300, 100, 257, 200, 43), (50, 1, 2, 49, 48)]:
        for name, x, esz in contraction_boxes(N, i0, j0, bi, bj, incoming=True):
            assert (x * esz) % 16 == 0
        i_base, j_base = i0 & ~7, j0 & ~7
        tiles_i = (i0 + bi - i_base + BM - 1) // BM
        tiles_j = (j0 + bj - j_base + BN - 1) // BN
        assert i_base + tiles_i * BM >= i0 + bi and j_base + tiles_j * BN >= j0 + bj
        assert 0 <= i0 - i_base < 8 and 0 <= j0 - j_base < 8


# --------------------------------------------------------------------------- triangle attention

def _box(name):
    """A Box constant {d0, d1, d2, esz} from the kernels' header, so the replay uses the real shapes."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "pair_representation_boltz_b300", "csrc",
                            "tm_kernels.h")).read()
    m = re.search(r"constexpr Box " + name + r"\{(\d+), (\d+), (\d+), (\d+)\}", hdr)
    assert m, name
    return tuple(int(g) for g in m.groups())


def attention_boxes(N, i, jp):
    """Yield (tensor, barrier, iteration, (x, y, z) start, box) for every copy of one attention CTA (row i,
    query tiles 2 jp and 2 jp + 1), in the order the kernel issues them: Q of both tiles at the first block
    of each head pair on q_full; per iteration t (head t // kblocks, key block t % kblocks of 64 keys) K,
    the bias tiles of both query tiles and v on the stage's barrier."""
    q, kbox, vb, bb = _box("kBoxTaQK"), _box("kBoxTaK"), _box("kBoxTaV"), _box("kBoxTaBias")
    kblocks = (N + 63) // 64
    for t in range(4 * kblocks):
        h, kb = divmod(t, kblocks)
        if kb == 0 and h % 2 == 0:
            for g in range(2):
                yield ("q", "q", h, (64 * (h // 2), (2 * jp + g) * 128, i), q)
        yield ("k", "kv", t, (64 * (h // 2), kb * 64, i), kbox)
        for g in range(2):
            yield ("bias", "kv", t, (kb * 64, (2 * jp + g) * 128, h), bb)
        yield ("v", "kv", t, (kb * 64, 32 * h, i), vb)


@pytest.mark.parametrize("N", [1, 7, 64, 127, 128, 129, 200, 300, 768, 1025, 3605])
def test_attention_boxes(N):
    """Every attention copy starts at a non-negative, 16-byte-aligned inner coordinate, and the bytes each
    barrier expects per phase equal the boxes it receives (a load past the grid still moves a whole,
    zero-filled box): 2 Q boxes per head pair; per block of 64 keys K, two bias boxes and one v box."""
    kq, kk, kb_, kv = 64 * 128 * 2, 64 * 64 * 2, 64 * 128 * 2, 64 * 32 * 2     # kQBytes, kKBytes, kBBytes, kVBytes
    expect_q = 2 * kq
    expect_kv = kk + 2 * kb_ + kv                                              # kStageBytes
    jpairs = ((N + 127) // 128 + 1) // 2
    rows = sorted({0, N // 2, N - 1})
    for i in rows:
        for jp in sorted({0, jpairs - 1}):
            got = {"q": {}, "kv": {}}
            for name, bar, t, (x, y, z), (d0, d1, d2, esz) in attention_boxes(N, i, jp):
                assert x >= 0 and y >= 0 and z >= 0 and (x * esz) % 16 == 0, (N, name, x)
                got[bar][t] = got[bar].get(t, 0) + d0 * d1 * d2 * esz
            kblocks = (N + 63) // 64
            assert got["q"] == {0: expect_q, 2: expect_q}, (N, got["q"])
            assert got["kv"] == {t: expect_kv for t in range(4 * kblocks)}, N


# --------------------------------------------------------------------------- backward L2 prefetch ranges

def _up(v, a):
    return (v + a - 1) // a * a


def _prefetch(base, b0, b1, alloc):
    a0, a1 = b0 & ~15, (b1 + 15) & ~15
    if a1 > a0:
        assert (base + a0) % 16 == 0 and base + a0 >= 0 and base + a1 <= alloc, (base, a0, a1, alloc)


def _backward_blocks(N, B):
    """The block edge the backward uses (B >= N: the whole grid) and its block rows."""
    B = min(B, N)
    return B, [(r0, min(B, N - r0)) for r0 in range(0, N, B)]


@pytest.mark.parametrize("N,B", [(128, 128), (129, 129), (200, 200), (255, 255), (256, 256), (257, 257),
                                 (511, 511), (768, 768), (1023, 1023), (1025, 1025), (3605, 3605),
                                 (300, 128), (1025, 256), (3605, 1536)])
def test_backward_prefetch_ranges_stay_aligned_and_inside(N, B):
    """The per-pair backward kernels prefetch into L2, for the next tile of 128 pairs: the output stage
    (over a block bi x bj of x [128][bi][ldxB]) row segments of each channel of x and, for whole grid
    rows, the tile's span of z, dout and the LayerNorm statistics; the projection stage (over the pairs
    of rb whole rows, dV [128][rb][ldx], the row block's dzh pair-major [rb N][128]) row segments of dV,
    the tile's dzh rows, z and the statistics. Every widened range must start on 16 bytes and end inside
    its allocation."""
    P = N * N
    B, rows = _backward_blocks(N, B)
    ldxN, ldxB = _up(N, 32), _up(B, 32)
    xalloc = _up(128 * B * (ldxN if len(rows) == 1 else ldxB) * 4, 256)
    valloc = _up(128 * B * ldxN * 4, 256)
    hb, zst, zb = _up(128 * B * N * 4, 256), _up(P * 8, 256), P * 256
    ldx = ldxN if len(rows) == 1 else ldxB
    # output stage, one block
    for (i0, bi) in rows[:2] + rows[-1:]:
        for (j0, bj) in rows[:1] + rows[-1:]:
            PB = bi * bj
            tiles = (PB + 127) // 128
            if bj < 128:
                continue
            for tn in sorted(set(range(0, tiles, max(1, tiles // 61))) | {tiles - 1}):
                q0, q1 = tn * 128, min(tn * 128 + 128, PB)
                il, jl = divmod(q0, bj)
                n1 = min(q1 - q0, bj - jl)
                for c in (0, 1, 127):
                    base = c * bi * ldx * 4
                    _prefetch(base + il * ldx * 4, 4 * jl, 4 * (jl + n1), xalloc)
                    if q0 + n1 < q1:
                        assert il + 1 < bi
                        _prefetch(base + (il + 1) * ldx * 4, 0, 4 * (q1 - q0 - n1), xalloc)
                if bj == N:
                    g0, g1 = i0 * N + q0, i0 * N + q1
                    _prefetch(0, g0 * 256, g1 * 256, zb)
                    _prefetch(0, g0 * 8, g1 * 8, zst)
    # projection stage, one block row
    for (r0, rb) in rows[:2] + rows[-1:]:
        Pr = rb * N
        tiles = (Pr + 127) // 128
        for tn in sorted(set(range(0, tiles, max(1, tiles // 61))) | {tiles - 1}):
            q0, q1 = tn * 128, min(tn * 128 + 128, Pr)
            il, k0 = divmod(q0, N)
            n1 = min(q1 - q0, N - k0)
            for c in (0, 1, 127):
                base = c * rb * ldxN * 4
                _prefetch(base + il * ldxN * 4, 4 * k0, 4 * (k0 + n1), valloc)
                if q0 + n1 < q1:
                    assert il + 1 < rb
                    _prefetch(base + (il + 1) * ldxN * 4, 0, 4 * (q1 - q0 - n1), valloc)
            for c in (0, 1, 127):                      # channel planes B N pairs apart (dzh_P)
                _prefetch(0, (c * B * N + q0) * 4, (c * B * N + q1) * 4, hb)
            g0, g1 = r0 * N + q0, r0 * N + q1
            _prefetch(0, g0 * 256, g1 * 256, zb)
            _prefetch(0, g0 * 8, g1 * 8, zst)


@pytest.mark.parametrize("N", [1, 37, 128, 129, 200, 1023, 3605])
@pytest.mark.parametrize("grid", [1, 148])
def test_attention_prefetch_ranges_stay_aligned_and_inside(N, grid):
    """The triangle attention's per-pair kernels prefetch into L2 the rows of the CTA's next tile of 128
    pairs: the projection (starting node) and the output stage as one request over the tile's contiguous
    rows of z (bf16) or o (fp16), 256 bytes per pair; the projection of the ending node one 256-byte
    request per pair at its transposed row. Every request must start on 16 bytes, span a multiple of 16
    bytes and lie inside the N^2 x 256-byte buffer."""
    P = N * N
    alloc = P * 256
    tiles = (P + 127) // 128
    for t in sorted(set(range(0, tiles, max(1, tiles // 97))) | {tiles - 1}):
        n0 = (t + grid) * 128
        if n0 < P:
            n1 = min(n0 + 128, P)
            b0, nbytes = n0 * 256, (n1 - n0) * 256
            assert b0 % 16 == 0 and nbytes % 16 == 0 and 0 < nbytes <= 32768 and b0 + nbytes <= alloc
        for r in (0, 1, 127):
            pn = t * 128 + r + grid * 128
            if pn < P:
                i_n, j_n = divmod(pn, N)
                b0 = (j_n * N + i_n) * 256
                assert b0 % 16 == 0 and b0 + 256 <= alloc
