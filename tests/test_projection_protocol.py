"""Host-side replay of the projection kernel's barrier protocol (no GPU needed).

The projection (csrc/k1_project.cu, k1_project) is a persistent CTA whose roles meet at mbarriers: a TMA
warp fills two z stages (and the weights once), one thread issues the MMAs of a tile into one of two
accumulators, four statistics warps read each z tile for the pairs' LayerNorm statistics and hand them to
the epilogue through two buffers, and sixteen epilogue warps read an accumulator and a statistics buffer
per tile. This model restates each role's waits and arrivals in the kernel's order and runs them under
random interleavings (copies landing and MMAs completing, in issue order, at random later times). It
checks that nothing deadlocks, that every wait passes on the phase the kernel means, and that every read
sees the data it means: the MMAs and the statistics read the z stage of their own tile, a z stage is
refilled only after both have read it, the epilogue reads the statistics and the accumulator of its own
tile, and neither is overwritten before all sixteen epilogue warps have read it.
"""
import random

import pytest

STAGES, STAT_WARPS, EPI_WARPS = 2, 4, 16


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.phase, self.pending, self.tx = name, count, 0, count, 0

    def expect(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, self.name
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.phase & 1) != parity


class Always:
    """A step that needs no barrier: a role's work between a wait and the reads it guards, which the
    scheduler may interleave with anything else."""
    name = "work"

    def passes(self, _parity):
        return True


WORK = (Always(), 0, None)


class Model:
    ZEMPTY_COUNT = 1 + STAT_WARPS
    STATS_RELEASE_Z = True

    def __init__(self, tiles, seed):
        self.rng = random.Random(seed)
        self.tiles = tiles
        B = Barrier
        self.zfull = [B(f"zfull{s}", 1) for s in range(STAGES)]
        self.zempty = [B(f"zempty{s}", self.ZEMPTY_COUNT) for s in range(STAGES)]
        self.tfull = [B(f"tfull{b}", 1) for b in range(2)]
        self.tempty = [B(f"tempty{b}", EPI_WARPS) for b in range(2)]
        self.sfull = [B(f"sfull{b}", STAT_WARPS) for b in range(2)]
        self.sempty = [B(f"sempty{b}", EPI_WARPS) for b in range(2)]
        self.wfull, self.fin = B("wfull", 1), B("fin", 1)
        self.zstage = [None] * STAGES
        self.acc = [None, None]
        self.stats = [dict(), dict()]           # per buffer: statistics warp -> tile
        self.read_acc = [set(), set()]
        self.read_stats = [set(), set()]
        self.copies, self.mma = [], []

    def producer(self):
        self.wfull.expect(1)
        self.copies.append(("w", None, None))
        s, ph = 0, 0
        for u in range(self.tiles):
            yield (self.zempty[s], ph ^ 1, ("zempty", s))
            self.zfull[s].expect(1)
            self.copies.append(("z", s, u))
            s += 1
            if s == STAGES:
                s, ph = 0, ph ^ 1

    def issuer(self):
        yield (self.wfull, 0, ("wfull",))
        s, ph = 0, 0
        for local in range(self.tiles):
            buf, use = local & 1, local >> 1
            yield (self.tempty[buf], (use & 1) ^ 1, ("tempty", buf))
            yield (self.zfull[s], ph, ("zfull", s))
            self.mma.append(("mma", local, s, buf))
            self.mma.append(("commit", self.zempty[s]))
            self.mma.append(("commit", self.tfull[buf]))
            s += 1
            if s == STAGES:
                s, ph = 0, ph ^ 1
        self.mma.append(("commit", self.fin))
        yield (self.fin, 0, ("fin",))

    def statistics(self, w):
        s, ph = 0, 0
        for local in range(self.tiles):
            sb, sph = local & 1, (local >> 1) & 1
            yield (self.zfull[s], ph, ("zfull", s))
            yield WORK
            assert self.zstage[s] == local, ("statistics read another tile's z", local, self.zstage[s])
            if self.STATS_RELEASE_Z:
                self.zempty[s].arrive()
            s += 1
            if s == STAGES:
                s, ph = 0, ph ^ 1
            yield (self.sempty[sb], sph ^ 1, ("sempty", sb))
            if local >= 2:
                assert all((local - 2, e) in self.read_stats[sb] for e in range(EPI_WARPS)), \
                    ("statistics overwritten before every epilogue warp read them", local)
            self.stats[sb][w] = local
            self.sfull[sb].arrive()

    def epilogue(self, e):
        for local in range(self.tiles):
            buf, use, sb, sph = local & 1, local >> 1, local & 1, (local >> 1) & 1
            yield (self.sfull[sb], sph, ("sfull", sb))
            yield (self.tfull[buf], use & 1, ("tfull", buf))
            yield WORK
            assert all(self.stats[sb].get(w) == local for w in range(STAT_WARPS)), ("stale statistics", local)
            assert self.acc[buf] == local, ("stale accumulator", local, self.acc[buf])
            self.read_acc[buf].add((local, e))
            self.read_stats[sb].add((local, e))
            self.tempty[buf].arrive()
            self.sempty[sb].arrive()

    def step_copy(self):
        kind, s, u = self.copies.pop(self.rng.randrange(len(self.copies)))
        if kind == "w":
            self.wfull.complete_tx(1)
        else:
            self.zstage[s] = u
            self.zfull[s].complete_tx(1)

    def step_mma(self):
        op = self.mma.pop(0)
        if op[0] == "mma":
            _, local, s, buf = op
            assert self.zstage[s] == local, ("MMA reads another tile's z", local, self.zstage[s])
            if local >= 2:
                assert all((local - 2, e) in self.read_acc[buf] for e in range(EPI_WARPS)), \
                    ("accumulator overwritten before every epilogue warp read it", local)
            self.acc[buf] = local
        else:
            op[1].arrive()

    def run(self):
        roles = {"tma": self.producer(), "mma": self.issuer()}
        roles.update({f"st{w}": self.statistics(w) for w in range(STAT_WARPS)})
        roles.update({f"epi{e}": self.epilogue(e) for e in range(EPI_WARPS)})
        waiting, done, count, meant = {}, set(), {}, {}
        producer_side = {"zempty", "tempty", "sempty"}       # waits that pass at once on a first use

        def advance(k):
            try:
                waiting[k] = next(roles[k])
                if waiting[k][2] is not None:
                    key = (k, waiting[k][2])
                    count[key] = count.get(key, -1) + 1
                    meant[k] = count[key] if waiting[k][2][0] in producer_side else count[key] + 1
            except StopIteration:
                done.add(k)

        for k in roles:
            advance(k)
        for _ in range(10 ** 6):
            if len(done) == len(roles) and not self.mma and not self.copies:
                return
            ready = [k for k in roles if k not in done and waiting[k][0].passes(waiting[k][1])]
            choices = ready + (["copy"] if self.copies else []) + (["tc"] if self.mma else [])
            assert choices, "deadlock: " + ", ".join(f"{k} on {waiting[k][0].name}" for k in roles if k not in done)
            c = self.rng.choice(choices)
            if c == "copy":
                self.step_copy()
            elif c == "tc":
                self.step_mma()
            else:
                bar = waiting[c][0]
                if waiting[c][2] is not None:
                    assert bar.phase == meant[c], ("a wait passed on another phase", c, bar.name, bar.phase, meant[c])
                advance(c)
        raise AssertionError("no progress")


@pytest.mark.parametrize("tiles", [1, 2, 3, 7, 12])
@pytest.mark.parametrize("seed", range(8))
def test_projection_protocol(tiles, seed):
    Model(tiles, seed).run()


def test_the_model_catches_statistics_released_before_the_epilogue_read_them():
    """A planted mistake: a statistics buffer's release counted for fewer warps than read it (eight, the
    epilogue's earlier warp count), so the statistics of a tile can be overwritten while the other eight
    epilogue warps still need them."""
    class Broken(Model):
        def __init__(self, tiles, seed):
            super().__init__(tiles, seed)
            self.sempty = [Barrier(f"sempty{b}", EPI_WARPS // 2) for b in range(2)]
    caught = 0
    for seed in range(30):
        try:
            Broken(8, seed).run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_the_model_catches_a_z_stage_released_by_the_mma_alone():
    """A planted mistake: the z stage's release counted for the MMA only, so the producer can refill it
    while a statistics warp still reads the tile before."""
    class Broken(Model):
        ZEMPTY_COUNT = 1
        STATS_RELEASE_Z = False
    caught = 0
    for seed in range(60):
        try:
            Broken(16, seed).run()
        except AssertionError:
            caught += 1
    assert caught > 0
