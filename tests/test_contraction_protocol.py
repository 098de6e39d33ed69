"""Host-side replay of the contraction kernel's CTA-pair barrier protocol (no GPU needed).

The contraction (csrc/k2_contract.cu, k2_contract) runs on clusters of two CTAs: a TMA warp in each CTA
fills its half of a six-stage ring, the first CTA's "full" barrier counts the bytes of both CTAs' copies,
one thread of the first CTA issues the pair's MMAs and commits each stage's release to both CTAs' "empty"
barriers and each finished accumulator to both CTAs' "full accumulator" barriers, and the epilogue warps of
both CTAs hand each of the two accumulators back on the first CTA's "empty accumulator" barrier. This
model restates each role's waits and arrivals in the kernel's order and runs them under random
interleavings, the copies landing and the tensor core completing the MMAs (in issue order) at random later
times. It checks that nothing deadlocks, that every wait passes on the phase the kernel means, and that
every read sees the data it means: the MMAs of a k-block read both CTAs' copies of that k-block, a stage
is overwritten only after its MMAs ran, the epilogue reads an accumulator only after its tile's last MMA
and the next tile's MMAs write it only after both CTAs' epilogues read it.
"""
import random

import pytest

STAGES, EPI_WARPS = 6, 4


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.phase, self.pending, self.tx = name, count, 0, count, 0

    def expect(self, nbytes):            # arrive.expect_tx
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
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
    def __init__(self, tiles, KB, seed):
        self.rng = random.Random(seed)
        self.tiles, self.KB = tiles, KB
        B = Barrier
        # full: first CTA only (its producer's arrival + both CTAs' bytes); empty, tfull: both CTAs
        self.full = [B(f"full{s}", 1) for s in range(STAGES)]
        self.empty = [[B(f"empty{r}{s}", 1) for s in range(STAGES)] for r in range(2)]
        self.tfull = [[B(f"tfull{r}{b}", 1) for b in range(2)] for r in range(2)]
        self.tempty = [B(f"tempty{b}", 2 * EPI_WARPS) for b in range(2)]
        self.fin = B("fin", 1)
        self.stage = [[None] * STAGES for _ in range(2)]     # per CTA: the (tile, k-block) a stage holds
        self.acc = [None, None]                               # per accumulator: (tile, k-blocks summed)
        self.read = [[set(), set()] for _ in range(2)]        # per CTA and accumulator: tiles read out
        self.copies = []                                      # copies in flight: (cta, stage, tile, kb)
        self.mma = []                                         # tensor core queue, in issue order

    def producer(self, r):
        s, ph = 0, 0
        for t in range(self.tiles):
            for kb in range(self.KB):
                yield (self.empty[r][s], ph ^ 1, ("empty", r, s))
                if r == 0:
                    self.full[s].expect(2)
                self.copies.append((r, s, t, kb))
                s += 1
                if s == STAGES:
                    s, ph = 0, ph ^ 1

    def issuer(self):
        s, ph = 0, 0
        for local in range(self.tiles):
            buf, use = local & 1, local >> 1
            yield (self.tempty[buf], (use & 1) ^ 1, ("tempty", buf))
            for kb in range(self.KB):
                yield (self.full[s], ph, ("full", s))
                self.mma.append(("mma", local, kb, s, buf))
                self.mma.append(("commit", [self.empty[0][s], self.empty[1][s]]))
                s += 1
                if s == STAGES:
                    s, ph = 0, ph ^ 1
            self.mma.append(("commit", [self.tfull[0][buf], self.tfull[1][buf]]))
        self.mma.append(("commit", [self.fin]))
        yield (self.fin, 0, ("fin",))

    def epilogue(self, r, w):
        for local in range(self.tiles):
            buf, use = local & 1, local >> 1
            yield (self.tfull[r][buf], use & 1, ("tfull", r, buf))
            yield WORK
            assert self.acc[buf] == (local, self.KB), ("epilogue reads an unfinished accumulator", local, self.acc[buf])
            self.read[r][buf].add((local, w))
            self.tempty[buf].arrive()

    def step_copy(self):
        r, s, t, kb = self.copies.pop(self.rng.randrange(len(self.copies)))
        self.stage[r][s] = (t, kb)
        self.full[s].complete_tx(1)

    def step_mma(self):
        op = self.mma.pop(0)
        if op[0] == "mma":
            _, local, kb, s, buf = op
            assert self.stage[0][s] == (local, kb) and self.stage[1][s] == (local, kb), \
                ("MMA reads a stage that does not hold its k-block", local, kb, self.stage[0][s], self.stage[1][s])
            if kb == 0:
                prev = local - 2
                if prev >= 0:
                    assert all((prev, w) in self.read[r][buf] for r in (0, 1) for w in range(EPI_WARPS)), \
                        ("accumulator overwritten before both epilogues read it", local)
                self.acc[buf] = (local, 1)
            else:
                assert self.acc[buf] == (local, kb), ("MMA accumulates into the wrong tile", local, kb)
                self.acc[buf] = (local, kb + 1)
        else:
            for bar in op[1]:
                bar.arrive()

    def run(self):
        roles = {"prod0": self.producer(0), "prod1": self.producer(1), "mma": self.issuer()}
        for r in (0, 1):
            for w in range(EPI_WARPS):
                roles[f"epi{r}{w}"] = self.epilogue(r, w)
        waiting, done, meant_phase = {}, set(), {}
        counters = {}

        def advance(k):
            try:
                waiting[k] = next(roles[k])
                key = waiting[k][2]
                if key is not None:
                    counters[(k, key)] = counters.get((k, key), -1) + 1
                    meant_phase[k] = counters[(k, key)]
            except StopIteration:
                done.add(k)
                waiting[k] = None

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
                # each role waits on a given barrier once per phase, in order: the n-th wait means phase n
                # (the producers' waits on "empty" start one phase early, as the first pass finds it free)
                if waiting[c][2] is not None:
                    n = meant_phase[c]
                    expect = n if waiting[c][2][0] == "empty" or waiting[c][2][0] == "tempty" else n + 1
                    assert bar.phase == expect, ("a wait passed on another phase", c, bar.name, bar.phase, expect)
                advance(c)
        raise AssertionError("no progress")


@pytest.mark.parametrize("tiles,KB", [(1, 1), (1, 7), (3, 2), (5, 6), (4, 13)])
@pytest.mark.parametrize("seed", range(10))
def test_contraction_protocol(tiles, KB, seed):
    Model(tiles, KB, seed).run()


def test_the_model_catches_a_release_before_the_mma():
    """A planted mistake: the stage's release committed before its MMAs, letting the producer overwrite
    operands the tensor core has not read yet."""
    class Broken(Model):
        def issuer(self):
            s, ph = 0, 0
            for local in range(self.tiles):
                buf, use = local & 1, local >> 1
                yield (self.tempty[buf], (use & 1) ^ 1, ("tempty", buf))
                for kb in range(self.KB):
                    yield (self.full[s], ph, ("full", s))
                    self.empty[0][s].arrive()
                    self.empty[1][s].arrive()
                    self.mma.append(("mma", local, kb, s, buf))
                    s += 1
                    if s == STAGES:
                        s, ph = 0, ph ^ 1
                self.mma.append(("commit", [self.tfull[0][buf], self.tfull[1][buf]]))
            self.mma.append(("commit", [self.fin]))
            yield (self.fin, 0, ("fin",))
    caught = 0
    for seed in range(30):
        try:
            Broken(3, 9, seed).run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_the_model_catches_an_accumulator_handed_back_by_one_cta():
    """A planted mistake: the accumulator hand-back counted for the first CTA's epilogue only, so the next
    tile's MMAs can overwrite it while the second CTA's epilogue still reads it."""
    class Broken(Model):
        def __init__(self, tiles, KB, seed):
            super().__init__(tiles, KB, seed)
            self.tempty = [Barrier(f"tempty{b}", EPI_WARPS) for b in range(2)]

        def epilogue(self, r, w):
            for local in range(self.tiles):
                buf, use = local & 1, local >> 1
                yield (self.tfull[r][buf], use & 1, ("tfull", r, buf))
                yield WORK
                assert self.acc[buf] == (local, self.KB), ("epilogue reads an unfinished accumulator", local)
                self.read[r][buf].add((local, w))
                if r == 0:
                    self.tempty[buf].arrive()
    caught = 0
    for seed in range(40):
        try:
            Broken(6, 2, seed).run()
        except AssertionError:
            caught += 1
    assert caught > 0
