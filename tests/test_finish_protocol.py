"""Host-side replay of the finish kernels' barrier protocols (no GPU needed).

The finish kernel with fp16 x (csrc/k3_finish.cu, k3_finish_x16) is a persistent CTA whose roles meet at
mbarriers: a TMA thread fills two x slots and one z stage per tile (and the weights once), one thread
issues a tile's MMAs into one of two accumulators, four statistics warps read each x slot for the pairs'
LayerNorm_out statistics and hand them to the epilogue through one buffer, and eight epilogue warps read
the statistics and an accumulator, write their rows of the output into their own staging rows and store
them with an asynchronous TMA store, waiting for their previous store to have read the rows before they
write them again. This model restates each role's waits and arrivals in the kernel's order and runs them
under random interleavings (copies landing, the tensor core completing the MMAs in issue order, and the
stores reading their staging rows, each at random later times). It checks that nothing deadlocks, that
every wait passes on the phase the kernel means, and that every read sees the data it means: the MMAs
and the statistics warps read the x slot of their own tile, the MMAs the z of their own tile; a slot or
the z stage is refilled only after all its readers are done; the epilogue reads the statistics and the
accumulator of its own tile, neither overwritten before all eight epilogue warps read it; and a store
reads the rows its warp wrote for that tile.
"""
import random

import pytest

LN_WARPS, EPI_WARPS = 4, 8


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
    """A step that needs no barrier: the role's work between a wait and the reads it guards, which the
    scheduler may interleave with anything else."""
    name = "work"

    def passes(self, _parity):
        return True


WORK = (Always(), 0, None)


class StoreDrained:
    """bulk_wait_read of one epilogue warp: its store in flight (if any) has read the staging rows."""

    def __init__(self, model, e):
        self.model, self.e, self.name = model, e, f"store{e}"

    def passes(self, _parity):
        return self.model.pending_store[self.e] is None


class Model:
    XEMPTY_COUNT = 1 + LN_WARPS
    STATS_RELEASE_X = True
    WAIT_FOR_STORE = True

    def __init__(self, tiles, seed):
        self.rng = random.Random(seed)
        self.tiles = tiles
        B = Barrier
        self.xfull = [B(f"xfull{s}", 1) for s in range(2)]
        self.xempty = [B(f"xempty{s}", self.XEMPTY_COUNT) for s in range(2)]
        self.zfull, self.zempty = B("zfull", 1), B("zempty", 1)
        self.tfull = [B(f"tfull{b}", 1) for b in range(2)]
        self.tempty = [B(f"tempty{b}", EPI_WARPS) for b in range(2)]
        self.sfull, self.sempty = B("sfull", LN_WARPS), B("sempty", EPI_WARPS)
        self.wfull, self.fin = B("wfull", 1), B("fin", 1)
        self.xslot, self.zstage, self.acc = [None, None], None, [None, None]
        self.x_read = [set(), set()]          # per slot: (tile, reader) reads done
        self.z_read = set()
        self.st = {}                          # statistics warp -> tile its statistics in the buffer belong to
        self.st_read = set()                  # (tile, epilogue warp)
        self.acc_read = [set(), set()]
        self.staging = [None] * EPI_WARPS     # per epilogue warp: the tile its staging rows hold
        self.pending_store = [None] * EPI_WARPS
        self.copies, self.mma = [], []

    # ------------------------------------------------------------------ roles
    def producer(self):
        self.wfull.expect(1)
        self.copies.append(("w",))
        ph = 0
        for local in range(self.tiles):
            xsl = local & 1
            yield (self.xempty[xsl], ((local >> 1) & 1) ^ 1, ("xempty", xsl))
            self.xfull[xsl].expect(1)
            self.copies.append(("x", xsl, local))
            yield (self.zempty, ph ^ 1, ("zempty",))
            self.zfull.expect(1)
            self.copies.append(("z", local))
            ph ^= 1

    def issuer(self):
        yield (self.wfull, 0, ("wfull",))
        ph = 0
        for local in range(self.tiles):
            buf = xsl = local & 1
            use = local >> 1
            yield (self.tempty[buf], (use & 1) ^ 1, ("tempty", buf))
            yield (self.xfull[xsl], use & 1, ("xfull", xsl))
            yield (self.zfull, ph, ("zfull",))
            self.mma.append(("mma", local, xsl, buf))
            self.mma.append(("commit", self.xempty[xsl]))
            self.mma.append(("commit", self.zempty))
            self.mma.append(("commit", self.tfull[buf]))
            ph ^= 1
        self.mma.append(("commit", self.fin))
        yield (self.fin, 0, ("fin",))

    def statistics(self, w):
        for local in range(self.tiles):
            xsl = local & 1
            yield (self.xfull[xsl], (local >> 1) & 1, ("xfull", xsl))
            yield WORK
            assert self.xslot[xsl] == local, ("statistics read another tile's x", local, self.xslot[xsl])
            self.x_read[xsl].add((local, w))
            if self.STATS_RELEASE_X:
                self.xempty[xsl].arrive()
            yield (self.sempty, (local & 1) ^ 1, ("sempty",))
            if local >= 1:
                assert all((local - 1, e) in self.st_read for e in range(EPI_WARPS)), \
                    ("statistics overwritten before every epilogue warp read them", local)
            self.st[w] = local
            self.sfull.arrive()

    def epilogue(self, e):
        for local in range(self.tiles):
            buf, use = local & 1, local >> 1
            yield (self.sfull, local & 1, ("sfull",))
            yield (self.tfull[buf], use & 1, ("tfull", buf))
            yield WORK
            assert all(self.st.get(w) == local for w in range(LN_WARPS)), ("stale statistics", local)
            self.st_read.add((local, e))
            self.sempty.arrive()
            if self.WAIT_FOR_STORE:
                yield (StoreDrained(self, e), 0, None)
            yield WORK
            assert self.acc[buf] == local, ("stale accumulator", local, self.acc[buf])
            self.acc_read[buf].add((local, e))
            self.staging[e] = local
            self.tempty[buf].arrive()
            if self.pending_store[e] is None:
                self.pending_store[e] = local
            else:                                   # only reachable without the wait above
                self.pending_store[e] = ("overrun", self.pending_store[e], local)

    # ------------------------------------------------------------------ asynchronous units
    def step_copy(self):
        op = self.copies.pop(self.rng.randrange(len(self.copies)))
        if op[0] == "w":
            self.wfull.complete_tx(1)
        elif op[0] == "x":
            _, s, u = op
            if u >= 2:
                readers = ["mma"] + list(range(LN_WARPS))
                assert all((u - 2, who) in self.x_read[s] for who in readers), \
                    ("x slot refilled before all its readers were done", u)
            self.xslot[s] = u
            self.xfull[s].complete_tx(1)
        else:
            _, u = op
            if u >= 1:
                assert u - 1 in self.z_read, ("z refilled before the MMAs read it", u)
            self.zstage = u
            self.zfull.complete_tx(1)

    def step_mma(self):
        op = self.mma.pop(0)
        if op[0] == "mma":
            _, local, xsl, buf = op
            assert self.xslot[xsl] == local, ("MMA reads another tile's x", local, self.xslot[xsl])
            assert self.zstage == local, ("MMA reads another tile's z", local, self.zstage)
            if local >= 2:
                assert all((local - 2, e) in self.acc_read[buf] for e in range(EPI_WARPS)), \
                    ("accumulator overwritten before every epilogue warp read it", local)
            self.acc[buf] = local
            self.x_read[xsl].add((local, "mma"))
            self.z_read.add(local)
        else:
            op[1].arrive()

    def step_store(self):
        e = self.rng.choice([k for k in range(EPI_WARPS) if self.pending_store[k] is not None])
        tile = self.pending_store[e]
        assert not isinstance(tile, tuple), ("staging rows rewritten before the store read them", tile)
        assert self.staging[e] == tile, ("a store read rows of another tile", tile, self.staging[e])
        self.pending_store[e] = None

    # ------------------------------------------------------------------ scheduler
    def _roles(self):
        roles = {"tma": self.producer(), "mma": self.issuer()}
        roles.update({f"st{w}": self.statistics(w) for w in range(LN_WARPS)})
        roles.update({f"epi{e}": self.epilogue(e) for e in range(EPI_WARPS)})
        return roles

    def run(self):
        roles = self._roles()
        waiting, done, count, meant = {}, set(), {}, {}
        # waits that pass at once on a first use
        producer_side = {"xempty", "zempty", "tempty", "sempty", "hempty"}

        def advance(k):
            try:
                waiting[k] = next(roles[k])
                key = waiting[k][2]
                if key is not None:
                    count[(k, key)] = count.get((k, key), -1) + 1
                    meant[k] = count[(k, key)] if key[0] in producer_side else count[(k, key)] + 1
            except StopIteration:
                done.add(k)

        for k in roles:
            advance(k)
        for _ in range(10 ** 6):
            stores = any(s is not None for s in self.pending_store)
            if len(done) == len(roles) and not self.mma and not self.copies and not stores:
                return
            ready = [k for k in roles if k not in done and waiting[k][0].passes(waiting[k][1])]
            choices = ready + (["copy"] if self.copies else []) + (["tc"] if self.mma else []) + \
                (["store"] if stores else [])
            assert choices, "deadlock: " + ", ".join(f"{k} on {waiting[k][0].name}" for k in roles if k not in done)
            c = self.rng.choice(choices)
            if c == "copy":
                self.step_copy()
            elif c == "tc":
                self.step_mma()
            elif c == "store":
                self.step_store()
            else:
                bar, _, key = waiting[c]
                if key is not None:
                    assert bar.phase == meant[c], ("a wait passed on another phase", c, bar.name, bar.phase, meant[c])
                advance(c)
        raise AssertionError("no progress")


@pytest.mark.parametrize("tiles", [1, 2, 3, 7, 12])
@pytest.mark.parametrize("seed", range(8))
def test_finish_protocol(tiles, seed):
    Model(tiles, seed).run()


def _caught(cls, tiles=8, seeds=30):
    caught = 0
    for seed in range(seeds):
        try:
            cls(tiles, seed).run()
        except AssertionError:
            caught += 1
    return caught


def test_the_model_catches_an_x_slot_released_by_the_mma_alone():
    """A planted mistake: the x slot's release counted for the MMA only (the statistics warps do not
    arrive), so the producer can refill it while a statistics warp still reads the tile before."""
    class Broken(Model):
        XEMPTY_COUNT = 1
        STATS_RELEASE_X = False

    assert _caught(Broken, tiles=16, seeds=60) > 0


def test_the_model_catches_staging_rewritten_under_a_store():
    """A planted mistake: the epilogue writes its staging rows without waiting for its previous TMA store
    to have read them."""
    class Broken(Model):
        WAIT_FOR_STORE = False

    assert _caught(Broken) > 0


class ModelX32:
    """The float32-x form (k3_finish_x32): one x slot, read by the four LayerNorm warps (after their z
    statistics for the same tile), which write the normalised fp16 x-hat operand; the MMA reads x-hat and
    z; the x-hat buffer is then the epilogue's staging, handed back to the LayerNorm warps through
    hempty once every epilogue warp's TMA store has read its rows."""
    HEMPTY_AFTER_STORE = True

    def __init__(self, tiles, seed):
        self.rng = random.Random(seed)
        self.tiles = tiles
        B = Barrier
        self.xfull, self.xempty = B("xfull", 1), B("xempty", LN_WARPS)
        self.zfull, self.zempty = B("zfull", 1), B("zempty", 1)
        self.hfull, self.hempty = B("hfull", LN_WARPS), B("hempty", EPI_WARPS)
        self.tfull = [B(f"tfull{b}", 1) for b in range(2)]
        self.tempty = [B(f"tempty{b}", EPI_WARPS) for b in range(2)]
        self.sfull, self.sempty = B("sfull", LN_WARPS), B("sempty", EPI_WARPS)
        self.wfull, self.fin = B("wfull", 1), B("fin", 1)
        self.xslot = self.zstage = None
        self.x_read, self.z_read = set(), set()
        self.owner, self.owner_set = None, set()    # x-hat buffer: ("ln" | "epi", tile) and who wrote
        self.xh_mma_read = -1
        self.acc, self.acc_read = [None, None], [set(), set()]
        self.st, self.st_read = {}, set()
        self.pending_store = [None] * EPI_WARPS
        self.copies, self.mma = [], []

    def producer(self):
        self.wfull.expect(1)
        self.copies.append(("w",))
        ph = 0
        for local in range(self.tiles):
            yield (self.xempty, ph ^ 1, ("xempty",))
            self.xfull.expect(1)
            self.copies.append(("x", local))
            yield (self.zempty, ph ^ 1, ("zempty",))
            self.zfull.expect(1)
            self.copies.append(("z", local))
            ph ^= 1

    def issuer(self):
        yield (self.wfull, 0, ("wfull",))
        ph = 0
        for local in range(self.tiles):
            buf, use = local & 1, local >> 1
            yield (self.tempty[buf], (use & 1) ^ 1, ("tempty", buf))
            yield (self.hfull, ph, ("hfull",))
            yield (self.zfull, ph, ("zfull",))
            self.mma.append(("mma", local, buf))
            self.mma.append(("commit", self.zempty))
            self.mma.append(("commit", self.tfull[buf]))
            ph ^= 1
        self.mma.append(("commit", self.fin))
        yield (self.fin, 0, ("fin",))

    def layernorm(self, w):
        ph = 0
        for local in range(self.tiles):
            yield (self.zfull, ph, ("zfull",))
            yield WORK
            assert self.zstage == local, ("z statistics of another tile", local, self.zstage)
            self.z_read.add((local, w))
            yield (self.sempty, (local & 1) ^ 1, ("sempty",))
            if local >= 1:
                assert all((local - 1, e) in self.st_read for e in range(EPI_WARPS)), \
                    ("statistics overwritten before every epilogue warp read them", local)
            self.st[w] = local
            self.sfull.arrive()
            yield (self.xfull, ph, ("xfull",))
            yield WORK
            assert self.xslot == local, ("LayerNorm read another tile's x", local, self.xslot)
            self.x_read.add((local, w))
            yield (self.hempty, ph ^ 1, ("hempty",))
            yield WORK
            if self.owner != ("ln", local):
                if local >= 1:
                    assert self.owner == ("epi", local - 1) and self.owner_set == set(range(EPI_WARPS)), \
                        ("x-hat written over rows the epilogue still stages", local, self.owner)
                    assert all(s is None for s in self.pending_store), \
                        ("x-hat written before the stores read the staging rows", local)
                self.owner, self.owner_set = ("ln", local), set()
            self.owner_set.add(w)
            self.xempty.arrive()
            self.hfull.arrive()
            ph ^= 1

    def epilogue(self, e):
        for local in range(self.tiles):
            buf, use = local & 1, local >> 1
            yield (self.sfull, local & 1, ("sfull",))
            yield (self.tfull[buf], use & 1, ("tfull", buf))
            yield WORK
            assert all(self.st.get(w) == local for w in range(LN_WARPS)), ("stale statistics", local)
            self.st_read.add((local, e))
            self.sempty.arrive()
            assert self.acc[buf] == local, ("stale accumulator", local, self.acc[buf])
            self.acc_read[buf].add((local, e))
            # the staging rows are the x-hat buffer: the MMA of this tile must have read it
            assert self.xh_mma_read >= local, ("staging written over x-hat the MMA still reads", local)
            if self.owner != ("epi", local):
                self.owner, self.owner_set = ("epi", local), set()
            self.owner_set.add(e)
            self.tempty[buf].arrive()
            self.pending_store[e] = local
            if self.HEMPTY_AFTER_STORE:
                yield (StoreDrained(self, e), 0, None)
            self.hempty.arrive()

    def step_copy(self):
        op = self.copies.pop(self.rng.randrange(len(self.copies)))
        if op[0] == "w":
            self.wfull.complete_tx(1)
        elif op[0] == "x":
            u = op[1]
            if u >= 1:
                assert all((u - 1, w) in self.x_read for w in range(LN_WARPS)), ("x refilled early", u)
            self.xslot = u
            self.xfull.complete_tx(1)
        else:
            u = op[1]
            if u >= 1:
                assert (u - 1, "mma") in self.z_read and all((u - 1, w) in self.z_read for w in range(LN_WARPS)), \
                    ("z refilled before all its readers were done", u)
            self.zstage = u
            self.zfull.complete_tx(1)

    def step_mma(self):
        op = self.mma.pop(0)
        if op[0] == "mma":
            _, local, buf = op
            assert self.owner == ("ln", local) and self.owner_set == set(range(LN_WARPS)), \
                ("MMA reads an incomplete or foreign x-hat", local, self.owner)
            assert self.zstage == local, ("MMA reads another tile's z", local, self.zstage)
            if local >= 2:
                assert all((local - 2, e) in self.acc_read[buf] for e in range(EPI_WARPS)), \
                    ("accumulator overwritten before every epilogue warp read it", local)
            self.acc[buf] = local
            self.xh_mma_read = local
            self.z_read.add((local, "mma"))
        else:
            op[1].arrive()

    def step_store(self):
        e = self.rng.choice([k for k in range(EPI_WARPS) if self.pending_store[k] is not None])
        tile = self.pending_store[e]
        assert self.owner == ("epi", tile) and e in self.owner_set, \
            ("a store read staging rows that were overwritten", tile, self.owner)
        self.pending_store[e] = None

    run = Model.run

    def _roles(self):
        roles = {"tma": self.producer(), "mma": self.issuer()}
        roles.update({f"ln{w}": self.layernorm(w) for w in range(LN_WARPS)})
        roles.update({f"epi{e}": self.epilogue(e) for e in range(EPI_WARPS)})
        return roles


@pytest.mark.parametrize("tiles", [1, 2, 3, 7, 12])
@pytest.mark.parametrize("seed", range(8))
def test_finish_x32_protocol(tiles, seed):
    ModelX32(tiles, seed).run()


def test_the_model_catches_x_hat_handed_back_before_the_stores_read_it():
    """A planted mistake in the float32-x form: hempty arrived when the store is issued rather than once
    it has read the staging rows, so the LayerNorm warps can write the next x-hat under it."""
    class Broken(ModelX32):
        HEMPTY_AFTER_STORE = False

    assert _caught(Broken, tiles=12, seeds=40) > 0
