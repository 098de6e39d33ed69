"""Host-side replay of the triangle-attention kernel's barrier protocol (no GPU needed).

The attend kernel (csrc/k_attention.cu, k_ta_attend) is a set of roles that meet only at mbarriers: a TMA
warp filling four stages of K / bias / v (and Q per head pair), one MMA warp per query tile issuing S into
three TMEM buffers and P V into the running output, and four softmax warps per tile. This model restates,
role by role and in the kernel's order, every wait (barrier, parity) and every arrival or commit, and runs
the roles under many random interleavings, with the tensor core completing each MMA warp's operations in
issue order at random later times. It checks that

* every role finishes (no interleaving leaves a role waiting for ever: the kernel would time out);
* a parity wait never passes on a phase other than the one the kernel means (the hardware's parity test
  accepts any completed phase of that parity, so a wait that can fall two phases behind is a bug: the
  model keeps phase numbers and flags it);
* the data each role reads is the data it means: the softmax reads S of block t only after S(t) has been
  computed and before S(t + 3) overwrites the buffer; the P V product of block t reads P(t) after the
  softmax stored it; the running output is finalised or rescaled only when every product before it is
  complete and before the next one starts; Q of the second head pair replaces the first only after every
  S of heads 0 and 1 ran.
"""
import random

import pytest

STAGES, SBUF, GROUPS, SM_WARPS = 4, 3, 2, 4


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.phase = 0          # phases completed so far
        self.pending = count

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, self.name
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        """The hardware's test: the phase of this parity has completed (the current phase differs)."""
        return (self.phase & 1) != parity


class Always:
    """A step that needs no barrier: a role's work between a wait and the reads it guards, which the
    scheduler may interleave with anything else."""
    name = "work"

    def passes(self, _parity):
        return True


WORK = (Always(), 0, None)


class Model:
    def __init__(self, KB, seed):
        self.rng = random.Random(seed)
        self.KB, self.T = KB, 4 * KB
        B = Barrier
        self.q_full, self.q_free, self.go1 = B("q_full", 1), B("q_free", GROUPS), B("go1", SM_WARPS)
        self.kv_full = [B(f"kv_full{s}", 1) for s in range(STAGES)]
        self.kv_empty = [B(f"kv_empty{s}", GROUPS + SM_WARPS * GROUPS) for s in range(STAGES)]
        self.s_full = [[B(f"s_full{g}{b}", 1) for b in range(SBUF)] for g in range(GROUPS)]
        self.p_full = [[B(f"p_full{g}{b}", SM_WARPS) for b in range(SBUF)] for g in range(GROUPS)]
        self.pv_done = [[B(f"pv_done{g}{b}", 1) for b in range(2)] for g in range(GROUPS)]
        self.pv_last = [B(f"pv_last{g}", 1) for g in range(GROUPS)]
        # data state
        self.stage_block = [None] * STAGES     # the block whose K / bias / v a stage holds (after its copy lands)
        self.q_pair = None                     # the head pair whose Q is in shared memory
        self.s_buf = [[None] * SBUF for _ in range(GROUPS)]       # ("S", t) or ("P", t)
        self.pv_completed = [set() for _ in range(GROUPS)]        # products that have run
        self.s_completed = [set() for _ in range(GROUPS)]
        self.mma_queue = [[] for _ in range(GROUPS)]             # per MMA warp, in issue order

    # ------------------------------------------------------------------ tensor core
    def mma_step(self, g):
        """Run the oldest operation of MMA warp g (in issue order)."""
        op = self.mma_queue[g].pop(0)
        kind = op[0]
        if kind == "S":
            t, b, st = op[1], op[2], op[3]
            h = t // self.KB
            assert self.stage_block[st] == t, ("S reads the wrong stage", t)
            assert self.q_pair == h // 2, ("S reads the wrong Q", t)
            self.s_buf[g][b] = ("S", t)
            self.s_completed[g].add(t)
        elif kind == "PV":
            t, b, st = op[1], op[2], op[3]
            assert self.s_buf[g][b] == ("P", t), ("P V reads something other than P of its block", t, self.s_buf[g][b])
            assert self.stage_block[st] == t, ("P V reads the wrong v", t)
            self.pv_completed[g].add(t)
        elif kind == "commit":
            op[1].arrive()

    # ------------------------------------------------------------------ roles (generators yield a wait)
    def tma(self):
        for t in range(self.T):
            h, kb, st, use = t // self.KB, t % self.KB, t % STAGES, t // STAGES
            if kb == 0 and h % 2 == 0:
                if h == 2:
                    yield (self.q_free, 0, None)
                    for g in range(GROUPS):
                        assert all(s in self.s_completed[g] for s in range(2 * self.KB)), "Q replaced early"
                self.q_pair = h // 2
                self.q_full.arrive()
            if use >= 1:
                yield (self.kv_empty[st], (use - 1) & 1, ("kv_empty", st, use - 1))
            self.stage_block[st] = t
            self.kv_full[st].arrive()

    def issuer(self, g):
        KB, T = self.KB, self.T

        def issue_s(t):
            h, kb, st, b = t // KB, t % KB, t % STAGES, t % SBUF
            if kb == 0 and h % 2 == 0:
                yield (self.q_full, (h // 2) & 1, ("q_full", h // 2))
            yield (self.kv_full[st], (t // STAGES) & 1, ("kv_full", st, t // STAGES))
            if g == 1 and t == 0:
                yield (self.go1, 0, ("go1", 0))
            self.mma_queue[g].append(("S", t, b, st))
            self.mma_queue[g].append(("commit", self.s_full[g][b]))
            if t == 2 * KB - 1:
                self.mma_queue[g].append(("commit", self.q_free))

        def issue_pv(t):
            b, st = t % SBUF, t % STAGES
            yield (self.p_full[g][b], (t // SBUF) & 1, ("p_full", g, b, t // SBUF))
            self.mma_queue[g].append(("PV", t, b, st))
            self.mma_queue[g].append(("commit", self.kv_empty[st]))
            self.mma_queue[g].append(("commit", self.pv_done[g][t & 1]))

        for t in range(SBUF):
            yield from issue_s(t)
        for t in range(T):
            yield from issue_pv(t)
            if t + SBUF < T:
                yield from issue_s(t + SBUF)
        self.mma_queue[g].append(("commit", self.pv_last[g]))

    def softmax(self, g, w):
        KB, T = self.KB, self.T
        for t in range(T):
            h, kb, st, b = t // KB, t % KB, t % STAGES, t % SBUF
            yield (self.s_full[g][b], (t // SBUF) & 1, ("s_full", g, b, t // SBUF))
            yield (self.kv_full[st], (t // STAGES) & 1, ("kv_full", st, t // STAGES))
            yield WORK
            assert self.s_buf[g][b] == ("S", t) or self.s_buf[g][b] == ("P", t), ("softmax reads stale S", t)
            assert self.stage_block[st] == t, ("softmax reads the wrong bias", t)
            if t >= 1 and kb == 0:
                yield (self.pv_done[g][(t - 1) & 1], ((t - 1) >> 1) & 1, ("pv_done", g, (t - 1) & 1, (t - 1) >> 1))
                assert all(s in self.pv_completed[g] for s in range(t)), ("finalised before its products", t)
            self.kv_empty[st].arrive()
            if self.rng.random() < 0.1 and kb != 0:          # the reference moved: rescale the running output
                yield (self.pv_done[g][(t - 1) & 1], ((t - 1) >> 1) & 1, ("pv_done", g, (t - 1) & 1, (t - 1) >> 1))
                assert all(s in self.pv_completed[g] for s in range(t)), ("rescaled before a product", t)
                assert t not in self.pv_completed[g]
            yield WORK                                         # the pass over S, then P stored over it
            assert self.s_buf[g][b] == ("S", t) or self.s_buf[g][b] == ("P", t), ("S overwritten during the pass", t)
            if w == SM_WARPS - 1:                              # the last warp's store completes P of the row block
                self.s_buf[g][b] = ("P", t)
            self.p_full[g][b].arrive()
            if g == 0 and t == 0:
                self.go1.arrive()
        yield (self.pv_last[g], 0, ("pv_last", g, 0))
        assert self.pv_completed[g] == set(range(T)), "finalised before the last product"

    # ------------------------------------------------------------------ scheduler
    def run(self):
        roles = {"tma": self.tma()}
        for g in range(GROUPS):
            roles[f"mma{g}"] = self.issuer(g)
            for w in range(SM_WARPS):
                roles[f"sm{g}{w}"] = self.softmax(g, w)
        waiting = {k: None for k in roles}       # the (barrier, parity, meant phase) a role waits on
        done = set()

        def advance(k):
            try:
                waiting[k] = next(roles[k])
            except StopIteration:
                done.add(k)
                waiting[k] = None

        for k in roles:
            advance(k)
        steps = 0
        while len(done) < len(roles) or any(self.mma_queue):
            steps += 1
            assert steps < 10 ** 6, "no progress"
            ready = [k for k in roles if k not in done and waiting[k][0].passes(waiting[k][1])]
            mma_ready = [g for g in range(GROUPS) if self.mma_queue[g]]
            choices = ready + [("mma", g) for g in mma_ready]
            assert choices, "deadlock: " + ", ".join(f"{k} on {waiting[k][0].name}" for k in roles if k not in done)
            c = self.rng.choice(choices)
            if isinstance(c, tuple):
                self.mma_step(c[1])
                continue
            bar, parity, meant = waiting[c]
            if meant is not None:
                # the phase the kernel means must be the one that completed, not one two phases on or behind
                phase_meant = meant[-1]
                assert bar.phase == phase_meant + 1, ("a wait passed on another phase", c, bar.name, bar.phase, phase_meant)
            advance(c)


@pytest.mark.parametrize("KB", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("seed", range(12))
def test_attention_protocol(KB, seed):
    Model(KB, seed).run()


def test_the_model_catches_a_two_phase_parity_wait():
    """A planted form of a bug the kernel once had: the last product waited through the alternating
    product barrier, whose phase can already be two on when the softmax gets there."""
    class Broken(Model):
        def softmax(self, g, w):
            gen = super().softmax(g, w)
            for item in gen:
                if item[0] is self.pv_last[g]:
                    T = self.T
                    item = (self.pv_done[g][(T - 1) & 1], ((T - 3) >> 1) & 1, ("pv_done", g, (T - 1) & 1, (T - 3) >> 1))
                yield item
    caught = 0
    for seed in range(40):
        try:
            Broken(4, seed).run()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_the_model_catches_s_issued_before_the_product_it_overwrites():
    """A planted reordering: S of block t + 3 issued before the P V product of block t, into the buffer
    that product reads (P lies over S), which the model must flag."""
    class Broken(Model):
        def issuer(self, g):
            KB, T = self.KB, self.T
            for t in range(SBUF):
                st, b = t % STAGES, t % SBUF
                if t % KB == 0 and (t // KB) % 2 == 0:
                    yield (self.q_full, ((t // KB) // 2) & 1, ("q_full", (t // KB) // 2))
                yield (self.kv_full[st], (t // STAGES) & 1, ("kv_full", st, t // STAGES))
                if g == 1 and t == 0:
                    yield (self.go1, 0, ("go1", 0))
                self.mma_queue[g] += [("S", t, b, st), ("commit", self.s_full[g][b])]
            for t in range(T):
                b, st = t % SBUF, t % STAGES
                yield (self.p_full[g][b], (t // SBUF) & 1, ("p_full", g, b, t // SBUF))
                if t + SBUF < T:
                    u = t + SBUF
                    su = u % STAGES
                    if u % KB == 0 and (u // KB) % 2 == 0:
                        yield (self.q_full, ((u // KB) // 2) & 1, ("q_full", (u // KB) // 2))
                    yield (self.kv_full[su], (u // STAGES) & 1, ("kv_full", su, u // STAGES))
                    self.mma_queue[g] += [("S", u, u % SBUF, su), ("commit", self.s_full[g][u % SBUF])]
                    if u == 2 * KB - 1:
                        self.mma_queue[g].append(("commit", self.q_free))
                self.mma_queue[g] += [("PV", t, b, st), ("commit", self.kv_empty[st]),
                                      ("commit", self.pv_done[g][t & 1])]
            self.mma_queue[g].append(("commit", self.pv_last[g]))
    with pytest.raises(AssertionError):
        Broken(3, 0).run()
