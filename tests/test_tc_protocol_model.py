"""CPU model of the synchronisation protocol of the tensor-core sparse kernel (sparse_tc.cu).

The kernel's roles, as one entity each (their threads move in lockstep with respect to the
barriers): the producers, the MMA-issuing thread, and the softmax warps.  Each waits on
mbarriers by parity, exactly as the kernel does (a wait for phase k passes once the barrier's
completed-phase count has parity k + 1), and the tensor cores run the issued MMAs in order, each
finishing at an arbitrary later moment; tcgen05.commit arrives once all earlier MMAs of the
issuing thread have finished.  Random interleavings of these steps are explored and every one
must finish (no deadlock) without a buffer being reused while an earlier user may still read it:

- a stage is refilled only after the S and P.V MMAs of the tile it held have finished;
- S(t) is written into its buffer only after the softmax has read S(t - 2) from it;
- the softmax reads S(t) only after that MMA finished and the stage's rows have landed;
- P(t) is written only after the P.V of tile t - 2 (which read that P buffer) finished;
- the O accumulator is rescaled only while no P.V is issued but unfinished;
- each wait passes on the phase it means, never on a later phase of the same parity.

This is a model of the design written from the kernel's structure, not shared code: it checks
the protocol (stage count, the order S(t+1) before P.V(t), the barriers and their parities).
Two of the kernel's waits turn out to be implied by the others, and removing either from the
model changes nothing: the S buffer's free barrier (S(t+2) is issued only after the MMA thread
has seen p_ready(t), which the softmax posts after reading S(t)) and the wait for P.V(t-2)
before P(t) is written (the softmax reads S(t) only after its commit, and a commit covers every
earlier MMA of the thread, P.V(t-2) included).  The kernel keeps both as checks that pass at
once.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.completed = 0        # phases completed so far

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def passes(self, phase):
        """A parity wait for phase `phase` (phase -1: the one before the first)."""
        ok = (self.completed & 1) == ((phase + 1) & 1)
        if ok:
            # the wait must mean this phase, not one two phases later of the same parity
            assert self.completed in (phase + 1, phase + 2) or phase < 0, (self.completed, phase)
            assert self.completed >= phase + 1 or phase < 0
        return ok and self.completed >= phase + 1


class Model:
    def __init__(self, ntiles, stages, rescale_tiles, rng):
        self.n, self.S, self.rng = ntiles, stages, rng
        self.rescale = rescale_tiles            # tiles at which the softmax rescales O
        self.full = [Barrier(1) for _ in range(stages)]
        self.empty = [Barrier(1) for _ in range(stages)]
        self.s_ready = [Barrier(1), Barrier(1)]
        self.s_free = [Barrier(1), Barrier(1)]
        self.p_ready = [Barrier(1), Barrier(1)]
        self.pv_done = [Barrier(1), Barrier(1)]
        self.q_ready = Barrier(1)
        # shared state
        self.stage_tile = [None] * stages       # tile whose rows are in the stage
        self.stage_landed = [False] * stages
        self.sbuf = [None, None]                # tile whose S is in the buffer
        self.sbuf_read = [True, True]
        self.pbuf = [None, None]
        self.queue = []                         # issued MMAs not finished: (kind, tile)
        self.done_mma = set()
        self.commits = []                       # (barrier, number of MMAs issued before it)
        self.issued = 0
        self.finished = 0
        self.in_flight_copies = []              # stages whose copies have not landed
        # role programs
        self.roles = [self.producer(), self.mma(), self.softmax()]
        self.alive = [True, True, True]

    # --- tensor cores and copies ------------------------------------------------------------
    def async_step(self):
        moves = []
        if self.queue:
            moves.append("mma")
        if self.in_flight_copies:
            moves.append("copy")
        if not moves:
            return False
        m = self.rng.choice(moves)
        if m == "mma":
            kind, t = self.queue.pop(0)
            self.finished += 1
            self.done_mma.add((kind, t))
            if kind == "S":
                self.sbuf[t & 1] = t
                self.sbuf_read[t & 1] = False
            still = []
            for bar, n in self.commits:
                if self.finished >= n:
                    bar.arrive()
                else:
                    still.append((bar, n))
            self.commits = still
        else:
            s = self.in_flight_copies.pop(self.rng.randrange(len(self.in_flight_copies)))
            self.stage_landed[s] = True
            self.full[s].arrive()               # the hardware-published stage
        return True

    def issue(self, kind, t):
        self.queue.append((kind, t))
        self.issued += 1

    def commit(self, bar):
        if self.finished >= self.issued:
            bar.arrive()
        else:
            self.commits.append((bar, self.issued))

    # --- roles: generators that yield a barrier wait (barrier, phase) or None (a plain step) ---
    def producer(self):
        for t in range(self.n):
            s = t % self.S
            yield (self.empty[s], t // self.S - 1)
            old = self.stage_tile[s]
            if old is not None:
                assert ("S", old) in self.done_mma and ("PV", old) in self.done_mma, \
                    f"stage {s} refilled with tile {t} while tile {old} may still be read"
            self.stage_tile[s] = t
            self.stage_landed[s] = False
            self.in_flight_copies.append(s)
            yield None

    def mma(self):
        yield (self.q_ready, 0)

        def issue_s(t):
            s, sb = t % self.S, t & 1
            yield (self.full[s], t // self.S)
            if t >= 2:
                yield (self.s_free[sb], (t - 2) // 2)
            assert self.stage_tile[s] == t and self.stage_landed[s], "S reads a stage not ready"
            assert self.sbuf_read[sb], \
                f"S({t}) would overwrite S({self.sbuf[sb]}) before it was read"
            self.issue("S", t)
            self.commit(self.s_ready[sb])

        yield from issue_s(0)
        for t in range(self.n):
            if t + 1 < self.n:
                yield from issue_s(t + 1)
            s, pb = t % self.S, t & 1
            yield (self.p_ready[pb], t // 2)
            assert self.pbuf[pb] == t, "P.V of a tile whose weights are not written"
            self.issue("PV", t)
            self.commit(self.pv_done[pb])
            self.commit(self.empty[s])
            yield None

    def softmax(self):
        self.q_ready.arrive()
        yield None
        for t in range(self.n):
            s, sb = t % self.S, t & 1
            yield (self.full[s], t // self.S)
            yield (self.s_ready[sb], t // 2)
            assert self.sbuf[sb] == t, f"softmax({t}) reads S({self.sbuf[sb]})"
            self.sbuf_read[sb] = True
            self.s_free[sb].arrive()
            yield None
            if t in self.rescale and t >= 1:
                yield (self.pv_done[(t - 1) & 1], (t - 1) // 2)
                assert all(k != "PV" for k, _ in self.queue), "O rescaled while a P.V runs"
            if t >= 2:
                yield (self.pv_done[sb], (t - 2) // 2)
                assert ("PV", t - 2) in self.done_mma
            self.pbuf[sb] = t
            self.p_ready[sb].arrive()
            yield None
        yield (self.pv_done[(self.n - 1) & 1], (self.n - 1) // 2)
        assert ("PV", self.n - 1) in self.done_mma

    # --- scheduler -----------------------------------------------------------------------------
    def run(self, max_steps=100000):
        waiting = [None, None, None]
        for _ in range(max_steps):
            ready = []
            for i, alive in enumerate(self.alive):
                if not alive:
                    continue
                w = waiting[i]
                if w is None or w[0].passes(w[1]):
                    ready.append(i)
            choices = ready + (["async"] if (self.queue or self.in_flight_copies) else [])
            if not choices:
                assert not any(self.alive), f"deadlock: waiting on {waiting}"
                return
            c = self.rng.choice(choices)
            if c == "async":
                self.async_step()
                continue
            try:
                waiting[c] = next(self.roles[c])
            except StopIteration:
                self.alive[c] = False
                waiting[c] = None
        raise AssertionError("no progress bound reached")


@pytest.mark.parametrize("stages", [4, 8])          # head dim 128 and 64
@pytest.mark.parametrize("ntiles", list(range(1, 9)))
def test_protocol_finishes_without_early_reuse(stages, ntiles):
    for seed in range(60):
        rng = random.Random(1000 * stages + 17 * ntiles + seed)
        rescale = {t for t in range(ntiles) if rng.random() < 0.4}
        Model(ntiles, stages, rescale, rng).run()


def test_model_catches_a_publish_lag_deadlock():
    """The checker is not vacuous: a producer that publishes a stage only after issuing two
    more tiles (the lag first tried in the kernel) deadlocks with four stages and eight tiles,
    because the MMA thread needs tile t + 1 before it issues the P.V that frees a stage."""

    class Lagged(Model):
        def producer(self):
            lag = self.S - 1
            issued = []
            for t in range(self.n):
                s = t % self.S
                yield (self.empty[s], t // self.S - 1)
                self.stage_tile[s] = t
                self.stage_landed[s] = True
                issued.append(s)
                if len(issued) > lag:
                    self.full[issued.pop(0)].arrive()
                yield None
            for s in issued:
                self.full[s].arrive()

    with pytest.raises(AssertionError, match="deadlock"):
        Lagged(8, 4, set(), random.Random(3)).run()


def test_model_catches_a_rescale_that_does_not_wait():
    """The checker is not vacuous for the accumulator either: rescaling O without first waiting
    for the previous tile's P.V is caught as a rescale while a P.V may still run."""

    class Eager(Model):
        def softmax(self):
            self.q_ready.arrive()
            yield None
            for t in range(self.n):
                s, sb = t % self.S, t & 1
                yield (self.full[s], t // self.S)
                yield (self.s_ready[sb], t // 2)
                self.sbuf_read[sb] = True
                self.s_free[sb].arrive()
                yield None
                if t >= 1:     # every tile rescales, without the wait on the previous P.V
                    assert all(k != "PV" for k, _ in self.queue), "O rescaled while a P.V runs"
                if t >= 2:
                    yield (self.pv_done[sb], (t - 2) // 2)
                self.pbuf[sb] = t
                self.p_ready[sb].arrive()
                yield None
            yield (self.pv_done[(self.n - 1) & 1], (self.n - 1) // 2)

    caught = 0
    for seed in range(50):
        try:
            Eager(8, 4, set(), random.Random(seed)).run()
        except AssertionError as e:
            assert "rescaled while a P.V runs" in str(e)
            caught += 1
    assert caught > 0
