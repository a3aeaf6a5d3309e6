"""The synchronisation protocol of the backward cluster passes, checked on the host.

A cluster of c CTAs walks a list of units (ny loop supertiles each).  Per CTA
three agents run: the TMA producer, the MMA issuer and the epilogue.  They meet
on mbarriers: the operand ring (full / empty per stage), the TMEM logit buffer
(tfull / tempty), the accumulator (accfull / accempty) and the grad-tile ring
(gready[writer][slot] in every CTA, gfree[slot] in the writer, G_SLOTS slots per
writer).  This model replays the kernel's program order for every agent of
every CTA under many random interleavings and checks that

  * every run finishes (no deadlock: the kernel's bounded waits would turn one
    into status 590), and
  * no barrier ever runs two phases ahead of a waiter.  A wait on mbarrier
    phase i is a parity test: it passes when phase i has completed and phase
    i+1 has not.  If phase i+1 could complete first, the waiter would block on
    the wrong parity (or later pass on a stale one).

Operation order mirrors k_bwd.cu; TMA and MMA completions are modelled as
immediate, which only removes delays.
"""
import random

import pytest

NST, G_SLOTS = 4, 2


class Bar:
    def __init__(self, expected):
        self.expected, self.count, self.phases = expected, 0, 0

    def arrive(self):
        self.count += 1
        if self.count == self.expected:
            self.count = 0
            self.phases += 1


class Violation(Exception):
    pass


def _wait(bar, i):
    """Wait for phase index i (i = -1: the phase before the first, already done)."""
    while True:
        if bar.phases >= i + 2:
            raise Violation(f"barrier ran two phases past a waiter (phase {i}, now {bar.phases})")
        if bar.phases == i + 1:
            return
        yield


def _schedule(nys, c):
    """Steps of the kernel loop: (cur, prev) with cur/prev = (k, r, ny) or None."""
    rounds = [(k, r, ny) for k, ny in enumerate(nys) for r in range((ny + c - 1) // c)]
    steps = []
    for i in range(len(rounds) + 1):
        steps.append((rounds[i] if i < len(rounds) else None, rounds[i - 1] if i > 0 else None))
    return steps


def _cta_agents(j, c, nys, nk, B):
    steps = _schedule(nys, c)
    nrounds = {k: (ny + c - 1) // c for k, ny in enumerate(nys)}

    def producer():
        k_acq = 0
        cnt = [0] * c

        def acquire():
            nonlocal k_acq
            s, u = k_acq % NST, k_acq // NST
            yield from _wait(B[j]["empty"][s], u - 1)
            B[j]["full"][s].arrive()           # expect_tx + the TMA's bytes
            k_acq += 1

        for cur, prev in steps:
            if cur is not None:
                k, r, ny = cur
                if r * c + j < ny:
                    for _ in range(nk):
                        yield from acquire()
            if prev is not None:
                k, r, ny = prev
                for yy in range(r * c, min(r * c + c, ny)):
                    wr = yy - r * c
                    g, u = cnt[wr] % G_SLOTS, cnt[wr] // G_SLOTS
                    yield from _wait(B[j]["gready"][wr][g], u)
                    for _ in range(4):
                        yield from acquire()
                    cnt[wr] += 1

    def mma():
        k_con = 0
        m_all = 0
        cnt = [0] * c

        def consume():
            nonlocal k_con
            s, u = k_con % NST, k_con // NST
            yield from _wait(B[j]["full"][s], u)
            k_con += 1
            return s

        for cur, prev in steps:
            if cur is not None:
                k, r, ny = cur
                if r * c + j < ny:
                    yield from _wait(B[j]["tempty"], m_all - 1)
                    for _ in range(nk):
                        s = yield from consume()
                        B[j]["empty"][s].arrive()
                    B[j]["tfull"].arrive()
                    m_all += 1
            if prev is not None:
                k, r, ny = prev
                if r == 0:
                    yield from _wait(B[j]["accempty"], k - 1)
                for yy in range(r * c, min(r * c + c, ny)):
                    wr = yy - r * c
                    g = cnt[wr] % G_SLOTS
                    for q in range(4):
                        s = yield from consume()
                        if q == 3:
                            B[wr]["gfree"][g].arrive()
                        B[j]["empty"][s].arrive()
                    cnt[wr] += 1
                if r == nrounds[k] - 1:
                    B[j]["accfull"].arrive()

    def epilogue():
        # Units in order; the next unit's first own tile is formed before this
        # unit's accumulator is stored (as in the kernel).
        m_all = 0

        def tile():
            nonlocal m_all
            g, u = m_all % G_SLOTS, m_all // G_SLOTS
            yield from _wait(B[j]["gfree"][g], u - 1)
            yield from _wait(B[j]["tfull"], m_all)
            B[j]["tempty"].arrive()
            for q in range(c):
                B[q]["gready"][j][g].arrive()
            m_all += 1

        def n_own(ny):
            return (ny - j + c - 1) // c if j < ny else 0

        m0 = 0
        for k, ny in enumerate(nys):
            for _ in range(m0, n_own(ny)):
                yield from tile()
            m0 = 0
            if k + 1 < len(nys) and n_own(nys[k + 1]) > 0:
                yield from tile()
                m0 = 1
            yield from _wait(B[j]["accfull"], k)
            B[j]["accempty"].arrive()

    return [producer(), mma(), epilogue()]


def _run(c, nys, nk, seed, gfree_arrivals=None):
    B = [{"full": [Bar(1) for _ in range(NST)], "empty": [Bar(1) for _ in range(NST)],
          "tfull": Bar(1), "tempty": Bar(1), "accfull": Bar(1), "accempty": Bar(1),
          "gready": [[Bar(1) for _ in range(G_SLOTS)] for _ in range(c)],
          "gfree": [Bar(gfree_arrivals or c) for _ in range(G_SLOTS)]} for _ in range(c)]
    agents = [a for j in range(c) for a in _cta_agents(j, c, nys, nk, B)]
    rng = random.Random(seed)
    live = list(range(len(agents)))
    stalled = 0
    while live:
        i = rng.choice(live)
        try:
            before = [(b.phases, b.count) for cta in B for b in _all_bars(cta)]
            next(agents[i])
            after = [(b.phases, b.count) for cta in B for b in _all_bars(cta)]
            stalled = 0 if after != before else stalled + 1
        except StopIteration:
            live.remove(i)
            stalled = 0
        if stalled > 200 * len(agents) + 1000:
            raise AssertionError(f"deadlock: agents {live} cannot progress")


def _all_bars(cta):
    yield from cta["full"]
    yield from cta["empty"]
    yield cta["tfull"]
    yield cta["tempty"]
    yield cta["accfull"]
    yield cta["accempty"]
    for row in cta["gready"]:
        yield from row
    yield from cta["gfree"]


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("nys", [[9, 8, 9], [3, 5, 1, 7], [1], [2, 1, 2, 1], [16, 16], [13]])
def test_protocol_finishes_without_phase_overrun(c, nys):
    for seed in range(6):
        _run(c, nys, nk=3, seed=seed)


@pytest.mark.parametrize("nys", [[20, 17, 3], [16], [40]])
def test_protocol_clusters_of_16(nys):
    for seed in range(2):
        _run(16, nys, nk=2, seed=seed)


@pytest.mark.parametrize("seed", range(4))
def test_protocol_long_units(seed):
    # the Qwen3 head shape's d_hidden split (66-67 supertiles per unit) and a
    # d_weight-like walk of many short units
    _run(4, [66, 67, 66], nk=16, seed=seed)
    _run(4, [8] * 7, nk=16, seed=seed)


def test_model_detects_a_missing_release():
    """A planted mistake -- every slot release one arrival short -- must
    deadlock in the model, or the checks above prove nothing."""
    with pytest.raises(AssertionError, match="deadlock"):
        _run(2, [6], nk=3, seed=0, gfree_arrivals=3)


def test_model_detects_a_phase_overrun():
    """A planted mistake -- a single grad slot per writer, filled again before
    every CTA has loaded it when the loaders' gready waits lag -- is caught by
    the parity check: with one ready barrier per writer and two tiles in
    flight, a lagging loader can see the barrier two phases ahead."""
    global G_SLOTS
    saved = G_SLOTS
    try:
        G_SLOTS = 1
        found = False
        for seed in range(40):
            try:
                _run(2, [8], nk=1, seed=seed, gfree_arrivals=1)   # release after one loader only
            except Violation:
                found = True
                break
            except AssertionError:
                pass
        assert found
    finally:
        G_SLOTS = saved
