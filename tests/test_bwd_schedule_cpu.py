"""The synchronisation protocol of the backward group passes, checked on the host.

A group of c CTA pairs walks a list of units (ny loop supertiles each).  The
two CTAs of a pair act as one MMA unit and meet on the same barriers at the
same points of their program, so the model takes one agent set per pair
(the pair's barriers complete when both CTAs have arrived, which only delays
them).  Per pair three agents run: the TMA producer, the MMA issuer and the
epilogue, plus a poller that watches the group's publish counts and hands
them to the producer through shared memory.  Inside a pair they meet on mbarriers: the operand ring (full /
empty per stage), the TMEM logit buffer (tfull / tempty) and the accumulator
(accfull / accempty).  Between the pairs of the group, the grad-tile ring
(G_SLOTS slots per writer)
is handed over through two monotonic counters per slot in global memory: the
writer adds to `ready` once per tile (the kernel: one add per epilogue warp,
four per tile) and a loader's poller waits until it reaches the fill it needs,
then raises the loader's shared count of that writer's published tiles; every
loader's MMA issuer adds to `free` once its loads of the tile have landed,
and the writer waits for c adds per earlier fill before writing the slot
again.  This model replays the kernel's program order for every agent of
every CTA under many random interleavings and checks that

  * every run finishes (no deadlock: the kernel's bounded waits would turn one
    into status 590);
  * no mbarrier ever runs two phases ahead of a waiter.  A wait on mbarrier
    phase i is a parity test: it passes when phase i has completed and phase
    i+1 has not.  If phase i+1 could complete first, the waiter would block on
    the wrong parity (or later pass on a stale one);
  * every load of a grad slot reads the tile it expects: the writer has
    written that fill and not yet a later one (no read before the write, no
    read of an overwritten slot), and a writer never writes a slot that a
    loader has still to read.

Operation order mirrors k_bwp.cu; TMA and MMA completions are modelled as
immediate, which only removes delays.
"""
import random

import pytest

NST, G_SLOTS = 6, 2


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


def _cta_agents(j, c, nys, nk, B, S, free_short=0, ready_short=0):
    steps = _schedule(nys, c)
    nrounds = {k: (ny + c - 1) // c for k, ny in enumerate(nys)}

    def _until(cond):
        while not cond():
            yield

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
                    # the poller has seen the writer's tile published
                    yield from _until(lambda: S["seen"][j][wr] >= cnt[wr] + 1)
                    for _ in range(4):
                        yield from acquire()
                        # the quarter is read now (the model's TMA completes at once)
                        if S["fills"][wr][g] != u + 1:
                            raise Violation(f"CTA {j} read slot {g} of writer {wr} holding fill "
                                            f"{S['fills'][wr][g] - 1}, expected {u}")
                    S["loaded"][j][wr][g] += 1
                    cnt[wr] += 1

    def poller():
        cnt = [0] * c
        for k, r, ny in (p for _, p in steps if p is not None):
            for yy in range(r * c, min(r * c + c, ny)):
                wr = yy - r * c
                g, u = cnt[wr] % G_SLOTS, cnt[wr] // G_SLOTS
                # the writer's u-th tile in slot g is published
                yield from _until(lambda: S["ready"][wr][g] >= u + 1 - ready_short)
                S["seen"][j][wr] = cnt[wr] + 1
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
                            S["free"][wr][g] += 1     # this CTA's loads of the tile have landed
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
            # every CTA of the group has loaded this slot's earlier fills
            yield from _until(lambda: S["free"][j][g] >= c * u - free_short)
            yield from _wait(B[j]["tfull"], m_all)
            for q in range(c):
                if S["loaded"][q][j][g] < u:
                    raise Violation(f"CTA {j} wrote fill {u} of slot {g} before CTA {q} read fill "
                                    f"{S['loaded'][q][j][g]}")
            S["fills"][j][g] += 1
            B[j]["tempty"].arrive()
            S["ready"][j][g] += 1
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

    return [producer(), poller(), mma(), epilogue()]


def _run(c, nys, nk, seed, free_short=0, ready_short=0):
    B = [{"full": [Bar(1) for _ in range(NST)], "empty": [Bar(1) for _ in range(NST)],
          "tfull": Bar(1), "tempty": Bar(1), "accfull": Bar(1), "accempty": Bar(1)} for _ in range(c)]
    S = {"ready": [[0] * G_SLOTS for _ in range(c)], "free": [[0] * G_SLOTS for _ in range(c)],
         "fills": [[0] * G_SLOTS for _ in range(c)], "seen": [[0] * c for _ in range(c)],
         "loaded": [[[0] * G_SLOTS for _ in range(c)] for _ in range(c)]}
    agents = [a for j in range(c) for a in _cta_agents(j, c, nys, nk, B, S, free_short, ready_short)]
    rng = random.Random(seed)
    live = list(range(len(agents)))
    stalled = 0

    def state():
        return ([(b.phases, b.count) for cta in B for b in _all_bars(cta)], str(S))
    while live:
        i = rng.choice(live)
        try:
            before = state()
            next(agents[i])
            stalled = 0 if state() != before else stalled + 1
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


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("nys", [[9, 8, 9], [3, 5, 1, 7], [1], [2, 1, 2, 1], [16, 16], [13]])
def test_protocol_finishes_without_phase_overrun(c, nys):
    for seed in range(6):
        _run(c, nys, nk=3, seed=seed)


@pytest.mark.parametrize("nys", [[20, 17, 3], [16], [40]])
def test_protocol_groups_of_16(nys):
    for seed in range(2):
        _run(16, nys, nk=2, seed=seed)


@pytest.mark.parametrize("seed", range(4))
def test_protocol_long_units(seed):
    # the Qwen3 head shape's d_hidden split (66-67 supertiles per unit) and a
    # d_weight-like walk of many short units
    _run(4, [66, 67, 66], nk=16, seed=seed)
    _run(4, [8] * 7, nk=16, seed=seed)


def test_model_detects_a_short_free_count():
    """A planted mistake -- the writer waiting for one release fewer than the
    group's loads -- lets it overwrite a slot a loader has still to read; the
    model must catch it, or the checks above prove nothing."""
    found = False
    for seed in range(40):
        try:
            _run(3, [9], nk=1, seed=seed, free_short=1)
        except Violation:
            found = True
            break
    assert found


def test_model_detects_a_short_ready_count():
    """A planted mistake -- a loader waiting for one publication fewer than
    the fill it needs -- lets it read a slot before the tile is written."""
    found = False
    for seed in range(40):
        try:
            _run(2, [8], nk=1, seed=seed, ready_short=1)
        except Violation:
            found = True
            break
    assert found
