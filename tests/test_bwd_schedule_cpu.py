"""The grad-slot hand-over protocol of the backward clusters, checked on the host.

In the d_hidden / d_weight passes a cluster of c CTAs walks units of ny loop
tiles; tile y of a unit is produced by CTA y % c into grad slot y % R (R
divides c).  A slot is refilled only after every CTA has consumed its previous
tile: the consumers of tile yy signal the CTA that fills slot yy % R next --
CTA (yy + R) % c of the same unit, or, after the unit's last tile in the slot,
CTA s of the cluster's next unit (if that unit has a tile s).  A producer waits
for a signal before every own tile y with y >= R, and before its first tile of
a unit when the previous unit had a tile in its slot.  These tests check, for
ragged unit sizes, that every signal has exactly one waiter and that each
producer's waits match its signals in order (the kernel counts them to pick the
mbarrier parity).  A missing signal is a deadlock (the bounded wait reports it
as status 590); an extra one releases a slot early.
"""
import pytest


def _signals_and_waits(c, R, nys):
    sent, waits = [], []
    for k, ny in enumerate(nys):
        ny_next = nys[k + 1] if k + 1 < len(nys) else 0
        ny_prev = nys[k - 1] if k > 0 else 0
        for yy in range(ny):                       # consumption order
            s = yy % R
            if yy + R < ny:
                sent.append(((yy + R) % c, (k, yy + R)))
            elif s < ny_next:
                sent.append((s, (k + 1, s)))
        for j in range(c):
            for y in range(j, ny, c):
                if y >= R or (k > 0 and ny_prev > j % R):
                    waits.append((j, (k, y)))
    return sent, waits


def _slots(c):
    return max(r for r in (4, 3, 2, 1) if c % r == 0)


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("nys", [[131, 132, 131, 132], [132, 131, 131], [3, 5, 4], [1, 2, 7],
                                 [16, 16, 16], [9, 8], [2, 1, 2, 1], [250]])
def test_every_signal_has_one_waiter(c, nys):
    R = _slots(c)
    sent, waits = _signals_and_waits(c, R, nys)
    assert sorted(sent) == sorted(waits)
    # per producer, the signals arrive in the order its tiles are produced
    for j in range(c):
        mine = [t for cta, t in sent if cta == j]
        assert mine == sorted(mine) == [t for cta, t in waits if cta == j]


def test_last_tile_of_a_slot_can_precede_the_last_round():
    # 131 tiles, 4 slots: slot 3's last tile (127) is in round 31, not in the
    # last round 32 -- its hand-over to the next unit must still be sent.
    sent, _ = _signals_and_waits(4, 4, [131, 131])
    assert (3, (1, 3)) in sent
