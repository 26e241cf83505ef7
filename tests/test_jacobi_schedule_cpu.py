"""The round-robin schedule of the SOAP block-Jacobi solve and the split of a round's A
rotations into the block pairs the next round's subproblems read ("critical") and the rest.

The formulas below restate, in Python, the ones the rotation kernels use (circle pairing of
the nb 32-index blocks, the inverse map from a block to its pair, the critical test of the
second launch, the canonical-owner test of the first).  The checks are what the schedule must
satisfy for the two launches to be correct for every size: each round pairs every block once,
each pair of blocks meets once per sweep, the two launches partition the block pairs, every
block the next round's subproblems read comes from the first launch, and no block pair is run
twice by it.  The GPU tests then compare the solve's results with the fp64 oracle.
"""
import pytest


def circle_pair(nb, r, i):
    if i == 0:
        return nb - 1, r
    return (r + i) % (nb - 1), (r - i + (nb - 1)) % (nb - 1)


def pair_of(nb, r, x):
    m, half = nb - 1, nb // 2
    if x == nb - 1 or x == r:
        return 0
    d = x - r
    if d < 0:
        d += m
    return d if d <= half - 1 else m - d


def partner_of(nb, r, x):
    a, b = circle_pair(nb, r, pair_of(nb, r, x))
    return b if a == x else a


def next_round(nb, r):
    return 0 if r + 1 == nb - 1 else r + 1


def critical_pair(nb, r, p, q):
    """The second launch's test: (p, q) belongs to the first launch."""
    if p == q:
        return True
    rn = next_round(nb, r)
    b0, b1 = circle_pair(nb, r, p)
    return (pair_of(nb, r, partner_of(nb, rn, b0)) == q or
            pair_of(nb, r, partner_of(nb, rn, b1)) == q)


def first_launch(nb, r):
    """Block pairs the first launch's 2P CTAs run (None where a CTA returns at once)."""
    P = nb // 2
    rn = next_round(nb, r)
    out = []
    for bid in range(2 * P):
        if bid < P:
            out.append((bid, bid))
            continue
        pp = bid - P
        x, y = circle_pair(nb, rn, pp)
        px, py = pair_of(nb, r, x), pair_of(nb, r, y)
        if px == py:
            out.append(None)
            continue
        x2 = partner_of(nb, r, x)
        p2 = pair_of(nb, rn, x2)
        if p2 < pp and pair_of(nb, r, partner_of(nb, rn, x2)) == py:
            out.append(None)
            continue
        out.append((min(px, py), max(px, py)))
    return out


SIZES = [2, 4, 6, 8, 10, 12, 24, 36, 48, 72, 96]


@pytest.mark.parametrize("nb", SIZES)
def test_round_robin_pairs_every_block_once_per_round_and_every_pair_once_per_sweep(nb):
    seen = set()
    for r in range(nb - 1):
        blocks = []
        for a in range(nb // 2):
            x, y = circle_pair(nb, r, a)
            assert pair_of(nb, r, x) == a and pair_of(nb, r, y) == a
            assert partner_of(nb, r, x) == y and partner_of(nb, r, y) == x
            blocks += [x, y]
            seen.add((min(x, y), max(x, y)))
        assert sorted(blocks) == list(range(nb))
    assert len(seen) == nb * (nb - 1) // 2


@pytest.mark.parametrize("nb", SIZES)
def test_the_two_launches_partition_the_block_pairs_and_feed_the_next_round(nb):
    P = nb // 2
    every = {(p, q) for p in range(P) for q in range(p, P)}
    for r in range(nb - 1):
        first = [c for c in first_launch(nb, r) if c is not None]
        assert len(first) == len(set(first)), "a block pair run twice"
        second = {(p, q) for (p, q) in every if not critical_pair(nb, r, p, q)}
        assert set(first) | second == every
        assert not (set(first) & second)
        # the next round's subproblem of pair pp reads blocks (x, x), (x, y), (y, y)
        rn = next_round(nb, r)
        for pp in range(P):
            x, y = circle_pair(nb, rn, pp)
            for u, v in ((x, x), (x, y), (y, y)):
                a, b = pair_of(nb, r, u), pair_of(nb, r, v)
                assert (min(a, b), max(a, b)) in first, (nb, r, pp, u, v)
