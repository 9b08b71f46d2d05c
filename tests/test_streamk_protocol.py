"""The wait-free stream-K fix-up, modelled on the host under random
interleavings of its workers' steps.

The kernels cut the stream-K region's k blocks into one contiguous range per
worker (cut k at position k * W / G).  Each cut has a state word and two
slots: the part of the tile right of the cut (published by whoever holds it)
and the piece of worker k - 1 left of it.  A worker whose piece ends inside
a tile settles that cut first: it adds the right part if it is already
published, else publishes its own piece and swaps its tag into the state
word, going on only if the right part arrived meanwhile.  Whoever holds a
sum that starts inside the tile then publishes it as the right part of the
cut at its start and swaps; if the left piece was there first, it adds it
and carries the sum on to the next cut to the left.  This model takes those
steps one atomic action at a time, in random orders, and checks what the
kernels rely on: every tile is stored exactly once, every slot is written at
most once, and each tile is summed as p0 + (p1 + (p2 + ...)) over its pieces
in k order (fp32 addition is commutative but not associative, so that is
what makes the bits independent of the order of arrival).
"""
import random

import pytest


def items_of(c, G, T, nkb):
    """Worker c's pieces (tile, kb0, kb1) of T tiles of nkb k blocks on G workers."""
    W = T * nkb
    s, e = c * W // G, (c + 1) * W // G
    out, pos = [], s
    while pos < e:
        t = pos // nkb
        lo = t * nkb
        out.append((t, pos - lo, min(e, lo + nkb) - lo))
        pos = lo + out[-1][2]
    return out


def run_once(G, T, nkb, rng):
    W = T * nkb
    cut_pos = lambda k: k * W // G
    state, right, left, written, stored = {}, {}, {}, set(), {}

    def write(slot, value, store):
        assert slot not in written, ("slot written twice", slot)
        written.add(slot)
        store[slot[1]] = value

    def worker(c):
        for (t, kb0, kb1) in items_of(c, G, T, nkb):
            val = ("p", t, kb0, kb1)     # this worker's own piece
            holds = True
            yield
            if kb1 < nkb:                 # the cut at the piece's end, k = c + 1
                k = c + 1
                if rng.random() < 0.5 and state.get(k) == "T":      # peek: right part there
                    val = ("+", val, right[k])
                    state[k] = 0
                else:
                    write(("left", k), val, left)
                    yield
                    old, state[k] = state.get(k), "H"
                    if old == "T":
                        val = ("+", val, right[k])
                        state[k] = 0
                    else:
                        holds = False
            k, inside = c, kb0 > 0
            while holds and inside:       # the cuts to the left
                yield
                write(("right", k), val, right)
                yield
                old, state[k] = state.get(k), "T"
                if old != "H":
                    holds = False
                    break
                state[k] = 0
                val = ("+", left[k], val)
                inside = cut_pos(k - 1) > t * nkb
                k -= 1
            if holds:
                assert t not in stored, ("tile stored twice", t)
                stored[t] = val
            yield

    gens = [worker(c) for c in range(G)]
    live = list(range(G))
    while live:
        c = rng.choice(live)
        try:
            next(gens[c])
        except StopIteration:
            live.remove(c)
    return stored


def canonical(v):
    """The sum tree up to commutativity of each addition."""
    if v[0] == "+":
        a, b = canonical(v[1]), canonical(v[2])
        return ("+",) + tuple(sorted([a, b], key=repr))
    return v


@pytest.mark.parametrize("G,T,nkb", [
    (152, 104, 13),   # tiles cut once or twice (ranges shorter than a tile)
    (48, 16, 256),    # three pieces a tile
    (128, 32, 128),   # four pieces a tile
    (96, 48, 64),     # two pieces a tile
    (5, 3, 9), (7, 4, 11), (3, 2, 8),
])
def test_every_tile_summed_once_in_k_order(G, T, nkb):
    assert T * nkb // G >= 2
    rng = random.Random(G * 1000 + T)
    for _ in range(40):
        stored = run_once(G, T, nkb, rng)
        assert sorted(stored) == list(range(T))
        for t, v in stored.items():
            pieces = sorted((p for c in range(G) for p in items_of(c, G, T, nkb) if p[0] == t),
                            key=lambda p: p[1])
            want = ("p",) + pieces[-1]
            for p in reversed(pieces[:-1]):
                want = ("+", ("p",) + p, want)
            assert canonical(v) == canonical(want), (t, v)
