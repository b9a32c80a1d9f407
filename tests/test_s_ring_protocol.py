"""A model of the forward kernel's hand-off protocol between its roles, checked under random
interleavings, for both orders the kernel uses:

  D = 128  one S/P buffer per query tile; per key tile j the MMA warp issues PV_0(j) (two
           halves), S_0(j+1), PV_1(j), S_1(j+1); the hand-off barriers are per tile.
  D = 64   three S/P buffers rotating between the tiles: S product k of a CTA (issue order: the
           tiles alternate while both have key tiles, then tile 1 alone) goes to buffer k mod 3;
           the MMA warp issues the PV product of S number k - 3, then S number k; the hand-off
           barriers are per buffer.

The roles:

  TMA producer   K_j and V_j into a ring of stages (K/V "full" and "empty" barriers);
  MMA warp       as above; tcgen05 commits arrive on barriers when every MMA issued before them
                 has finished (an in-order tensor pipe, modelled as a queue);
  softmax t      per key step j: wait for S_t(j); optionally rescale O_t, which needs every PV
                 product of tile t before step j finished (D = 64 first waits for the previous
                 PV product on a per-tile barrier; D = 128 needs no wait); release the two
                 halves of P_t(j);
  epilogue t     wait for the last PV product of tile t.

An mbarrier is modelled by its count of completed phases; a parity wait is only meaningful while
the barrier is at most one phase past the awaited one, so the model fails any wait on a barrier
two or more phases ahead (the kernel would then wait for a later phase and time out). It also
fails an S product issued into a buffer whose P has not been read by an issued PV product, a
rescale of O while a PV product of the tile is unfinished, and a deadlock.

The D = 64 kernel keys its barriers by buffer, which is safe for any key-tile counts n0 <= n1.
Keying them by tile, with two barriers alternating between even and odd key steps, is not: when
tile 1 has two or more key tiles more than tile 0, its softmax, alone on the three buffers, may
run two steps ahead of its PV products. (Causal launches give tile 1 at most one key tile more,
but the protocol does not rely on that.) Without its wait for the previous PV product, the D = 64
rescale would touch O while that product still runs."""
import random

import pytest


class Barrier:
    def __init__(self, name):
        self.name, self.completed = name, 0

    def arrive(self):
        # one arrival completes a phase (a softmax warpgroup's 128 arrivals in the kernel)
        self.completed += 1

    def done(self, phase: int) -> bool:
        if self.completed >= phase + 2:
            raise AssertionError(f"{self.name}: wait on phase {phase}, barrier {self.completed} "
                                 f"phases in")
        return self.completed > phase


def s_seq(t: int, j: int, n0: int) -> int:
    """Issue number of S_t(j) in the D = 64 order."""
    return 2 * j + t if j < n0 else n0 + j


def simulate(n0: int, n1: int, stages: int, rng: random.Random, rescale_p: float,
             pipe_p: float, ring: bool = True, per_buffer: bool = True,
             rescale_wait: bool = True) -> None:
    assert 1 <= n0 <= n1
    bars = {}
    pipe = []               # in-order tensor pipe: ("pv", t, j, half), ("s", t, j), ("commit", b)
    pv_issued = set()       # (t, j) of PV products issued (both halves)
    pv_done = set()         # ... and finished
    buf_of = {}             # (t, j) -> S/P buffer

    def bar(name):
        if name not in bars:
            bars[name] = Barrier(name)
        return bars[name]

    def hand(kind, t, j):
        """(barrier, phase) of the hand-off of tile t's step j."""
        if not ring:
            return bar((kind, t)), j
        k = s_seq(t, j, n0)
        if per_buffer:
            return bar((kind, k % 3)), k // 3
        return bar((kind, t, j & 1)), j >> 1

    def producer():
        for j in range(n1):
            st, use = j % stages, j // stages
            while use > 0 and not bar(("K_EMPTY", st)).done(use - 1):
                yield
            bar(("K_FULL", st)).arrive()
            yield
            while use > 0 and not bar(("V_EMPTY", st)).done(use - 1):
                yield
            bar(("V_FULL", st)).arrive()
            yield

    def issue_pv(t, j):
        """Both halves of PV_t(j), each after its P half is released."""
        st = j % stages
        while not bar(("V_FULL", st)).done(j // stages):
            yield
        for h, kind in enumerate(("P_HALF", "P_FULL")):
            b, ph = hand(kind, t, j)
            while not b.done(ph):
                yield
            pipe.append(("pv", t, j, h))
            yield
        pv_issued.add((t, j))
        if ring:
            pipe.append(("commit", ("O_DONE", t)))
        if j + 1 == (n0, n1)[t]:
            pipe.append(("commit", ("O_READY", t)))
        if t == 1:
            pipe.append(("commit", ("V_EMPTY", st)))

    def issue_s(t, j, buf):
        st = j % stages
        while not bar(("K_FULL", st)).done(j // stages):
            yield
        # the buffer's previous S/P must have been read by an issued PV product
        prev = [tj for tj, b in buf_of.items() if b == buf]
        assert all(tj in pv_issued for tj in prev), "S product issued over an unread P"
        for tj in prev:
            del buf_of[tj]
        buf_of[(t, j)] = buf
        pipe.append(("s", t, j))
        pipe.append(("commit", hand("S_FULL", t, j)[0].name))
        if t == 1:
            pipe.append(("commit", ("K_EMPTY", st)))

    def mma():
        if ring:
            def seq_at(k):
                return (k & 1, k >> 1) if k < 2 * n0 else (1, k - n0)
            total = n0 + n1
            for k in range(total + 3):
                if k >= 3:
                    yield from issue_pv(*seq_at(k - 3))
                if k < total:
                    yield from issue_s(*seq_at(k), k % 3)
                yield
        else:
            yield from issue_s(0, 0, 0)
            yield from issue_s(1, 0, 1)
            for j in range(n1):
                for t in range(2):
                    if j >= (n0, n1)[t]:
                        continue
                    yield from issue_pv(t, j)
                    if j + 1 < (n0, n1)[t]:
                        yield from issue_s(t, j + 1, t)
                    yield

    def softmax(t):
        for j in range((n0, n1)[t]):
            b, ph = hand("S_FULL", t, j)
            while not b.done(ph):
                yield
            for _ in range(rng.randint(0, 3)):
                yield
            if j > 0 and rng.random() < rescale_p:
                if ring and rescale_wait:
                    while not bar(("O_DONE", t)).done(j - 1):
                        yield
                assert all((t, i) in pv_done for i in range(j)), "O rescaled while a PV runs"
            hand("P_HALF", t, j)[0].arrive()
            yield
            hand("P_FULL", t, j)[0].arrive()
            yield
        while not bar(("O_READY", t)).done(0):
            yield

    alive = [producer(), mma(), softmax(0), softmax(1)]
    idle = 0
    while alive or pipe:
        if pipe and (not alive or rng.random() < pipe_p):
            op = pipe.pop(0)
            if op[0] == "commit":
                bar(op[1]).arrive()
            elif op[0] == "pv" and op[3] == 1:
                pv_done.add((op[1], op[2]))   # the product's second half has run
            idle = 0
            continue
        role = rng.choice(alive)
        try:
            next(role)
        except StopIteration:
            alive.remove(role)
        idle += 1
        assert idle < 20000 or pipe, "deadlock"


def random_case(rng, max_extra=4):
    n0 = rng.randint(1, 9)
    n1 = n0 + rng.choice([0, 0, 1, 1, max_extra])
    return n0, n1, rng.choice([2, 4]), rng.choice([0.0, 0.3, 1.0]), rng.choice([0.05, 0.3, 0.9])


@pytest.mark.parametrize("seed", range(4))
def test_buffer_keyed_ring_is_safe(seed):
    rng = random.Random(seed)
    for _ in range(500):
        n0, n1, stages, rescale_p, pipe_p = random_case(rng)
        simulate(n0, n1, stages, rng, rescale_p, pipe_p)


@pytest.mark.parametrize("seed", range(2))
def test_two_buffer_order_is_safe(seed):
    """The D = 128 order with per-tile barriers and no wait before a rescale, on the key-tile
    counts the kernel gives it (equal, or one more for tile 1 under causal masking)."""
    rng = random.Random(100 + seed)
    for _ in range(500):
        n0, n1, stages, rescale_p, pipe_p = random_case(rng, max_extra=1)
        simulate(n0, n1, stages, rng, rescale_p, pipe_p, ring=False)


def test_tile_keyed_ring_can_run_two_phases_ahead():
    rng = random.Random(1)
    with pytest.raises(AssertionError, match="phases in"):
        for _ in range(2000):
            n0 = rng.randint(1, 9)
            simulate(n0, n0 + 2, rng.choice([2, 4]), rng, 0.3, rng.choice([0.05, 0.3, 0.9]),
                     per_buffer=False)


def test_ring_rescale_needs_its_wait():
    rng = random.Random(2)
    with pytest.raises(AssertionError, match="O rescaled while a PV runs"):
        for _ in range(2000):
            n0, n1, stages, _, pipe_p = random_case(rng)
            simulate(n0, n1, stages, rng, 1.0, pipe_p, rescale_wait=False)
