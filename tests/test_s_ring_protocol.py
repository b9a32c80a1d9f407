"""A model of the forward kernel's hand-off protocol at D = 64, where the S products of the two
query tiles rotate through three TMEM buffers (S product k of a CTA, in issue order, in buffer
k mod 3), checked under random interleavings of its four roles:

  TMA producer   K_j and V_j into a ring of stages (K/V "full" and "empty" barriers);
  MMA warp       for k = 0, 1, ...: the PV product of S number k - 3 (its two halves after the
                 softmax releases them), then S number k; tcgen05 commits arrive on barriers when
                 every MMA issued before them has finished (an in-order tensor pipe);
  softmax t      per key step j: wait for S_t(j), optionally wait for PV_t(j-1) to finish (a
                 rescale of O), release the two halves of P_t(j);
  epilogue t     wait for the last PV of tile t.

An mbarrier is modelled by its count of completed phases; a parity wait is only meaningful while
the barrier is at most one phase past the awaited one, so the model fails any wait on a barrier
two or more phases ahead (the kernel would then wait for a later phase and time out). It also
fails an S product issued into a buffer whose previous PV has not been issued, and a deadlock.

The kernel keys the S-full and P-half/P-full barriers by buffer, which is safe for any key-tile
counts n0 <= n1. The second test shows that keying them by tile, with two barriers alternating
between even and odd key steps, is not: when tile 1 has two or more key tiles more than tile 0,
its softmax, alone on the three buffers, may run two steps ahead of its PV products. (Causal
launches give tile 1 at most one key tile more, but the protocol does not rely on that.)"""
import random

import pytest


class Barrier:
    def __init__(self, count: int, name):
        self.count, self.name, self.pending, self.completed = count, name, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.completed += 1

    def done(self, phase: int) -> bool:
        if self.completed >= phase + 2:
            raise AssertionError(f"{self.name}: wait on phase {phase}, barrier {self.completed} "
                                 f"phases in")
        return self.completed > phase


def s_seq(t: int, j: int, n0: int) -> int:
    """Issue number of S_t(j): the tiles alternate while both have key tiles, then tile 1."""
    return 2 * j + t if j < n0 else n0 + j


def simulate(n0: int, n1: int, stages: int, rng: random.Random, rescale_p: float,
             pipe_p: float, per_buffer: bool = True) -> None:
    assert 1 <= n0 <= n1
    bars = {}

    def bar(name, count=1):
        # one arrival completes a phase (a softmax warpgroup's 128 arrivals in the kernel)
        if name not in bars:
            bars[name] = Barrier(count, name)
        return bars[name]

    def hand(kind, t, j):
        """(barrier, phase) of the hand-off of tile t's step j."""
        k = s_seq(t, j, n0)
        if per_buffer:
            return bar((kind, k % 3)), k // 3
        return bar((kind, t, j & 1)), j >> 1

    pipe = []          # in-order tensor pipe: MMAs and commits
    pv_issued = set()

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

    def seq_at(k):
        return (k & 1, k >> 1) if k < 2 * n0 else (1, k - n0)

    def mma():
        total = n0 + n1
        for k in range(total + 3):
            if k >= 3:
                t, j = seq_at(k - 3)
                st = j % stages
                while not bar(("V_FULL", st)).done(j // stages):
                    yield
                b, ph = hand("P_HALF", t, j)
                while not b.done(ph):
                    yield
                pipe.append(("mma",))
                yield
                b, ph = hand("P_FULL", t, j)
                while not b.done(ph):
                    yield
                pipe.append(("mma",))
                pv_issued.add(k - 3)
                pipe.append(("commit", ("O_DONE", t)))
                if j + 1 == (n0, n1)[t]:
                    pipe.append(("commit", ("O_READY", t)))
                if t == 1:
                    pipe.append(("commit", ("V_EMPTY", st)))
                yield
            if k < total:
                t, j = seq_at(k)
                st = j % stages
                while not bar(("K_FULL", st)).done(j // stages):
                    yield
                assert k < 3 or (k - 3) in pv_issued, "S product issued over an unread P"
                pipe.append(("mma",))
                b, _ = hand("S_FULL", t, j)
                pipe.append(("commit", b.name))
                if t == 1:
                    pipe.append(("commit", ("K_EMPTY", st)))
                yield

    def softmax(t):
        for j in range((n0, n1)[t]):
            b, ph = hand("S_FULL", t, j)
            while not b.done(ph):
                yield
            for _ in range(rng.randint(0, 3)):
                yield
            if j > 0 and rng.random() < rescale_p:
                while not bar(("O_DONE", t)).done(j - 1):
                    yield
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
            idle = 0
            continue
        role = rng.choice(alive)
        try:
            next(role)
        except StopIteration:
            alive.remove(role)
        idle += 1
        assert idle < 20000 or pipe, "deadlock"


def random_case(rng):
    n0 = rng.randint(1, 9)
    n1 = n0 + rng.choice([0, 0, 1, 1, 4])
    return n0, n1, rng.choice([2, 4]), rng.choice([0.0, 0.3, 1.0]), rng.choice([0.05, 0.3, 0.9])


@pytest.mark.parametrize("seed", range(4))
def test_buffer_keyed_hand_offs_are_safe(seed):
    rng = random.Random(seed)
    for _ in range(500):
        n0, n1, stages, rescale_p, pipe_p = random_case(rng)
        simulate(n0, n1, stages, rng, rescale_p, pipe_p)


def test_tile_keyed_hand_offs_can_run_two_phases_ahead():
    rng = random.Random(1)
    with pytest.raises(AssertionError, match="phases in"):
        for _ in range(2000):
            n0 = rng.randint(1, 9)
            simulate(n0, n0 + 2, rng.choice([2, 4]), rng, 0.3, rng.choice([0.05, 0.3, 0.9]),
                     per_buffer=False)
