"""The stage ring of the multi-token query's wide kernel, modelled on the CPU.

Two consumer groups take alternate stages of a 3-deep ring; each stage has a "full" barrier
(one arrival per producer warp plus the copied bytes) and an "empty" barrier (one arrival per
consumer warp of the group that read it).  A wait names a barrier phase only by its parity.
The model lands copies in random order and checks that a group reads a stage only once the
fill it expects is complete -- with the kernel's order of waits (the previous fill's release,
then the fill), and, as a control, that waiting on the fill's parity alone can read early."""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.completed, self.tx = count, count, 0, 0

    def arrive(self):
        self.pending -= 1
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def parity_done(self, parity):  # mbarrier try_wait.parity: the phase of that parity is complete
        return (self.completed & 1) != parity


def run_ring(nstages, nst, ng, warps, producers, release_first, seed):
    """None if every read saw its own fill; else a description of the first early read or stall."""
    rng = random.Random(seed)
    full = [Barrier(producers) for _ in range(nst)]
    empty = [Barrier(warps) for _ in range(nst)]
    landed, content, pending = {}, [None] * nst, []

    def producer():
        for k in range(nstages):
            s = k % nst
            if k >= nst:
                yield empty[s], ((k // nst) - 1) & 1
            full[s].tx += 1
            full[s].arrive()

            def land(s=s, k=k):
                landed[(s, k)] = landed.get((s, k), 0) + 1
                if landed[(s, k)] == producers:
                    content[s] = k
                full[s].tx -= 1
                full[s]._complete()
            pending.append(land)

    def consumer(g):
        for k in range(g, nstages, ng):
            s = k % nst
            if release_first and nst % ng and k >= nst:
                yield empty[s], ((k // nst) - 1) & 1
            yield full[s], (k // nst) & 1
            if content[s] != k:
                raise AssertionError(f"group {g} read stage {s} for fill {k} holding fill {content[s]}")
            empty[s].arrive()

    agents = [producer() for _ in range(producers)] + [consumer(g) for g in range(ng) for _ in range(warps)]
    waits = [None] * len(agents)
    live = set(range(len(agents)))
    try:
        while live:
            ready = [a for a in live if waits[a] is None or waits[a][0].parity_done(waits[a][1])]
            if pending and (not ready or rng.random() < 0.5):
                pending.pop(rng.randrange(len(pending)))()
                continue
            if not ready:
                return "stall"
            a = rng.choice(ready)
            try:
                waits[a] = next(agents[a])
            except StopIteration:
                live.discard(a)
    except AssertionError as e:
        return str(e)
    return None


@pytest.mark.parametrize("producers", [1, 2])
def test_kernel_wait_order_never_reads_early(producers):
    for seed in range(300):
        assert run_ring(24, 3, 2, 2, producers, True, seed) is None, seed


def test_parity_alone_can_read_early():
    """The control: without the release wait some interleaving reads a stage before its fill."""
    assert any(run_ring(24, 3, 2, 2, 1, False, seed) is not None for seed in range(300))


def test_ring_depth_a_multiple_of_the_groups_needs_no_release_wait():
    for seed in range(200):
        assert run_ring(24, 4, 2, 2, 2, False, seed) is None, seed
