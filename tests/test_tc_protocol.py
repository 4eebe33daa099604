"""The barrier protocol of the tcgen05 multi-token kernel, modelled on the CPU.

Roles as in the kernel: two K producer warps (3-deep ring) and two V producer warps (2-deep
ring) whose copies land in random order; one MMA issuer that, whenever it looks, issues the
P.V product of the oldest tile whose probabilities are written and whose V has landed, else
the score product of the next tile whose K has landed and whose score buffer (of two) has been
read; eight softmax warps that read a tile's scores, release the buffer, wait until the
previous P.V product has finished with P^T, and write the tile's probabilities.  Products
complete in random order relative to everything else, and every wait names its barrier phase
only by parity (mbarrier try_wait.parity), so a protocol that let a phase be taken for another
would show up as a role reading or overwriting the wrong data.  The checks: every stage, score
buffer and P^T is read holding the tile the reader expects and is never overwritten while an
unfinished product reads it; no schedule stalls; each planted mistake is caught."""
import random

import pytest

NK, NV, NMATH = 3, 2, 8


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

    def parity_done(self, parity):  # try_wait.parity: the phase of that parity is complete
        return (self.completed & 1) != parity


def run_tc(nt, seed, plant=None):
    """None if the schedule ran to the end with every check holding; else the first failure."""
    rng = random.Random(seed)
    kfull, kempty = [Barrier(2) for _ in range(NK)], [Barrier(1) for _ in range(NK)]
    vfull, vempty = [Barrier(2) for _ in range(NV)], [Barrier(1) for _ in range(NV)]
    sfull, sfree = [Barrier(1) for _ in range(2)], [Barrier(NMATH) for _ in range(2)]
    pfull, pfree, done = Barrier(NMATH), Barrier(1), Barrier(1)
    st = dict(k=[None] * NK, v=[None] * NV, s=[None] * 2, k_reads=[0] * NK, v_reads=[0] * NV,
              s_loaded=[[None] * NMATH for _ in range(2)], p=[None] * NMATH, pv_busy=0, busy=0)
    landed, pending, errors = {}, [], []

    def fail(msg):
        if not errors:
            errors.append(msg)

    def producer(is_v, pw):
        ring_full, ring_empty, n = (vfull, vempty, NV) if is_v else (kfull, kempty, NK)
        content, reads = (st["v"], st["v_reads"]) if is_v else (st["k"], st["k_reads"])
        for j in range(nt):
            s = j % n
            if j >= n and plant != "no_empty_wait":
                yield ring_empty[s], ((j // n) - 1) & 1
            ring_full[s].tx += 1
            ring_full[s].arrive()

            def land(s=s, j=j):
                if reads[s]:
                    fail(f"{'V' if is_v else 'K'} stage {s} overwritten while a product reads it")
                landed[(is_v, s, j)] = landed.get((is_v, s, j), 0) + 1
                if landed[(is_v, s, j)] == 2:
                    content[s] = j
                ring_full[s].tx -= 1
                ring_full[s]._complete()
            pending.append(land)

    def mma():
        js = jp = 0
        while jp < nt:
            if (jp < js and pfull.parity_done(jp & 1) and vfull[jp % NV].parity_done((jp // NV) & 1)):
                vs = jp % NV
                if st["v"][vs] != jp or any(x != jp for x in st["p"]):
                    fail(f"P.V({jp}) issued on V of {st['v'][vs]} / P of {st['p']}")
                st["v_reads"][vs] += 1
                st["pv_busy"] += 1
                st["busy"] += 1

                def pv_done(vs=vs):
                    st["v_reads"][vs] -= 1
                    st["pv_busy"] -= 1
                    st["busy"] -= 1
                    vempty[vs].arrive()
                    pfree.arrive()
                pending.append(pv_done)
                jp += 1
            elif (js < nt and kfull[js % NK].parity_done((js // NK) & 1) and
                  (js < 2 or plant == "no_sfree_wait" or sfree[js & 1].parity_done(((js >> 1) - 1) & 1))):
                ks, b = js % NK, js & 1
                if st["k"][ks] != js:
                    fail(f"S({js}) issued on K of {st['k'][ks]}")
                st["k_reads"][ks] += 1
                st["busy"] += 1

                def s_done(ks=ks, b=b, j=js):
                    if j >= 2 and any(x != j - 2 for x in st["s_loaded"][b]):
                        fail(f"score buffer {b} overwritten by S({j}) before every warp read S({j - 2})")
                    st["s"][b] = j
                    st["k_reads"][ks] -= 1
                    st["busy"] -= 1
                    kempty[ks].arrive()
                    sfull[b].arrive()
                pending.append(s_done)
                js += 1
            else:
                yield None  # nothing ready: look again later

        def all_done():  # the final commit: every product issued so far is complete
            if st["busy"]:
                pending.append(all_done)
            else:
                done.arrive()
        pending.append(all_done)

    def math(w):
        for j in range(nt):
            b = j & 1
            yield sfull[b], (j >> 1) & 1
            if st["s"][b] != j:
                fail(f"warp {w} read scores of {st['s'][b]} for tile {j}")
            st["s_loaded"][b][w] = j
            sfree[b].arrive()
            if j > 0 and plant != "no_pfree_wait":
                yield pfree, (j - 1) & 1
            if st["pv_busy"]:
                fail(f"warp {w} wrote P({j}) while a P.V product reads P^T")
            st["p"][w] = j
            pfull.arrive()
        yield done, 0

    roles = [producer(v, pw) for v in (False, True) for pw in (0, 1)] + [mma()] + [math(w) for w in range(NMATH)]
    waits = {}  # role -> the (barrier, parity) it is blocked on, or None: it polls (the MMA issuer)
    for i, r in enumerate(roles):
        try:
            waits[i] = next(r)
        except StopIteration:
            pass
    unseen = True  # the state changed since the issuer last looked
    while (waits or pending) and not errors:
        blocked = {i: w for i, w in waits.items() if w is not None}
        ready = [i for i, w in blocked.items() if w[0].parity_done(w[1])]
        polls = [i for i, w in waits.items() if w is None]
        if not ready and not pending and not (polls and unseen):
            return "stall: no role can proceed and nothing is in flight"
        choices = ready + (polls if unseen else []) + (["event"] * (len(pending) > 0))
        c = rng.choice(choices)
        if c == "event":
            pending.pop(rng.randrange(len(pending)))()
            unseen = True
            continue
        polled = waits[c] is None
        try:
            waits[c] = next(roles[c])
        except StopIteration:
            del waits[c]
        unseen = not (polled and waits.get(c, 0) is None)
    return errors[0] if errors else None


@pytest.mark.parametrize("nt", [1, 2, 3, 5, 8])
def test_tc_protocol_holds(nt):
    for seed in range(60):
        assert run_tc(nt, seed) is None, (nt, seed, run_tc(nt, seed))


@pytest.mark.parametrize("plant", ["no_pfree_wait", "no_sfree_wait", "no_empty_wait"])
def test_tc_protocol_catches_planted_mistakes(plant):
    found = [run_tc(nt, seed, plant) for nt in (3, 5, 8) for seed in range(40)]
    assert any(f is not None for f in found), plant
