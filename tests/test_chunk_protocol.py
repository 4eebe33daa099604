"""The barrier protocol of the prompt-chunk kernel (multi-token query past 64 rows per kv head),
modelled on the CPU.

Roles as in the kernel: one K producer warp and one V producer warp (three-deep rings) whose
copies land at random times; one MMA issuer that, whenever it looks, issues P(jp) V(jp) once the
tile's probabilities are written and its V has landed, else S(js) once K(js) has landed and
P(js - 2) V -- the last reader of the score buffer js % 2 -- is complete; four softmax warps
that, per tile, wait for their scores, sometimes (a moved reference maximum) wait for the
previous P.V to rescale their O rows, and write P over the scores they read.  The products run
on the tensor pipe in issue order, each finishing at a random time relative to every other
role; every wait names its barrier phase only by parity (mbarrier try_wait.parity).  Checks:
every stage and score buffer holds what its reader expects and is not overwritten while an
unfinished product reads it; O is not rescaled while a product accumulates into it; no
schedule stalls; each planted mistake is caught."""
import random

import pytest

NK, NV, NMATH = 3, 3, 4


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


def run_chunk(nt, seed, plant=None):
    """None if the schedule ran to the end with every check holding; else the first failure."""
    rng = random.Random(seed)
    kfull, kempty = [Barrier(1) for _ in range(NK)], [Barrier(1) for _ in range(NK)]
    vfull, vempty = [Barrier(1) for _ in range(NV)], [Barrier(1) for _ in range(NV)]
    nbuf_p = 1 if plant == "one_pfull" else 2
    sfull = [Barrier(1) for _ in range(2)]
    pfull = [Barrier(NMATH) for _ in range(nbuf_p)]
    pfree = [Barrier(1) for _ in range(2)]
    done = Barrier(1)
    # buffer b: what it holds -- ("S", j) once S(j) lands, ("P", j, warps written) after the warps
    st = dict(k=[None] * NK, v=[None] * NV, buf=[None, None], k_reads=[0] * NK, v_reads=[0] * NV,
              buf_reads=[0, 0], o_writes=0, o_applied=-1)
    pipe, pending, errors = [], [], []  # pipe: products issued, in order; pending: landings

    def fail(msg):
        if not errors:
            errors.append(msg)

    def producer(is_v):
        full, empty, n = (vfull, vempty, NV) if is_v else (kfull, kempty, NK)
        content, reads = (st["v"], st["v_reads"]) if is_v else (st["k"], st["k_reads"])
        for j in range(nt):
            s = j % n
            if j >= n and plant != "no_empty_wait":
                yield empty[s], ((j // n) - 1) & 1
            full[s].tx += 1
            full[s].arrive()

            def land(s=s, j=j):
                if reads[s]:
                    fail(f"{'V' if is_v else 'K'} stage {s} overwritten while a product reads it")
                content[s] = j
                full[s].tx -= 1
                full[s]._complete()
            pending.append(land)

    def mma():
        js = jp = 0
        while jp < nt:
            pb = jp & 1 if nbuf_p == 2 else 0
            if (jp < js and pfull[pb].parity_done((jp >> 1) & 1 if nbuf_p == 2 else jp & 1) and
                    vfull[jp % NV].parity_done((jp // NV) & 1)):
                b, vs = jp & 1, jp % NV
                if st["v"][vs] != jp:
                    fail(f"P.V({jp}) issued on V of {st['v'][vs]}")
                if st["buf"][b] != ("P", jp, NMATH):
                    fail(f"P.V({jp}) issued on buffer {b} holding {st['buf'][b]}")
                st["v_reads"][vs] += 1
                st["buf_reads"][b] += 1
                st["o_writes"] += 1

                def pv_done(b=b, vs=vs, j=jp):
                    if st["o_applied"] != j - 1:
                        fail(f"P.V({j}) accumulated after P.V({st['o_applied']})")
                    st["o_applied"] = j
                    st["v_reads"][vs] -= 1
                    st["buf_reads"][b] -= 1
                    st["o_writes"] -= 1
                    vempty[vs].arrive()
                    pfree[b].arrive()
                pipe.append(pv_done)
                jp += 1
            elif (js < nt and kfull[js % NK].parity_done((js // NK) & 1) and
                  (js < 2 or plant == "no_pfree_before_s" or pfree[js & 1].parity_done(((js >> 1) - 1) & 1))):
                ks, b = js % NK, js & 1
                if st["k"][ks] != js:
                    fail(f"S({js}) issued on K of {st['k'][ks]}")
                st["k_reads"][ks] += 1

                def s_done(ks=ks, b=b, j=js):
                    if st["buf_reads"][b]:
                        fail(f"S({j}) wrote buffer {b} while P.V({j - 2}) reads its P")
                    if j >= 2 and st["buf"][b] != ("P", j - 2, NMATH):
                        fail(f"S({j}) overwrote buffer {b} holding {st['buf'][b]}")
                    st["buf"][b] = ("S", j)
                    st["k_reads"][ks] -= 1
                    kempty[ks].arrive()
                    sfull[b].arrive()
                pipe.append(s_done)
                js += 1
            else:
                yield None  # nothing ready: look again later

        pipe.append(lambda: done.arrive())  # the final commit: after every product issued

    def math(w):
        for j in range(nt):
            b = j & 1
            yield sfull[b], (j >> 1) & 1
            held = st["buf"][b]
            if not (held == ("S", j) or (held[0] == "P" and held[1] == j)):
                fail(f"warp {w} read buffer {b} holding {held} for tile {j}")
            if j > 0 and rng.random() < 0.5:  # the reference moved: rescale this warp's O rows
                if plant != "no_pfree_before_rescale":
                    yield pfree[(j - 1) & 1], ((j - 1) >> 1) & 1
                if st["o_writes"]:
                    fail(f"warp {w} rescaled O while a P.V accumulates into it")
            cur = st["buf"][b]
            st["buf"][b] = ("P", j, (cur[2] if cur[0] == "P" else 0) + 1)
            pfull[b if nbuf_p == 2 else 0].arrive()
        yield done, 0

    roles = [producer(False), producer(True), mma()] + [math(w) for w in range(NMATH)]
    waits = {}  # role -> the (barrier, parity) it is blocked on, or None: it polls (the MMA issuer)
    for i, r in enumerate(roles):
        try:
            waits[i] = next(r)
        except StopIteration:
            pass
    unseen = True
    while (waits or pending or pipe) and not errors:
        blocked = {i: w for i, w in waits.items() if w is not None}
        ready = [i for i, w in blocked.items() if w[0].parity_done(w[1])]
        polls = [i for i, w in waits.items() if w is None]
        if not ready and not pending and not pipe and not (polls and unseen):
            return "stall: no role can proceed and nothing is in flight"
        choices = ready + (polls if unseen else []) + (["land"] * (len(pending) > 0)) + (["mma"] * (len(pipe) > 0))
        c = rng.choice(choices)
        if c == "land":
            pending.pop(rng.randrange(len(pending)))()
            unseen = True
            continue
        if c == "mma":  # the oldest product on the tensor pipe completes
            pipe.pop(0)()
            unseen = True
            continue
        polled = waits[c] is None
        try:
            waits[c] = next(roles[c])
        except StopIteration:
            del waits[c]
        unseen = not (polled and waits.get(c, 0) is None)
    return errors[0] if errors else None


@pytest.mark.parametrize("nt", [1, 2, 3, 4, 7, 10])
def test_chunk_protocol_holds(nt):
    for seed in range(60):
        assert run_chunk(nt, seed) is None, (nt, seed, run_chunk(nt, seed))


@pytest.mark.parametrize("plant", ["no_pfree_before_s", "no_pfree_before_rescale", "no_empty_wait", "one_pfull"])
def test_chunk_protocol_catches_planted_mistakes(plant):
    found = [run_chunk(nt, seed, plant) for nt in (3, 5, 8) for seed in range(60)]
    assert any(f is not None for f in found), plant
