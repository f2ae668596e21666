"""The tensor-core kernel's ring protocol, checked on the host.

The kernel (`moe_tc_kernel`) moves every stage through three rings of shared
or tensor memory, each slot guarded by mbarriers that are waited on by phase
parity: a weight-code ring (a TMA producer fills it, three dequantising
warpgroups read it), the A ring in tensor memory (the warpgroups write it, the
MMA issuers read it) and the token-row B ring (a TMA producer fills it, the
MMA issuers read it); the accumulators are handed between the issuers and the
epilogue by two more barriers.  A parity wait cannot tell the phase it waits
for from the one two phases earlier, so the protocol is only right if no
waiter can ever run two phases ahead of a barrier.

This test runs the protocol as a discrete-event model with random
interleavings: every agent (producers, warpgroups, issuers) is a generator
that waits on barriers by parity exactly as the kernel does; copies complete
in any order, MMAs and commits in issue order (one tensor pipe).  Every slot
records which stage it holds and which stage last read it, and every
successful wait is checked against the stage the waiter expects.  The
kernel's arrangement (stages dealt to the warpgroups by global number, rings
whose depths are those of the kernel, MMA issuers that each walk every stage
in order) must never fail; two known-wrong arrangements must be caught:
issuers that own alternate stages (MMAs out of stage order), and a code ring
whose depth is not a multiple of the three warpgroups.
"""
import random

import pytest


class Violation(AssertionError):
    pass


def check(cond, what):
    if not cond:
        raise Violation(what)


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; a parity wait passes
    when the phase of that parity is the last completed one."""

    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0

    def arrive(self, n=1):
        self.pending += n
        check(self.pending <= self.count, "more arrivals than the phase expects")
        if self.pending == self.count:
            self.done += 1
            self.pending = 0

    def test(self, parity):
        return parity != (self.done & 1)


def run(items, kps, kA, kC, issuers, seed, n_issuers=2):
    """One CTA's items (kps stages each) through the rings.  issuers:
    "per_matrix" (the kernel: n_issuers issuers, each issuing its matrix of
    every stage in order; two for gate/up, one for down) or "alternate"
    (two issuers, issuer i owning the stages g = i mod 2)."""
    if issuers == "alternate":
        n_issuers = 2
    rng = random.Random(seed)
    kB = kA
    S = items * kps
    G = 3  # dequantising warpgroups
    c_full = [Barrier(1) for _ in range(kC)]
    c_free = [Barrier(4) for _ in range(kC)]       # one arrival per warp
    a_full = [Barrier(4) for _ in range(kA)]
    ab_free = [Barrier(n_issuers) for _ in range(kA)]  # one commit per issuer
    b_full = [Barrier(1) for _ in range(kB)]
    acc_full, acc_free = Barrier(n_issuers), Barrier(4 * G)
    # slot contents: the stage written last, and the last stage read
    code_slot = [None] * kC
    code_read = [set() for _ in range(kC)]
    a_slot = [None] * kA
    b_slot = [None] * kB
    mma_done = set()        # stages whose MMAs (both issuers') have completed
    issued = {}             # stage -> issuers that issued its MMAs
    copies = []             # in flight: (kind, slot, stage)
    pipe = []               # tensor pipe, in issue order: ("mma", g, i) / ("commit", bar)

    def wait(bar, parity):  # a blocked agent names what it waits for
        while not bar.test(parity):
            yield (bar, parity)

    def code_producer():
        for g in range(S):
            c = g % kC
            yield from wait(c_free[c], ((g // kC) & 1) ^ 1)
            # the slot's previous stage has been read by all its warps
            check(g < kC or (g - kC) in code_read[c], f"code slot {c} refilled before stage {g - kC} was read")
            copies.append(("code", c, g))

    def rows_producer():
        for g in range(S):
            s = g % kB
            yield from wait(ab_free[s], ((g // kB) & 1) ^ 1)
            check(g < kB or (g - kB) in mma_done, f"B slot {s} refilled before stage {g - kB}'s MMAs")
            copies.append(("b", s, g))

    def warpgroup(w):
        for it in range(items):
            for g in range(it * kps, (it + 1) * kps):
                if g % G != w:
                    continue
                c, s = g % kC, g % kA
                yield from wait(c_full[c], (g // kC) & 1)
                check(code_slot[c] == g, f"warpgroup {w} read code slot {c} holding {code_slot[c]}, wanted {g}")
                code_read[c].add(g)
                c_free[c].arrive(4)
                yield
                yield from wait(ab_free[s], ((g // kA) & 1) ^ 1)
                check(g < kA or (g - kA) in mma_done, f"A slot {s} overwritten before stage {g - kA}'s MMAs")
                a_slot[s] = g
                yield
                a_full[s].arrive(4)
            yield from wait(acc_full, it & 1)
            check(all(x in mma_done for x in range(it * kps, (it + 1) * kps)),
                  f"epilogue of item {it} before all its MMAs")
            yield
            acc_free.arrive(4)

    def issuer(i):
        for it in range(items):
            yield from wait(acc_free, (it & 1) ^ 1)
            for g in range(it * kps, (it + 1) * kps):
                if issuers == "alternate" and g % 2 != i:
                    continue
                s = g % kA
                yield from wait(b_full[s], (g // kB) & 1)
                yield from wait(a_full[s], (g // kA) & 1)
                check(b_slot[s] == g, f"issuer {i}: B slot {s} holds {b_slot[s]}, wanted {g}")
                check(a_slot[s] == g, f"issuer {i}: A slot {s} holds {a_slot[s]}, wanted {g}")
                pipe.append(("mma", g, i))
                if issuers == "alternate":  # the one owner commits twice
                    pipe.append(("commit", ab_free[s]))
                pipe.append(("commit", ab_free[s]))
                yield
            pipe.append(("commit", acc_full))

    agents = [code_producer(), rows_producer()] + [warpgroup(w) for w in range(G)]
    agents += [issuer(i) for i in range(n_issuers)]
    # Each run gives every agent its own speed and the copies and the tensor
    # pipe their own rates, so that skewed schedules (one warpgroup or one
    # issuer far behind the others) are explored as well as even ones.
    speed = {id(a): rng.expovariate(1.0) + 1e-3 for a in agents}
    p_copy, p_pipe = rng.uniform(0.05, 0.45), rng.uniform(0.05, 0.45)
    live = {id(a): [a, None] for a in agents}  # agent, the wait it is blocked on

    def runnable():
        return [v for v in live.values() if v[1] is None or v[1][0].test(v[1][1])]

    while live or copies or pipe:
        r = rng.random()
        if copies and r < p_copy:
            kind, slot, g = copies.pop(rng.randrange(len(copies)))  # any order
            if kind == "code":
                code_slot[slot] = g
                c_full[slot].arrive()
            else:
                b_slot[slot] = g
                b_full[slot].arrive()
            continue
        if pipe and r < p_copy + p_pipe:
            op = pipe.pop(0)  # in issue order
            if op[0] == "mma":
                _, g, i = op
                issued.setdefault(g, set()).add(i)
                need = set(range(n_issuers)) if issuers == "per_matrix" else {g % 2}
                if issued[g] >= need:
                    mma_done.add(g)
            else:
                op[1].arrive()
            continue
        ready = runnable()
        if not ready:
            check(copies or pipe, "deadlock: every agent waits and nothing is in flight")
            continue
        v = rng.choices(ready, weights=[speed[id(x[0])] for x in ready])[0]
        try:
            v[1] = next(v[0])
        except StopIteration:
            del live[id(v[0])]


@pytest.mark.parametrize("kA,kC,n_issuers", [(4, 6, 2), (4, 9, 1)])
def test_kernel_protocol_holds(kA, kC, n_issuers):
    """The kernel's rings (gate/up: code ring 6 and two issuers, down: 9 and
    one; A and B rings 4): no wait ever passes on a stale phase and no slot is
    overwritten early, over many random interleavings."""
    for seed in range(400):
        run(items=2, kps=32, kA=kA, kC=kC, issuers="per_matrix", seed=seed, n_issuers=n_issuers)


def test_alternate_stage_issuers_are_caught():
    """Issuers that own alternate stages issue MMAs out of stage order; some
    interleaving lets a waiter take a phase two uses old."""
    with pytest.raises(Violation):
        for seed in range(2000):
            run(items=2, kps=32, kA=4, kC=6, issuers="alternate", seed=seed)


def test_code_ring_not_multiple_of_warpgroups_is_caught():
    """A code ring of 4 slots (not a multiple of the three warpgroups) lets a
    warpgroup that runs ahead read a slot whose copy is still landing."""
    with pytest.raises(Violation):
        for seed in range(2000):
            run(items=2, kps=32, kA=4, kC=4, issuers="per_matrix", seed=seed)
