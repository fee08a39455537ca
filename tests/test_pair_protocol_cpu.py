"""A CPU model of the stage protocol of the tensor-core GEMM run as CTA pairs
(lq_gemm_tma.cu: gemm_tma_kernel with PAIR), run under random interleavings.

Each CTA c of the pair has a ring of S stages; stage ks lives in slot ks mod S
with phase (ks / S) mod 2. In each CTA the producer waits for the slot's
`empty` phase (from the second lap on), then its A half-tile copy lands at a
random later time and counts as one arrival on `full`; each of the four
converter warps of the stage's group waits for `empty` too, writes its
quarter of the W slot and arrives on `full`. Rank 1's gate warp waits for its
own `full` and sends one arrival to rank 0's `pfull` (a remote arrive that
lands at a random later time); rank 0's gate warp waits for `pfull` and
arrives on rank 0's `full`, which therefore counts 1 + 4 + 1 arrivals. Rank
0's MMA thread waits for its `full`, reads both CTAs' A halves and W slots of
the stage, and its commit arrives on both CTAs' `empty` once the MMAs have
completed (again later, in issue order: a commit tracks every earlier MMA of
its thread). Barriers follow the parity rule of mbarrier waits.

Checked: every MMA reads the stage it expects from all four places (both A
halves, both W slots), nothing overwrites a slot an MMA in flight still
reads, and the run ends. Planted mistakes must be caught: rank 0's `full`
without the gate's arrival (count 5), rank 1's gate not waiting for its own
`full`, and the commit arriving on rank 0's `empty` only (a deadlock).
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.done & 1) != parity


def run(S, nk, seed, full0_count=6, gate1_waits=True, multicast=True, max_steps=400000):
    rng = random.Random(seed)
    full = [[Barrier(full0_count) for _ in range(S)], [Barrier(5) for _ in range(S)]]
    empty = [[Barrier(1) for _ in range(S)] for _ in range(2)]
    pfull = [Barrier(1) for _ in range(S)]
    A = [[None] * S for _ in range(2)]
    W = [[[None] * 4 for _ in range(S)] for _ in range(2)]
    reading = {}                  # slot -> stage of the MMA in flight on it
    events = []                   # (kind, args) in flight
    prod = [0, 0]                 # next stage each producer issues
    convq = [[[g] * 4 for g in range(2)] for _ in range(2)]  # per warp of each group
    gate = [0, 0]
    mma = {"ks": 0}
    issues = []

    def fail(msg):
        issues.append(msg)

    def slot_free(c, ks):
        st = ks % S
        return ks < S or empty[c][st].passed(((ks // S) - 1) & 1)

    def write_check(st, ks):
        if st in reading and reading[st] != ks:
            fail(f"slot {st} overwritten with stage {ks} while MMA {reading[st]} reads it")

    def actions():
        acts = []
        for c in range(2):
            if prod[c] < nk and slot_free(c, prod[c]):
                acts.append(("prod", c))
            for g in range(2):
                for q in range(4):
                    ks = convq[c][g][q]
                    if ks < nk and slot_free(c, ks):
                        acts.append(("conv", c, g, q))
        ks = gate[1]
        if ks < nk and (not gate1_waits or full[1][ks % S].passed((ks // S) & 1)):
            acts.append(("gate1",))
        ks = gate[0]
        if ks < nk and pfull[ks % S].passed((ks // S) & 1):
            acts.append(("gate0",))
        ks = mma["ks"]
        if ks < nk and full[0][ks % S].passed((ks // S) & 1):
            acts.append(("mma",))
        # copies and remote arrives land in any order; a commit arrives once
        # every MMA the thread issued before it has completed, so commits land
        # in issue order
        first_commit = next((i for i, e in enumerate(events) if e[0] == "commit"), None)
        for i in range(len(events)):
            if events[i][0] != "commit" or i == first_commit:
                acts.append(("land", i))
        return acts

    steps = 0
    while True:
        if mma["ks"] == nk and not events and all(p == nk for p in prod):
            break
        acts = actions()
        if not acts:
            return "deadlock", issues
        steps += 1
        if steps > max_steps:
            return "timeout", issues
        a = rng.choice(acts)
        if a[0] == "prod":
            c = a[1]
            ks = prod[c]
            events.append(("a_lands", (c, ks)))
            prod[c] += 1
        elif a[0] == "conv":
            _, c, g, q = a
            ks = convq[c][g][q]
            st = ks % S
            write_check(st, ks)
            W[c][st][q] = ks
            full[c][st].arrive()
            convq[c][g][q] += 2
        elif a[0] == "gate1":
            ks = gate[1]
            events.append(("remote", ks % S))
            gate[1] += 1
        elif a[0] == "gate0":
            ks = gate[0]
            if full0_count == 6:
                full[0][ks % S].arrive()
            gate[0] += 1
        elif a[0] == "mma":
            ks = mma["ks"]
            st = ks % S
            for c in range(2):
                if A[c][st] != ks:
                    fail(f"MMA {ks} reads A half of CTA {c} holding stage {A[c][st]}")
                if any(x != ks for x in W[c][st]):
                    fail(f"MMA {ks} reads W slot of CTA {c} holding {W[c][st]}")
            reading[st] = ks
            events.append(("commit", st))
            mma["ks"] += 1
        else:
            kind, arg = events.pop(a[1])
            if kind == "a_lands":
                c, ks = arg
                st = ks % S
                write_check(st, ks)
                A[c][st] = ks
                full[c][st].arrive()
            elif kind == "remote":
                pfull[arg].arrive()
            else:  # the stage's MMAs completed: the commit's arrivals
                reading.pop(arg, None)
                for c in ((0, 1) if multicast else (0,)):
                    empty[c][arg].arrive()
    return "ok", issues


@pytest.mark.parametrize("S", [2, 3, 4])
@pytest.mark.parametrize("nk", [1, 2, 5, 16, 17])
def test_pair_protocol_reads_the_right_stages(S, nk):
    for seed in range(25):
        status, issues = run(S, nk, seed)
        assert status == "ok", (S, nk, seed, status)
        assert not issues, (S, nk, seed, issues[:3])


def test_pair_protocol_model_catches_planted_mistakes():
    def caught(**kw):
        for seed in range(200):
            status, issues = run(3, 12, seed, **kw)
            if status != "ok" or issues:
                return True
        return False
    assert caught(full0_count=5)          # rank 0's full without the gate
    assert caught(gate1_waits=False)      # rank 1's gate not waiting for its own full
    assert caught(multicast=False)        # commit to rank 0's empty only: rank 1 stalls
