"""A CPU model of the weight-ring protocols of the decode chain
(lq_gemv_chain.cu), the streaming GEMV (lq_gemv.cu) and the batched decode
kernel (lq_gemv_batch.cu), run under random interleavings.

The model keeps the kernel's rules: global stage g lives in ring slot g mod S
with phase (g / S) mod 2, belongs to row-group g mod nr (S a multiple of nr)
and is finished by K-group (g / nr) mod nk. Every K-group warp of the row-group
waits for the slot's `full` phase, reads the slot, writes its partial into the
partials buffer of (phase, slot), arrives on `red_full` and on `empty` at once
(the slot goes back to the producer before the reduction); the finisher then
waits for `red_full` and reads every K-group's partial. The producer refills a
slot once its previous `empty` phase completed; the copy lands later, at a
random time. Barriers follow the parity rule of mbarrier waits: a wait for
parity P passes once the phase with parity P is the last one completed.

Checked: each warp reads the stage it expects from the slot (never a refill
or a stale copy), each finisher reads partials of its own stage only, and the
run never deadlocks. The streaming GEMV differs in its release (the finisher
hands the slot back after reading the partials, one buffer per slot), the
batched kernel in having no producer (the finisher refills the slot after
reading the partials). Three planted mistakes must be caught: the chain with
one partials buffer per slot, a ring whose slot count is not a multiple of the
row-groups, and the batched kernel's refill issued before the read.
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


def run(S, nr, nk, stages, seed, phase_buffers=2, mode="chain", max_steps=200000):
    """mode "chain": every warp releases the slot right after posting its
    partial (partials double-buffered by phase); "stream" (lq_gemv.cu): the
    finisher releases the slot after reading the partials (one buffer per
    slot); "batch" (lq_gemv_batch.cu): no producer, the finisher issues the
    stage S further on into the slot after reading the partials;
    "batch-early": the same with the refill issued before the read."""
    rng = random.Random(seed)
    full = [Barrier(1) for _ in range(S)]
    empty = [Barrier(nk) for _ in range(S)]
    red_full = [Barrier(nk) for _ in range(S)]
    slot = [None] * S
    red = {}                      # (buffer, slot, kgroup) -> stage
    in_flight = []                # (slot, stage) copies issued, not landed
    prod = {"g": 0}
    # each warp (rg, kg): its next stage and where it is in that stage's steps
    warps = {(rg, kg): {"g": rg, "step": 0} for rg in range(nr) for kg in range(nk)}

    def buf(g):
        return ((g // S) & 1) if phase_buffers == 2 else 0

    if mode.startswith("batch"):
        phase_buffers = 1
        for g in range(min(S, stages)):
            in_flight.append((g % S, g))
        prod["g"] = stages  # no producer: the finishers refill

    def producer_step():
        g = prod["g"]
        if g >= stages:
            return False
        s, lap = g % S, g // S
        if lap > 0 and not empty[s].passed((lap - 1) & 1):
            return False
        in_flight.append((s, g))
        prod["g"] += 1
        return True

    def land_step():
        if not in_flight:
            return False
        i = rng.randrange(len(in_flight))
        s, g = in_flight.pop(i)
        slot[s] = g
        full[s].arrive()
        return True

    def warp_step(key):
        rg, kg = key
        w = warps[key]
        g = w["g"]
        if g >= stages:
            return False
        s, ph, kf = g % S, (g // S) & 1, (g // nr) % nk
        if w["step"] == 0:                      # wait for the slot, read it
            if not full[s].passed(ph):
                return False
            assert slot[s] == g, f"warp {key} read stage {slot[s]} in slot {s}, expected {g}"
            w["step"] = 1
            return True
        if w["step"] == 1:                      # partial, red_full (and empty)
            red[(buf(g), s, kg)] = g
            red_full[s].arrive()
            if mode == "chain" or (mode == "stream" and kg != kf):
                empty[s].arrive()
            w["step"] = 2 if kg == kf else 3
            return True
        if w["step"] == 2:                      # finisher: every K-group's partial
            if not red_full[s].passed(ph):
                return False
            if mode == "batch-early":
                if g + S < stages:
                    in_flight.append((s, g + S))  # refill first (the planted mistake)
                w["step"] = 4                   # ... and read in a later step
                return True
            w["step"] = 4
        if w["step"] == 4:
            for k in range(nk):
                got = red[(buf(g), s, k)]
                assert got == g, f"finisher of stage {g} read K-group {k}'s partial of stage {got}"
            if mode == "stream":
                empty[s].arrive()
            if mode == "batch" and g + S < stages:
                in_flight.append((s, g + S))    # the refill, after the read
            w["step"] = 3
            return True
        w["g"] = g + nr                         # next stage of this row-group
        w["step"] = 0
        return True

    actors = [producer_step, land_step] + [lambda k=k: warp_step(k) for k in warps]
    for _ in range(max_steps):
        if prod["g"] >= stages and not in_flight and all(w["g"] >= stages for w in warps.values()):
            return
        order = actors[:]
        rng.shuffle(order)
        if not any(a() for a in order):
            raise AssertionError("deadlock")
    raise AssertionError("did not finish")


@pytest.mark.parametrize("mode", ["chain", "stream", "batch"])
@pytest.mark.parametrize("S,nr,nk", [(4, 4, 4), (8, 4, 4), (16, 4, 4), (2, 1, 16), (8, 2, 8), (6, 2, 8),
                                     (32, 8, 2)])
def test_ring_protocol_under_random_interleavings(S, nr, nk, mode):
    stages = 5 * S + 3
    for seed in range(40):
        run(S, nr, nk, stages, seed, mode=mode)


def test_single_partials_buffer_is_caught():
    """With the slot released before the reduction, one partials buffer per
    slot lets the next use of the slot overwrite partials the finisher has not
    read yet: the model must find such an interleaving."""
    caught = 0
    for seed in range(300):
        try:
            run(4, 4, 4, 40, seed, phase_buffers=1)
        except AssertionError as e:
            assert "partial" in str(e)
            caught += 1
    assert caught > 0


def test_ring_not_a_multiple_of_row_groups_is_caught():
    """The planner keeps S a multiple of nr so that each slot serves one
    row-group, whose warps visit it in order. With S = 6 and nr = 4 a slot
    passes between row-groups, and a parity wait can pass on an older phase:
    the model must see a stale read or a deadlock."""
    caught = 0
    for seed in range(200):
        try:
            run(6, 4, 2, 40, seed)
        except AssertionError:
            caught += 1
    assert caught > 0


def test_batch_refill_before_reading_the_partials_is_caught():
    """The batched kernel's first version refilled the slot before its
    finisher had read the partials, and lost parity at M = 4: the next stage
    in the slot wrote over them. The model must find that interleaving."""
    caught = 0
    for seed in range(300):
        try:
            run(4, 4, 4, 40, seed, mode="batch-early")
        except AssertionError as e:
            assert "partial" in str(e)
            caught += 1
    assert caught > 0


def _cta_rows(b, G, N):
    r0 = (b * N) // G
    return r0, ((b + 1) * N) // G - r0


@pytest.mark.parametrize("S,nr,nk,RS", [(4, 4, 4, 8), (8, 4, 4, 5), (16, 4, 4, 2), (2, 1, 16, 8),
                                        (6, 2, 8, 8), (32, 8, 2, 1)])
def test_incremental_stage_walk_matches_the_closed_forms(S, nr, nk, RS):
    """Each consumer warp of the chain walks its row-group's global stages
    rg, rg + nr, ... through all problems, advancing slot, ring phase and
    finisher incrementally (no divisions per problem). Over random problem
    lists (CTAs with no rows of some problems included) the walk must visit
    exactly the stages g = rg mod nr of every problem, with slot g mod S,
    phase (g / S) mod 2 and finisher (g / nr) mod nk."""
    rng = random.Random(S * 100 + nr * 10 + RS)
    G = 152
    for _ in range(20):
        Ns = [rng.choice([0, 1, 5, 100, 151, 152, 153, 4096, 11008]) for _ in range(rng.randint(1, 12))]
        for b in (0, 1, 75, 151):
            nsts = [(_cta_rows(b, G, N)[1] + RS - 1) // RS for N in Ns]
            visited = set()
            for rg in range(nr):
                gw, s, ph, kf, g0 = rg, rg, 0, 0, 0
                for j, nst in enumerate(nsts):
                    st = gw - g0
                    assert 0 <= st < nr  # the warp's next stage is in this problem's first nr
                    while st < nst:
                        g = g0 + st
                        assert (s, ph, kf) == (g % S, (g // S) & 1, (g // nr) % nk)
                        assert g % nr == rg
                        visited.add((j, st))
                        s += nr
                        if s >= S:
                            s -= S
                            ph ^= 1
                        kf = kf + 1 if kf + 1 < nk else 0
                        gw += nr
                        st += nr
                    g0 += nst
            assert visited == {(j, st) for j, nst in enumerate(nsts) for st in range(nst)}
