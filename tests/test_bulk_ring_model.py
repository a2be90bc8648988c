"""CPU model of the shared-memory ring of the bulk-fed capped sync
(csrc/fsdp_bulk.cu): its protocol, not its arithmetic.

A producer fills chunk q into stage q % nst and record q % (nst + 2) after
the stage's previous chunk was released; one or two groups of folding warps
take alternate chunks, wait on the stage's "full" barrier with a parity
wait, read the chunk's record, release the stage's data slot, then store
using the record. A stage's copies land some time after the producer's
arrival, in any order across stages.

An mbarrier parity wait only tells the current phase from the one before
it: it returns at once when the barrier is one phase *behind* the one the
waiter wants. The model checks, over random schedules, that no group ever
passes a wait before its chunk has landed and that no record is rewritten
while a group may still read it, for every stage count the kernel uses (a
multiple of the group count, so a stage always serves the same group), and
that an odd stage count with two groups breaks the first property (the
fault the kernel's rule prevents)."""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.completed = 0  # phases completed so far

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def test_wait(self, parity):
        # true iff the phase of this parity has completed, i.e. the current
        # (incomplete) phase has the other parity
        return (self.completed & 1) != parity


def run_ring(nst, groups, nchunks, seed):
    rnd = random.Random(seed)
    full = [Barrier(1) for _ in range(nst)]
    empty = [Barrier(1) for _ in range(nst)]  # one group's release counts once here
    nrec = nst + 2
    records = [None] * nrec
    landed = {}
    in_flight = []  # (chunk, stage): arrived, copies not landed yet
    readers = {}  # record -> chunk a group may still read it for
    prod = {"q": 0, "stage": 0, "ph": 0, "rec": 0}
    cons = [{"q": g, "stage": g, "ph": 0, "rec": g, "state": "wait"} for g in range(groups)]
    for _ in range(10 ** 6):
        actors = (["P"] if prod["q"] < nchunks else []) + (["L"] if in_flight else []) + \
            [g for g in range(groups) if cons[g]["q"] < nchunks]
        if not actors:
            return
        a = rnd.choice(actors)
        if a == "L":
            q, s = in_flight.pop(rnd.randrange(len(in_flight)))
            full[s].arrive()
            landed[q] = s
        elif a == "P":
            s = prod["stage"]
            if not empty[s].test_wait(prod["ph"] ^ 1):
                continue
            r = prod["rec"]
            assert r not in readers, f"record {r} rewritten while chunk {readers[r]} may read it"
            records[r] = prod["q"]
            in_flight.append((prod["q"], s))
            prod["q"] += 1
            prod["rec"] = (r + 1) % nrec
            prod["stage"] += 1
            if prod["stage"] == nst:
                prod["stage"], prod["ph"] = 0, prod["ph"] ^ 1
        else:
            c = cons[a]
            if c["state"] == "wait":
                if not full[c["stage"]].test_wait(c["ph"]):
                    continue
                assert landed.get(c["q"]) == c["stage"], f"group {a} passed the wait of chunk {c['q']} early"
                assert records[c["rec"]] == c["q"]
                readers[c["rec"]] = c["q"]
                c["state"] = "release"
            elif c["state"] == "release":  # data slot read: release it
                empty[c["stage"]].arrive()
                c["stage"] += groups
                if c["stage"] >= nst:
                    c["stage"] -= nst
                    c["ph"] ^= 1
                c["state"] = "store"
            else:  # stores done: the record is free
                del readers[c["rec"]]
                c["rec"] = (c["rec"] + groups) % nrec
                c["q"] += groups
                c["state"] = "wait"
    raise AssertionError("no progress")


@pytest.mark.parametrize("groups", [1, 2])
def test_ring_protocol_holds_for_the_kernels_stage_counts(groups):
    for nst in range(2, 25):
        if nst % groups:
            continue
        for seed in range(60):
            run_ring(nst, groups, 40, seed)


def test_odd_ring_with_two_groups_is_caught():
    with pytest.raises(AssertionError, match="passed the wait"):
        for seed in range(400):
            run_ring(3, 2, 60, seed)
