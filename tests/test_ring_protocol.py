"""A model of the shared-memory ring that feeds the persistent decode kernels
(kda_decode_stream_kernel, kda_decode_packed_kernel, kda_decode_tokens_kernel
and kda_decode_tokens_wy_kernel), run on the CPU.

The protocol, as the kernels implement it: a CTA's local heads j = 0, 1, ...
go to consumer group j % G in order; head j lives in stage j % NST as that
stage's use n = j // NST. Thread 0 fills stages 0 .. NST-1 at the start.
The consumer of head j waits on the stage's `issued` mbarrier for phase n - 1
(n > 0: the refill for use n was issued), then on its `full` mbarrier for
phase n (the bytes of use n landed), reads the stage, and after its group
barrier refills the stage with head j + NST and arrives on `issued`.

An mbarrier wait names a phase only by its parity: it returns once the
barrier's completed-phase count has a parity other than the one waited on.
So a wait for phase k is correct only if, whenever it runs, at most k + 1
phases have completed; two beyond would look like none. The model runs the
groups and the copy engine under many random schedules and checks that no
wait ever sees that aliasing, that every head reads the bytes of its own
fill, and that the ring never deadlocks, for the stage counts and group
counts the kernels use (NST 2-8, G 1, 2 and 4 with NST >= G) and ragged
head counts.
"""
import random

import pytest


class Barrier:
    """An mbarrier reduced to its completed-phase count."""

    def __init__(self):
        self.completed = 0

    def wait_ready(self, phase):
        # hardware: try_wait.parity(phase & 1) is true iff the current phase
        # parity differs from it, i.e. completed % 2 != phase % 2
        return self.completed % 2 != phase % 2


def run_ring(NST, G, K, rng):
    """One random schedule of a CTA with K local heads. Returns the head each
    consumer read, in head order; raises AssertionError on an aliased wait
    or a deadlock."""
    full = [Barrier() for _ in range(NST)]
    issued = [Barrier() for _ in range(NST)]
    stage_data = [None] * NST           # which head's bytes a stage holds
    in_flight = []                      # (stage, head) copies issued, not landed
    for s in range(min(NST, K)):        # initial fills (use 0 of each stage)
        in_flight.append((s, s))
    next_head = list(range(G))          # each group's next local head
    step = [0] * G                      # 0: waiting on issued, 1: waiting on full
    read = {}

    def land(idx):
        s, head = in_flight.pop(idx)
        stage_data[s] = head
        full[s].completed += 1

    for _ in range(100000):
        if all(h >= K for h in next_head) and not in_flight:
            return [read[j] for j in range(K)]
        actors = [("copy", i) for i in range(len(in_flight))]
        actors += [("group", g) for g in range(G) if next_head[g] < K]
        kind, who = rng.choice(actors)
        if kind == "copy":
            land(who)
            continue
        g, j = who, next_head[who]
        s, n = j % NST, j // NST
        if step[g] == 0:
            if n > 0:
                # the wait for issued phase n - 1 must not see phase n + 1 done
                assert issued[s].completed <= n, "issued wait aliased (head %d)" % j
                if not issued[s].wait_ready(n - 1):
                    continue
            step[g] = 1
            continue
        assert full[s].completed <= n + 1, "full wait aliased (head %d)" % j
        if not full[s].wait_ready(n):
            continue
        read[j] = stage_data[s]
        # group barrier, then thread 0 refills the stage with head j + NST
        if j + NST < K:
            in_flight.append((s, j + NST))
            issued[s].completed += 1
        next_head[g] += G
        step[g] = 0
    raise AssertionError("ring deadlocked: NST=%d G=%d K=%d" % (NST, G, K))


@pytest.mark.parametrize("NST", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_ring_reads_every_head_once_without_aliasing(NST, G):
    if G == 4 and NST % G:
        pytest.skip("four groups run with a multiple of four stages (see the next test)")
    rng = random.Random(1000 * NST + G)
    for K in [1, 2, NST - 1, NST, NST + 1, 2 * NST + 1, 3 * NST + G, 37]:
        if K < 1:
            continue
        for _ in range(60):
            assert run_ring(NST, G, K, rng) == list(range(K))


def test_model_catches_a_ring_too_shallow_for_its_waits():
    """The check has teeth: a consumer that refills before it has read (the
    refill issued ahead of the group barrier, modelled as a stage that is
    overwritten early) reads another head's bytes in some schedule."""
    rng = random.Random(7)

    def run_early_refill(NST, K):
        full = [Barrier() for _ in range(NST)]
        stage_data = [None] * NST
        in_flight = [(s, s) for s in range(min(NST, K))]
        j, read, waiting = 0, [], True
        for _ in range(10000):
            if j >= K and not in_flight:
                return read
            acts = ["copy"] * len(in_flight) + (["c"] if j < K else [])
            a = rng.choice(acts)
            if a == "copy":
                s, h = in_flight.pop(rng.randrange(len(in_flight)))
                stage_data[s] = h
                full[s].completed += 1
                continue
            s, n = j % NST, j // NST
            if waiting:
                if not full[s].wait_ready(n):
                    continue
                waiting = False
                if j + NST < K:                      # refill first ...
                    in_flight.append((s, j + NST))
                continue
            read.append(stage_data[s])               # ... read afterwards
            j, waiting = j + 1, True
        return None

    bad = 0
    for _ in range(200):
        r = run_early_refill(2, 8)
        if r is not None and r != list(range(8)):
            bad += 1
    assert bad > 0


def test_four_groups_need_a_stage_count_that_is_a_multiple_of_four():
    """With four groups and five stages, head j + 5 belongs to another group
    than head j, whose consumer refills its stage; a group far enough ahead
    then waits on a parity two phases old and reads stale bytes. The packed
    kernel therefore rounds its stage count down to a multiple of the group
    count; this pins that the model sees the hazard."""
    rng = random.Random(7)
    failed = False
    for _ in range(300):
        try:
            if run_ring(5, 4, 37, rng) != list(range(37)):
                failed = True
        except AssertionError:
            failed = True
    assert failed
