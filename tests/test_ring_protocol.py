"""The decode kernel's ring protocol, modelled on the host.

One ring of R = 12 shared-memory slots carries a CTA's weight tiles and K,V
history stages in queue order.  Copy k goes to slot k mod R and completes
phase k div R of that slot's full barrier; its consumers release it by
completing the same phase of the slot's empty barrier.  The producer issues
copy k once copy k - R was released (its slot is free) and copy k - cap has
landed (at most cap copies in flight).  Consumers take the copies in order:
a GEMV task's tiles one row block at a time, in pairs within the row block
(both waits first, then both tiles, then both releases) or one by one (the
rolled int4 loop), an attention task's stages a chunk of up to four at a
time, released together at the chunk's end.

For random queues, landing delays and every cap from 1 to R, the model
checks that every run completes, that no copy is issued into a slot whose
previous copy was not yet released, that the copies in flight never exceed
the cap, and that the (slot, phase) each consumer waits on is the one the
producer filled with that copy.  It restates the kernel's arithmetic; it
shares no code with it.
"""
import random

import pytest

R = 12            # ring slots
CHUNK = 4         # K,V stages an attention chunk holds at once


def consumer_groups(rng):
    """A random queue as the consumers take it: a list of groups of copy
    counts; the copies of one group are waited for together and released
    together."""
    groups = []
    for _ in range(rng.randint(3, 12)):
        kind = rng.choice(["gemv_pairs", "gemv_single", "attn", "merge"])
        if kind == "merge":           # no ring copies
            continue
        if kind == "attn":
            stages = rng.randint(0, 30)
            while stages > 0:
                take = min(CHUNK, stages)
                groups.append(take)
                stages -= take
            continue
        nkt = rng.randint(1, 8)
        for _ in range(rng.randint(1, 5)):          # row blocks
            if kind == "gemv_single":
                groups.extend([1] * nkt)
            else:
                kt = 0
                while kt < nkt:
                    two = kt + 1 < nkt
                    groups.append(2 if two else 1)
                    kt += 2
    return groups


def run(groups, cap, rng):
    total = sum(groups)
    issued = 0
    landed = [False] * total
    released = [False] * total
    land_at = {}
    slot_copy = [None] * R            # copy currently held by each slot
    slot_uses = [0] * R               # copies each slot has held (its barrier phases)
    phase_of = [None] * total         # the phase copy k completes
    clock = 0
    g = 0                             # next consumer group
    first = 0                         # its first copy
    idle = 0
    while g < len(groups):
        clock += 1
        progress = False
        # copies land after a random delay
        for k, t in list(land_at.items()):
            if t <= clock:
                landed[k] = True
                del land_at[k]
                progress = True
        # the producer issues at most a few copies per tick
        for _ in range(rng.randint(0, 3)):
            k = issued
            if k >= total:
                break
            slot_free = k < R or released[k - R]
            cap_ok = k < cap or landed[k - cap]
            if not (slot_free and cap_ok):
                break
            s = k % R
            assert slot_copy[s] is None or released[slot_copy[s]], "slot overwritten before release"
            slot_copy[s] = k
            phase_of[k] = slot_uses[s] & 1
            slot_uses[s] += 1
            land_at[k] = clock + rng.randint(1, 6)
            issued += 1
            progress = True
            in_flight = sum(1 for j in range(issued) if not landed[j])
            assert in_flight <= cap, f"{in_flight} copies in flight above cap {cap}"
        # the consumers finish the current group once all its copies landed
        n = groups[g]
        if n == 0 or all(k < issued and landed[k] for k in range(first, first + n)):
            for k in range(first, first + n):
                # the consumer's (slot, phase) of copy k: (k mod R, (k div R) mod 2)
                assert slot_copy[k % R] == k, "consumer waits on a slot the copy is not in"
                assert phase_of[k] == (k // R) & 1, "consumer waits on the wrong phase"
                released[k] = True
            first += n
            g += 1
            progress = True
        idle = 0 if progress else idle + 1
        assert idle < 100, f"deadlock: copy {issued} of {total} issued, group {g} of {len(groups)}"
    assert issued == total and all(released)


@pytest.mark.parametrize("cap", list(range(1, R + 1)))
def test_ring_protocol_completes(cap):
    rng = random.Random(1000 + cap)
    for _ in range(40):
        run(consumer_groups(rng), cap, rng)


def test_a_chunk_fits_the_ring():
    """An attention chunk holds its stages together: the ring must hold a
    whole chunk plus the pair a GEMV consumer may hold before it."""
    assert CHUNK <= R and 2 <= R
