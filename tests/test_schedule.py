"""The schedule builder and its safety gate (host only).

* Every real lowering (five workloads, several CTA counts and knobs) is
  accepted, covers every row of every matrix exactly once per layer and
  balances the bytes each CTA streams.
* Adversarial schedules made by mutating real ones: the validator never
  accepts one that the brute-force ground truth (tests/schedule_model.py)
  finds unsafe.  The mutations follow the failure classes the AMK safety
  gate is meant to catch: cycles, thresholds outside [1, #producers],
  dropped producers, consumers queued before producers, unjoined
  multi-producer counters, unordered writers, unreachable outputs and
  dangling ids.
"""
import random

import pytest

from workload import configs as wc

from . import schedule_model as sm


@pytest.fixture(scope="module")
def amk():
    from decode_megakernel_gb300 import build
    build.build()
    from decode_megakernel_gb300 import amk as m
    return m


def lowered(amk, model, max_seq, **knobs):
    cfg = amk.make_config(model, max_seq)
    return amk.amk_build_schedule(cfg, amk.make_schedule_config(**knobs))


REAL = [("tiny", [1, 2, 7, 152]), ("llama1b", [61, 152]),
        ("llama8b-bf16", [152]), ("llama8b-int8", [152]), ("llama8b-int4", [132])]


@pytest.mark.parametrize("name,ctas", REAL)
def test_real_lowerings_accepted(amk, name, ctas):
    w = wc.workload(name)
    for n in ctas:
        blob = lowered(amk, w.model, w.max_seq, num_ctas=n)
        st, rep = amk.amk_validate_serialized(blob)
        assert st == amk.AMK_OK, rep


@pytest.mark.parametrize("knobs", [dict(num_ctas=19, attn_splits=3, max_rows_per_task=16),
                                   dict(num_ctas=152, attn_splits=1),
                                   dict(num_ctas=64, attn_splits=200, max_rows_per_task=100)])
def test_knob_lowerings_accepted(amk, knobs):
    for model in (wc.TINY, wc.with_format(wc.TINY, "int8")):
        st, rep = amk.amk_validate_serialized(lowered(amk, model, 40, **knobs))
        assert st == amk.AMK_OK, rep


def test_lowering_structure_8b(amk):
    """Rows covered once per layer; per-CTA streamed bytes balanced."""
    m = wc.LLAMA_8B_BF16
    s = sm.parse(lowered(amk, m, 2176, num_ctas=152))
    T_QKV, T_O, T_GU, T_DOWN, T_LM = 0, 2, 3, 4, 5
    # row block sizes (bf16, Kt = 2048 -> 4 rows of 2048 per 16 KB tile)
    rows = {T_QKV: 6144, T_O: 4096, T_GU: 28672, T_DOWN: 4096, T_LM: 128256}
    rt = 4
    for typ, nrows in rows.items():
        layers = range(m.n_layers) if typ != T_LM else [m.n_layers - 1]
        for l in layers:
            cov = [0] * (nrows // rt)
            for t in s.tasks:
                if t.type == typ and t.layer == l:
                    for rb in range(t.a[0], t.a[1]):
                        cov[rb] += 1
            assert set(cov) == {1}, (typ, l)
    # bytes per CTA over the whole step: every GEMV task streams (a1 - a0) row blocks
    rb_bytes = {T_QKV: 2 * 16384, T_O: 2 * 16384, T_GU: 2 * 16384, T_DOWN: 7 * 16384,
                T_LM: 2 * 16384}
    per = [0] * 152
    for t in s.tasks:
        if t.type in rb_bytes:
            per[t.queue] += (t.a[1] - t.a[0]) * rb_bytes[t.type]
    assert max(per) / min(per) < 1.01
    # one attention task per (kv head, split), one combine per kv head and layer
    assert sum(t.type == 1 for t in s.tasks) == m.n_layers * 8 * 19
    assert sum(t.type == 6 for t in s.tasks) == m.n_layers * 8


def test_ground_truth_agrees_on_real_lowerings(amk):
    s = sm.parse(lowered(amk, wc.TINY, 24, num_ctas=3))
    ok, why = sm.truth(s)
    assert ok, why
    # and the Python round trip is lossless
    assert sm.serialize(s) == lowered(amk, wc.TINY, 24, num_ctas=3)


# ------------------------------------------------------------ adversarial

def _rand_task(s, rng, pred=lambda t: True):
    ids = [i for i, t in enumerate(s.tasks) if pred(t)]
    return rng.choice(ids) if ids else None


def mutate(s, rng):
    """One structural mutation; returns its name."""
    kind = rng.randrange(14)
    T = len(s.tasks)
    if kind == 0:   # cycle: an early task waits on the last counter
        t = _rand_task(s, rng, lambda t: t.queue >= 0)
        c = max(range(len(s.counters)), key=lambda c: max(
            (i for i, x in enumerate(s.tasks) if x.signal == c), default=-1))
        s.tasks[t].waits = [(c, s.counters[c][0])]
        return "cycle"
    if kind == 1:   # threshold 0 or above #producers
        t = _rand_task(s, rng, lambda t: bool(t.waits))
        c, th = s.tasks[t].waits[0]
        s.tasks[t].waits[0] = (c, rng.choice([0, s.counters[c][0] + 1, -3]))
        return "threshold"
    if kind == 2:   # drop a producer, keep the counter consistent
        t = _rand_task(s, rng, lambda t: t.signal >= 0 and t.queue >= 0)
        c = s.tasks[t].signal
        s.tasks[t].signal = -1
        s.counters[c][0] -= 1
        for x in s.tasks:
            x.waits = [(cc, min(th, s.counters[cc][0])) for cc, th in x.waits]
        return "drop-producer"
    if kind == 3:   # drop a producer, inconsistent count
        t = _rand_task(s, rng, lambda t: t.signal >= 0)
        s.tasks[t].signal = -1
        return "dangling-producer"
    if kind == 4:   # consumer before its producer in one queue: swap neighbours
        q = rng.randrange(len(s.queues))
        if len(s.queues[q]) >= 2:
            i = rng.randrange(len(s.queues[q]) - 1)
            s.queues[q][i], s.queues[q][i + 1] = s.queues[q][i + 1], s.queues[q][i]
        return "swap"
    if kind == 5:   # unjoined multi-producer counter: threshold below #producers
        t = _rand_task(s, rng, lambda t: bool(t.waits) and s.counters[t.waits[0][0]][0] > 1)
        if t is not None:
            c, th = s.tasks[t].waits[0]
            s.tasks[t].waits[0] = (c, rng.randrange(1, th))
        return "partial-wait"
    if kind == 6:   # remove a wait
        t = _rand_task(s, rng, lambda t: bool(t.waits))
        s.tasks[t].waits = []
        return "no-wait"
    if kind == 7:   # widen a write so that two writers overlap
        t = _rand_task(s, rng, lambda t: any(a[3] for a in t.acc))
        acc = list(s.tasks[t].acc)
        j = rng.choice([k for k, a in enumerate(acc) if a[3]])
        b, lo, hi, w = acc[j]
        acc[j] = (b, max(0, lo - rng.randrange(1, 64)), min(s.buffers[b][0], hi + rng.randrange(1, 64)), w)
        s.tasks[t].acc = acc
        return "overlap"
    if kind == 8:   # unreachable output: drop the writes of one LM-head task
        t = _rand_task(s, rng, lambda t: t.type == 5)
        s.tasks[t].acc = [a for a in s.tasks[t].acc if not a[3]] + [(0, 0, 1, 0)]
        return "uncovered-output"
    if kind == 9:   # dangling ids
        t = rng.randrange(T)
        which = rng.randrange(3)
        if which == 0:
            s.tasks[t].signal = len(s.counters) + 5
        elif which == 1 and s.tasks[t].acc:
            b, lo, hi, w = s.tasks[t].acc[0]
            s.tasks[t].acc[0] = (len(s.buffers) + 1, lo, hi, w)
        else:
            s.queues[rng.randrange(len(s.queues))].append(T + 3)
        return "dangling-id"
    if kind == 10:  # move a task to the front of another queue
        t = _rand_task(s, rng, lambda t: t.queue >= 0)
        q0 = s.tasks[t].queue
        q1 = rng.randrange(len(s.queues))
        s.queues[q0].remove(t)
        s.body[q0] = min(s.body[q0], len(s.queues[q0]))
        s.queues[q1].insert(rng.randrange(len(s.queues[q1]) + 1), t)
        s.tasks[t].queue = q1
        s.body[q1] = min(s.body[q1] + 1, len(s.queues[q1]))
        return "move"
    if kind == 11:  # a completion task that waits, or loses its trigger
        t = _rand_task(s, rng, lambda t: t.queue == -1)
        if t is not None:
            if rng.random() < 0.5:
                s.tasks[t].waits = [(0, 1)]
            else:
                for c in s.counters:
                    if c[1] == t:
                        c[1] = -1
        return "completion"
    if kind == 12:  # prefill body that needs the LM head, or a body cut short
        q = rng.randrange(len(s.queues))
        s.body[q] = rng.randrange(len(s.queues[q]) + 2)
        return "body"
    # random field tweak
    t = rng.randrange(T)
    if s.tasks[t].waits:
        c, th = s.tasks[t].waits[0]
        s.tasks[t].waits[0] = (rng.randrange(len(s.counters)), th)
    return "retarget"


def test_adversarial_no_false_accepts(amk):
    rng = random.Random(1234)
    bases = [sm.parse(lowered(amk, m, 20, num_ctas=n))
             for m in (wc.TINY, wc.with_format(wc.TINY, "int8"))
             for n in (2, 3, 4)]
    stats = {"unsafe": 0, "safe": 0, "rejected_safe": 0}
    for i in range(1500):
        s = sm.clone(rng.choice(bases))
        names = [mutate(s, rng) for _ in range(rng.choice([1, 1, 2, 3]))]
        st, rep = amk.amk_validate_serialized(sm.serialize(s))
        ok, why = sm.truth(s)
        if ok:
            stats["safe"] += 1
            stats["rejected_safe"] += int(st != amk.AMK_OK)
        else:
            stats["unsafe"] += 1
            assert st != amk.AMK_OK, f"false accept after {names}: truth says {why}"
    print(stats)
    assert stats["unsafe"] > 1000
