"""The schedule builder and its safety gate (host only).

* Every real lowering (five workloads, several CTA counts and knobs) is
  accepted, covers every row of every matrix exactly once per layer and
  balances the bytes each CTA streams.
* Adversarial schedules made by mutating real ones: the validator never
  accepts one that the brute-force ground truth (tests/schedule_model.py)
  finds unsafe.  The mutations follow the failure classes the AMK safety
  gate is meant to catch, restated for version-tagged data: cycles
  (waiting for a later version), unsatisfiable waits (a version nobody
  writes), dropped or duplicated producers, consumers queued before their
  producers, readers that may find the next version already written,
  unordered writers, unreachable outputs and dangling ids.
"""
import random

import numpy as np
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
    """Rows covered once per layer; per-CTA streamed bytes balanced; every
    tagged word written once per version."""
    m = wc.LLAMA_8B_BF16
    s = sm.parse(lowered(amk, m, 2176, num_ctas=152))
    T_QKV, T_ATTN, T_O, T_GU, T_DOWN, T_LM, T_COMB = 0, 1, 2, 3, 4, 5, 6
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
    # one attention task per (kv head, split), one merge per query head and layer
    assert sum(t.type == T_ATTN for t in s.tasks) == m.n_layers * 8 * 19
    assert sum(t.type == T_COMB for t in s.tasks) == m.n_layers * 32
    assert s.versions == m.n_layers
    # tagged buffers: each version written exactly once per element
    for b, (size, kind) in enumerate(s.buffers):
        if kind != sm.TAGGED:
            continue
        for v in range(1, s.versions + 1):
            cnt = np.zeros(size, dtype=np.int64)
            for t in s.tasks:
                for bb, lo, hi, wr, ver in t.acc:
                    if bb == b and wr and ver == v:
                        cnt[lo:hi] += 1
            assert (cnt == 1).all(), (b, v)


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


def _tagged(s, a):
    return 0 <= a[0] < len(s.buffers) and s.buffers[a[0]][1] == sm.TAGGED


def _pick_access(s, rng, write):
    cand = [(i, j) for i, t in enumerate(s.tasks) for j, a in enumerate(t.acc)
            if bool(a[3]) == write and _tagged(s, a)]
    return rng.choice(cand) if cand else (None, None)


def mutate(s, rng):
    """One structural mutation; returns its name."""
    kind = rng.randrange(15)
    T = len(s.tasks)
    if kind == 0:   # cycle: an early reader waits for a later version
        i, j = _pick_access(s, rng, write=False)
        if i is not None:
            b, lo, hi, wr, v = s.tasks[i].acc[j]
            s.tasks[i].acc[j] = (b, lo, hi, wr, min(s.versions, v + rng.randrange(1, 3)))
        return "later-version"
    if kind == 1:   # stale read: wait for an older version
        i, j = _pick_access(s, rng, write=False)
        if i is not None:
            b, lo, hi, wr, v = s.tasks[i].acc[j]
            s.tasks[i].acc[j] = (b, lo, hi, wr, max(1, v - 1))
        return "older-version"
    if kind == 2:   # drop a write: some version of some element is never written
        i, j = _pick_access(s, rng, write=True)
        if i is not None and len(s.tasks[i].acc) > 1:
            del s.tasks[i].acc[j]
        return "drop-write"
    if kind == 3:   # a writer writes the wrong version
        i, j = _pick_access(s, rng, write=True)
        if i is not None:
            b, lo, hi, wr, v = s.tasks[i].acc[j]
            s.tasks[i].acc[j] = (b, lo, hi, wr, rng.choice([max(1, v - 1), min(s.versions, v + 1)]))
        return "write-version"
    if kind == 4:   # consumer before its producer in one queue: swap neighbours
        q = rng.randrange(len(s.queues))
        if len(s.queues[q]) >= 2:
            i = rng.randrange(len(s.queues[q]) - 1)
            s.queues[q][i], s.queues[q][i + 1] = s.queues[q][i + 1], s.queues[q][i]
        return "swap"
    if kind == 5:   # duplicate writer: copy a write into another task
        i, j = _pick_access(s, rng, write=True)
        t2 = rng.randrange(T)
        if i is not None:
            s.tasks[t2].acc.append(s.tasks[i].acc[j])
        return "duplicate-write"
    if kind == 6:   # remove a read (the task no longer waits, keeps running early)
        i, j = _pick_access(s, rng, write=False)
        if i is not None:
            del s.tasks[i].acc[j]
        return "drop-read"
    if kind == 7:   # widen a write so that two writers overlap
        i, j = _pick_access(s, rng, write=True)
        if i is not None:
            b, lo, hi, wr, v = s.tasks[i].acc[j]
            s.tasks[i].acc[j] = (b, max(0, lo - rng.randrange(1, 64)),
                                 min(s.buffers[b][0], hi + rng.randrange(1, 64)), wr, v)
        return "overlap"
    if kind == 8:   # unreachable output: drop the writes of one LM-head task
        t = _rand_task(s, rng, lambda t: t.type == 5)
        if t is not None:
            s.tasks[t].acc = [a for a in s.tasks[t].acc if not a[3]] + [(0, 0, 1, 1, s.versions)]
        return "uncovered-output"
    if kind == 9:   # dangling ids
        t = rng.randrange(T)
        which = rng.randrange(3)
        if which == 0:
            s.tasks[t].queue = len(s.queues) + 2
        elif which == 1 and s.tasks[t].acc:
            b, lo, hi, wr, v = s.tasks[t].acc[0]
            s.tasks[t].acc[0] = (len(s.buffers) + 1, lo, hi, wr, v)
        else:
            s.queues[rng.randrange(len(s.queues))].append(T + 3)
        return "dangling-id"
    if kind == 10:  # move a task to another queue position
        t = rng.randrange(T)
        q0 = s.tasks[t].queue
        q1 = rng.randrange(len(s.queues))
        s.queues[q0].remove(t)
        s.body[q0] = min(s.body[q0], len(s.queues[q0]))
        s.queues[q1].insert(rng.randrange(len(s.queues[q1]) + 1), t)
        s.tasks[t].queue = q1
        s.body[q1] = min(s.body[q1] + 1, len(s.queues[q1]))
        return "move"
    if kind == 11:  # retarget a read to another tagged buffer's range
        i, j = _pick_access(s, rng, write=False)
        if i is not None:
            b, lo, hi, wr, v = s.tasks[i].acc[j]
            b2 = rng.choice([k for k, x in enumerate(s.buffers) if x[1] == sm.TAGGED])
            size = s.buffers[b2][0]
            lo2 = rng.randrange(size)
            s.tasks[i].acc[j] = (b2, lo2, min(size, lo2 + (hi - lo)), wr, v)
        return "retarget"
    if kind == 12:  # prefill body cut short or extended
        q = rng.randrange(len(s.queues))
        s.body[q] = rng.randrange(len(s.queues[q]) + 2)
        return "body"
    if kind == 13:  # version bookkeeping
        s.versions = rng.choice([0, s.versions - 1, s.versions + 1, 200])
        return "versions"
    # shrink a write (a hole in some version)
    i, j = _pick_access(s, rng, write=True)
    if i is not None:
        b, lo, hi, wr, v = s.tasks[i].acc[j]
        if hi - lo > 1:
            s.tasks[i].acc[j] = (b, lo + 1, hi, wr, v)
    return "shrink-write"


def test_adversarial_no_false_accepts(amk):
    rng = random.Random(1234)
    bases = [sm.parse(lowered(amk, m, 20, num_ctas=n, attn_splits=sp))
             for m in (wc.TINY, wc.with_format(wc.TINY, "int8"))
             for n, sp in ((2, 0), (3, 2), (4, 0))]
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


def _alias_case(reader_first: bool):
    """A 1-element tagged buffer written at versions 1..20 by a chain of
    tasks on queue 0, and a reader of version 20.  Alone on queue 1, the
    reader may start while the word still holds version 0 (the previous
    step's last), 20 versions behind: with 4-bit tags that aliases.  Queued
    after the writer of version 20, it finds at worst version 19."""
    V = 20
    bufs = [(1, sm.TAGGED), (1, sm.OUTPUT), (1, sm.OUTPUT)]
    tasks = [sm.Task(0, 0, 0, acc=[(0, 0, 1, 1, v)]) for v in range(1, V + 1)]
    r = sm.Task(0, 0, 1 if reader_first else 0, acc=[(0, 0, 1, 0, V), (1, 0, 1, 1, 0)])
    other = sm.Task(0, 0, 1, acc=[(2, 0, 1, 1, 0)])
    tasks += [r, other]
    if reader_first:
        queues = [list(range(V)), [V, V + 1]]
    else:
        queues = [list(range(V + 1)), [V + 1]]
    return sm.Schedule(bufs, tasks, queues, [len(q) for q in queues], V)


@pytest.mark.parametrize("reader_first", [True, False])
def test_tag_alias_gate(amk, reader_first):
    s = _alias_case(reader_first)
    ok, why = sm.truth(s)
    st, rep = amk.amk_validate_serialized(sm.serialize(s))
    assert ok == (not reader_first), why
    assert (st == amk.AMK_OK) == ok, rep
    if reader_first:
        assert "alias" in rep and "alias" in why


# --------------------------------------------------- re-queued lowerings

@pytest.mark.parametrize("knobs", [dict(num_ctas=8), dict(num_ctas=37, attn_splits=5, max_rows_per_task=32)])
def test_requeued_lowerings(amk, knobs):
    """amk_validate_requeued (the gate of amk_load_weights_requeued): the
    library's own lowering and placement-only edits of it pass; an edit
    whose queue order deadlocks, a task that is not the lowering's, a lost
    or duplicated task and an LM-head task inside a body are refused."""
    from decode_megakernel_gb300 import schedule_ir as ir
    from decode_megakernel_gb300 import tune
    c = amk.make_config(wc.TINY, 48)
    sched = amk.make_schedule_config(**knobs)
    blob = amk.amk_build_schedule(c, sched)
    s = ir.parse(blob)
    assert ir.serialize(s) == blob
    assert amk.amk_validate_requeued(c, sched, blob)[0] == amk.AMK_OK
    for edit in ("rotate_queues:1", "rotate_queues:3", "spread_combines:1", "spread_combines:2"):
        st, rep = amk.amk_validate_requeued(c, sched, tune.apply_edit(blob, edit))
        assert st == amk.AMK_OK, (edit, rep)
    st, rep = amk.amk_validate_requeued(c, sched, tune.apply_edit(blob, "hoist_next_layer"))
    assert st == amk.AMK_ERR_SCHEDULE_INVALID and "cycle" in rep
    foreign = ir.parse(blob)
    foreign.tasks[0].params[0] += 1
    assert amk.amk_validate_requeued(c, sched, ir.serialize(foreign))[0] == amk.AMK_ERR_SCHEDULE_INVALID
    lost = ir.parse(blob)
    q = next(i for i, items in enumerate(lost.queues) if len(items) > 1)
    lost.queues[q].pop(0)
    lost.body[q] -= 1
    st, rep = amk.amk_validate_requeued(c, sched, ir.serialize(lost))
    assert st == amk.AMK_ERR_SCHEDULE_INVALID and "no queue" in rep
    dup = ir.parse(blob)
    dup.queues[q].insert(0, dup.queues[q][0])
    dup.body[q] += 1
    assert amk.amk_validate_requeued(c, sched, ir.serialize(dup))[0] == amk.AMK_ERR_SCHEDULE_INVALID
    lm_in_body = ir.parse(blob)
    q = next(i for i, items in enumerate(lm_in_body.queues)
             if any(lm_in_body.tasks[t].type == ir.T_LMHEAD for t in items))
    lm_in_body.body[q] = len(lm_in_body.queues[q])
    st, rep = amk.amk_validate_requeued(c, sched, ir.serialize(lm_in_body))
    assert st == amk.AMK_ERR_SCHEDULE_INVALID and "LM-head" in rep
    assert amk.amk_validate_requeued(c, sched, b"\x00" * 16)[0] == amk.AMK_ERR_SCHEDULE_INVALID
