"""The serialised task schedule (amk_build_schedule) as Python data, and the
structural edits the schedule search proposes.

A schedule lists tasks (type, layer, parameters, the queue of the CTA that
runs it, its memory accesses) and per queue the order of its tasks and the
length of its body (the part a prefill step runs, without the LM head).
The edits here change only placement: which CTA runs a task and in which
order.  They may produce schedules that deadlock; the library's safety gate
(amk_validate_requeued) decides, before anything is launched.  The format is
documented in csrc/schedule.hpp; this module only moves words around.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MAGIC = 0x414D4B53
FORMAT = 2
T_QKV, T_ATTN, T_OPROJ, T_GATEUP, T_DOWN, T_LMHEAD, T_COMBINE = range(7)


@dataclass
class Task:
    type: int
    layer: int
    queue: int
    params: list
    acc: list = field(default_factory=list)   # [(buffer, lo, hi, write, version)]


@dataclass
class Schedule:
    buffers: list
    tasks: list
    queues: list      # per queue: task ids in order
    body: list        # per queue: body length
    versions: int


def parse(blob: bytes) -> Schedule:
    w = np.frombuffer(blob, dtype=np.int64)
    if len(w) < 8 or w[0] != MAGIC or w[1] != FORMAT:
        raise ValueError("not a serialised schedule")
    nt, nq, nb, na, ni, nv = (int(x) for x in w[2:8])
    p = 8
    buffers = [(int(w[p + 2 * i]), int(w[p + 2 * i + 1])) for i in range(nb)]
    p += 2 * nb
    rows = w[p:p + 9 * nt].reshape(nt, 9)
    p += 9 * nt
    accs = w[p:p + 5 * na].reshape(na, 5)
    p += 5 * na
    qrows = w[p:p + 3 * nq].reshape(nq, 3)
    p += 3 * nq
    items = w[p:p + ni]
    tasks = [Task(int(r[0]), int(r[1]), int(r[2]), [int(x) for x in r[5:9]],
                  [tuple(int(v) for v in a) for a in accs[r[3]:r[3] + r[4]]]) for r in rows]
    queues = [[int(x) for x in items[q[0]:q[0] + q[1]]] for q in qrows]
    return Schedule(buffers, tasks, queues, [int(q[2]) for q in qrows], nv)


def serialize(s: Schedule) -> bytes:
    out = [MAGIC, FORMAT, len(s.tasks), len(s.queues), len(s.buffers),
           sum(len(t.acc) for t in s.tasks), sum(len(q) for q in s.queues), s.versions]
    for b in s.buffers:
        out += list(b)
    ab = 0
    for t in s.tasks:
        out += [t.type, t.layer, t.queue, ab, len(t.acc)] + list(t.params)
        ab += len(t.acc)
    for t in s.tasks:
        for a in t.acc:
            out += list(a)
    ib = 0
    for q, b in zip(s.queues, s.body):
        out += [ib, len(q), b]
        ib += len(q)
    for q in s.queues:
        out += q
    return np.array(out, dtype=np.int64).tobytes()


def _requeue(s: Schedule, queues: list) -> Schedule:
    """A copy of s with new queue contents (task ids per queue); bodies
    recounted as the non-LM prefix of each queue."""
    tasks = [Task(t.type, t.layer, t.queue, list(t.params), list(t.acc)) for t in s.tasks]
    body = []
    for q, items in enumerate(queues):
        for i in items:
            tasks[i].queue = q
        body.append(sum(1 for i in items if tasks[i].type != T_LMHEAD))
    return Schedule(list(s.buffers), tasks, [list(q) for q in queues], body, s.versions)


def rotate_queues(s: Schedule, k: int) -> Schedule:
    """Queue q's tasks run on CTA (q + k) mod C: another SM assignment of
    the same per-CTA work."""
    C = len(s.queues)
    queues = [None] * C
    for q in range(C):
        queues[(q + k) % C] = list(s.queues[q])
    return _requeue(s, queues)


def spread_combines(s: Schedule, stride: int) -> Schedule:
    """Each split-merge task moves to the end of the attention tasks of the
    queue `stride` CTAs further on (the same layer's merge, run by another
    CTA)."""
    C = len(s.queues)
    queues = [list(q) for q in s.queues]
    moved = [(q, i) for q in range(C) for i in queues[q] if s.tasks[i].type == T_COMBINE]
    for q, i in moved:
        queues[q].remove(i)
    for q, i in moved:
        dst = (q + stride) % C
        layer = s.tasks[i].layer
        # after the last attention task of that layer in the destination queue
        pos = 0
        for j, t in enumerate(queues[dst]):
            tk = s.tasks[t]
            if tk.layer < layer or (tk.layer == layer and tk.type in (T_QKV, T_ATTN, T_COMBINE)):
                pos = j + 1
            else:
                break
        queues[dst].insert(pos, i)
    return _requeue(s, queues)


def hoist_next_layer(s: Schedule) -> Schedule:
    """Moves the first layer-1 task of a queue that also runs a layer-0 down
    projection to the front of that queue, ahead of layer-0 work whose
    outputs it reads: an edit the safety gate must reject (the queue order
    and the data dependence form a cycle)."""
    queues = [list(q) for q in s.queues]
    queue = next(q for q, items in enumerate(queues)
                 if any(s.tasks[i].layer == 0 and s.tasks[i].type == T_DOWN for i in items)
                 and any(s.tasks[i].layer == 1 and s.tasks[i].type != T_LMHEAD for i in items))
    items = queues[queue]
    first = next(i for i in items if s.tasks[i].layer == 1 and s.tasks[i].type != T_LMHEAD)
    items.remove(first)
    items.insert(0, first)
    return _requeue(s, queues)
