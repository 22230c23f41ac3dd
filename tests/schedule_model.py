"""Python view of the serialised schedule and an independent ground truth.

The ground truth decides safety by brute force, written separately from
the C++ validator: deadlock by running every queue to a fixpoint (counters
only grow, so greedy order does not matter), races by the happens-before
relation of "wait until any t of n producers signalled" (a task X is
guaranteed done before the consumer when X precedes, or is, at least
n - t + 1 of the n producers: any t finished producers then include one
that X precedes), and output coverage by marking every element.  A cycle
in the producer -> consumer graph is unsafe by definition (the gate
requires an acyclic DAG).  The safety conditions are the ones the AutoMegaKernel safety
gate names: acyclic/satisfiable waits with 1 <= t <= #producers, valid
queue orders, joined multi-producer counters, happens-before-respecting
memory accesses, reachable outputs and referential integrity.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field

import numpy as np

MAGIC = 0x414D4B53
NTASKF = 12


@dataclass
class Task:
    type: int
    layer: int
    queue: int
    waits: list = field(default_factory=list)     # [(counter, threshold)]
    signal: int = -1
    acc: list = field(default_factory=list)       # [(buffer, lo, hi, write)]
    a: list = field(default_factory=lambda: [0, 0, 0, 0])


@dataclass
class Schedule:
    buffers: list    # [(size, kind)]
    counters: list   # [[producers, completion]]
    tasks: list
    queues: list     # [[task ids]]
    body: list       # per queue


def parse(blob: bytes) -> Schedule:
    w = np.frombuffer(blob, dtype=np.int64)
    assert w[0] == MAGIC and w[1] == 1
    nt, nc, nq, nb, nw, na, ni = (int(x) for x in w[2:9])
    p = 9
    buffers = [(int(w[p + 2 * i]), int(w[p + 2 * i + 1])) for i in range(nb)]
    p += 2 * nb
    counters = [[int(w[p + 2 * i]), int(w[p + 2 * i + 1])] for i in range(nc)]
    p += 2 * nc
    trows = w[p:p + nt * NTASKF].reshape(nt, NTASKF)
    p += nt * NTASKF
    waits = w[p:p + 2 * nw].reshape(nw, 2)
    p += 2 * nw
    accs = w[p:p + 4 * na].reshape(na, 4)
    p += 4 * na
    qrows = w[p:p + 3 * nq].reshape(nq, 3)
    p += 3 * nq
    items = w[p:p + ni]
    tasks = []
    for r in trows:
        t = Task(int(r[0]), int(r[1]), int(r[2]))
        t.waits = [(int(a), int(b)) for a, b in waits[r[3]:r[3] + r[4]]]
        t.signal = int(r[5])
        t.acc = [tuple(int(v) for v in a) for a in accs[r[6]:r[6] + r[7]]]
        t.a = [int(v) for v in r[8:12]]
        tasks.append(t)
    queues = [[int(x) for x in items[q[0]:q[0] + q[1]]] for q in qrows]
    body = [int(q[2]) for q in qrows]
    return Schedule(buffers, counters, tasks, queues, body)


def serialize(s: Schedule) -> bytes:
    nw = sum(len(t.waits) for t in s.tasks)
    na = sum(len(t.acc) for t in s.tasks)
    ni = sum(len(q) for q in s.queues)
    out = [MAGIC, 1, len(s.tasks), len(s.counters), len(s.queues), len(s.buffers), nw, na, ni]
    for b in s.buffers:
        out += list(b)
    for c in s.counters:
        out += list(c)
    wb = ab = 0
    for t in s.tasks:
        out += [t.type, t.layer, t.queue, wb, len(t.waits), t.signal, ab, len(t.acc)] + list(t.a)
        wb += len(t.waits)
        ab += len(t.acc)
    for t in s.tasks:
        for wt in t.waits:
            out += list(wt)
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


def clone(s: Schedule) -> Schedule:
    return copy.deepcopy(s)


# ------------------------------------------------------------ ground truth

def truth(s: Schedule):
    """(safe, reason) by brute force."""
    T, NC, NQ, NB = len(s.tasks), len(s.counters), len(s.queues), len(s.buffers)
    prods = [[] for _ in range(NC)]
    for i, t in enumerate(s.tasks):
        if not (-1 <= t.queue < NQ) or not (-1 <= t.signal < NC) or not (0 <= t.type < 7):
            return False, "bad id"
        if t.signal >= 0:
            prods[t.signal].append(i)
        for c, th in t.waits:
            if not (0 <= c < NC):
                return False, "bad wait counter"
        for b, lo, hi, wr in t.acc:
            if not (0 <= b < NB) or lo < 0 or hi <= lo or hi > s.buffers[b][0]:
                return False, "bad access"
    completion_of = [-1] * T
    for c, (n, comp) in enumerate(s.counters):
        if n != len(prods[c]):
            return False, "producer count mismatch"
        if comp != -1:
            if not (0 <= comp < T) or s.tasks[comp].queue != -1 or completion_of[comp] != -1:
                return False, "bad completion"
            if s.tasks[comp].waits or n == 0:
                return False, "bad completion"
            completion_of[comp] = c
    seen = [0] * T
    if len(s.body) != NQ:
        return False, "bad body"
    for q, items in enumerate(s.queues):
        if not (0 <= s.body[q] <= len(items)):
            return False, "bad body"
        for t in items:
            if not (0 <= t < T) or s.tasks[t].queue != q:
                return False, "bad queue item"
            seen[t] += 1
    for i, t in enumerate(s.tasks):
        if t.queue >= 0 and seen[i] != 1:
            return False, "task not queued once"
        if t.queue == -1 and completion_of[i] == -1:
            return False, "orphan completion task"
        for c, th in t.waits:
            if not (1 <= th <= len(prods[c])):
                return False, "threshold outside [1, producers]"

    # deadlock: fixpoint of the queues (also gives an execution order)
    val = [0] * NC
    head = [0] * NQ
    order = []

    def fire(t):
        stack = [t]
        while stack:
            k = stack.pop()
            order.append(k)
            c = s.tasks[k].signal
            if c >= 0:
                val[c] += 1
                if val[c] == len(prods[c]) and s.counters[c][1] >= 0:
                    stack.append(s.counters[c][1])

    progress = True
    while progress:
        progress = False
        for q in range(NQ):
            while head[q] < len(s.queues[q]):
                t = s.queues[q][head[q]]
                if all(val[c] >= th for c, th in s.tasks[t].waits):
                    head[q] += 1
                    fire(t)
                    progress = True
                else:
                    break
    if any(head[q] < len(s.queues[q]) for q in range(NQ)) or len(order) != T:
        return False, "deadlock"

    # prefill (body only) must not depend on skipped tasks
    in_body = [False] * T
    for q, items in enumerate(s.queues):
        for t in items[:s.body[q]]:
            in_body[t] = True
    for i in range(T):
        if s.tasks[i].queue == -1:
            ps = prods[completion_of[i]]
            if any(in_body[p] for p in ps) and not all(in_body[p] for p in ps):
                return False, "completion mixes body and skipped"
            in_body[i] = all(in_body[p] for p in ps)
    for i, t in enumerate(s.tasks):
        if in_body[i]:
            for c, _ in t.waits:
                if any(not in_body[p] for p in prods[c]):
                    return False, "body waits on skipped"

    # the producer -> consumer graph (with queue order) must be acyclic
    succ = [[] for _ in range(T)]
    indeg = [0] * T
    prev = {}
    for items in s.queues:
        for a, b in zip(items, items[1:]):
            prev[b] = a
            succ[a].append(b)
            indeg[b] += 1
    for i, t in enumerate(s.tasks):
        srcs = [p for c, _ in t.waits for p in prods[c]]
        if completion_of[i] >= 0:
            srcs += prods[completion_of[i]]
        for p in srcs:
            succ[p].append(i)
            indeg[i] += 1
    topo = [i for i in range(T) if indeg[i] == 0]
    for i in topo:
        for j in succ[i]:
            indeg[j] -= 1
            if indeg[j] == 0:
                topo.append(j)
    if len(topo) != T:
        return False, "cyclic dependency"

    # happens-before in topological order.  A wait for any t of n producers
    # guarantees X is done iff X precedes (or is) at least n - t + 1 of them.
    before = [None] * T   # tasks guaranteed complete before t starts
    for t in topo:
        pre = set()
        if t in prev:
            pre |= before[prev[t]] | {prev[t]}
        for c, th in s.tasks[t].waits:
            ps = prods[c]
            need = len(ps) - th + 1
            cand = {}
            for p in ps:
                for x in before[p] | {p}:
                    cand[x] = cand.get(x, 0) + 1
            pre |= {x for x, k in cand.items() if k >= need}
        if completion_of[t] >= 0:
            for p in prods[completion_of[t]]:
                pre |= before[p] | {p}
        before[t] = pre

    for b in range(NB):
        accs = [(i, lo, hi, wr) for i, t in enumerate(s.tasks) for (bb, lo, hi, wr) in t.acc if bb == b]
        for x in range(len(accs)):
            for y in range(x + 1, len(accs)):
                i, lo1, hi1, w1 = accs[x]
                j, lo2, hi2, w2 = accs[y]
                if i == j or not (w1 or w2) or hi1 <= lo2 or hi2 <= lo1:
                    continue
                if i not in before[j] and j not in before[i]:
                    return False, f"race on buffer {b}"
    for b, (size, kind) in enumerate(s.buffers):
        if kind == 1:
            cov = np.zeros(size, dtype=bool)
            for t in s.tasks:
                for bb, lo, hi, wr in t.acc:
                    if bb == b and wr:
                        cov[lo:hi] = True
            if not cov.all():
                return False, "output not covered"
    return True, "safe"
