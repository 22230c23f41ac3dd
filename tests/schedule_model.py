"""Python view of the serialised schedule and an independent ground truth.

The schedule synchronises through tagged data: each element of a tagged
buffer is written once per version, and a read of version v polls the
elements until they carry v.  The ground truth decides safety by brute
force, element by element, written separately from the C++ validator
(which works on intervals, adjacent versions and vector clocks):

* integrity: ids, ranges, versions, every task queued exactly once;
* every element of a tagged buffer has exactly one writer per version, for
  every version 1..V, all of them in the prefill body;
* no deadlock: the graph of queue order + writer -> reader edges is
  acyclic (a cycle is unsafe by definition) and the queues run to
  completion when each task starts once every writer it reads finished;
* happens-before (sets of tasks guaranteed complete before a task starts,
  built in topological order): for every element, every access of version
  u is ordered before every write of a later version and after every write
  of an earlier one; untagged buffers: every write ordered against every
  overlapping access;
* tags cycle with period 15: when a reader starts (its queue predecessor
  done), every element it polls already holds a version at most 14 behind
  the awaited one (the previous step's last version counts as version 0);
* every element of an output buffer is written.

These are the AutoMegaKernel safety-gate conditions (acyclic, satisfiable
waits, valid queue orders, joined producers, happens-before-respecting
memory accesses, reachable outputs, referential integrity) restated for
counters of one producer fused with the data.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field

import numpy as np

MAGIC = 0x414D4B53
FORMAT = 2
NTASKF = 9
NACCF = 5
TAGGED, OUTPUT, STATE = 0, 1, 2
MAX_VERSIONS = 4096
MAX_TAG_GAP = 14


@dataclass
class Task:
    type: int
    layer: int
    queue: int
    acc: list = field(default_factory=list)       # [(buffer, lo, hi, write, version)]
    a: list = field(default_factory=lambda: [0, 0, 0, 0])


@dataclass
class Schedule:
    buffers: list    # [(size, kind)]
    tasks: list
    queues: list     # [[task ids]]
    body: list       # per queue
    versions: int


def parse(blob: bytes) -> Schedule:
    w = np.frombuffer(blob, dtype=np.int64)
    assert w[0] == MAGIC and w[1] == FORMAT
    nt, nq, nb, na, ni, nv = (int(x) for x in w[2:8])
    p = 8
    buffers = [(int(w[p + 2 * i]), int(w[p + 2 * i + 1])) for i in range(nb)]
    p += 2 * nb
    trows = w[p:p + nt * NTASKF].reshape(nt, NTASKF)
    p += nt * NTASKF
    accs = w[p:p + NACCF * na].reshape(na, NACCF)
    p += NACCF * na
    qrows = w[p:p + 3 * nq].reshape(nq, 3)
    p += 3 * nq
    items = w[p:p + ni]
    tasks = []
    for r in trows:
        t = Task(int(r[0]), int(r[1]), int(r[2]))
        t.acc = [tuple(int(v) for v in a) for a in accs[r[3]:r[3] + r[4]]]
        t.a = [int(v) for v in r[5:9]]
        tasks.append(t)
    queues = [[int(x) for x in items[q[0]:q[0] + q[1]]] for q in qrows]
    body = [int(q[2]) for q in qrows]
    return Schedule(buffers, tasks, queues, body, nv)


def serialize(s: Schedule) -> bytes:
    na = sum(len(t.acc) for t in s.tasks)
    ni = sum(len(q) for q in s.queues)
    out = [MAGIC, FORMAT, len(s.tasks), len(s.queues), len(s.buffers), na, ni, s.versions]
    for b in s.buffers:
        out += list(b)
    ab = 0
    for t in s.tasks:
        out += [t.type, t.layer, t.queue, ab, len(t.acc)] + list(t.a)
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


def clone(s: Schedule) -> Schedule:
    return copy.deepcopy(s)


# ------------------------------------------------------------ ground truth

def truth(s: Schedule):
    """(safe, reason) by brute force over elements."""
    T, NQ, NB, V = len(s.tasks), len(s.queues), len(s.buffers), s.versions
    if not (1 <= V <= MAX_VERSIONS):
        return False, "bad version count"
    for size, kind in s.buffers:
        if size <= 0 or kind not in (TAGGED, OUTPUT, STATE):
            return False, "bad buffer"
    for t in s.tasks:
        if not (0 <= t.queue < NQ) or not (0 <= t.type < 7):
            return False, "bad id"
        if not any(a[3] for a in t.acc):
            return False, "writes nothing"
        for b, lo, hi, wr, ver in t.acc:
            if not (0 <= b < NB) or lo < 0 or hi <= lo or hi > s.buffers[b][0]:
                return False, "bad access"
            if s.buffers[b][1] == TAGGED:
                if not (1 <= ver <= V):
                    return False, "bad version"
            elif ver != 0:
                return False, "bad version"
    if len(s.body) != NQ:
        return False, "bad body"
    seen = [0] * T
    for q, items in enumerate(s.queues):
        if not (0 <= s.body[q] <= len(items)):
            return False, "bad body"
        for t in items:
            if not (0 <= t < T) or s.tasks[t].queue != q:
                return False, "bad queue item"
            seen[t] += 1
    if any(c != 1 for c in seen):
        return False, "task not queued once"
    in_body = [False] * T
    for q, items in enumerate(s.queues):
        for t in items[:s.body[q]]:
            in_body[t] = True

    # per-element writers of every version of every tagged buffer
    writer = {}   # (b, e, v) -> task
    for i, t in enumerate(s.tasks):
        for b, lo, hi, wr, ver in t.acc:
            if wr and s.buffers[b][1] == TAGGED:
                if not in_body[i]:
                    return False, "tagged write outside the body"
                for e in range(lo, hi):
                    if (b, e, ver) in writer:
                        return False, "two writers of one version"
                    writer[(b, e, ver)] = i
    for b, (size, kind) in enumerate(s.buffers):
        if kind == TAGGED:
            for e in range(size):
                for v in range(1, V + 1):
                    if (b, e, v) not in writer:
                        return False, "version not written"

    # writer -> reader edges and queue order
    preds = [set() for _ in range(T)]
    for i, t in enumerate(s.tasks):
        for b, lo, hi, wr, ver in t.acc:
            if not wr and s.buffers[b][1] == TAGGED:
                for e in range(lo, hi):
                    w = writer[(b, e, ver)]
                    if w == i:
                        return False, "waits for its own write"
                    preds[i].add(w)
    prev = {}
    for items in s.queues:
        for a, b in zip(items, items[1:]):
            prev[b] = a
    for i in range(T):
        if in_body[i] and any(not in_body[w] for w in preds[i]):
            return False, "body waits on skipped"

    # deadlock: start a task once its queue predecessor and writers are done
    done = [False] * T
    head = [0] * NQ
    progress = True
    while progress:
        progress = False
        for q in range(NQ):
            while head[q] < len(s.queues[q]):
                t = s.queues[q][head[q]]
                if all(done[w] for w in preds[t]):
                    done[t] = True
                    head[q] += 1
                    progress = True
                else:
                    break
    if not all(done):
        return False, "deadlock"

    # happens-before sets in a topological order of the same graph
    succ = [[] for _ in range(T)]
    indeg = [0] * T
    for i in range(T):
        srcs = set(preds[i])
        if i in prev:
            srcs.add(prev[i])
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
    before = [None] * T
    for t in topo:
        pre = set()
        srcs = set(preds[t])
        if t in prev:
            srcs.add(prev[t])
        for p in srcs:
            pre |= before[p] | {p}
        before[t] = pre

    for b in range(NB):
        accs = [(i, lo, hi, wr, ver) for i, t in enumerate(s.tasks)
                for (bb, lo, hi, wr, ver) in t.acc if bb == b]
        tagged = s.buffers[b][1] == TAGGED
        for x in range(len(accs)):
            for y in range(len(accs)):
                i, lo1, hi1, w1, v1 = accs[x]
                j, lo2, hi2, w2, v2 = accs[y]
                if i == j or not w2 or hi1 <= lo2 or hi2 <= lo1:
                    continue
                # accs[y] is a write overlapping accs[x]
                if tagged:
                    if v1 < v2 and i not in before[j]:
                        return False, f"buffer {b}: access of an older version not before a newer write"
                    if v1 > v2 and j not in before[i]:
                        return False, f"buffer {b}: write of an older version not before a newer access"
                    if v1 == v2 and not w1 and j not in before[i]:
                        return False, f"buffer {b}: read before its writer"
                elif i not in before[j] and j not in before[i]:
                    return False, f"race on buffer {b}"
    # tag aliasing: per element, the newest version surely written when the
    # reader starts (its queue predecessor and everything before it done)
    for i, t in enumerate(s.tasks):
        done_at_start = (before[prev[i]] | {prev[i]}) if i in prev else set()
        for b, lo, hi, wr, ver in t.acc:
            if wr or s.buffers[b][1] != TAGGED:
                continue
            for e in range(lo, hi):
                held = max([u for u in range(1, ver) if writer[(b, e, u)] in done_at_start],
                           default=0)
                if ver - held > MAX_TAG_GAP:
                    return False, "tags may alias"
    for b, (size, kind) in enumerate(s.buffers):
        if kind == OUTPUT:
            cov = np.zeros(size, dtype=bool)
            for t in s.tasks:
                for bb, lo, hi, wr, ver in t.acc:
                    if bb == b and wr:
                        cov[lo:hi] = True
            if not cov.all():
                return False, "output not covered"
    return True, "safe"
