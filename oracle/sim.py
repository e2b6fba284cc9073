"""Queue simulator (TEST INFRASTRUCTURE ONLY).

* ``deadlock_check`` -- runs static per-worker queues in order against event
  counters: a worker may retire its head task once every wait of that task is
  met; if no worker can move while tasks remain, the plan deadlocks and the
  blocked heads are reported.
* the toy network of the lecture's correctness demo ("CMU 15-779 Lecture 7
  notes", sections 6.2 and 6.5): GEMV -> blockwise tanh -> GEMV -> split-K
  GEMV, executed by a multi-worker interpreter that picks a random ready
  worker at every step.  Split-K partials are added into the output in
  execution order, so results differ bit for bit between interleavings while
  staying correct; deleting one dependency makes some interleavings wrong,
  never a single worker.

The toy's sizes are not printed; the ones here are the only ones consistent
with what the notes do print (28 tasks, 52 pairwise edges, 9 events after
merging identical dependency sets, a tanh task depending on the 3 GEMV tasks
that cover its 24 elements, a split-K segment depending on the 2 tasks that
write its 16 elements, and an edge GEMV3[7] -> GEMV4[3]): GEMV1 12 tasks of 8
rows, tanh 4 tasks of 24, GEMV3 8 tasks of 8 rows reading all 96 values,
GEMV4 4 K-segments of 16.
"""
from __future__ import annotations

import random
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Set, Tuple

import numpy as np

from . import rules


# ---------------------------------------------------------------------------
# deadlock check over counters
# ---------------------------------------------------------------------------

@dataclass
class SimResult:
    ok: bool
    counters: List[int]
    blocked: List[Tuple[int, int]]   # (worker, task) heads that could not move
    order: List[int]                 # retirement order of tasks


def deadlock_check(queues: Sequence[Sequence[int]], waits: Dict[int, List[Tuple]],
                   signals: Dict[int, List[Tuple[int, int]]], n_events: int, steps: int = 1,
                   rng: Optional[random.Random] = None) -> SimResult:
    """Run ``steps`` back-to-back passes of the queues (counters never reset).

    ``waits[t]`` holds (event, threshold[, epoch offset]); the target at step s
    is threshold x (s + 1 + offset).  ``-1`` entries are NoOps.  With ``rng``
    the ready worker to advance is picked at random, else the lowest index.
    """
    counters = [0] * n_events
    order: List[int] = []
    for s in range(steps):
        pos = [0] * len(queues)

        def head(w):
            while pos[w] < len(queues[w]) and queues[w][pos[w]] < 0:
                pos[w] += 1
            return queues[w][pos[w]] if pos[w] < len(queues[w]) else None

        def ready(t):
            for wt in waits.get(t, []):
                ev, thr = wt[0], wt[1]
                off = wt[2] if len(wt) > 2 else 0
                if counters[ev] < thr * (s + 1 + off):
                    return False
            return True

        while True:
            cand = [w for w in range(len(queues)) if head(w) is not None and ready(head(w))]
            if not cand:
                break
            w = rng.choice(cand) if rng else cand[0]
            t = head(w)
            for ev, inc in signals.get(t, []):
                counters[ev] += inc
            order.append(t)
            pos[w] += 1
        blocked = [(w, head(w)) for w in range(len(queues)) if head(w) is not None]
        if blocked:
            return SimResult(False, counters, blocked, order)
    return SimResult(True, counters, [], order)


# ---------------------------------------------------------------------------
# toy network of the correctness demo
# ---------------------------------------------------------------------------

TOY_K0 = 32      # input length of GEMV1 (not printed; any value works)
TOY_OUT = 16     # outputs of the split-K GEMV (not printed; any value works)


def toy_graph():
    """The toy network as MPK-style ops/edges (grid cuts per tensor dim)."""
    ops = [rules.Op("gemv1", (12, 1, 1)), rules.Op("tanh", (4, 1, 1)),
           rules.Op("gemv3", (8, 1, 1)), rules.Op("gemv4", (4, 1, 1))]
    edges = [rules.Edge("gemv1", "tanh", (0, -1, -1), (0, -1, -1)),     # y1[96]
             rules.Edge("tanh", "gemv3", (0, -1, -1), (-1, -1, -1)),    # y2[96], read whole
             rules.Edge("gemv3", "gemv4", (0, -1, -1), (0, -1, -1))]    # y3[64], K segments
    return ops, edges


def toy_pairwise_deps() -> Dict[Tuple[str, int], Set[Tuple[str, int]]]:
    """Dependencies derived from read/write regions (the lecture's analysis):
    task B depends on task A when A's output range overlaps B's input range."""
    out = {("gemv1", i): (8 * i, 8 * i + 8) for i in range(12)}
    out.update({("tanh", i): (24 * i, 24 * i + 24) for i in range(4)})
    out.update({("gemv3", i): (8 * i, 8 * i + 8) for i in range(8)})
    inp = {("tanh", i): ("gemv1", (24 * i, 24 * i + 24)) for i in range(4)}
    inp.update({("gemv3", i): ("tanh", (0, 96)) for i in range(8)})
    inp.update({("gemv4", i): ("gemv3", (16 * i, 16 * i + 16)) for i in range(4)})
    deps: Dict[Tuple[str, int], Set[Tuple[str, int]]] = {("gemv1", i): set() for i in range(12)}
    for t, (src, (a, b)) in inp.items():
        deps[t] = {p for p, (c, d) in out.items() if p[0] == src and c < b and a < d}
    return deps


def merge_identical_dep_sets(deps) -> int:
    """Number of events when tasks with identical (non-empty) dependency sets
    share one event."""
    return len({frozenset(s) for s in deps.values() if s})


@dataclass
class ToyData:
    x: np.ndarray
    w1: np.ndarray
    w3: np.ndarray
    w4: np.ndarray


def toy_data(seed: int = 0) -> ToyData:
    r = np.random.default_rng(seed)
    return ToyData(r.standard_normal(TOY_K0), r.standard_normal((96, TOY_K0)) * 0.3,
                   r.standard_normal((64, 96)) * 0.3, r.standard_normal((TOY_OUT, 64)) * 0.3)


def toy_direct(d: ToyData) -> np.ndarray:
    y1 = d.w1 @ d.x
    y2 = np.tanh(y1)
    y3 = d.w3 @ y2
    return d.w4 @ y3


def toy_interpreter(d: ToyData, n_workers: int, deps, rng: random.Random) -> np.ndarray:
    """Round-robin AOT queues over the tasks in topological order; at every step
    a random worker whose head task has all its dependencies retired executes
    it atomically.  The split-K GEMV adds its partial into the output."""
    order = ([("gemv1", i) for i in range(12)] + [("tanh", i) for i in range(4)] +
             [("gemv3", i) for i in range(8)] + [("gemv4", i) for i in range(4)])
    queues = [[] for _ in range(n_workers)]
    for i, t in enumerate(order):
        queues[i % n_workers].append(t)
    y1 = np.full(96, np.nan)
    y2 = np.full(96, np.nan)
    y3 = np.full(64, np.nan)
    out = np.zeros(TOY_OUT)
    done: Set[Tuple[str, int]] = set()
    pos = [0] * n_workers
    while any(pos[w] < len(queues[w]) for w in range(n_workers)):
        cand = [w for w in range(n_workers)
                if pos[w] < len(queues[w]) and deps[queues[w][pos[w]]] <= done]
        if not cand:
            raise RuntimeError("toy interpreter deadlocked")
        w = rng.choice(cand)
        kind, i = queues[w][pos[w]]
        if kind == "gemv1":
            y1[8 * i:8 * i + 8] = d.w1[8 * i:8 * i + 8] @ d.x
        elif kind == "tanh":
            y2[24 * i:24 * i + 24] = np.tanh(y1[24 * i:24 * i + 24])
        elif kind == "gemv3":
            y3[8 * i:8 * i + 8] = d.w3[8 * i:8 * i + 8] @ y2
        else:
            seg = slice(16 * i, 16 * i + 16)
            part = d.w4[:, seg] @ y3[seg]
            out += part      # accumulation order follows execution order
        done.add((kind, i))
        pos[w] += 1
    return out
