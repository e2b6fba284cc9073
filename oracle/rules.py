"""Planner rules, written out plainly (TEST INFRASTRUCTURE ONLY; see package doc).

Sources (page title, section):

* "MPK code walkthrough" (Mirage Persistent Kernel), section on the
  fine-grained pipeline: ``build_partition``, the per-dimension gcd event
  partition, the fork-producer and join-consumer lcm normalisation with its
  F/A/B/G worked example and the four gcd examples; section on building the
  SM-level DAG: the per-event task creation that makes each event's successor
  tasks contiguous, and the event record {num_triggers, first_task_id,
  last_task_id}.
* "MegaRTP megakernel article", section 4 (TaskGraph): the whole / tile /
  tile_cover / tile_reduce pairing strategies and their thresholds;
  section 4 (KernelPlan): round-robin queues padded with NoOp.
* "CMU 15-779 Lecture 7 notes: Mega-Kernel", sections 6.3-6.4: ahead-of-time
  round-robin queues, and longest-first placement for unequal tasks.

Pins: the F/A/B/G example, the four gcd examples and the build_partition
example (values the page prints, in ``tests/golden/mpk_examples.json``); the
Llama-1B layer counts of the lecture (1,984 tasks, 15 events, 3,968
task-event edges, about 380k pairwise edges); the GLM plan of the MegaRTP
article (732 tasks, 70 events, [148, 5, 32] queue, 140x5 + 8x4).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from itertools import product as _iproduct
from typing import Callable, Dict, List, Optional, Sequence, Tuple

MAX_TENSOR_DIMS = 4


# ---------------------------------------------------------------------------
# graph description
# ---------------------------------------------------------------------------

@dataclass
class Op:
    """An operator with a launch grid of up to three axes (x, y, z).

    ``exists`` optionally removes grid points (ragged grids such as per-sequence
    attention splits); removed points create no task and trigger nothing.
    ``cost`` gives the bytes a task streams (used only for queue balancing).
    """
    name: str
    grid: Tuple[int, int, int]
    exists: Optional[Callable[[Tuple[int, int, int]], bool]] = None
    cost: Optional[Callable[[Tuple[int, int, int]], int]] = None


@dataclass
class Edge:
    """A tensor dependency ``prod -> cons``.

    ``out_map[a]`` is the tensor dimension that the producer's grid axis ``a``
    cuts (-1: the axis does not cut the tensor, e.g. a split-K axis);
    ``in_map[a]`` is the same for the consumer's grid axes.
    """
    prod: str
    cons: str
    out_map: Tuple[int, int, int]
    in_map: Tuple[int, int, int]


def build_partition(grid: Sequence[int], dim_map: Sequence[int]) -> List[int]:
    """How many pieces the grid cuts each tensor dimension into (1 if uncut).

    MPK walkthrough, fine-grained pipeline: grid (128,1,1) with map
    (1,-1,-1) gives [1,128,1,1].
    """
    part = [1] * MAX_TENSOR_DIMS
    for axis, d in enumerate(dim_map):
        if d >= 0:
            part[d] *= grid[axis]
    return part


def bids(grid: Sequence[int]):
    """Grid points in lexicographic order, x the most significant axis."""
    return list(_iproduct(range(grid[0]), range(grid[1]), range(grid[2])))


def piece_index(bid: Sequence[int], grid: Sequence[int], dim_map: Sequence[int], d: int) -> int:
    """Index of the piece of tensor dim ``d`` that grid point ``bid`` touches.

    When several grid axes cut the same dimension they combine in axis order
    (x most significant).
    """
    idx = 0
    for axis, dd in enumerate(dim_map):
        if dd == d:
            idx = idx * grid[axis] + bid[axis]
    return idx


def _lcm(a: int, b: int) -> int:
    return a * b // math.gcd(a, b)


@dataclass
class EdgeEvents:
    event_dim: List[int]
    prod_part: List[int]
    cons_part: List[int]

    def prod_group(self, d):  # producer pieces per event along d
        return self.prod_part[d] // self.event_dim[d]

    def cons_group(self, d):  # consumer pieces per event along d
        return self.cons_part[d] // self.event_dim[d]


def edge_event_dims(ops: Dict[str, Op], edges: List[Edge]) -> List[EdgeEvents]:
    """gcd event partition per edge, then fork and join lcm normalisation.

    MPK walkthrough: ``event_dim[d] = gcd(prod_part[d], cons_part[d])``.
    Fork (a producer with several out-edges): the producer-side group sizes
    ``prod_part/event_dim`` are lcm'd across the edges; if the lcm divides the
    producer's cut, each edge's ``event_dim`` becomes ``prod_part/lcm``.
    Join (a consumer with several in-edges): the same on the consumer side.
    When the lcm does not divide the cut the page only names a safety check;
    we then fall back to one whole-producer event for that group.
    """
    ee = []
    for e in edges:
        pp = build_partition(ops[e.prod].grid, e.out_map)
        cp = build_partition(ops[e.cons].grid, e.in_map)
        ee.append(EdgeEvents([math.gcd(a, b) for a, b in zip(pp, cp)], pp, cp))

    def normalise(idx: List[int], side: str):
        parts = [ee[i].prod_part if side == "prod" else ee[i].cons_part for i in idx]
        if any(p != parts[0] for p in parts):
            for i in idx:
                ee[i].event_dim = [1] * MAX_TENSOR_DIMS
            return
        part = parts[0]
        new_dim = []
        for d in range(MAX_TENSOR_DIMS):
            l = 1
            for i in idx:
                l = _lcm(l, part[d] // ee[i].event_dim[d])
            if part[d] % l != 0:
                for i in idx:
                    ee[i].event_dim = [1] * MAX_TENSOR_DIMS
                return
            new_dim.append(part[d] // l)
        for i in idx:
            ee[i].event_dim = list(new_dim)

    fork_members, join_members = set(), set()
    for name in ops:
        out_idx = [i for i, e in enumerate(edges) if e.prod == name]
        if len(out_idx) > 1:
            normalise(out_idx, "prod")
            fork_members.update(out_idx)
    for name in ops:
        in_idx = [i for i, e in enumerate(edges) if e.cons == name]
        if len(in_idx) > 1:
            if fork_members.intersection(in_idx):
                raise NotImplementedError("an edge that is both in a fork and in a join")
            normalise(in_idx, "cons")
            join_members.update(in_idx)
    return ee


# ---------------------------------------------------------------------------
# task graph construction (linearisation with contiguous successors)
# ---------------------------------------------------------------------------

@dataclass
class Task:
    op: str
    bid: Tuple[int, int, int]
    trigger_event: Optional[int] = None
    dependent_event: Optional[int] = None


@dataclass
class Event:
    num_triggers: int
    first_task_id: int
    last_task_id: int  # exclusive


@dataclass
class TaskGraph:
    tasks: List[Task]
    events: List[Event]
    first_tasks: List[int]
    edge_events: List[EdgeEvents] = field(default_factory=list)

    def pairwise_edges(self) -> int:
        """Task-to-task dependency pairs that the events stand for."""
        return sum(ev.num_triggers * (ev.last_task_id - ev.first_task_id) for ev in self.events)

    def task_event_edges(self) -> int:
        n = 0
        for t in self.tasks:
            n += (t.trigger_event is not None) + (t.dependent_event is not None)
        return n


def _unravel(i: int, radix: Sequence[int]) -> List[int]:
    out = [0] * len(radix)
    for d in range(len(radix) - 1, -1, -1):
        out[d] = i % radix[d]
        i //= radix[d]
    return out


def _in_event(bid, grid, dim_map, part, event_dim, coords) -> bool:
    for d in range(MAX_TENSOR_DIMS):
        g = part[d] // event_dim[d]
        if piece_index(bid, grid, dim_map, d) // g != coords[d]:
            return False
    return True


def build_task_graph(ops_list: List[Op], edges: List[Edge], order: Optional[List[str]] = None) -> TaskGraph:
    """MPK walkthrough, 'building the SM-level DAG'.

    Walk the op-level linearisation.  An op with no in-edge puts its tasks in
    lexicographic grid order (first tasks).  Otherwise, for every event of the
    incoming edge (or of the fork bundle / join group it belongs to), in
    mixed-radix order over the tensor dims: record ``first_task_id``, create
    the consumer tasks that fall in the event's box (for a fork bundle, those
    of every consumer in the bundle), record ``last_task_id``, then mark every
    producer task in the event's producer-side box with this trigger event and
    count it in ``num_triggers``.
    """
    ops = {o.name: o for o in ops_list}
    order = order or [o.name for o in ops_list]
    ee = edge_event_dims(ops, edges)
    tasks: List[Task] = []
    events: List[Event] = []
    tid: Dict[Tuple[str, Tuple[int, int, int]], int] = {}
    done = set()

    def exists(op: Op, bid) -> bool:
        return op.exists is None or op.exists(bid)

    def add_task(op: Op, bid, dep):
        tid[(op.name, bid)] = len(tasks)
        tasks.append(Task(op.name, bid, None, dep))

    for name in order:
        if name in done:
            continue
        op = ops[name]
        in_idx = [i for i, e in enumerate(edges) if e.cons == name]
        if not in_idx:
            for bid in bids(op.grid):
                if exists(op, bid):
                    add_task(op, bid, None)
            done.add(name)
            continue
        if len(in_idx) > 1:  # join consumer
            edim = ee[in_idx[0]].event_dim
            for k in range(math.prod(edim)):
                coords = _unravel(k, edim)
                ev_id = len(events)
                first = len(tasks)
                for bid in bids(op.grid):
                    if exists(op, bid) and _in_event(bid, op.grid, edges[in_idx[0]].in_map,
                                                     ee[in_idx[0]].cons_part, edim, coords):
                        add_task(op, bid, ev_id)
                n_trig = 0
                for i in in_idx:
                    e = edges[i]
                    prod = ops[e.prod]
                    for pbid in bids(prod.grid):
                        if exists(prod, pbid) and _in_event(pbid, prod.grid, e.out_map, ee[i].prod_part, edim, coords):
                            tasks[tid[(prod.name, pbid)]].trigger_event = ev_id
                            n_trig += 1
                events.append(Event(n_trig, first, len(tasks)))
            done.add(name)
            continue
        e0 = edges[in_idx[0]]
        prod = ops[e0.prod]
        bundle = [i for i, e in enumerate(edges) if e.prod == e0.prod]
        for i in bundle:
            if len([j for j, e in enumerate(edges) if e.cons == edges[i].cons]) != 1:
                raise NotImplementedError("fork bundle consumer with several in-edges")
        # consumers of the bundle in the order they appear in the linearisation
        bundle.sort(key=lambda i: order.index(edges[i].cons))
        edim = ee[bundle[0]].event_dim
        for k in range(math.prod(edim)):
            coords = _unravel(k, edim)
            ev_id = len(events)
            first = len(tasks)
            for i in bundle:
                cop = ops[edges[i].cons]
                for bid in bids(cop.grid):
                    if exists(cop, bid) and _in_event(bid, cop.grid, edges[i].in_map, ee[i].cons_part, edim, coords):
                        add_task(cop, bid, ev_id)
            n_trig = 0
            for pbid in bids(prod.grid):
                if exists(prod, pbid) and _in_event(pbid, prod.grid, e0.out_map, ee[bundle[0]].prod_part, edim, coords):
                    tasks[tid[(prod.name, pbid)]].trigger_event = ev_id
                    n_trig += 1
            events.append(Event(n_trig, first, len(tasks)))
        for i in bundle:
            done.add(edges[i].cons)
    first_tasks = [i for i, t in enumerate(tasks) if t.dependent_event is None]
    return TaskGraph(tasks, events, first_tasks, ee)


# ---------------------------------------------------------------------------
# MegaRTP pairing strategies
# ---------------------------------------------------------------------------

WHOLE, TILE, TILE_COVER, TILE_REDUCE = "whole", "tile", "tile_cover", "tile_reduce"


def pairing(strategy: str, n_publishers: int, k: int = 1) -> List[int]:
    """Thresholds of the events one producer->consumer pairing creates.

    MegaRTP article, TaskGraph: ``whole`` -- one event, every producer adds
    one, the consumer waits for all of them; ``tile`` -- one event per
    producer region, threshold 1; ``tile_cover`` -- k disjoint producer
    regions cover one consumer region, threshold k; ``tile_reduce`` -- k
    partials reduce into one consumer region, threshold k.  The counter only
    counts; on the device cover and reduce are the same mechanism.
    """
    if strategy == WHOLE:
        return [n_publishers]
    if strategy == TILE:
        return [1] * n_publishers
    if strategy in (TILE_COVER, TILE_REDUCE):
        if k <= 0 or n_publishers % k:
            raise ValueError("k must divide the number of publishing tiles")
        return [k] * (n_publishers // k)
    raise ValueError(strategy)


def check_cover(regions: List[Tuple[int, int]], target: Tuple[int, int]) -> bool:
    """tile_cover host check: disjoint half-open regions whose union is target."""
    rs = sorted(regions)
    pos = target[0]
    for a, b in rs:
        if a != pos:
            return False
        pos = b
    return pos == target[1]


def check_reduce(regions: List[Tuple[int, int]], target: Tuple[int, int]) -> bool:
    """tile_reduce host check: every partial covers exactly the target region."""
    return all(r == tuple(target) for r in regions)


# ---------------------------------------------------------------------------
# static queues
# ---------------------------------------------------------------------------

def round_robin(n_tasks: int, n_workers: int) -> List[List[int]]:
    """Task i goes to worker i mod n_workers (MegaRTP KernelPlan)."""
    q = [[] for _ in range(n_workers)]
    for i in range(n_tasks):
        q[i % n_workers].append(i)
    return q


def greedy_balance(order: Sequence[int], cost: Sequence[int], n_workers: int) -> List[List[int]]:
    """Deal tasks, in the given (topological) order, each to the worker with the
    least accumulated cost so far (ties: lowest worker index).  With equal costs
    this is round-robin; every queue stays a subsequence of ``order``."""
    load = [0] * n_workers
    q = [[] for _ in range(n_workers)]
    for t in order:
        w = min(range(n_workers), key=lambda i: (load[i], i))
        q[w].append(t)
        load[w] += cost[t]
    return q


def longest_first_within(groups: List[Tuple[int, int]], cost: Sequence[int]) -> List[int]:
    """Within each contiguous [first, last) range reorder tasks by descending
    cost (stable), the longest-first placement of the lecture's AOT/JIT study;
    ranges are kept contiguous so event successors stay contiguous."""
    out: List[int] = []
    for a, b in groups:
        out.extend(sorted(range(a, b), key=lambda t: -cost[t]))
    return out


def pad_queues(queues: List[List[int]], noop: int = -1) -> Tuple[List[List[int]], int]:
    """Pad every queue to the longest with NoOp entries (MegaRTP KernelPlan)."""
    lmax = max((len(q) for q in queues), default=0)
    return [q + [noop] * (lmax - len(q)) for q in queues], lmax


def expected_counters(thresholds: Sequence[int], steps: int) -> List[int]:
    """Counters are never reset between steps (monotone epochs, as in the
    GEMM+AllToAll post's ready epochs): after ``steps`` steps every event's
    counter equals steps x (increments it receives per step)."""
    return [steps * t for t in thresholds]
