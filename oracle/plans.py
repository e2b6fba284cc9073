"""Whole-plan statements built on ``rules`` (TEST INFRASTRUCTURE ONLY).

* ``llama_step_plan`` -- the tile expansion of one decode step of a dense
  Llama-style decoder into per-op grids and tensor edges, run through the MPK
  gcd/lcm event rule, then queued.  The op set is the lecture's seven fused
  instruction types ("CMU 15-779 Lecture 7 notes", section 5.1): RMSNorm+QKV,
  attention (+ reduction), O-projection+residual, RMSNorm+gate/up+SiLU,
  down+residual with its intermediate split into K chunks that each have a
  counter, RMSNorm+LM head.  An embedding-gather task starts the step.
* ``megartp_glm_plan`` -- the MegaRTP article's GLM pre-attention plan
  (section 4, TaskGraph and KernelPlan): fixed per-op tile counts and the
  publications / waits the article lists.

The tile-expansion reading (which tensor dimension each grid axis cuts, the
cost model used to balance queues) is this project's; both this file and the
C++ planner state it independently and must agree bit for bit.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

from . import rules
from .rules import Edge, Op


@dataclass
class LlamaShape:
    L: int
    H: int
    Hq: int
    Hkv: int
    D: int
    F: int
    V: int


@dataclass
class Knobs:
    rows_qkv: int
    rows_o: int
    rows_up: int      # gate rows (= up rows) per MLP-up tile
    rows_down: int
    kchunk_down: int  # K extent of one down-projection tile
    rows_lm: int
    attn_split: int   # cache positions per attention task
    wbytes: int = 2   # bytes per projection weight: 2 (bf16), 1 (e4m3); the LM head stays bf16


def _ceil(a, b):
    return -(-a // b)


@dataclass
class PlannedTask:
    op: str
    kind: str
    layer: int
    bid: Tuple[int, int, int]
    cost: int
    waits: List[Tuple[int, int, int]]   # (event, threshold, epoch offset)
    signals: List[Tuple[int, int]]      # (event, increment)


@dataclass
class Plan:
    tasks: List[PlannedTask]
    thresholds: List[int]
    queues: List[List[int]]   # task ids, -1 = NoOp
    lmax: int
    graph: rules.TaskGraph


def llama_step_ops(shape: LlamaShape, k: Knobs, B: int, seq0: Sequence[int], max_steps: int):
    G = shape.Hq // shape.Hkv
    rows_group = (G + 2) * shape.D
    assert rows_group % k.rows_qkv == 0 and shape.F % k.rows_up == 0 and shape.F % k.kchunk_down == 0
    nsplit = [_ceil(seq0[b] + max_steps, k.attn_split) for b in range(B)]
    ns_max = max(nsplit)

    def attn_rows(bid):
        g, b, s = bid
        last_pos = seq0[b] + max_steps - 1          # cached rows at the last step
        return max(0, min(k.attn_split, last_pos - s * k.attn_split))

    wb = k.wbytes

    def rows_cost(n_rows, rows, kdim, mult=1, wbytes=wb):
        def f(bid):
            r0 = bid[0] * rows
            return mult * min(rows, n_rows - r0) * kdim * wbytes
        return f

    ops: List[Op] = [Op("embed", (1, 1, 1), cost=lambda bid: B * shape.H * 2)]
    kinds = {"embed": ("embed", -1)}
    edges: List[Edge] = []
    prev = "embed"
    for l in range(shape.L):
        qkv, attn, o, up, down = (f"{n}{l}" for n in ("qkv", "attn", "o", "up", "down"))
        ops.append(Op(qkv, (shape.Hkv, rows_group // k.rows_qkv, 1),
                      cost=lambda bid: k.rows_qkv * shape.H * wb))
        ops.append(Op(attn, (shape.Hkv, B, ns_max), exists=lambda bid: bid[2] < nsplit[bid[1]],
                      cost=lambda bid: 2 * shape.D * 2 * attn_rows(bid)))
        ops.append(Op(o, (_ceil(shape.H, k.rows_o), 1, 1), cost=rows_cost(shape.H, k.rows_o, shape.Hq * shape.D)))
        ops.append(Op(up, (shape.F // k.rows_up, 1, 1), cost=lambda bid: 2 * k.rows_up * shape.H * wb))
        ops.append(Op(down, (_ceil(shape.H, k.rows_down), shape.F // k.kchunk_down, 1),
                      cost=rows_cost(shape.H, k.rows_down, k.kchunk_down)))
        for n, kind in ((qkv, "qkv"), (attn, "attn"), (o, "o"), (up, "up"), (down, "down")):
            kinds[n] = (kind, l)
        # h [B, H] -> qkv reads all of it
        edges.append(Edge(prev, qkv, (1, -1, -1), (-1, -1, -1)))
        # qkv [B, Hkv, rows_group]: producer cuts group and rows, consumer cuts batch and group
        edges.append(Edge(qkv, attn, (1, 2, -1), (1, 0, -1)))
        # attn_out [B, Hkv, G*D]: O reads all of it; the split axis is a reduction
        edges.append(Edge(attn, o, (1, 0, -1), (-1, -1, -1)))
        # h after O -> MLP-up reads all of it
        edges.append(Edge(o, up, (1, -1, -1), (-1, -1, -1)))
        # act [B, F]: up cuts F by tiles, down cuts F by K chunks
        edges.append(Edge(up, down, (1, -1, -1), (-1, 1, -1)))
        prev = down
    ops.append(Op("lm", (_ceil(shape.V, k.rows_lm), 1, 1), cost=rows_cost(shape.V, k.rows_lm, shape.H, wbytes=2)))
    kinds["lm"] = ("lm", -1)
    edges.append(Edge(prev, "lm", (1, -1, -1), (-1, -1, -1)))
    # the embed op writes all of h with one task: its out_map cuts nothing
    edges[0] = Edge("embed", "qkv0", (-1, -1, -1), (-1, -1, -1))
    return ops, edges, kinds


def _round_up(x, a):
    return -(-x // a) * a


def llama_knobs(shape: LlamaShape, B: int, seq0: Sequence[int], max_steps: int, n_workers: int,
                smem_per_cta: int, fp8: bool = False) -> Knobs:
    """Tile knobs of a plan of GEMV tiles (batch 1..8), from the stated rules.

    * FP8 projections (batch 1, every projection K = 2048): the same knobs as
      bf16 (the row-per-warp tiles then hold 32 e4m3 rows per 64 KB page), one
      byte per projection weight in the task costs.

    * Rows per tile: the most rows (a power of two) of K bf16 values that fit a
      64 KB tile (128 KB when every K is a multiple of 512 at batch above 1:
      the warp-level tensor-core tiles take two pages), at most 16 (8 at batch
      above 4 without those tiles), MLP-up half of that; MLP-down's K chunk is
      the largest multiple of 8 up to 2048 that divides the ffn.
    * The page: 64 KB when three fit beside the fixed buffers (two activation
      buffers of batch x the longest K in fp32 when both fit in 32 KB, else
      one; two slots for the attention staging and the O residual rows; the
      attention scores and 4 reduction buffers; barriers and flags), else
      32 KB, else 16 KB; the tensor-core tiles at K = 4096 take 64 KB pages of
      8 rows with a single activation buffer.
    * Batch 1 with pages of exactly 16 rows: QKV 32 rows, MLP-up 64 gate rows,
      MLP-down 64 rows, LM head one tile per worker (whole pages).
    * Batch above 4 without the tensor-core tiles' pages: at most 8 rows (MLP-up 4).
    * Attention: 16384 / (2 head_dim) positions, doubled up to 512 while the
      attention tasks outnumber the workers.
    """
    H, Hq, Hkv, D, F, V = shape.H, shape.Hq, shape.Hkv, shape.D, shape.F, shape.V
    G = Hq // Hkv
    WARPS, TILE_ROWS, RESID, NRED, MBAR, CTRL = 8, 16, 16, 4, 512, 256

    def pow2_floor(v):
        r = 1
        while r * 2 <= v:
            r *= 2
        return r

    clamp = lambda v, lo, hi: max(lo, min(hi, v))
    mma = H % 512 == 0 and (Hq * D) % 512 == 0 and min(F, 2048) % 512 == 0
    rcap = 8 if B > 4 and not mma else 16
    tile = 2 * 65536 if mma else 65536
    qkv = pow2_floor(clamp(tile // (2 * H), 1, rcap))
    o = pow2_floor(clamp(tile // (2 * Hq * D), 1, rcap))
    up = pow2_floor(clamp(tile // (4 * H), 1, rcap // 2))
    kc = 8
    for c in range(8, min(F, 2048) + 1, 8):
        if F % c == 0:
            kc = c
    down = pow2_floor(clamp(tile // (2 * kc), 1, rcap))
    lm = pow2_floor(clamp(tile // (2 * H), 1, rcap))
    T = clamp(16384 // (2 * D), 16, 256)
    while 2 * T <= 512 and sum(_ceil(s + max_steps, T) for s in seq0) * Hkv > n_workers:
        T *= 2
    # shared memory beside the pages
    kmax = max(H, Hq * D, kc)
    abuf = _round_up(B * kmax * 4, 128)
    act = _round_up((G * (D + 16) + 2 * D) * 4 + B * RESID * 4, 128)
    maxb = 1 if B <= 1 else 2 if B <= 2 else 4 if B <= 4 else 8
    red = _round_up(WARPS * TILE_ROWS * maxb * 4, 128)
    aux = _round_up((WARPS * _ceil(T, WARPS // G) + 32) * 4, 128) + NRED * red
    nbuf = 2 if 2 * abuf <= 32768 else 1
    fixed = nbuf * abuf + 2 * act + aux + MBAR + CTRL
    page = 16384
    for pb in (65536, 32768):
        if (smem_per_cta - fixed) // pb >= 3:
            page = pb
            break
    if mma and page < 16 * kmax and nbuf == 2 and 16 * kmax <= 65536 and \
            (smem_per_cta - (fixed - abuf)) // (16 * kmax) >= 3:
        page = 16 * kmax
    multi = lambda K: B == 1 and K % 256 == 0 and K <= 2048 and page == 32 * K
    if multi(H):
        lm = 16 * min(64, _ceil(_ceil(V, 16), n_workers))
        if F % 64 == 0:
            up = 64
        if D % 32 == 0:
            qkv = 32
    if multi(kc) and H % 64 == 0:
        down = 64
    mma_pages = mma and all(page // (2 * K) >= 8 and K % 512 == 0 for K in (H, Hq * D, kc))
    if B > 4 and not mma_pages:
        qkv, o, down, lm, up = min(qkv, 8), min(o, 8), min(down, 8), min(lm, 8), min(up, 4)
    return Knobs(qkv, o, up, down, kc, lm, T, 1 if fp8 else 2)


@dataclass
class TcKnobs:
    ksplit_qkv: int   # K splits of the QKV tiles
    ksplit_o: int     # K splits of the O tiles
    kchunk_down: int  # K extent of one MLP-down tile
    attn_split: int   # cache positions per attention task


TC_M, TC_SEG, TC_KS = 128, 64, 128   # tile rows, segment rows, K columns per stage


def tc_knobs(shape: LlamaShape, B: int, seq0: Sequence[int], max_steps: int, n_workers: int) -> TcKnobs:
    """Tile knobs of a tensor-core plan, from the stated rules: a K split is
    the largest power of two up to 8 that keeps the op's tasks within the
    workers with whole 128-column stages; the MLP-down K chunk is the largest
    of 1024, 512, 256 dividing the ffn that gives at least half as many
    tasks as workers (else the smallest that divides); the attention split is
    16384 / (2 head_dim) positions, doubled up to 512 while the attention
    tasks outnumber the workers."""
    G = shape.Hq // shape.Hkv

    def ksplit(tiles, K):
        k = 1
        while k < 8 and tiles * k * 2 <= n_workers and K % (k * 2) == 0 and (K // (k * 2)) % TC_KS == 0:
            k *= 2
        return k

    kc = 0
    for c in (1024, 512, 256):
        if shape.F % c == 0:
            kc = c
            if (shape.H // TC_M) * (shape.F // c) * 2 >= n_workers:
                break
    T = max(16, min(256, 16384 // (2 * shape.D)))
    while 2 * T <= 512 and sum(_ceil(s + max_steps, T) for s in seq0) * shape.Hkv > n_workers:
        T *= 2
    return TcKnobs(ksplit(shape.Hkv * (G + 2) * shape.D // TC_M, shape.H), ksplit(shape.H // TC_M, shape.Hq * shape.D),
                   kc, T)


def llama_tc_step_ops(shape: LlamaShape, k: TcKnobs, B: int, seq0: Sequence[int], max_steps: int):
    """The decode step on tensor-core tiles of 128 weight rows: per layer an
    RMSNorm task per sequence, QKV tiles (K split), attention, O tiles (K
    split, added into the residual), the MLP RMSNorm, MLP-up tiles of 64 gate
    + 64 up rows, MLP-down tiles per K chunk; then the final RMSNorm and the
    LM-head tiles.  The same rules (gcd / lcm events) turn it into a plan."""
    G = shape.Hq // shape.Hkv
    rows_group = (G + 2) * shape.D
    nsplit = [_ceil(s + max_steps, k.attn_split) for s in seq0[:B]]
    ns_max = max(nsplit)
    H, QD = shape.H, shape.Hq * shape.D

    def attn_rows(bid):
        g, b, s = bid
        return max(0, min(k.attn_split, seq0[b] + max_steps - 1 - s * k.attn_split))

    ops: List[Op] = [Op("embed", (1, 1, 1), cost=lambda bid: B * H * 2)]
    kinds = {"embed": ("embed", -1)}
    edges: List[Edge] = []
    whole = lambda a, b: edges.append(Edge(a, b, (-1, -1, -1), (-1, -1, -1)))
    prev = "embed"
    for l in range(shape.L):
        na, qkv, attn, o, nm, up, down = (f"{n}{l}" for n in ("norma", "qkv", "attn", "o", "normm", "up", "down"))
        ops.append(Op(na, (B, 1, 1), cost=lambda bid: H * 2))
        ops.append(Op(qkv, (shape.Hkv, rows_group // TC_M, k.ksplit_qkv), cost=lambda bid: TC_M * (H // k.ksplit_qkv) * 2))
        ops.append(Op(attn, (shape.Hkv, B, ns_max), exists=lambda bid: bid[2] < nsplit[bid[1]],
                      cost=lambda bid: 2 * shape.D * 2 * attn_rows(bid)))
        ops.append(Op(o, (H // TC_M, k.ksplit_o, 1), cost=lambda bid: TC_M * (QD // k.ksplit_o) * 2))
        ops.append(Op(nm, (B, 1, 1), cost=lambda bid: H * 2))
        ops.append(Op(up, (shape.F // TC_SEG, 1, 1), cost=lambda bid: TC_M * H * 2))
        ops.append(Op(down, (H // TC_M, shape.F // k.kchunk_down, 1), cost=lambda bid: TC_M * k.kchunk_down * 2))
        for n, kind in ((na, "norm"), (qkv, "qkv"), (attn, "attn"), (o, "o"), (nm, "norm"), (up, "up"),
                        (down, "down")):
            kinds[n] = (kind, l)
        whole(prev, na)                                   # the residual, read whole
        whole(na, qkv)                                    # x^, read whole
        edges.append(Edge(qkv, attn, (1, 2, -1), (1, 0, -1)))   # the K-split axis reduces
        edges.append(Edge(attn, o, (1, 0, -1), (-1, -1, -1)))
        whole(o, nm)
        whole(nm, up)
        edges.append(Edge(up, down, (1, -1, -1), (-1, 1, -1)))
        prev = down
    ops.append(Op("normf", (B, 1, 1), cost=lambda bid: H * 2))
    ops.append(Op("lm", (_ceil(shape.V, TC_M), 1, 1), cost=lambda bid: min(TC_M, shape.V - bid[0] * TC_M) * H * 2))
    kinds["normf"] = ("norm", -1)
    kinds["lm"] = ("lm", -1)
    whole(prev, "normf")
    whole("normf", "lm")
    return ops, edges, kinds


def _queue(tasks: List[PlannedTask], graph: rules.TaskGraph, n_workers: int) -> Tuple[List[List[int]], int]:
    q = rules.greedy_balance(range(len(tasks)), [t.cost for t in tasks], n_workers)
    return rules.pad_queues(q)


def llama_step_plan(shape: LlamaShape, k, B: int, seq0: Sequence[int], max_steps: int,
                    n_workers: int) -> Plan:
    """Plan one decode step; the same plan serves ``max_steps`` consecutive steps.
    ``k`` is a ``Knobs`` (GEMV tiles) or a ``TcKnobs`` (tensor-core tiles).

    Tasks inside each event's successor range are placed longest-first (only
    attention tasks differ in size), then dealt to workers greedily by bytes in
    that order.  The step ends with an extra event that every LM-head task
    triggers; the next step's embedding task waits on it one epoch back.
    """
    if isinstance(k, TcKnobs):
        ops, edges, kinds = llama_tc_step_ops(shape, k, B, seq0, max_steps)
    else:
        ops, edges, kinds = llama_step_ops(shape, k, B, seq0, max_steps)
    g = rules.build_task_graph(ops, edges)
    opmap = {o.name: o for o in ops}
    cost = [opmap[t.op].cost(t.bid) for t in g.tasks]
    # longest-first inside every successor range (stable), then renumber
    ranges = [(0, len(g.first_tasks))] + [(e.first_task_id, e.last_task_id) for e in g.events]
    order = rules.longest_first_within(sorted(ranges), cost)
    new_id = {old: new for new, old in enumerate(order)}
    step_done = len(g.events)
    thresholds = [e.num_triggers for e in g.events] + [0]
    tasks: List[PlannedTask] = []
    for old in order:
        t = g.tasks[old]
        kind, layer = kinds[t.op]
        waits, signals = [], []
        if t.dependent_event is not None:
            waits.append((t.dependent_event, g.events[t.dependent_event].num_triggers, 0))
        if t.trigger_event is not None:
            signals.append((t.trigger_event, 1))
        if kind == "lm":
            signals.append((step_done, 1))
            thresholds[step_done] += 1
        tasks.append(PlannedTask(t.op, kind, layer, t.bid, cost[old], waits, signals))
    # the embedding task waits for the previous step's LM head (epoch offset -1)
    for t in tasks:
        if t.kind == "embed":
            t.waits.append((step_done, thresholds[step_done], -1))
    # remap event first/last ids are unchanged by a within-range permutation
    assert sorted(new_id.values()) == list(range(len(order)))
    queues, lmax = _queue(tasks, g, n_workers)
    return Plan(tasks, thresholds, queues, lmax, g)


# ---------------------------------------------------------------------------
# MegaRTP GLM pre-attention plan (M=16, KV=8192)
# ---------------------------------------------------------------------------

GLM_TILE_COUNTS = {"A0": 16, "B0": 84, "C0": 48, "B1": 8, "D1": 128, "D0": 128, "D2": 256, "E1": 64}


def megartp_glm_plan(n_workers: int = 148):
    """The article's plan: tiles A0 16, B0 1*21*4, C0 1*12*4, B1 8, D1 1*32*4,
    D0 1*64*2, D2 1*64*4, E1 4*16 (732), listed in that order.  Publications:
    event0 (A0's 16 hidden/scale rows, whole) feeds B0 and B1; event1 (A0's 16
    norm rows, whole) feeds C0; event2 (16 final B0 Q/scale tiles) feeds D0
    and D1; event3 (48 C0 partials, tile_reduce) feeds D1; events 4-67 (D0's
    128 tiles, tile_cover in pairs, one per head) feed D2; event68 (32 D1
    Indexer-Q tiles) and event69 (B1's cache write, threshold 1) feed E1.

    Which 16 of B0's and 32 of D1's tiles publish is not stated; the last ones
    are taken (parity unpinned for that mapping).
    """
    order = list(GLM_TILE_COUNTS)
    base, n = {}, 0
    for op in order:
        base[op] = n
        n += GLM_TILE_COUNTS[op]
    thresholds: List[int] = []
    waits: Dict[int, List[Tuple[int, int]]] = {i: [] for i in range(n)}
    signals: Dict[int, List[Tuple[int, int]]] = {i: [] for i in range(n)}

    def publish(op, publishers, strategy, k, consumers):
        ths = rules.pairing(strategy, len(publishers), k)
        first = len(thresholds)
        thresholds.extend(ths)
        per = len(publishers) // len(ths)
        for j, t in enumerate(publishers):
            signals[base[op] + t].append((first + j // per, 1))
        for cop in consumers:
            nc = GLM_TILE_COUNTS[cop]
            cper = nc // len(ths)
            for c in range(nc):
                ev = first + c // cper
                waits[base[cop] + c].append((ev, thresholds[ev]))

    a0 = list(range(16))
    publish("A0", a0, rules.WHOLE, 16, ["B0", "B1"])                       # event 0
    publish("A0", a0, rules.WHOLE, 16, ["C0"])                             # event 1
    publish("B0", list(range(84 - 16, 84)), rules.WHOLE, 16, ["D0", "D1"])  # event 2
    publish("C0", list(range(48)), rules.TILE_REDUCE, 48, ["D1"])          # event 3
    publish("D0", list(range(128)), rules.TILE_COVER, 2, ["D2"])           # events 4..67
    publish("D1", list(range(128 - 32, 128)), rules.WHOLE, 32, ["E1"])     # event 68
    publish("B1", [7], rules.WHOLE, 1, ["E1"])                             # event 69
    queues = rules.round_robin(n, n_workers)
    padded, lmax = rules.pad_queues(queues)
    return {"n_tasks": n, "thresholds": thresholds, "waits": waits, "signals": signals,
            "queues": padded, "lmax": lmax, "base": base}
