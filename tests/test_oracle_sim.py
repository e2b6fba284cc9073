"""Pins of the queue simulator and the lecture's race demo."""
import json
import os
import random

import numpy as np

from conftest import GOLDEN
from oracle import plans, rules, sim

with open(os.path.join(GOLDEN, "plan_counts.json")) as f:
    TOY = json.load(f)["toy_net"]


def test_toy_net_counts():
    deps = sim.toy_pairwise_deps()
    assert len(deps) == TOY["tasks"]
    assert sum(len(s) for s in deps.values()) == TOY["pairwise_edges"]
    assert sim.merge_identical_dep_sets(deps) == TOY["events"]
    assert all(len(deps[("tanh", i)]) == TOY["tanh_deps"] for i in range(4))
    assert all(len(deps[("gemv4", i)]) == TOY["segment_deps"] for i in range(4))
    a, i, b, j = TOY["deleted_edge"]
    assert (a, i) in deps[(b, j)]
    # the gcd rule on the same network gives the same 9 events
    ops, edges = sim.toy_graph()
    g = rules.build_task_graph(ops, edges)
    assert len(g.tasks) == TOY["tasks"] and len(g.events) == TOY["events"]
    assert g.pairwise_edges() == TOY["pairwise_edges"]


def test_race_demo():
    d = sim.toy_data(0)
    ref = sim.toy_direct(d)
    deps = sim.toy_pairwise_deps()
    outs = [sim.toy_interpreter(d, TOY["workers"], deps, random.Random(s)) for s in range(TOY["interleavings"])]
    assert all(np.max(np.abs(o - ref)) < 1e-12 for o in outs)
    # split-K partials land in execution order: bitwise results differ between interleavings
    assert len({o.tobytes() for o in outs}) > 1
    a, i, b, j = TOY["deleted_edge"]
    broken = {k: set(v) for k, v in deps.items()}
    broken[(b, j)].discard((a, i))
    wrong = 0
    for s in range(TOY["interleavings"]):
        o = sim.toy_interpreter(d, TOY["workers"], broken, random.Random(s))
        wrong += not np.all(np.abs(o - ref) < 1e-9)
    assert 0 < wrong < TOY["interleavings"]
    # one worker runs the queue in topological order: never wrong
    for s in range(5):
        o = sim.toy_interpreter(d, 1, broken, random.Random(s))
        assert np.max(np.abs(o - ref)) < 1e-12


def _plan_waits(p):
    waits = {i: t.waits for i, t in enumerate(p.tasks)}
    sigs = {i: t.signals for i, t in enumerate(p.tasks)}
    return waits, sigs


def test_llama_plan_is_deadlock_free_over_steps():
    shape = plans.LlamaShape(L=2, H=256, Hq=4, Hkv=2, D=64, F=688, V=1024)
    kn = plans.Knobs(rows_qkv=16, rows_o=16, rows_up=8, rows_down=16, kchunk_down=688, rows_lm=16, attn_split=32)
    p = plans.llama_step_plan(shape, kn, 2, [64, 40], 3, 7)
    waits, sigs = _plan_waits(p)
    r = sim.deadlock_check(p.queues, waits, sigs, len(p.thresholds), steps=3)
    assert r.ok
    assert r.counters == rules.expected_counters(p.thresholds, 3)
    for s in range(5):
        r = sim.deadlock_check(p.queues, waits, sigs, len(p.thresholds), steps=3, rng=random.Random(s))
        assert r.ok


def test_deadlock_detected():
    # two workers, each waiting first for what the other signals later
    waits = {0: [(1, 1)], 1: [], 2: [(0, 1)], 3: []}
    sigs = {0: [], 1: [(0, 1)], 2: [], 3: [(1, 1)]}
    r = sim.deadlock_check([[0, 1], [2, 3]], waits, sigs, 2)
    assert not r.ok and sorted(r.blocked) == [(0, 0), (1, 2)]
    # an unreachable threshold blocks too
    r = sim.deadlock_check([[0]], {0: [(0, 2)]}, {}, 1)
    assert not r.ok
    # a queue that is not a subsequence of a topological order can deadlock on one worker
    r = sim.deadlock_check([[2, 1]], {2: [(0, 1)], 1: []}, {1: [(0, 1)], 2: []}, 1)
    assert not r.ok


def test_waits_target_the_current_epoch():
    """Counters are never reset: at step s a wait of threshold t needs t x (s + 1).
    Worker 0's consumer must wait for worker 1's producer in every step, not
    only the first."""
    waits = {0: [(0, 1)], 1: []}
    sigs = {0: [], 1: [(0, 1)]}
    r = sim.deadlock_check([[0], [1]], waits, sigs, 1, steps=3)
    assert r.ok and r.order == [1, 0, 1, 0, 1, 0] and r.counters == [3]


def test_wait_one_epoch_back():
    """A wait with epoch offset -1 at step s needs t x s: nothing at the first
    step, the previous step's signals after that."""
    waits = {0: [(0, 1, -1)], 1: []}
    sigs = {0: [], 1: [(0, 1)]}
    r = sim.deadlock_check([[0], [1]], waits, sigs, 1, steps=2)
    assert r.ok and r.order == [0, 1, 0, 1]
