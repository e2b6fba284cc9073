"""Pins of the oracle's planner rules against values the pages print."""
import json
import math
import os

from conftest import GOLDEN
from oracle import plans, rules, tail


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


MPK = _golden("mpk_examples.json")
COUNTS = _golden("plan_counts.json")


def test_build_partition_example():
    ex = MPK["build_partition"]
    assert rules.build_partition(ex["grid"], ex["map"]) == ex["part"]


def _fabg():
    g = MPK["fork_join"]["grids"]
    ops = [rules.Op(n, tuple(g[n])) for n in ("F", "A", "B", "G")]
    x = (0, -1, -1)
    edges = [rules.Edge("F", "A", x, x), rules.Edge("F", "B", x, x),
             rules.Edge("A", "G", x, x), rules.Edge("B", "G", x, x)]
    return ops, edges


def test_raw_gcd_per_edge():
    ops, edges = _fabg()
    opm = {o.name: o for o in ops}
    raw = MPK["fork_join"]["raw_event_dim_x"]
    for e in edges:
        pp = rules.build_partition(opm[e.prod].grid, e.out_map)
        cp = rules.build_partition(opm[e.cons].grid, e.in_map)
        assert math.gcd(pp[0], cp[0]) == raw[f"{e.prod}->{e.cons}"]


def test_fork_join_worked_example():
    ops, edges = _fabg()
    ex = MPK["fork_join"]
    g = rules.build_task_graph(ops, edges)
    ee = g.edge_events
    # fork: both F edges end with 2 events; join: both G edges end with 2
    assert ee[0].event_dim[0] == ee[1].event_dim[0] == ex["fork_events"]
    assert ee[2].event_dim[0] == ee[3].event_dim[0] == ex["join_events"]
    assert ee[0].prod_group(0) == ex["fork_lcm"] and ee[2].cons_group(0) == ex["join_lcm"]
    t = g.tasks
    # fork events: F tasks {0,1} trigger event 0, {2,3} event 1
    f_trig = {}
    for tt in t:
        if tt.op == "F":
            f_trig.setdefault(tt.trigger_event, []).append(tt.bid[0])
    assert sorted(f_trig.values()) == ex["fork_event_producers"]
    ev0 = g.events[f_trig_key(f_trig, [0, 1])]
    fired = {}
    for i in range(ev0.first_task_id, ev0.last_task_id):
        fired.setdefault(t[i].op, []).append(t[i].bid[0])
    assert fired == ex["fork_event0_fires"]
    # join events
    g_events = sorted({tt.dependent_event for tt in t if tt.op == "G"})
    assert [g.events[e].num_triggers for e in g_events] == ex["join_num_triggers"]
    rel = [[t[i].bid[0] for i in range(g.events[e].first_task_id, g.events[e].last_task_id)] for e in g_events]
    assert rel == ex["join_event_releases"]["G"]
    # successors of every event are contiguous and every non-first task has one
    for i, tt in enumerate(t):
        if tt.dependent_event is not None:
            ev = g.events[tt.dependent_event]
            assert ev.first_task_id <= i < ev.last_task_id


def f_trig_key(d, members):
    return [k for k, v in d.items() if v == members][0]


def test_gcd_examples():
    for ex in MPK["gcd_examples"]:
        ops = [rules.Op("P", (ex["prod"], 1, 1)), rules.Op("C", (ex["cons"], 1, 1))]
        g = rules.build_task_graph(ops, [rules.Edge("P", "C", (0, -1, -1), (0, -1, -1))])
        assert len(g.events) == ex["events"]
        assert all(e.num_triggers == ex["producers_per_event"] for e in g.events)
        # every consumer task waits on exactly one event
        assert sum(e.last_task_id - e.first_task_id for e in g.events) == ex["cons"]


def test_fork_with_coprime_consumer_groups_merges_to_one_event():
    # producer cut 6; consumers cut 4 and 3 -> producer groups 3 and 2 -> lcm 6 divides 6 -> one event
    ops = [rules.Op("P", (6, 1, 1)), rules.Op("A", (4, 1, 1)), rules.Op("B", (3, 1, 1))]
    x = (0, -1, -1)
    g = rules.build_task_graph(ops, [rules.Edge("P", "A", x, x), rules.Edge("P", "B", x, x)])
    assert len(g.events) == 1 and g.events[0].num_triggers == 6
    # producer cut 4; consumers 4 and 3 -> groups 1 and 4 -> lcm 4 divides 4 -> 1 event
    ops = [rules.Op("P", (4, 1, 1)), rules.Op("A", (4, 1, 1)), rules.Op("B", (3, 1, 1))]
    g = rules.build_task_graph(ops, [rules.Edge("P", "A", x, x), rules.Edge("P", "B", x, x)])
    assert len(g.events) == 1


def test_pairing_strategies():
    assert rules.pairing(rules.WHOLE, 16) == [16]
    assert rules.pairing(rules.TILE, 3) == [1, 1, 1]
    assert rules.pairing(rules.TILE_COVER, 128, 2) == [2] * 64
    assert rules.pairing(rules.TILE_REDUCE, 48, 48) == [48]
    assert rules.check_cover([(0, 8), (8, 16)], (0, 16))
    assert not rules.check_cover([(0, 8), (4, 16)], (0, 16))
    assert rules.check_reduce([(0, 16)] * 3, (0, 16))
    assert not rules.check_reduce([(0, 16), (0, 8)], (0, 16))


def test_megartp_glm_plan_counts():
    ex = COUNTS["megartp_glm"]
    p = plans.megartp_glm_plan(ex["workers"])
    assert p["n_tasks"] == ex["n_tasks"] == sum(ex["tile_counts"].values())
    th = p["thresholds"]
    assert len(th) == ex["n_events"]
    assert th[:4] == ex["thresholds_head"]
    assert th[4:68] == [ex["d0_pair_threshold"]] * ex["d0_pair_events"]
    assert th[68] == ex["event68_threshold"] and th[69] == ex["event69_threshold"]
    q = p["queues"]
    assert [len(q), p["lmax"], 32] == ex["queue_shape"]
    lens = [sum(1 for t in row if t >= 0) for row in q]
    assert lens.count(5) == ex["workers_with_5"] and lens.count(4) == ex["workers_with_4"]
    # D1 joins B0 and C0: it waits on event2 >= 16 and event3 >= 48
    d1 = p["base"]["D1"]
    assert p["waits"][d1] == [(2, 16), (3, 48)]
    e1 = p["base"]["E1"]
    assert p["waits"][e1] == [(68, 32), (69, 1)]
    # every publication reaches its threshold exactly
    from collections import Counter
    got = Counter(ev for s in p["signals"].values() for ev, _ in s)
    assert [got[i] for i in range(len(th))] == th


LLAMA1B = plans.LlamaShape(L=16, H=2048, Hq=32, Hkv=8, D=64, F=8192, V=128256)
KN = plans.Knobs(rows_qkv=16, rows_o=16, rows_up=8, rows_down=16, kchunk_down=2048, rows_lm=16, attn_split=64)


def test_llama1b_layer_counts():
    """Lecture section 6.2: one Llama-1B layer = 1,984 tasks, 15 events,
    3,968 task-event edges, about 380k pairwise edges (attention over 1024
    cached positions in 16 splits)."""
    ex = COUNTS["llama1b_layer"]
    shape = plans.LlamaShape(L=2, **{k: getattr(LLAMA1B, k) for k in ("H", "Hq", "Hkv", "D", "F", "V")})
    ops, edges, kinds = plans.llama_step_ops(shape, KN, 1, [1023], 1)
    g = rules.build_task_graph(ops, edges)
    layer1 = [i for i, t in enumerate(g.tasks) if kinds[t.op][1] == 1]
    assert len(layer1) == ex["tasks"]
    evs = sorted({g.tasks[i].dependent_event for i in layer1})
    assert len(evs) == ex["events"]
    edges_te = sum((g.tasks[i].dependent_event is not None) + (g.tasks[i].trigger_event is not None) for i in layer1)
    assert edges_te == ex["task_event_edges"]
    pairwise = sum(g.events[e].num_triggers * (g.events[e].last_task_id - g.events[e].first_task_id) for e in evs)
    assert abs(pairwise - ex["pairwise_edges_approx"]) / ex["pairwise_edges_approx"] < 0.01
    assert pairwise == 379904
    assert sum(1 for i in layer1 if kinds[g.tasks[i].op][0] == "qkv") == ex["qkv_tasks"]


def test_llama1b_forward_task_count():
    ex = COUNTS["llama1b_layer"]
    p = plans.llama_step_plan(LLAMA1B, KN, 1, [1023], 1, 132)
    n = len(p.tasks)
    assert abs(n - ex["forward_tasks_approx"]) / ex["forward_tasks_approx"] < 0.01
    # every queue is a subsequence of the task order, which is topological
    for row in p.queues:
        ids = [t for t in row if t >= 0]
        assert ids == sorted(ids)


def test_tail_model():
    ex = COUNTS["tail"]
    m = tail.tail_model(ex["n_tasks"], ex["n_sms"], ex["tile_bytes"], ex["bw"], latency_us=1.1)
    assert (m.waves, m.busy_last_wave, m.idle_last_wave) == (ex["waves"], ex["busy_last"], ex["idle_last"])
    assert round(m.ideal_us, 2) == ex["ideal_us"]
    assert round(m.kernel_us, 2) == ex["kernel_us"]
    assert abs(m.per_task_us - ex["task_read_us_approx"]) < 0.05
    tasks = 3072 // ex["alt_rows"]
    assert tasks == ex["alt_tasks"]
    m2 = tail.tail_model(tasks, ex["n_sms"], ex["alt_tile_bytes"], ex["bw"])
    assert m2.waves == 1 and m2.idle_last_wave == ex["alt_idle"]
    assert abs(m2.kernel_us - ex["alt_us_approx"]) < 0.1
    assert tail.prefetch_depth(ex["pages"], ex["pages_per_task"]) == ex["depth"]
    assert tail.prefetch_depth(ex["pages"], ex["alt_pages_per_task"]) == ex["alt_depth"]


def test_expected_counters():
    assert rules.expected_counters([16, 2, 1], 3) == [48, 6, 3]


def test_attention_splits_cover_every_position():
    """Split-KV: a sequence's splits are 0..n-1 of T positions each and cover
    every position up to the last step's new token, with no split left empty
    (checked on ragged lengths, where rounding matters)."""
    shape = plans.LlamaShape(L=1, H=256, Hq=4, Hkv=2, D=64, F=688, V=1024)
    for seq0, steps, T in (([1000], 1, 64), ([5, 64, 130], 4, 32)):
        kn = plans.Knobs(rows_qkv=16, rows_o=16, rows_up=8, rows_down=16, kchunk_down=688, rows_lm=16,
                         attn_split=T)
        ops, edges, kinds = plans.llama_step_ops(shape, kn, len(seq0), seq0, steps)
        g = rules.build_task_graph(ops, edges)
        for b, s0 in enumerate(seq0):
            splits = sorted({t.bid[2] for t in g.tasks if kinds[t.op][0] == "attn" and t.bid[1] == b})
            assert splits == list(range(len(splits)))
            assert len(splits) * T >= s0 + steps
            assert (len(splits) - 1) * T < s0 + steps
