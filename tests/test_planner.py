"""libmk host side on CPU: exported symbols, and the C++ planner against the
oracle's independent statement of the same rules -- bit for bit."""
import os
import re

from dataclasses import replace

import numpy as np
import pytest

from conftest import ROOT
from oracle import plans, rules, sim
from persistent_megakernel_decode_gb300 import runtime as rt
from persistent_megakernel_decode_gb300 import synth

GB300 = dict(num_sms=152, smem_per_cta=232448)


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_megakernel_decode_gb300 import build
    build.build()


def test_library_exports_every_declared_function():
    hdr = open(os.path.join(ROOT, "include", "mk.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    names = set(re.findall(r"\b(mk_[a-z_]+)\s*\(", hdr))
    assert names == set(rt.EXPORTED)
    lib = rt.load()
    for n in names:
        assert hasattr(lib, n), n


PAGE_TITLES = ("MegaRTP megakernel article", "GEMM + AllToAll fusion post", "CMU 15-779 Lecture 7 notes",
               "MPK code walkthrough")


def test_every_declaration_cites_its_passage():
    """Each exported function's comment names the page (and section) that
    defines the operation, or says that the pages have no counterpart."""
    hdr = open(os.path.join(ROOT, "include", "mk.h")).read()
    decl = re.compile(r"^(?:int|void|int32_t|const char \*)\s*\*?\s*(mk_[a-z_]+)\s*\(", re.M)
    prev_end = 0
    for m in decl.finditer(hdr):
        # the comment text between the previous declaration and this one
        between = hdr[prev_end:m.start()]
        comments = " ".join(re.findall(r"/\*(.*?)\*/", between, flags=re.S))
        text = re.sub(r"\s*\*\s*", " ", comments)
        text = re.sub(r"\s+", " ", text)
        assert any(t in text for t in PAGE_TITLES) or "no counterpart" in text, m.group(1)
        prev_end = m.end()


def test_binding_decodes_argmax_keys_with_the_export():
    import inspect
    src = inspect.getsource(rt.argmax_index)
    assert "mk_argmax_index" in src and "0xFFFFFFFF" not in src
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 151936, 64)
    keys = (rng.integers(0, 2 ** 31, 64).astype(np.uint64) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - idx.astype(np.uint64))
    assert (rt.argmax_index(keys) == idx).all()


def test_build_and_bench_hash_cover_every_source():
    import bench
    from persistent_megakernel_decode_gb300 import build as b
    csrc = sorted(os.listdir(b.CSRC))
    assert sorted(b.SOURCES + b.HEADERS) == csrc
    h0 = bench.kernel_source_hash()
    assert isinstance(h0, str) and len(h0) == 16


def _oracle_knobs(info):
    return plans.Knobs(rows_qkv=info["rows_qkv"], rows_o=info["rows_o"], rows_up=info["rows_up"],
                       rows_down=info["rows_down"], kchunk_down=info["kchunk_down"], rows_lm=info["rows_lm"],
                       attn_split=info["attn_split"])


def _compare(shape, B, seq0, steps, workers=152, fp8=False, **kn):
    # the oracle deals tasks by bytes, the pages' rule (the default time-model
    # schedule is checked for validity below)
    p = rt.Plan.llama(shape, B, seq0, steps, max(seq0) + steps + 3, num_sms=workers, smem_per_cta=232448,
                      schedule=rt.SCHED_BYTES, fp8=fp8, **kn)
    info = p.info()
    assert info["weight_fp8"] == int(fp8)
    q, ids, th, tasks = p.export()
    osh = plans.LlamaShape(shape.L, shape.H, shape.Hq, shape.Hkv, shape.D, shape.F, shape.V)
    tile_knobs = {k: v for k, v in kn.items() if k != "tc_tiles"}
    if tile_knobs:  # a test that sets tile knobs itself: the oracle takes the same
        okn = _oracle_knobs(info)
    else:           # defaults: the oracle derives them from its own statement of the rules
        okn = plans.llama_knobs(osh, B, seq0, steps, workers, 232448, fp8=fp8)
        assert okn == replace(_oracle_knobs(info), wbytes=okn.wbytes), (okn, _oracle_knobs(info))
    op = plans.llama_step_plan(osh, okn, B, seq0, steps, workers)
    assert info["num_tasks"] == len(op.tasks)
    assert list(th) == op.thresholds
    for i, t in enumerate(op.tasks):
        r = tasks[i]
        assert rt.OP_NAMES[r[0]] == t.kind, i
        assert (r[1], r[2], r[3], r[4], r[5]) == (t.layer, *t.bid, t.cost), i
        assert [(r[7 + 3 * k], r[8 + 3 * k], r[9 + 3 * k]) for k in range(r[6])] == list(t.waits), i
        assert [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] == list(t.signals), i
    assert info["lmax"] == op.lmax
    assert ids.tolist() == op.queues
    # instruction words carry the same waits/signals as the task table
    for w in range(ids.shape[0]):
        for s in range(ids.shape[1]):
            t = ids[w, s]
            if t < 0:
                assert not q[w, s].any()
            else:
                assert q[w, s, 0] == tasks[t][0] and q[w, s, 3] == t
    return p, op


def _compare_tc(shape, B, seq0, steps, workers=152):
    """Tensor-core plans against the oracle's statement, which derives its own
    tile knobs (K splits, MLP-down K chunk, attention split) from the rules."""
    p = rt.Plan.llama(shape, B, seq0, steps, max(seq0) + steps + 3, num_sms=workers, smem_per_cta=232448,
                      schedule=rt.SCHED_BYTES)
    info = p.info()
    assert info["tc_tiles"] == 1
    q, ids, th, tasks = p.export()
    osh = plans.LlamaShape(shape.L, shape.H, shape.Hq, shape.Hkv, shape.D, shape.F, shape.V)
    kn = plans.tc_knobs(osh, B, seq0, steps, workers)
    assert (info["ksplit_qkv"], info["ksplit_o"], info["kchunk_down"], info["attn_split"]) == \
        (kn.ksplit_qkv, kn.ksplit_o, kn.kchunk_down, kn.attn_split)
    op = plans.llama_step_plan(osh, kn, B, seq0, steps, workers)
    assert info["num_tasks"] == len(op.tasks)
    assert list(th) == op.thresholds
    for i, t in enumerate(op.tasks):
        r = tasks[i]
        assert rt.OP_NAMES[r[0]] == t.kind, i
        assert (r[1], r[2], r[3], r[4], r[5]) == (t.layer, *t.bid, t.cost), i
        assert [(r[7 + 3 * k], r[8 + 3 * k], r[9 + 3 * k]) for k in range(r[6])] == list(t.waits), i
        assert [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] == list(t.signals), i
    assert info["lmax"] == op.lmax
    assert ids.tolist() == op.queues
    return p, op


def test_tc_planner_matches_oracle_small_shapes():
    _compare_tc(synth.TINY_TC, 16, [64 + 3 * b for b in range(16)], 4)
    _compare_tc(synth.SMALL_QK, 11, [40 + 17 * b for b in range(11)], 3, workers=37)


def test_tc_planner_matches_oracle_qwen3_8b_b16():
    w = synth.WORKLOADS["qwen3_8b_b16"]
    p, op = _compare_tc(synth.QWEN3_8B, 16, synth.seq_lengths(w), w.steps)
    info = p.info()
    assert (info["ksplit_qkv"], info["ksplit_o"], info["kchunk_down"]) == (2, 4, 1024)


def test_tc_planner_matches_oracle_llama1b_b8():
    w = synth.WORKLOADS["llama1b_b8"]
    p, op = _compare_tc(synth.LLAMA_1B, 8, synth.seq_lengths(w), w.steps)
    assert p.info()["kchunk_down"] == 1024


def test_tc_plan_needs_shapes_in_128s():
    # batch above 8 needs the tensor-core tiles; the tiny decoder's ffn of 688 does not allow them
    with pytest.raises(rt.MkError) as e:
        rt.Plan.llama(synth.TINY, 12, [10] * 12, 2, 20, **GB300)
    assert e.value.code == rt.MK_ERR_UNSUPPORTED
    with pytest.raises(rt.MkError):
        rt.Plan.llama(synth.TINY, 4, [10] * 4, 2, 20, tc_tiles=1, **GB300)
    # and batch 8 can still opt out of them
    p = rt.Plan.llama(synth.LLAMA_1B, 8, [100] * 8, 2, 120, tc_tiles=-1, **GB300)
    assert p.info()["tc_tiles"] == 0


def test_planner_matches_oracle_tiny():
    _compare(synth.TINY, 1, [64], 8)


def test_planner_matches_oracle_tiny_ragged_batch():
    _compare(synth.TINY, 3, [5, 64, 130], 4, workers=7, attn_split=32, rows_qkv=8, rows_o=4, rows_lm=8)


def test_planner_matches_oracle_llama1b_b1():
    p, op = _compare(synth.LLAMA_1B, 1, [1024], 128)
    assert p.info()["num_events"] == 16 * 15 + 2


def test_planner_matches_oracle_llama1b_b8_variable_lengths():
    # the warp-level tensor-core tiles (batch 8 takes tcgen05 tiles by default)
    w = synth.WORKLOADS["llama1b_b8"]
    _compare(synth.LLAMA_1B, 8, synth.seq_lengths(w), 64, tc_tiles=-1)


def test_planner_matches_oracle_qwen3_8b_b1():
    _compare(synth.QWEN3_8B, 1, [2048], 32, workers=148)


@pytest.mark.parametrize("name,shape,B,steps,want", [
    ("llama1b_b1", synth.LLAMA_1B, 1, 128, 128),   # 1152 positions / 128 = 9 splits x 8 kv heads = 72 tasks
    ("qwen3_8b_b1", synth.QWEN3_8B, 1, 32, 128),   # 2080 / 64 = 33 x 8 = 264 > 152; / 128 = 17 x 8 = 136
    ("llama1b_b8", synth.LLAMA_1B, 8, 64, 512),    # thousands of tasks: capped at 512 positions
    ("qwen3_8b_b16", synth.QWEN3_8B, 16, 32, 512), # 16 x 2080 / 256 = 9 x 16 x 8 = 1152 tasks: capped at 512
    ("tiny", synth.TINY, 1, 8, 128),               # 72 positions: one split per kv head
])
def test_attention_split_doubles_while_tasks_outnumber_workers(name, shape, B, steps, want):
    seq0 = synth.seq_lengths(synth.WORKLOADS[name])
    p = rt.Plan.llama(shape, B, seq0, steps, max(seq0) + steps + 1, **GB300)
    T = p.info()["attn_split"]
    assert T == want
    tasks = sum(-(-(s + steps) // T) for s in seq0) * shape.Hkv
    assert T == 512 or tasks <= GB300["num_sms"]
    if T > 16384 // (2 * shape.D):  # doubled: the half split gave more tasks than workers
        assert sum(-(-(s + steps) // (T // 2)) for s in seq0) * shape.Hkv > GB300["num_sms"]


def test_planner_queue_simulates_over_steps():
    p = rt.Plan.llama(synth.TINY, 2, [3, 70], 5, 80, **GB300)
    q, ids, th, tasks = p.export()
    waits = {i: [(r[7 + 3 * k], r[8 + 3 * k], r[9 + 3 * k]) for k in range(r[6])] for i, r in enumerate(tasks)}
    sigs = {i: [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] for i, r in enumerate(tasks)}
    res = sim.deadlock_check(ids.tolist(), waits, sigs, len(th), steps=5)
    assert res.ok and res.counters == rules.expected_counters(th.tolist(), 5)


@pytest.mark.parametrize("shape,B,seq0,workers", [
    (synth.TINY, 3, [5, 64, 130], 7),
    (synth.LLAMA_1B, 1, [1024], 152),
    (synth.LLAMA_1B, 8, [512, 4096, 700, 2300, 1500, 3999, 600, 2048], 152),
])
def test_timed_schedule_is_a_valid_deal_of_the_same_tasks(shape, B, seq0, workers):
    """The time-model schedule deals exactly the byte schedule's tasks, with the
    same waits and signals; the queues are subsequences of one topological
    order (queue order plus producer -> event -> consumer edges form no cycle)
    and deadlock-free over several steps."""
    steps = 3
    kw = dict(num_sms=workers, smem_per_cta=232448)
    pt = rt.Plan.llama(shape, B, seq0, steps, max(seq0) + steps + 3, schedule=rt.SCHED_TIMED, **kw)
    pb = rt.Plan.llama(shape, B, seq0, steps, max(seq0) + steps + 3, schedule=rt.SCHED_BYTES, **kw)
    qt, idt, tht, tt = pt.export()
    qb, idb, thb, tb = pb.export()
    assert (tt == tb).all() and (tht == thb).all()
    ids = idt.tolist()
    flat = sorted(t for row in ids for t in row if t >= 0)
    assert flat == list(range(len(tt)))
    waits = {i: [(r[7 + 3 * k], r[8 + 3 * k], r[9 + 3 * k]) for k in range(r[6])] for i, r in enumerate(tt)}
    sigs = {i: [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] for i, r in enumerate(tt)}
    n, ne = len(tt), len(tht)
    succ = [[] for _ in range(n + ne)]                   # task nodes 0..n-1, event nodes n..n+ne-1
    for row in ids:
        real = [t for t in row if t >= 0]
        assert all(t < 0 for t in row[len(real):])       # NoOps only pad the tail
        for a, b in zip(real, real[1:]):
            succ[a].append(b)
    for i in range(n):
        for e, _ in sigs[i]:
            succ[i].append(n + e)
        for e, _, off in waits[i]:
            if off >= 0:
                succ[n + e].append(i)
    indeg = [0] * (n + ne)
    for v in succ:
        for w in v:
            indeg[w] += 1
    stack = [v for v in range(n + ne) if indeg[v] == 0]
    seen = 0
    while stack:
        v = stack.pop()
        seen += 1
        for w in succ[v]:
            indeg[w] -= 1
            if indeg[w] == 0:
                stack.append(w)
    assert seen == n + ne                                # acyclic: one topological order holds every queue
    res = sim.deadlock_check(ids, waits, sigs, len(tht), steps=steps)
    assert res.ok and res.counters == rules.expected_counters(tht.tolist(), steps)


def test_graph_plan_fork_join_example():
    ops = [dict(grid=(4, 1, 1)), dict(grid=(4, 1, 1)), dict(grid=(2, 1, 1)), dict(grid=(4, 1, 1))]
    x = (0, -1, -1)
    edges = [dict(prod=0, cons=1, out_map=x, in_map=x), dict(prod=0, cons=2, out_map=x, in_map=x),
             dict(prod=1, cons=3, out_map=x, in_map=x), dict(prod=2, cons=3, out_map=x, in_map=x)]
    p = rt.Plan.graph(ops, edges, num_sms=3, smem_per_cta=65536)
    _, ids, th, tasks = p.export()
    g = rules.build_task_graph([rules.Op(n, tuple(o["grid"])) for n, o in zip("FABG", ops)],
                               [rules.Edge("FABG"[e["prod"]], "FABG"[e["cons"]], x, x) for e in edges])
    assert th.tolist() == [e.num_triggers for e in g.events] == [2, 2, 3, 3]
    for i, t in enumerate(g.tasks):
        r = tasks[i]
        assert "FABG"[r[21]] == t.op and r[2] == t.bid[0]
        assert (r[7] if r[6] else None) == t.dependent_event
        assert (r[17] if r[16] else None) == t.trigger_event


def test_graph_plan_gcd_examples():
    for cons, events in ((128, 128), (64, 64), (1, 1), (127, 1)):
        p = rt.Plan.graph([dict(grid=(128, 1, 1)), dict(grid=(cons, 1, 1))],
                          [dict(prod=0, cons=1, out_map=(0, -1, -1), in_map=(0, -1, -1))], num_sms=16,
                          smem_per_cta=65536)
        assert p.info()["num_events"] == events


def test_graph_plan_megartp_glm():
    """MegaRTP article: 732 tile tasks, 70 events, [148, 5, 32] queue, 8-op table of 1024 B."""
    counts = plans.GLM_TILE_COUNTS
    names = list(counts)
    ops = [dict(grid=(counts[n], 1, 1)) for n in names]
    ix = {n: i for i, n in enumerate(names)}
    pubs = [dict(prod=ix["A0"], num_pub=16, strategy=rt.PAIR_WHOLE, cons=[ix["B0"], ix["B1"]]),
            dict(prod=ix["A0"], num_pub=16, strategy=rt.PAIR_WHOLE, cons=[ix["C0"]]),
            dict(prod=ix["B0"], first_pub=68, num_pub=16, strategy=rt.PAIR_WHOLE, cons=[ix["D0"], ix["D1"]]),
            dict(prod=ix["C0"], num_pub=48, strategy=rt.PAIR_TILE_REDUCE, k=48, cons=[ix["D1"]]),
            dict(prod=ix["D0"], num_pub=128, strategy=rt.PAIR_TILE_COVER, k=2, cons=[ix["D2"]]),
            dict(prod=ix["D1"], first_pub=96, num_pub=32, strategy=rt.PAIR_WHOLE, cons=[ix["E1"]]),
            dict(prod=ix["B1"], first_pub=7, num_pub=1, strategy=rt.PAIR_WHOLE, cons=[ix["E1"]])]
    p = rt.Plan.graph(ops, pubs=pubs, round_robin=True, num_sms=148, smem_per_cta=232448)
    info = p.info()
    q, ids, th, tasks = p.export()
    ref = plans.megartp_glm_plan(148)
    assert info["num_tasks"] == 732 and info["num_events"] == 70
    assert list(q.shape) == [148, 5, 32]
    assert th.tolist() == ref["thresholds"]
    assert ids.tolist() == ref["queues"]
    assert info["num_ops"] * 16 * 8 == 1024
    for i in range(732):
        r = tasks[i]
        assert [(r[7 + 3 * k], r[8 + 3 * k]) for k in range(r[6])] == ref["waits"][i]
        assert [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] == ref["signals"][i]


def test_per_op_mode_segments():
    p = rt.Plan.llama(synth.TINY, 1, [64], 2, 80, mode=rt.MODE_PER_OP, **GB300)
    info = p.info()
    assert info["num_launches"] == info["num_ops"] == 2 + 5 * synth.TINY.L
    _, ids, th, tasks = p.export()
    got = sorted(int(t) for t in ids if t >= 0)
    assert got == list(range(info["num_tasks"]))


@pytest.mark.parametrize("bad,code", [
    (dict(batch=9), rt.MK_ERR_UNSUPPORTED),
    (dict(cache_slots=10), rt.MK_ERR_INVALID),
    (dict(rows_qkv=24), rt.MK_ERR_UNSUPPORTED),
    (dict(smem_per_cta=40000), rt.MK_ERR_UNSUPPORTED),
])
def test_planner_rejects(bad, code):
    B = bad.pop("batch", 1)
    cs = bad.pop("cache_slots", 80)
    tgt = dict(GB300)
    tgt.update(bad)
    with pytest.raises(rt.MkError) as e:
        rt.Plan.llama(synth.TINY, B, [64] * B, 8, cs, **tgt)
    assert e.value.code == code


def test_argmax_key_decoding():
    assert rt.load().mk_argmax_index(0xFFFFFFFF) == 0
    assert rt.load().mk_argmax_index((123 << 32) | (0xFFFFFFFF - 77)) == 77


def test_launch_probe_rejects_an_empty_grid():
    rc = rt.load().mk_launch_probe(0, 1, None)
    assert rc == rt.MK_ERR_INVALID and b"num_workers" in rt.load().mk_last_error()


def test_qwen3_8b_batch1_gemv_tiles_fit_the_wide_row_per_warp_path():
    """Every K = 4096 GEMV instruction of the Qwen3-8B batch-1 plan has the
    shape the wide row-per-warp tile takes (64 KB pages of 8 rows, two pages:
    16 rows, or 8 gate + 8 up rows); MLP-down K chunks of 2048 take the
    row-per-warp path with x in registers (16-row pages)."""
    W_P = 14
    P_NROWS, P_KC, P_RPP, P_NPG = W_P + 1, W_P + 3, W_P + 8, W_P + 9
    w = synth.WORKLOADS["qwen3_8b_b1"]
    p = rt.Plan.llama(w.shape, 1, [2048], 32, 2048 + 33, **GB300)
    assert p.info()["page_bytes"] == 65536
    q, ids, _, _ = p.export()
    words = q[ids >= 0]
    seen = set()
    for op in ("qkv", "o", "up", "lm", "down"):
        sel = words[words[:, 0] == rt.OPCODE[op]]
        assert len(sel)
        kc, rows, rpp, npg = sel[:, P_KC], sel[:, P_NROWS], sel[:, P_RPP], sel[:, P_NPG]
        if op == "down":
            assert (kc == 2048).all() and (rpp == 16).all()
        else:
            assert (kc == 4096).all() and (rpp == 8).all() and (npg == 2).all()
            assert ((rows == 8) if op == "up" else (rows == 16)).all()
        seen.add(op)
    assert seen == {"qkv", "o", "up", "lm", "down"}


def test_fp8_plan_matches_the_oracle_and_its_tiles():
    """FP8 projections (Llama-1B width, 2 layers, batch 1): the plan equals the
    oracle's (same knobs, one byte per projection weight in the costs), and
    every projection tile is marked e4m3 with 32 rows to a page, inside one
    128-row block; the LM head stays bf16; the algorithmic bytes count e4m3
    weights and their block scales."""
    from dataclasses import replace as rep
    sh = rep(synth.LLAMA_1B, L=2)
    p, op = _compare(sh, 1, [1024], 4, fp8=True)
    q, ids, th, tasks = p.export()
    P_W8, P_RPP, P_NPG, P_ROW0, P_NROWS = 26, 22, 23, 14, 15
    for w in q.reshape(-1, 32):
        kind = rt.OP_NAMES[w[0]]
        if kind in ("qkv", "o", "up", "down"):
            assert w[P_W8] == 1 and w[P_RPP] == 32, kind
            rows = (2 if kind == "up" else 1) * w[P_NROWS]
            assert w[P_NPG] == -(-rows // 32)
            assert w[P_ROW0] // 128 == (w[P_ROW0] + w[P_NROWS] - 1) // 128
        elif kind == "lm":
            assert w[P_W8] == 0 and w[P_RPP] == 16
    H, QD, KD, F, L, V = sh.H, sh.Hq * sh.D, sh.Hkv * sh.D, sh.F, sh.L, sh.V
    blocks = lambda n, k: -(-n // 128) * (k // 128)
    weights = L * (QD * H + 2 * KD * H + H * QD + 2 * F * H + H * F) + V * H * 2
    scales = L * 4 * (blocks(QD, H) + 2 * blocks(KD, H) + blocks(H, QD) + 2 * blocks(F, H) + blocks(H, F))
    kv = 2 * 1024 * sh.Hkv * sh.D * 2 * L + 2 * sh.Hkv * sh.D * 2 * L
    norms = (2 * L + 1) * H * 2
    assert p.info()["algorithmic_bytes_step"] == weights + scales + H * 2 + kv + norms


# ---------------------------------------------------------------- attention pools

def _pool_plan(B=8, steps=3, workers=152, **kn):
    shape = synth.LLAMA_1B
    seq0 = synth.seq_lengths(synth.WORKLOADS["llama1b_b8"])
    p = rt.Plan.llama(shape, B, seq0[:B], steps, max(seq0[:B]) + steps + 3, num_sms=workers, smem_per_cta=232448,
                      attn_pool=1, **kn)
    return shape, seq0[:B], p


@pytest.mark.parametrize("tc", [0, -1], ids=["tcgen05", "warp_mma"])
def test_attention_pools_one_per_worker_and_layer(tc):
    """attn_pool plans: no host-dealt attention task; every worker holds exactly
    one pool slot per layer; O waits for all of them (threshold = workers); a
    layer's pool waits for its whole QKV op."""
    shape, seq0, p = _pool_plan(tc_tiles=tc)
    info = p.info()
    q, ids, th, tasks = p.export()
    W = info["num_workers"]
    assert not (tasks[:, 0] == rt.OPCODE["attn"]).any()
    pool = tasks[:, 0] == rt.OPCODE["attn_pool"]
    assert pool.sum() == W * shape.L
    for l in range(shape.L):
        rows = np.where(pool & (tasks[:, 1] == l))[0]
        assert sorted(tasks[rows, 2].tolist()) == list(range(W))       # bid[0] = the worker
        ev = set(tasks[rows, 17].tolist())
        assert len(ev) == 1 and th[ev.pop()] == W                       # one event, W signals a step
        waits = {tuple(tasks[r, 7:10]) for r in rows}
        assert len(waits) == 1
        wev, wthr, woff = waits.pop()
        qkv = (tasks[:, 0] == rt.OPCODE["qkv"]) & (tasks[:, 1] == l)
        assert woff == 0 and wthr == qkv.sum() == th[wev]                 # the whole QKV op
    # each worker's queue holds its own pools (slot words carry the worker in the task table)
    for w in range(W):
        mine = [t for t in ids[w] if t >= 0 and tasks[t, 0] == rt.OPCODE["attn_pool"]]
        assert len(mine) == shape.L and all(tasks[t, 2] == w for t in mine)


def test_attention_pool_table_covers_each_task_once_longest_first():
    shape, seq0, p = _pool_plan()
    info = p.info()
    tab = p.attn_table()
    G, T = shape.Hq // shape.Hkv, info["attn_split"]
    nsplit = [-(-(s0 + 3) // T) for s0 in seq0]
    per_layer = shape.Hkv * sum(nsplit)
    assert tab.shape == (shape.L * per_layer, 32)
    P_G, P_B, P_SPLIT, P_T0, P_T, P_NSPLIT, P_LAYER, P_ATHR = range(14, 22)
    q, ids, th, tasks = p.export()
    for l in range(shape.L):
        rows = tab[l * per_layer:(l + 1) * per_layer]
        assert (rows[:, 0] == rt.OPCODE["attn"]).all() and (rows[:, 2] == 0).all()   # no waits, no signals
        keys = sorted((int(r[P_G]), int(r[P_B]), int(r[P_SPLIT])) for r in rows)
        assert keys == sorted((g, b, s) for g in range(shape.Hkv) for b in range(len(seq0)) for s in range(nsplit[b]))
        cached = [max(0, min(T, seq0[r[P_B]] + 3 - 1 - r[P_SPLIT] * T)) for r in rows]
        assert cached == sorted(cached, reverse=True)                                   # longest first
        assert (rows[:, P_LAYER] == l).all() and (rows[:, P_T0] == rows[:, P_SPLIT] * T).all()
        assert all(int(r[P_NSPLIT]) == nsplit[r[P_B]] for r in rows)
        pool_ev = {int(r[10]) for r in rows}
        assert len(pool_ev) == 1 and (rows[:, P_ATHR] == th[pool_ev.pop()]).all()


def test_attention_pools_need_a_batch():
    with pytest.raises(rt.MkError) as e:
        rt.Plan.llama(synth.LLAMA_1B, 1, [100], 3, 110, attn_pool=1, num_sms=152, smem_per_cta=232448)
    assert e.value.code == rt.MK_ERR_UNSUPPORTED


def test_attention_split_needs_its_k_pages_in_the_ring():
    """A task holds its K pages (at most 4), releases them, then waits for its
    V pages: 512 positions of head_dim 128 fit 32 KB pages (4 of K) and 64 KB
    pages (2), and the planner refuses a split whose K would take more than 4
    pages even where the pool has room for them."""
    p = rt.Plan.llama(synth.QWEN3_8B, 16, [2048] * 16, 2, 2060, attn_split=512, **GB300)
    info = p.info()
    assert info["attn_split"] == 512 and info["page_bytes"] == 32768 and info["num_pages"] >= 4
    p = rt.Plan.llama(synth.QWEN3_8B, 1, [2048], 2, 2060, attn_split=512, **GB300)
    assert p.info()["attn_split"] == 512 and p.info()["page_bytes"] == 65536
    p = rt.Plan.llama(synth.QWEN3_8B, 1, [2048], 2, 2060, attn_split=256, page_bytes=16384, **GB300)
    assert p.info()["num_pages"] >= 8  # 4 pages of K at 16 KB
    with pytest.raises(rt.MkError) as e:  # 8 pages of K
        rt.Plan.llama(synth.QWEN3_8B, 1, [2048], 2, 2060, attn_split=512, page_bytes=16384, **GB300)
    assert e.value.code == rt.MK_ERR_UNSUPPORTED and "page pool" in rt.load().mk_last_error().decode()
    with pytest.raises(rt.MkError) as e:
        rt.Plan.llama(synth.QWEN3_8B, 16, [2048] * 16, 2, 2060, attn_split=1024, **GB300)
    assert e.value.code == rt.MK_ERR_UNSUPPORTED
