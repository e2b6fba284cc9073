"""Host-side checks of the GLM block plan (no GPU): task counts, events and
thresholds, tile coverage of every FP8 matrix, RoPE tiles, waits, the
algorithmic byte count, and deadlock-free queues over several steps -- for
the warp-level MMA tiles (``tc_tiles=-1``) and the tcgen05 tiles (the
default at M = 16: 128 weight rows per task, the first GEMMs split over K)."""
import numpy as np

from oracle import rules, sim
from persistent_megakernel_decode_gb300 import runtime as rt
from persistent_megakernel_decode_gb300 import synth

W_ROW, W_P = 1, 14
P_ROW0, P_NROWS, P_KC, P_OUT0, P_KTOT, P_RPP, P_NPG = 14, 15, 17, 18, 21, 22, 23
P_GL_LD, P_GL_ROPE, P_GL_M, P_GL_T, P_GL_POS0 = 24, 25, 26, 27, 28
P_K0, P_GL_TCT, P_GL_SUM = 16, 29, 30


def _plan(steps=3, tc_tiles=-1, dims=synth.GLM):
    return rt.Plan.glm(dims, steps, num_sms=152, smem_per_cta=232448, tc_tiles=tc_tiles)


def _slots(q, ids):
    out = []
    for w in range(ids.shape[0]):
        for s in range(ids.shape[1]):
            if ids[w, s] >= 0:
                out.append((int(ids[w, s]), q[w, s]))
    return sorted(out, key=lambda x: x[0])


def test_glm_plan_counts_events_and_bytes():
    d = synth.GLM
    p = _plan()
    info = p.info()
    q, ids, th, tasks = p.export()
    nq = d.qlora + d.kvlora + d.rope
    n_fan = nq // 16 + d.gate_heads // 16 + d.idx_dim // 16
    n_second = (d.q_heads * d.q_head_dim + d.idx_heads * d.idx_dim) // 64
    assert info["num_tasks"] == d.M + n_fan + d.M + n_second == 432
    # A0 rows; QKV-A + Indexer-K tiles; FIN rows; Head-Gate + FIN + second GEMMs
    assert list(th) == [d.M, nq // 16 + d.idx_dim // 16, d.M, d.gate_heads // 16 + d.M + n_second]
    # algorithmic bytes, counted here from the shapes: e4m3 weights and fp32
    # block scales once; x, residual, residual out; outputs and cache rows;
    # each intermediate written once
    kb_h, kb_q = d.H // 128, d.qlora // 128
    mats = synth.glm_mat_shapes(d)
    weights = sum(n * k for n, k in mats.values())
    scales = sum(4 * ((n + 127) // 128) * (k // 128) for n, k in mats.values())
    io = d.M * d.H * 2 * 3 + d.H * 2 + d.M * (d.gate_heads + d.q_heads * d.q_head_dim + d.idx_heads * d.idx_dim) * 2 \
        + d.M * (d.kvlora + d.rope + d.idx_dim) * 2
    inter = d.M * (d.H + kb_h * 4 + (nq + d.idx_dim) * 2 + d.qlora + kb_q * 4)
    assert weights == 39_321_600
    assert info["algorithmic_bytes_step"] == weights + scales + io + inter == 40_680_768


def test_glm_plan_tiles_cover_each_matrix_once_with_rope_on_head_tails():
    d = synth.GLM
    q, ids, th, tasks = _plan().export()
    slots = _slots(q, ids)
    by_op = {}
    for t, w in slots:
        by_op.setdefault(int(w[W_ROW]), []).append(w)
    assert sorted(by_op) == list(range(7))
    assert all(int(w[0]) == rt.OPCODE["glm_a0"] for w in by_op[0])
    assert sorted(int(w[P_ROW0]) for w in by_op[0]) == list(range(d.M))
    assert sorted(int(w[P_ROW0]) for w in by_op[4]) == list(range(d.M))
    nq = d.qlora + d.kvlora + d.rope
    widths = {1: (nq, d.H, 0), 2: (d.gate_heads, d.H, 0), 3: (d.idx_dim, d.H, 0),
              5: (d.q_heads * d.q_head_dim, d.qlora, d.q_head_dim), 6: (d.idx_heads * d.idx_dim, d.qlora, d.idx_dim)}
    for op, (N, K, head) in widths.items():
        rows = np.zeros(N, int)
        for w in by_op[op]:
            assert int(w[0]) == rt.OPCODE["glm_gemm"]
            r0, nr = int(w[P_ROW0]), int(w[P_NROWS])
            rows[r0:r0 + nr] += 1
            assert int(w[P_KC]) == K == int(w[P_KTOT]) and int(w[P_OUT0]) == r0 and int(w[P_GL_LD]) == N
            rpp = int(w[P_RPP])
            assert rpp == 49152 // K and int(w[P_NPG]) == -(-nr // rpp)
            rope = bool(w[P_GL_ROPE])
            assert rope == (head > 0 and r0 % head == head - 64), (op, r0)
            assert int(w[P_GL_M]) == d.M and int(w[P_GL_T]) == d.T and int(w[P_GL_POS0]) == d.pos0
        assert (rows == 1).all(), op


def test_glm_plan_waits_and_deadlock_free_queues():
    steps = 3
    q, ids, th, tasks = _plan(steps).export()
    waits = {i: [(r[7 + 3 * k], r[8 + 3 * k], r[9 + 3 * k]) for k in range(r[6])] for i, r in enumerate(tasks)}
    sigs = {i: [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] for i, r in enumerate(tasks)}
    kinds = {i: rt.OP_NAMES[r[0]] for i, r in enumerate(tasks)}
    for i, k in kinds.items():
        if k == "glm_a0":
            assert waits[i] == [(3, th[3], -1)]     # the previous step's last tasks
        elif k == "glm_fin":
            assert waits[i] == [(1, th[1], 0)]
    res = sim.deadlock_check(ids.tolist(), waits, sigs, len(th), steps=steps)
    assert res.ok and res.counters == rules.expected_counters(th.tolist(), steps)


# ---------------------------------------------------------------- tcgen05 tiles

def _ceil(a, b):
    return -(-a // b)


def test_glm_tc_plan_is_the_default_at_m16_and_counts():
    d = synth.GLM
    p = _plan(tc_tiles=0)
    info = p.info()
    assert info["tc_tiles"] == 1 and info["page_bytes"] == 16384
    q, ids, th, tasks = p.export()
    nq = d.qlora + d.kvlora + d.rope
    row_tiles = _ceil(nq, 128) + _ceil(d.gate_heads, 128) + _ceil(d.idx_dim, 128)
    assert row_tiles == 19
    # the largest divisor of H / 128 = 48 with 19 x parts <= 152 workers and <= 12 stages a part
    ks = 8
    n_second = _ceil(d.q_heads * d.q_head_dim, 128) + _ceil(d.idx_heads * d.idx_dim, 128)
    assert info["num_tasks"] == d.M + row_tiles * ks + d.M + n_second == 16 + 152 + 16 + 128
    # Head-Gate's sums are rounded by FIN: its tiles count into FIN's event
    assert list(th) == [d.M, (_ceil(nq, 128) + _ceil(d.idx_dim, 128) + _ceil(d.gate_heads, 128)) * ks, d.M,
                        d.M + n_second]
    assert info["algorithmic_bytes_step"] == 40_680_768  # the same bytes, whatever the tiling
    # the warp-level tiles stay available
    assert _plan(tc_tiles=-1).info()["tc_tiles"] == 0


def test_glm_tc_tiles_cover_each_weight_block_once():
    d = synth.GLM
    q, ids, th, tasks = _plan(tc_tiles=0).export()
    by_op = {}
    for t, w in _slots(q, ids):
        by_op.setdefault(int(w[W_ROW]), []).append(w)
    nq = d.qlora + d.kvlora + d.rope
    widths = {1: (nq, d.H, 0, 8), 2: (d.gate_heads, d.H, 0, 8), 3: (d.idx_dim, d.H, 0, 8),
              5: (d.q_heads * d.q_head_dim, d.qlora, d.q_head_dim, 1), 6: (d.idx_heads * d.idx_dim, d.qlora, d.idx_dim, 1)}
    for op, (N, K, head, ks) in widths.items():
        cover = np.zeros((_ceil(N, 128), K // 128), int)
        for w in by_op[op]:
            assert int(w[0]) == rt.OPCODE["glm_gemm"] and int(w[P_GL_TCT]) == 1
            r0, nr, k0, kc = int(w[P_ROW0]), int(w[P_NROWS]), int(w[P_K0]), int(w[P_KC])
            assert r0 % 128 == 0 and nr == min(128, N - r0) and int(w[P_OUT0]) == r0 and int(w[P_GL_LD]) == N
            assert int(w[P_KTOT]) == K and kc == K // ks and k0 % kc == 0 and int(w[P_NPG]) == kc // 128 <= 12
            assert int(w[P_GL_SUM]) == (1 if op <= 3 else 0)  # the first GEMMs add into sums FIN rounds
            cover[r0 // 128, k0 // 128:(k0 + kc) // 128] += 1
            # RoPE: bit j for rows r0 + 64 j .. + 63 when they are a head's last 64 rows
            want = sum(1 << j for j in range(2)
                       if head > 0 and r0 + 64 * j < N and (r0 + 64 * j) % head == head - 64)
            assert int(w[P_GL_ROPE]) == want, (op, r0)
        assert (cover == 1).all(), op
    # FIN finalises the sums: it says so, with the Head-Gate width
    for w in by_op[4]:
        assert int(w[W_P + 6]) == 1 and int(w[W_P + 7]) == d.gate_heads


def test_glm_tc_queues_deadlock_free():
    steps = 3
    q, ids, th, tasks = _plan(steps, tc_tiles=0).export()
    waits = {i: [(r[7 + 3 * k], r[8 + 3 * k], r[9 + 3 * k]) for k in range(r[6])] for i, r in enumerate(tasks)}
    sigs = {i: [(r[17 + 2 * k], r[18 + 2 * k]) for k in range(r[16])] for i, r in enumerate(tasks)}
    res = sim.deadlock_check(ids.tolist(), waits, sigs, len(th), steps=steps)
    assert res.ok and res.counters == rules.expected_counters(th.tolist(), steps)


def test_glm_tc_needs_sixteen_rows():
    from dataclasses import replace
    small = replace(synth.GLM, T=4)
    assert _plan(tc_tiles=0, dims=small).info()["tc_tiles"] == 0  # the default falls back
    try:
        _plan(tc_tiles=1, dims=small)
    except rt.MkError as e:
        assert e.code == rt.MK_ERR_UNSUPPORTED
    else:
        raise AssertionError("tensor-core GLM tiles accepted M != 16")
