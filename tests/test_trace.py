"""Host-side trace summaries on a hand-made trace (no GPU)."""
import numpy as np
import pytest

from persistent_megakernel_decode_gb300 import trace as tr
from persistent_megakernel_decode_gb300.runtime import OPCODE


def _slot(t, w, i, opc, task, start, met, done, handed=0, pub=0, lstart=0):
    t[w, i, tr.T_OPC] = opc | (task << 32)
    t[w, i, tr.T_START] = start
    t[w, i, tr.T_MET] = met
    t[w, i, tr.T_DONE] = done
    t[w, i, tr.T_HANDED] = handed
    t[w, i, tr.T_PUB] = pub
    t[w, i, tr.T_LSTART] = lstart


@pytest.fixture
def fake():
    """Two workers, one layer: embed (task 0), qkv (1, 2), attn (3), o (4), lm (5).
    Times in ns from 1,000,000."""
    t = np.zeros((2, 4, 16), np.uint64)
    b = 1_000_000
    _slot(t, 0, 0, OPCODE["embed"], 0, b, b, b + 1000, pub=b + 1500)
    _slot(t, 0, 1, OPCODE["qkv"], 1, b + 1000, b + 2000, b + 5000, handed=b + 2500, pub=b + 5400, lstart=b)
    _slot(t, 1, 0, OPCODE["qkv"], 2, b, b + 2000, b + 6000, handed=b + 3000, pub=b + 6200, lstart=b)
    _slot(t, 1, 1, OPCODE["attn"], 3, b + 6000, b + 7000, b + 12000, handed=b + 7500, pub=b + 12500)
    _slot(t, 0, 2, OPCODE["o"], 4, b + 5000, b + 13000, b + 15000, handed=b + 13500, pub=b + 15200)
    _slot(t, 0, 3, OPCODE["lm"], 5, b + 15000, b + 16000, b + 20000, handed=b + 16000, pub=b + 20100)
    tasks = np.zeros((6, 24), np.int32)
    tasks[:, 1] = [-1, 0, 0, 0, 0, -1]
    return t, tasks


def test_summarize_shares_and_active_fraction(fake):
    t, _ = fake
    s = tr.summarize(t)
    assert s["span_us"] == pytest.approx(20.0)
    busy = {"embed": 1.0, "qkv": 4.0 + 6.0, "attn": 6.0, "o": 10.0, "lm": 5.0}
    total = sum(busy.values())
    assert s["sm_active_frac"] == pytest.approx(total / (2 * 20.0))
    for k, v in busy.items():
        assert s["ops"][k]["share"] == pytest.approx(v / total)
    assert s["ops"]["qkv"]["act_wait_us"] == pytest.approx((1.5 + 3.0) / 2)
    assert s["ops"]["qkv"]["publish_us"] == pytest.approx((0.4 + 0.2) / 2)
    assert s["ops"]["qkv"]["loader_lead_us"] == pytest.approx((1.0 + 0.0) / 2)
    assert s["ops"]["o"]["act_wait_us"] == pytest.approx(8.5)
    assert "inner_us" not in s["ops"]["qkv"]


def test_summarize_inner_stamps(fake):
    t, _ = fake
    b = 1_000_000
    t[1, 1, 6] = b + 8500     # attention: K pages 1 us after its hand-off at 7.5
    t[1, 1, 10] = b + 11500
    s = tr.summarize(t)
    assert s["ops"]["attn"]["inner_us"] == pytest.approx({"6": 1.0, "10": 4.0})


def test_timeline_rows(fake):
    t, tasks = fake
    rows = tr.timeline(t, tasks)
    assert [(r["layer"], r["op"]) for r in rows] == [(-1, "embed"), (0, "qkv"), (0, "attn"), (0, "o"), (-1, "lm")]
    q = rows[1]
    assert q["n"] == 2 and q["met_first"] == pytest.approx(2.0) and q["met_last"] == pytest.approx(2.0)
    assert q["done_last"] == pytest.approx(6.0) and q["pub_last"] == pytest.approx(6.2)
    assert q["task_us"] == pytest.approx((2.5 + 3.0) / 2)


def test_layer_profile_gaps(fake):
    t, tasks = fake
    prof = tr.layer_profile(tr.timeline(t, tasks))
    assert set(prof) == {"qkv", "attn", "o"}
    assert prof["qkv"]["gap_us"] is None                  # first op of the first layer
    assert prof["attn"]["gap_us"] == pytest.approx(1.0)    # ready at 7, qkv done at 6
    assert prof["o"]["gap_us"] == pytest.approx(1.0)       # ready at 13, attn done at 12
    assert prof["attn"]["span_us"] == pytest.approx(5.0)


def test_empty_trace():
    t = np.zeros((3, 5, 16), np.uint64)
    assert tr.summarize(t) == {}
    assert tr.timeline(t, np.zeros((1, 24), np.int32)) == []


def test_layer_profile_across_layers():
    """Two layers of qkv -> down: the second layer's qkv gap runs from the
    first layer's last down instruction done; means are over layers."""
    t = np.zeros((1, 4, 16), np.uint64)
    b = 1_000_000
    _slot(t, 0, 0, OPCODE["qkv"], 0, b, b + 1000, b + 3000)
    _slot(t, 0, 1, OPCODE["down"], 1, b + 3000, b + 4000, b + 8000)
    _slot(t, 0, 2, OPCODE["qkv"], 2, b + 8000, b + 10000, b + 13000)
    _slot(t, 0, 3, OPCODE["down"], 3, b + 13000, b + 14000, b + 20000)
    tasks = np.zeros((4, 24), np.int32)
    tasks[:, 1] = [0, 0, 1, 1]
    prof = tr.layer_profile(tr.timeline(t, tasks))
    assert prof["qkv"]["gap_us"] == pytest.approx(2.0)     # 10 - 8: only layer 1 has a previous op
    assert prof["down"]["gap_us"] == pytest.approx(1.0)    # (4 - 3 + 14 - 13) / 2
    assert prof["qkv"]["span_us"] == pytest.approx(2.5)    # (3 - 1 + 13 - 10) / 2
    assert prof["down"]["span_us"] == pytest.approx(5.0)   # (8 - 4 + 20 - 14) / 2
