"""Per-instruction trace summaries (runs with ``MK_RUN_TRACE``).

Per queue slot the kernel stamps globaltimer nanoseconds (uint64 [workers,
lmax, 16], see ``mk_read_trace``):

====  ======================================================================
[0]   opcode | task id << 32
[1]   consumer warp 0 reaches the slot
[2]   the activation loader has seen every wait of the slot met
[3]   consumer warp 0 is done with the slot
[4]   loader starts issuing the slot's weight pages, [5] has issued them
[6..10] stamps inside the op (attention: K pages ready, scores, V pages
      ready, P.V, partial written; tensor-core tiles: [7] pages ready, [9] K
      loop done, [10] reduction barrier passed)
[13]  the activation is handed to the consumers (0 when the slot skipped it)
[14]  the publisher has added the slot's signals, [15] it saw the slot done
====  ======================================================================

``summarize`` gives per-opcode time shares and the SM-active fraction;
``timeline`` gives, per (layer, op), when its first and last instructions had
their inputs, when the last one finished and when it was published -- the
step's critical path, op by op.
"""
from __future__ import annotations

from collections import defaultdict
from typing import Dict, List

import numpy as np

from .runtime import OP_NAMES

T_OPC, T_START, T_MET, T_DONE, T_LSTART, T_LEND, T_HANDED, T_PUB, T_SEEN = 0, 1, 2, 3, 4, 5, 13, 14, 15
T_INNER = (6, 7, 8, 9, 10)  # stamps inside an op (attention: K pages, scores, V pages, P.V, partial out)


def _valid(trace: np.ndarray) -> np.ndarray:
    op = (trace[..., T_OPC] & 0xFFFFFFFF).astype(np.int64)
    return (op > 0) & (trace[..., T_DONE] > 0) & (trace[..., T_START] > 0)


def summarize(trace: np.ndarray) -> dict:
    """Per-opcode busy time (consumer start to done), its share, the mean wait
    for the activation hand-off, the publish latency (done to published), the
    loader's lead (issue start before the consumers reach the slot) and the
    mean time of each stamp inside the op from the hand-off (``inner_us``);
    the SM-active fraction is the busy time over workers x span."""
    op = (trace[..., T_OPC] & 0xFFFFFFFF).astype(np.int64)
    t = trace.astype(np.float64)
    valid = _valid(trace)
    if not valid.any():
        return {}
    t0 = t[..., T_START][valid].min()
    span = t[..., T_DONE][valid].max() - t0
    per: Dict[str, Dict[str, float]] = defaultdict(lambda: defaultdict(float))
    for w, i in zip(*np.nonzero(valid)):
        r = t[w, i]
        d = per[OP_NAMES.get(int(op[w, i]), str(int(op[w, i])))]
        d["n"] += 1
        d["busy"] += r[T_DONE] - r[T_START]
        if r[T_HANDED] > 0:
            d["act_wait"] += max(0.0, r[T_HANDED] - r[T_START])
            d["n_handed"] += 1
        if r[T_PUB] > 0:
            d["publish"] += max(0.0, r[T_PUB] - r[T_DONE])
            d["n_pub"] += 1
        if r[T_LSTART] > 0:
            d["loader_lead"] += r[T_START] - r[T_LSTART]
            d["n_lead"] += 1
        base = max(r[T_START], r[T_HANDED])
        for k in T_INNER:
            if r[k] > 0:
                d[f"in{k}"] += r[k] - base
                d[f"n_in{k}"] += 1
    busy = sum(d["busy"] for d in per.values())
    out = {"span_us": span / 1e3, "workers": int(trace.shape[0]),
           "sm_active_frac": busy / (span * trace.shape[0]) if span > 0 else 0.0, "ops": {}}
    for k, d in sorted(per.items(), key=lambda kv: -kv[1]["busy"]):
        n = d["n"]
        e = {"n": int(n), "mean_us": d["busy"] / n / 1e3, "share": d["busy"] / busy if busy else 0.0}
        if d["n_handed"]:
            e["act_wait_us"] = d["act_wait"] / d["n_handed"] / 1e3
        if d["n_pub"]:
            e["publish_us"] = d["publish"] / d["n_pub"] / 1e3
        if d["n_lead"]:
            e["loader_lead_us"] = d["loader_lead"] / d["n_lead"] / 1e3
        inner = {str(j): d[f"in{j}"] / d[f"n_in{j}"] / 1e3 for j in T_INNER if d[f"n_in{j}"]}
        if inner:
            e["inner_us"] = inner
        out["ops"][k] = e
    return out


def timeline(trace: np.ndarray, tasks: np.ndarray) -> List[dict]:
    """One row per (layer, op) in the order the ops first became ready.

    ``tasks`` is the plan's exported task table (column 1 = layer).  Times are
    microseconds from the step's first consumer start: ``met_first`` /
    ``met_last`` -- first and last instruction of the op with every wait met;
    ``done_last`` -- its last instruction finished; ``pub_last`` -- the last
    signal published; ``task_us`` -- mean consumer time per instruction from
    the hand-off (or the slot start when there was none) to done."""
    valid = _valid(trace)
    if not valid.any():
        return []
    t = trace.astype(np.float64)
    t0 = t[..., T_START][valid].min()
    groups: Dict[tuple, Dict[str, list]] = defaultdict(lambda: defaultdict(list))
    for w, i in zip(*np.nonzero(valid)):
        r = t[w, i]
        opc = int(trace[w, i, T_OPC] & 0xFFFFFFFF)
        task = int(trace[w, i, T_OPC] >> 32)
        layer = int(tasks[task, 1]) if 0 <= task < len(tasks) else -1
        g = groups[(layer, opc)]
        g["met"].append(r[T_MET] if r[T_MET] > 0 else r[T_START])
        g["done"].append(r[T_DONE])
        g["pub"].append(r[T_PUB])
        g["task"].append(r[T_DONE] - max(r[T_START], r[T_HANDED]))
    rows = []
    for (layer, opc), g in groups.items():
        pub = [p for p in g["pub"] if p > 0]
        rows.append({
            "layer": layer, "op": OP_NAMES.get(opc, str(opc)), "n": len(g["done"]),
            "met_first": (min(g["met"]) - t0) / 1e3, "met_last": (max(g["met"]) - t0) / 1e3,
            "done_last": (max(g["done"]) - t0) / 1e3,
            "pub_last": (max(pub) - t0) / 1e3 if pub else None,
            "task_us": float(np.mean(g["task"])) / 1e3,
        })
    rows.sort(key=lambda r: (r["met_first"], r["layer"]))
    return rows


def layer_profile(rows: List[dict]) -> Dict[str, dict]:
    """Means over the decoder layers (layer >= 0) of each op's span: from its
    first instruction having its inputs to its last one done (``span_us``);
    the hand-over from the previous op of the same layer chain
    (``gap_us``: this op's first ready instruction minus the previous op's
    last one done; negative when they overlap); the mean consumer time per
    instruction (``task_us``)."""
    by_layer: Dict[int, List[dict]] = defaultdict(list)
    for r in rows:
        by_layer[r["layer"]].append(r)
    chains = [sorted(v, key=lambda r: r["met_first"]) for k, v in sorted(by_layer.items()) if k >= 0]
    acc: Dict[str, Dict[str, list]] = defaultdict(lambda: defaultdict(list))
    prev_done = None
    for chain in chains:
        for r in chain:
            a = acc[r["op"]]
            a["span"].append(r["done_last"] - r["met_first"])
            a["task"].append(r["task_us"])
            a["n"].append(r["n"])
            if prev_done is not None:
                a["gap"].append(r["met_first"] - prev_done)
            prev_done = r["done_last"]
    out = {}
    for op, a in acc.items():
        out[op] = {"n": float(np.mean(a["n"])), "span_us": float(np.mean(a["span"])),
                   "task_us": float(np.mean(a["task"])),
                   "gap_us": float(np.mean(a["gap"])) if a["gap"] else None}
    return out
