"""Per-instruction trace summaries (runs with ``MK_RUN_TRACE``).

The kernel stamps, per queue slot, the consumer start, the moment the
activation loader finished its waits, and the consumer end (globaltimer ns).
``summarize`` turns that into per-opcode time shares, the SM-active fraction
and the wait share -- the in-kernel view of where a step's time goes.
"""
from __future__ import annotations

from collections import defaultdict

import numpy as np

from .runtime import OP_NAMES


def summarize(trace: np.ndarray) -> dict:
    """trace: uint64 [workers, lmax, 4] = (opcode | task << 32, start, ready, done)."""
    op = (trace[..., 0] & 0xFFFFFFFF).astype(np.int64)
    start, ready, done = (trace[..., k].astype(np.float64) for k in (1, 2, 3))
    valid = (op > 0) & (done > 0)
    if not valid.any():
        return {}
    t0 = start[valid].min()
    t1 = done[valid].max()
    span = t1 - t0
    per = defaultdict(lambda: {"n": 0, "busy_ns": 0.0, "wait_ns": 0.0})
    for w in range(trace.shape[0]):
        prev_done = None
        for i in range(trace.shape[1]):
            if not valid[w, i]:
                continue
            name = OP_NAMES.get(int(op[w, i]), str(op[w, i]))
            d = per[name]
            d["n"] += 1
            d["busy_ns"] += done[w, i] - start[w, i]
            d["wait_ns"] += max(0.0, ready[w, i] - start[w, i]) if ready[w, i] > 0 else 0.0
    busy = sum(d["busy_ns"] for d in per.values())
    out = {"span_us": span / 1e3, "workers": int(trace.shape[0]),
           "sm_active_frac": busy / (span * trace.shape[0]) if span > 0 else 0.0, "ops": {}}
    for k, d in sorted(per.items(), key=lambda kv: -kv[1]["busy_ns"]):
        out["ops"][k] = {"n": d["n"], "mean_us": d["busy_ns"] / d["n"] / 1e3,
                         "share": d["busy_ns"] / busy if busy else 0.0,
                         "mean_wait_us": d["wait_ns"] / d["n"] / 1e3}
    return out
