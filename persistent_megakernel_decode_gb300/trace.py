"""Per-instruction trace summaries (runs with ``MK_RUN_TRACE``).

Per queue slot the kernel stamps (globaltimer ns): consumer start, the moment
the activation loader finished its waits, consumer end, loader issue start
and end, first and last weight page ready at the consumers.  ``summarize``
turns that into per-opcode time shares, the SM-active fraction, how long
instructions waited for their activation and for their pages, how far ahead
the loader ran, and the loader's issue pace.
"""
from __future__ import annotations

from collections import defaultdict

import numpy as np

from .runtime import OP_NAMES


def summarize(trace: np.ndarray) -> dict:
    """trace: uint64 [workers, lmax, 8]."""
    op = (trace[..., 0] & 0xFFFFFFFF).astype(np.int64)
    t = trace.astype(np.float64)
    start, ready, done, lstart, lend, pfirst, plast = (t[..., k] for k in (1, 2, 3, 4, 5, 6, 7))
    valid = (op > 0) & (done > 0)
    if not valid.any():
        return {}
    t0 = start[valid].min()
    span = done[valid].max() - t0
    per = defaultdict(lambda: defaultdict(float))
    for w in range(trace.shape[0]):
        prev_l = None
        for i in range(trace.shape[1]):
            if not valid[w, i]:
                continue
            d = per[OP_NAMES.get(int(op[w, i]), str(op[w, i]))]
            d["n"] += 1
            d["busy"] += done[w, i] - start[w, i]
            if ready[w, i] > 0:
                d["act_wait"] += max(0.0, ready[w, i] - start[w, i])
            if pfirst[w, i] > 0:
                d["page_wait"] += max(0.0, pfirst[w, i] - max(start[w, i], ready[w, i]))
                d["compute"] += done[w, i] - pfirst[w, i]
                d["n_pages"] += 1
            if lstart[w, i] > 0:
                d["loader_lead"] += start[w, i] - lstart[w, i]
                d["issue"] += lend[w, i] - lstart[w, i]
                if prev_l is not None:
                    d["loader_pace"] += lstart[w, i] - prev_l
                    d["n_pace"] += 1
                prev_l = lstart[w, i]
    busy = sum(d["busy"] for d in per.values())
    out = {"span_us": span / 1e3, "workers": int(trace.shape[0]),
           "sm_active_frac": busy / (span * trace.shape[0]) if span > 0 else 0.0, "ops": {}}
    for k, d in sorted(per.items(), key=lambda kv: -kv[1]["busy"]):
        n = d["n"]
        e = {"n": int(n), "mean_us": d["busy"] / n / 1e3, "share": d["busy"] / busy if busy else 0.0,
             "act_wait_us": d["act_wait"] / n / 1e3}
        if d["n_pages"]:
            e["page_wait_us"] = d["page_wait"] / d["n_pages"] / 1e3
            e["first_page_to_done_us"] = d["compute"] / d["n_pages"] / 1e3
        if d["n_pace"]:
            e["loader_lead_us"] = d["loader_lead"] / n / 1e3
            e["loader_issue_us"] = d["issue"] / n / 1e3
            e["loader_pace_us"] = d["loader_pace"] / d["n_pace"] / 1e3
        out["ops"][k] = e
    return out
