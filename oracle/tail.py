"""Wave-quantisation (tail) arithmetic of a kernel-per-op run (TEST INFRASTRUCTURE ONLY).

"CMU 15-779 Lecture 7 notes", section 3.1 (tail effect) and exercise 2: a
kernel of ``n_tasks`` equal tasks on ``n_sms`` SMs runs in
ceil(n_tasks / n_sms) waves; the last wave keeps only the remainder busy.
With every SM given an equal share of the HBM bandwidth, one task of
``tile_bytes`` takes tile_bytes / (bw / n_sms); the kernel takes
waves x that, plus a fixed start/finish latency.  The ideal time is all bytes
over the full bandwidth.  Section 4.2: with a page pool of ``pages`` pages
and tasks that use ``pages_per_task``, floor(pages / pages_per_task) tasks
fit ahead.

Pinned by the notes' printed figures: QKV 192 tasks x 64 KiB on 132 SMs at
3.35 TB/s -> 2 waves, 60 busy / 72 idle in the second, ideal 3.76 us,
6.26 us with a 1.1 us latency; 24-row tasks -> 128 tasks, one wave, 4 idle,
about 3.8 us; 13 pages / 4 per task -> 3 ahead, 6 per task -> 2.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass
class TailModel:
    waves: int
    busy_last_wave: int
    idle_last_wave: int
    ideal_us: float
    per_task_us: float
    kernel_us: float


def tail_model(n_tasks: int, n_sms: int, tile_bytes: int, bw_bytes_per_s: float,
               latency_us: float = 0.0) -> TailModel:
    waves = math.ceil(n_tasks / n_sms)
    busy = n_tasks - (waves - 1) * n_sms
    per_task = tile_bytes / (bw_bytes_per_s / n_sms) * 1e6
    ideal = n_tasks * tile_bytes / bw_bytes_per_s * 1e6
    return TailModel(waves, busy, n_sms - busy, ideal, per_task, waves * per_task + latency_us)


def prefetch_depth(pages: int, pages_per_task: int) -> int:
    return pages // pages_per_task
