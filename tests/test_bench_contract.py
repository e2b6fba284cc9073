"""The bench line's contract on the host: the reference arm (the CPU oracle)
prints one JSON line with the keys the driver reads; a non-zero rank prints
nothing and exits 0."""
import json
import os
import subprocess
import sys

from conftest import ROOT

CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny", "--steps", "2",
       "--warmup", "1"]


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run(CMD, capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run({"RANK": "0"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    for k in ("metric", "value", "n_gpus", "steps", "warmup", "ms_per_step", "scaling", "vs_baseline", "dtype", "data",
              "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work():
    r = _run({"RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_launch_chunks_cover_every_step_once():
    import bench
    for first, n, spl in [(5, 100, 16), (0, 3, 16), (3, 32, 16), (0, 7, 1), (2, 16, 16), (0, 0, 4)]:
        ch = bench.launch_chunks(first, n, spl)
        steps = [s for st, k in ch for s in range(st, st + k)]
        assert steps == list(range(first, first + n))
        assert all(1 <= k <= spl for _, k in ch)
        assert len(ch) == -(-n // spl)


def test_per_launch_bytes_follow_the_steps_each_launch_runs():
    """The roofline's per-launch figures scale the per-step bytes by the steps a
    timed launch actually runs, which the launch length only bounds."""
    import bench
    assert bench.steps_per_launch(bench.launch_chunks(5, 20, 128)) == 20    # one launch of every timed step
    assert bench.steps_per_launch(bench.launch_chunks(5, 128, 128)) == 128
    assert bench.steps_per_launch(bench.launch_chunks(0, 32, 16)) == 16
    assert bench.steps_per_launch(bench.launch_chunks(0, 100, 16)) == 100 / 7  # six of 16 and one of 4
    assert bench.steps_per_launch(bench.launch_chunks(0, 7, 1)) == 1
