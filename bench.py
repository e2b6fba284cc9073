"""Decode-step benchmark of the persistent megakernel (one JSON line on rank 0).

Default workload: Llama-3.2-1B shape, batch 1, KV cache pre-filled to 1024
tokens, random bf16 weights (synthetic; no trained weights, no dataset).  A
step is one decode step of the whole model: embedding, 16 layers, LM head and
argmax, run by the persistent kernel.  The timed region runs the steps in
cooperative launches of up to --steps-per-launch (default 16) steps each: the
next step's token is the previous step's greedy argmax, read on the device,
so no step is skipped or cached; --steps-per-launch 1 times one launch per
step (the side legs report both).  The end-to-end figure keeps one launch per
step with the token copied in and the argmax copied out each step.  Weights
(2.5 GB) exceed the 129 MB L2, so no flush is needed between steps.

Arms:
  --impl mk (default)   the CUDA path through the C ABI (libmk)
  --impl reference      the plain CPU oracle (fp32 twin) on the host cores
Multi-GPU: independent replicas, one per rank, no collective on the data path
(weak scaling); value = tokens of all ranks / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode step µs & tokens/s at 1 GB300; achieved HBM GB/s as % of roofline"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    from persistent_megakernel_decode_gb300 import build as _b
    for f in _b.SOURCES + _b.HEADERS:
        with open(os.path.join(ROOT, "persistent_megakernel_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(ROOT, "include", "mk.h"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()[:16]


def launch_chunks(first, n, spl):
    """Steps first .. first + n - 1 as (first step, steps) launches of at most spl steps."""
    return [(first + i, min(spl, n - i)) for i in range(0, n, spl)]


def steps_per_launch(chunks):
    """Mean decode steps of the timed launches (an int when they are all equal):
    the factor between the per-step and the per-launch byte figures."""
    total = sum(k for _, k in chunks)
    m = total / len(chunks)
    return int(m) if float(m).is_integer() else m


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"mk_interp_{workload}.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") == kernel_source_hash():
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch
    import torch.distributed as dist
    dist.init_process_group("nccl")
    rank = dist.get_rank()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
    return rank, dist.get_world_size(), dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def slowest_replica_ms(total_ms, dist, dev=None):
    """The timed region's length over all ranks: the maximum (the job is done
    when its slowest replica is).  NCCL reduces a device tensor, gloo a host one."""
    if dist is None:
        return total_ms
    import torch
    t = torch.tensor([total_ms], dtype=torch.float64,
                     device=dev if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, total_ms):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (total_ms / 1e3)


def side_measurements(args, w, dev, stream, weights, kc, vc, seq0, max_steps, first_free_step):
    """The comparison legs measured beside the megakernel in the same run: the
    same device code launched once per op (stream and CUDA-Graph variants), the
    megakernel's per-step launches replayed from a CUDA Graph, and an empty
    kernel's launch time (cooperative and plain, the interpreter's grid)."""
    import torch
    from persistent_megakernel_decode_gb300 import runtime as rt
    out = {}
    K = 16

    def timed_steps(sess, first, graph):
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for st in range(first, first + K):
                    sess.run(st, 1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for st in range(first, first + K):
                    sess.run(st, 1)
                e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / K

    for mode, name in ((rt.MODE_PER_OP, "per_op"), (rt.MODE_MEGAKERNEL, "megakernel")):
        try:
            sess = rt.Session(w.shape, weights, kc, vc, seq0, max_steps, stream=stream, mode=mode)
            sess.tokens[0] = torch.tensor([1] * w.batch, dtype=torch.int32, device=dev)
            with torch.cuda.stream(stream):
                for st in range(3):
                    sess.run(st, 1)
            sess.sync()
            launches = sess.plan.info()["num_launches"]
            ms_stream = timed_steps(sess, 3, False)
            ms_graph = timed_steps(sess, 3 + K, True)
            err = int(sess.sync().code)
            out[name] = {"launches_per_step": launches, "ms_per_step_stream": ms_stream,
                         "ms_per_step_cuda_graph": ms_graph, "device_error": err, "steps": K}
            del sess
        except Exception as e:  # a leg that cannot run is reported, not fatal
            out[name] = {"unavailable": str(e)[:200]}
    # several steps in one cooperative launch (MK_RUN_ONE_LAUNCH): ms per step
    # for 1, 4 and 16 steps per launch, beside the empty-launch probe below
    try:
        need = 3 + 1 + 4 + 16
        if max_steps < need:
            raise RuntimeError(f"needs a session of {need} steps")
        sess = rt.Session(w.shape, weights, kc, vc, seq0, max_steps, stream=stream)
        sess.tokens[0] = torch.tensor([1] * w.batch, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            for st in range(3):
                sess.run(st, 1)
        sess.sync()
        first, per = 3, {}
        for k in (1, 4, 16):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                sess.run(first, k, one_launch=True)
                e1.record(stream)
            stream.synchronize()
            per[str(k)] = e0.elapsed_time(e1) / k
            first += k
        out["megakernel_one_launch"] = {"ms_per_step_by_steps_per_launch": per,
                                        "device_error": int(sess.sync().code)}
        del sess
    except Exception as e:
        out["megakernel_one_launch"] = {"unavailable": str(e)[:200]}
    info = rt.Plan.llama(w.shape, w.batch, seq0, 1, kc.shape[3]).info()
    for coop in (True, False):
        n = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(10):
                rt.launch_probe(info["num_workers"], coop, stream)
            e0.record(stream)
            for _ in range(n):
                rt.launch_probe(info["num_workers"], coop, stream)
            e1.record(stream)
        stream.synchronize()
        out["empty_launch_us_" + ("cooperative" if coop else "plain")] = e0.elapsed_time(e1) / n * 1e3
    return out


def cpu_oracle_rate(w, steps, warmup=0, device_for_inputs=None, nthreads=None):
    """Time the oracle's fp32 twin on the host cores over `steps` decode steps."""
    import torch
    from oracle import forward as orc
    from persistent_megakernel_decode_gb300 import synth
    s = w.shape
    seq0 = synth.seq_lengths(w)
    dev = device_for_inputs or "cpu"
    wt = synth.make_weights(s, w.weight_seed, device=dev, fp8=w.fp8)
    hw = synth.host_weights(wt)
    del wt
    smax = max(seq0) + warmup + steps + 1
    dims = (s.L, w.batch, s.Hkv, smax, s.D)
    rng = np.random.default_rng(w.cache_seed)
    kc = rng.integers(0x3000, 0x3F80, size=dims, dtype=np.uint16)   # finite bf16 bit patterns
    vc = rng.integers(0x3000, 0x3F80, size=dims, dtype=np.uint16)
    shape = orc.Shape(s.L, s.H, s.Hq, s.Hkv, s.D, s.F, s.V, s.qk_norm, s.eps, s.theta)
    cores = nthreads or os.cpu_count() or 1
    toks = synth.first_tokens(w)
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        _, _, am = orc.decode_step(shape, hw, kc, vc, [x + i for x in seq0], toks, precision=32, nthreads=cores,
                                   want_hidden=False)
        dt = time.perf_counter() - t0
        toks = [int(x) for x in am]
        if i >= warmup:
            times.append(dt)
    return float(np.sum(times)), cores


def run_reference(args, w, rank):
    if rank != 0:
        return
    total, cores = cpu_oracle_rate(w, args.steps, args.warmup)
    tps = w.batch * args.steps / total
    sample = f"{args.steps} timed decode steps of {w.name} (fp32 oracle, all layers), after {args.warmup} warm-up"
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "seq_len": w.seq_len, "layers": w.shape.L},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_mk(args, w, rank, world, dist):
    import torch
    from persistent_megakernel_decode_gb300 import build, runtime as rt, synth
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    s = w.shape
    seq0 = synth.seq_lengths(w)
    steps_total = args.warmup + args.steps
    max_steps = max(w.steps, steps_total)
    weights = synth.make_weights(s, w.weight_seed, device=dev, fp8=w.fp8)
    smax = max(seq0) + max_steps + 1
    kc, vc = synth.make_cache(s, w.batch, smax, w.cache_seed, device=dev)
    stream = torch.cuda.Stream(dev)
    target = {"mode": rt.MODE_PER_OP} if args.mode == "per_op" else {}
    for kv in args.knob:
        k, v = kv.split("=")
        target[k] = int(v)
    # batched workloads: attention tasks dealt on the host by the time-model
    # scheduler (with 512-position splits measured faster than device-side
    # claims at batch 8 and 16); --knob attn_pool=1 claims them on the device
    sess = rt.Session(s, weights, kc, vc, seq0, max_steps, stream=stream, **target)
    info = sess.plan.info()
    sess.tokens[0] = torch.tensor(synth.first_tokens(w), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    # launches of up to `spl` decode steps each (MK_RUN_ONE_LAUNCH: the next
    # step's token is the previous step's argmax, on the device); the per-op
    # baseline mode launches per op and step
    spl = 1 if args.mode == "per_op" else max(1, args.steps_per_launch)

    def chunks(first, n):
        return launch_chunks(first, n, spl)

    # warm-up: launches of up to `spl` steps, like the timed ones
    with torch.cuda.stream(stream):
        for st, k in chunks(0, args.warmup):
            sess.run(st, k, one_launch=k > 1)
    sess.sync()
    # timed: events on the launching stream around every launch
    timed = chunks(args.warmup, args.steps)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(timed) + 1)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for j, (st, k) in enumerate(timed):
                sess.run(st, k, one_launch=k > 1)
                ev[j + 1].record(stream)
        stream.synchronize()
    rec = sess.sync()
    barrier(dist)
    # per step: each launch's time over its steps
    step_ms = np.concatenate([np.full(k, ev[j].elapsed_time(ev[j + 1]) / k) for j, (st, k) in enumerate(timed)])
    total_ms = slowest_replica_ms(float(ev[0].elapsed_time(ev[-1])), dist, dev)
    value = job_rate(w.batch * args.steps, world, total_ms)
    # end to end through the public API with host buffers: token in, argmax out
    e2e_steps = min(args.steps, 32)
    pinned_tok = torch.tensor(synth.first_tokens(w), dtype=torch.int32).pin_memory()
    pinned_key = torch.zeros(w.batch, dtype=torch.int64).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            sess.tokens[i].copy_(pinned_tok, non_blocking=True)
            sess.run(i, 1, host_tokens=True)
            pinned_key.copy_(sess.argmax[i], non_blocking=True)
            stream.synchronize()
            pinned_tok.copy_(torch.from_numpy(rt.argmax_index(pinned_key.numpy().view(np.uint64)).astype(np.int32)))
    e2e_s = time.perf_counter() - t0
    e2e = {"value": w.batch * e2e_steps / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * w.batch,
           "d2h_bytes_per_step": 8 * w.batch, "steps": e2e_steps}
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    alg = info["algorithmic_bytes_step"]
    avg_launch_s = float(np.mean(step_ms)) / 1e3
    achieved = alg / avg_launch_s / 1e9
    # per timed launch (its mean number of steps: at most `spl` each): every
    # step streams the whole model, so the one-step ncu traffic scales with
    # the steps a launch runs
    traffic = profiled_traffic(w.name)
    per_launch = steps_per_launch(timed)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic * per_launch if traffic is not None else None, "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": alg * per_launch, "steps_per_launch": per_launch,
                "algorithmic_bytes_per_step": alg, "traffic_per_step": traffic,
                "kernel": "mk_interp", "nominal_8tbs_frac": achieved / 8000.0}
    cpu = None
    if not args.no_cpu_baseline:
        cpu_steps = 2
        total, cores = cpu_oracle_rate(w, cpu_steps, 0, device_for_inputs=dev)
        cpu = {"value": w.batch * cpu_steps / total, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{cpu_steps} decode steps of {w.name} (fp32 oracle, all layers, batch {w.batch})"}
        total1, _ = cpu_oracle_rate(w, 1, 0, device_for_inputs=dev, nthreads=1)
        cpu["single_core"] = {"value": w.batch / total1, "unit": "tokens/s", "cores": 1,
                              "sample": f"1 decode step of {w.name} (fp32 oracle, one thread)"}
    side = None
    if not args.no_extras and world == 1:
        side = side_measurements(args, w, dev, stream, weights, kc, vc, seq0, max_steps, args.warmup + args.steps)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 projections, bf16 LM head" if w.fp8 else "bf16", "accumulate": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.seq_len, "layers": s.L, "hidden": s.H,
                   "vocab": s.V, "mode": args.mode, "weights": "fp8 e4m3, 128x128 block scales" if w.fp8 else "bf16",
                   "l2": f"weights ({alg / 1e9:.2f} GB) exceed L2 (129 MB); no flush",
                   "steps_per_launch": spl, "knobs": {k: v for k, v in target.items() if k != "mode"},
                   "parallelism": f"replicas{world}"},
        "step_us": {"median": float(np.median(step_ms)) * 1e3, "p10": float(np.percentile(step_ms, 10)) * 1e3,
                    "p90": float(np.percentile(step_ms, 90)) * 1e3},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": len(timed) * info["num_launches"], "side": side,
        "plan": {k: info[k] for k in ("num_workers", "lmax", "num_tasks", "num_events", "num_pages", "smem_bytes")},
        "device_error": int(rec.code),
    }
    print(json.dumps(line), flush=True)
    if args.trace_out:
        write_trace(args.trace_out, sess, stream, step_ms)


def write_trace(path, sess, stream, step_ms):
    """One traced step (step 1 after a fresh step 0, host tokens) and its
    summaries: per-opcode shares, the (layer, op) timeline and per-layer means.
    The stamps are global stores of their own, so the traced step runs a
    little slower than the timed ones; both spans are written."""
    import torch
    from persistent_megakernel_decode_gb300 import trace as tr
    with torch.cuda.stream(stream):
        sess.run(0, 1, host_tokens=True)
        sess.run(1, 1, host_tokens=True, trace=True)
    rec = sess.sync()
    t = sess.trace()
    tasks = sess.plan.export()[3]
    rows = tr.timeline(t, tasks)
    out = {"device_error": int(rec.code), "timed_step_us_median": float(np.median(step_ms)) * 1e3,
           "summary": tr.summarize(t), "layer_profile": tr.layer_profile(rows), "timeline": rows}
    with open(path, "w") as f:
        json.dump(out, f, indent=1)


def run_glm(args, rank, world, dist):
    """The GLM FP8 pre-attention block (M = 16 = 2 requests x 8 tokens,
    hidden 6144, 39.3 MB of e4m3 weights).  The weights fit in L2, so every
    timed step runs cold: an L2-sized buffer is overwritten before it, outside
    its events.  Warm figures are reported beside."""
    import torch
    from persistent_megakernel_decode_gb300 import build, runtime as rt, synth
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    d = synth.GLM
    steps_total = args.warmup + 2 * args.steps + 40
    inp = {k: v.to(dev) for k, v in synth.make_glm_inputs(d).items()}
    stream = torch.cuda.Stream(dev)
    target = {}
    for kv in args.knob:
        k, v = kv.split("=")
        target[k] = int(v)
    sess = rt.GlmSession(d, inp, max_steps=steps_total, stream=stream, **target)
    info = sess.plan.info()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for st in range(args.warmup):
            sess.run(st, 1)
    sess.sync()
    step = args.warmup
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xff)
                ev[i][0].record(stream)
                sess.run(step, 1)
                ev[i][1].record(stream)
                step += 1
        stream.synchronize()
    cold_ms = np.array([a.elapsed_time(b) for a, b in ev])
    # warm: back to back, weights L2-resident
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        sess.run(step, args.steps)
        e1.record(stream)
    stream.synchronize()
    step += args.steps
    warm_ms = e0.elapsed_time(e1) / args.steps
    rec = sess.sync()
    total_ms = slowest_replica_ms(float(cold_ms.sum()), dist, dev)
    value = job_rate(d.M * args.steps, world, total_ms)
    # end to end: x and residual from pinned host memory in, Q-B / Indexer-Q / Head-Gate out
    hx = inp["x"].cpu().pin_memory()
    hres = inp["res"].cpu().pin_memory()
    outs = [sess.out[k] for k in ("q", "iq", "gate")]
    hout = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    e2e_steps = 20
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            inp["x"].copy_(hx, non_blocking=True)
            inp["res"].copy_(hres, non_blocking=True)
            sess.run(step, 1)
            step += 1
            for o, h in zip(outs, hout):
                h.copy_(o, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e = {"value": d.M * e2e_steps / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": 2 * hx.numel() * 2, "d2h_bytes_per_step": sum(h.numel() * 2 for h in hout),
           "steps": e2e_steps}
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    alg = info["algorithmic_bytes_step"]
    achieved = alg / (float(np.mean(cold_ms)) / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic("glm52_preattn_m16"), "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": alg, "kernel": "mk_interp (GLM instance)",
                "nominal_8tbs_frac": achieved / 8000.0}
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import glm
        sh = glm.GlmShape(R=d.R, T=d.T, H=d.H, qlora=d.qlora, kvlora=d.kvlora, rope=d.rope, q_heads=d.q_heads,
                          q_head_dim=d.q_head_dim, gate_heads=d.gate_heads, idx_heads=d.idx_heads,
                          idx_dim=d.idx_dim, slots=d.slots, eps=d.eps, theta=d.theta)
        f = lambda t: t.detach().cpu().to(torch.float64).numpy()
        wts = {}
        for n in synth.GLM_MATS:
            wts[n] = inp["w_" + n].cpu().numpy()
            wts[n + "_s"] = inp["s_" + n].cpu().numpy()
        t0 = time.perf_counter()
        glm.forward(sh, f(inp["x"]), f(inp["res"]), f(inp["norm"]), wts)
        cpu_s = time.perf_counter() - t0
        cpu = {"value": d.M / cpu_s, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": "one forward of the block (numpy fp64 oracle)"}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "config": {"workload": "glm52_preattn_m16", "requests": d.R, "tokens": d.T, "hidden": d.H,
                   "cache_slots": d.slots, "l2": "weights (39.3 MB) fit in L2: a 256 MB buffer is overwritten "
                   "before every timed step, outside its events", "parallelism": f"replicas{world}"},
        "step_us": {"median": float(np.median(cold_ms)) * 1e3, "p10": float(np.percentile(cold_ms, 10)) * 1e3,
                    "p90": float(np.percentile(cold_ms, 90)) * 1e3, "warm_mean": warm_ms * 1e3},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(),
        "gpu_launches": args.steps * info["num_launches"],
        "plan": {k: info[k] for k in ("num_workers", "lmax", "num_tasks", "num_events", "num_pages", "smem_bytes")},
        "device_error": int(rec.code),
    }
    print(json.dumps(line), flush=True)


def run_glm_reference(args):
    """The numpy fp64 oracle of the GLM block on the host cores, a bounded sample of steps."""
    import torch
    from oracle import glm
    from persistent_megakernel_decode_gb300 import synth
    d = synth.GLM
    inp = synth.make_glm_inputs(d)
    sh = glm.GlmShape(R=d.R, T=d.T, H=d.H, qlora=d.qlora, kvlora=d.kvlora, rope=d.rope, q_heads=d.q_heads,
                      q_head_dim=d.q_head_dim, gate_heads=d.gate_heads, idx_heads=d.idx_heads, idx_dim=d.idx_dim,
                      slots=d.slots, eps=d.eps, theta=d.theta)
    f = lambda t: t.to(torch.float64).numpy()
    wts = {}
    for n in synth.GLM_MATS:
        wts[n] = inp["w_" + n].numpy()
        wts[n + "_s"] = inp["s_" + n].numpy()
    steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for _ in range(steps):
        glm.forward(sh, f(inp["x"]), f(inp["res"]), f(inp["norm"]), wts)
    total = time.perf_counter() - t0
    v = d.M * steps / total
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
                      "steps": steps, "warmup": 0, "ms_per_step": total / steps * 1e3, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": {"workload": "glm52_preattn_m16"},
                      "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                       "sample": f"{steps} forwards of the block (numpy fp64 oracle)"},
                      "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--workload", default="llama1b_b1")
    ap.add_argument("--mode", default="megakernel", choices=["megakernel", "per_op"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side legs (per-op and CUDA-Graph launches, empty-kernel probe)")
    ap.add_argument("--knob", action="append", default=[], help="planner knob, e.g. attn_split=512")
    ap.add_argument("--trace-out", default="",
                    help="after the bench line, run one traced step and write its timeline (JSON) here")
    ap.add_argument("--steps-per-launch", type=int, default=128,
                    help="decode steps per cooperative launch in the timed region, at most (1: one launch per "
                         "step; the default covers a whole 128-step decode)")
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only the first N decoder layers (a small case for profiling, not a bench line)")
    args = ap.parse_args()
    from dataclasses import replace
    from persistent_megakernel_decode_gb300 import synth
    if args.workload == "glm52_preattn_m16":
        if args.trace_out:
            ap.error("--trace-out covers the decoder workloads only")
        if args.impl == "reference":
            if int(os.environ.get("RANK", "0")) == 0:
                run_glm_reference(args)
            return
        rank, world, dist = dist_setup(args.gpus)
        run_glm(args, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
        return
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = replace(w, name=f"{w.name}_L{args.layers}", shape=replace(w.shape, L=args.layers))
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, w, rank)
        return
    rank, world, dist = dist_setup(args.gpus)
    run_mk(args, w, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
