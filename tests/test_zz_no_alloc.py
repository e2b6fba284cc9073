"""The allocation-free entry point, mk_run_static, against mk_run.

Some callers cannot allocate device memory (an application whose own
allocator owns the device, or a loop where cudaMalloc could block); for them
mk_run_static keeps the workspace in a fixed array inside the library.  This
test decodes the same two steps through both entry points, on separate copies
of the same seeded inputs, and checks that the outputs agree within the 1e-2
tolerance the parity tests use.  It runs last, and passes alone or after the
other tests (the static array keeps earlier contents; step 0 clears what must
start at zero).
"""
import numpy as np
import pytest
import torch

from persistent_megakernel_decode_gb300 import runtime as rt
from persistent_megakernel_decode_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(180)]


def _normwise(a, ref):
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-30))


def test_static_workspace_matches_allocated_workspace_two_calls():
    from persistent_megakernel_decode_gb300 import build
    build.build()
    shape = synth.TINY
    dev = torch.device("cuda:0")
    w = synth.make_weights(shape, 11, device=dev)
    kc, vc = synth.make_cache(shape, 2, 80, 111, device=dev)
    seq0 = [64, 20]
    ref = rt.Session(shape, w, kc.clone(), vc.clone(), seq0, 2, capture_hidden=True)
    nal = rt.Session(shape, w, kc.clone(), vc.clone(), seq0, 2, capture_hidden=True)
    assert nal.plan.info()["workspace_bytes"] <= rt.STATIC_WORKSPACE_BYTES
    for s in range(2):
        toks = torch.tensor([100 + s, 900 - s], dtype=torch.int32, device=dev)
        ref.tokens[s] = toks
        nal.tokens[s] = toks
        ref.run(s, 1, host_tokens=True)
        ref.sync()
        addr = nal.run_static(s, 1, host_tokens=True)
        rec = nal.sync_static(addr)
        assert rec.code == 0
        a, b = ref.logits.cpu().numpy(), nal.logits.cpu().numpy()
        assert _normwise(b, a) <= 1e-2
        assert _normwise(nal.hidden.cpu().numpy(), ref.hidden.cpu().numpy()) <= 1e-2
        assert list(ref.step_tokens(s)) == list(nal.step_tokens(s))
    # the appended KV entries agree too
    assert _normwise(nal.kcache.float().cpu().numpy(), ref.kcache.float().cpu().numpy()) <= 1e-2


def test_static_workspace_rejects_oversized_plans():
    from persistent_megakernel_decode_gb300 import build
    build.build()
    # a plan whose workspace exceeds the static array is refused before any GPU work
    p = rt.Plan.llama(synth.QWEN3_8B, 4, [2048] * 4, 32, 2081, num_sms=152, smem_per_cta=232448, attn_split=16)
    assert p.info()["workspace_bytes"] > rt.STATIC_WORKSPACE_BYTES
    addr = rt.C.c_uint64(0)
    rc = rt.load().mk_run_static(p.h, 0, 1, 0, 0, None, rt.C.byref(addr))
    assert rc == rt.MK_ERR_INVALID and b"static workspace" in rt.load().mk_last_error()


def test_static_workspace_alternating_plans():
    """Two plans take turns on the one static array: each call after a switch
    uploads that plan's queue again and must start at step 0 (the counters
    in the array are the other plan's); resuming at a later step after a
    switch is refused, and the same plan may go on once it owns the array."""
    from persistent_megakernel_decode_gb300 import build
    build.build()
    shape = synth.TINY
    dev = torch.device("cuda:0")
    w = synth.make_weights(shape, 12, device=dev)
    kc, vc = synth.make_cache(shape, 2, 80, 112, device=dev)
    k1, v1 = synth.make_cache(shape, 1, 80, 113, device=dev)
    cases = {"A": ([64, 20], kc, vc, [7, 300]), "B": ([33], k1, v1, [512])}
    ref, nal = {}, {}
    for n, (seq0, k, v, toks) in cases.items():
        ref[n] = rt.Session(shape, w, k.clone(), v.clone(), seq0, 2, capture_hidden=True)
        nal[n] = rt.Session(shape, w, k.clone(), v.clone(), seq0, 2, capture_hidden=True)
        for s in (ref[n], nal[n]):
            s.tokens[0] = torch.tensor(toks, dtype=torch.int32, device=dev)
            s.tokens[1] = torch.tensor(toks, dtype=torch.int32, device=dev) + 1
    snap = {}  # (plan, step) -> what mk_run left after that step
    for n in cases:
        for step in range(2):
            ref[n].run(step, 1, host_tokens=True)
            ref[n].sync()
            snap[n, step] = (ref[n].hidden.cpu().numpy(), ref[n].logits.cpu().numpy(), list(ref[n].step_tokens(step)))

    def check(n, step):
        h, lg, tok = snap[n, step]
        b = nal[n]
        assert _normwise(b.hidden.cpu().numpy(), h) <= 1e-2, (n, step)
        assert _normwise(b.logits.cpu().numpy(), lg) <= 1e-2, (n, step)
        assert list(b.step_tokens(step)) == tok, (n, step)

    lib = rt.load()
    for n in ("A", "B", "A"):
        # re-running step 0 rewrites the same cache slot with the same values
        addr = nal[n].run_static(0, 1, host_tokens=True)
        assert nal[n].sync_static(addr).code == 0
    check("A", 0)
    # B runs step 0, then A may not resume at step 1 on B's counters
    addr = nal["B"].run_static(0, 1, host_tokens=True)
    assert nal["B"].sync_static(addr).code == 0
    check("B", 0)
    out = rt.C.c_uint64(0)
    rc = lib.mk_run_static(nal["A"].plan.h, 1, 1, rt.RUN_HOST_TOKENS, 0,
                           rt.C.c_void_p(nal["A"].stream.cuda_stream), rt.C.byref(out))
    assert rc == rt.MK_ERR_INVALID and b"first_step 0" in lib.mk_last_error()
    # B still owns the array and goes on to step 1
    addr = nal["B"].run_static(1, 1, host_tokens=True)
    assert nal["B"].sync_static(addr).code == 0
    check("B", 1)
    # A starts over at step 0 and then continues
    for s in range(2):
        addr = nal["A"].run_static(s, 1, host_tokens=True)
        assert nal["A"].sync_static(addr).code == 0
    check("A", 1)
