"""Several decode steps in one cooperative launch (MK_RUN_ONE_LAUNCH) against
the same steps launched one by one -- which the parity tests check against
the oracle -- on every kernel instance: the lean batch-1 instance (the tiny
decoder, two layers of the Llama-1B width, and the full benchmarked plan at
16 steps per launch), the general instance (batch 3), the tensor-core
instance (batch 16) and the GLM block.

Within one launch every worker walks its queue once per step; the monotone
event epochs order the steps, the next step's embedding waits for the
previous step's LM head, and K/V rows appended by an earlier step of the
launch are read only after that step's attention event.  Tokens are fed on
the device (each step's argmax feeds the next), so a wrong step boundary
shows as a different token chain.  MLP-down and (tensor-core) O tiles add
into the residual with atomics, so the two runs agree to rounding, not bit
for bit: logits and residual snapshots within 1e-4 normwise, the appended
bf16 cache within one bf16 unit of its largest value (2^-8 normwise: an fp32
value that differs in its last bits may round to the neighbouring bf16),
identical tokens, and counters that are steps x increments.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from persistent_megakernel_decode_gb300 import runtime as rt
from persistent_megakernel_decode_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(600)]

STEPS = 6


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_megakernel_decode_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _normwise(a, ref):
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _run(shape, lengths, one_launch, seed):
    dev = torch.device("cuda:0")
    w = synth.make_weights(shape, seed, device=dev)
    kc, vc = synth.make_cache(shape, len(lengths), max(lengths) + STEPS + 1, seed + 100, device=dev)
    sess = rt.Session(shape, w, kc, vc, lengths, STEPS, capture_hidden=True)
    g = torch.Generator().manual_seed(seed + 200)
    sess.tokens[0] = torch.randint(0, shape.V, (len(lengths),), generator=g).to(torch.int32).to(dev)
    if one_launch:
        sess.run(0, STEPS, one_launch=True)
    else:
        for s in range(STEPS):
            sess.run(s, 1)
    assert sess.sync().code == 0
    return sess


@pytest.mark.parametrize("name,shape,lengths", [
    ("tiny_lean", synth.TINY, [64]),
    ("llama_width_lean", replace(synth.LLAMA_1B, L=2), [700]),
    ("tiny_general_b3", synth.TINY, [5, 64, 130]),
    ("tiny_tc_b16", synth.TINY_TC, [20 + 13 * b for b in range(16)]),
])
def test_one_launch_matches_step_launches(name, shape, lengths):
    a = _run(shape, lengths, False, 51)
    b = _run(shape, lengths, True, 51)
    assert np.array_equal(a.tokens.cpu().numpy(), b.tokens.cpu().numpy()), name
    assert _normwise(b.logits.cpu().numpy(), a.logits.cpu().numpy()) <= 1e-4
    assert _normwise(b.hidden.cpu().numpy(), a.hidden.cpu().numpy()) <= 1e-4
    for x, y in ((a.kcache, b.kcache), (a.vcache, b.vcache)):
        assert _normwise(y.float().cpu().numpy(), x.float().cpu().numpy()) <= 2.0 ** -8
    th = a.plan.export()[2]
    assert (a.counters() == STEPS * th).all() and (b.counters() == STEPS * th).all()


def test_benchmarked_plan_16_steps_in_one_launch():
    """The launch shape the benchmark times: the full 16-layer Llama-1B plan at
    batch 1 (1024 cached tokens), 16 steps in one launch against 16 launches."""
    wl = synth.WORKLOADS["llama1b_b1"]
    steps = 16
    dev = torch.device("cuda:0")

    def run(one_launch):
        w = synth.make_weights(wl.shape, wl.weight_seed, device=dev)
        kc, vc = synth.make_cache(wl.shape, 1, wl.seq_len + steps + 1, wl.cache_seed, device=dev)
        sess = rt.Session(wl.shape, w, kc, vc, [wl.seq_len], steps)
        sess.tokens[0] = torch.tensor(synth.first_tokens(wl), dtype=torch.int32, device=dev)
        if one_launch:
            sess.run(0, steps, one_launch=True)
        else:
            for s in range(steps):
                sess.run(s, 1)
        assert sess.sync().code == 0
        return sess

    a, b = run(False), run(True)
    assert np.array_equal(a.tokens.cpu().numpy(), b.tokens.cpu().numpy())
    assert _normwise(b.logits.cpu().numpy(), a.logits.cpu().numpy()) <= 1e-4
    for x, y in ((a.kcache, b.kcache), (a.vcache, b.vcache)):
        assert _normwise(y.float().cpu().numpy(), x.float().cpu().numpy()) <= 2.0 ** -8
    th = a.plan.export()[2]
    assert (a.counters() == steps * th).all() and (b.counters() == steps * th).all()


@pytest.mark.parametrize("tc_tiles", [0, -1], ids=["tcgen05", "warp_mma"])
def test_one_launch_glm_block(tc_tiles):
    """Bit for bit with the warp-level tiles; with the tcgen05 tiles (K-split
    parts added by atomics in arrival order) A0 bit for bit, the first GEMMs
    within one bf16 unit, and the rest bit for bit where those agree."""
    dev = torch.device("cuda:0")
    inp = {k: v.to(dev) for k, v in synth.make_glm_inputs(synth.GLM).items()}
    a = rt.GlmSession(synth.GLM, {k: v.clone() for k, v in inp.items()}, max_steps=4, tc_tiles=tc_tiles)
    b = rt.GlmSession(synth.GLM, {k: v.clone() for k, v in inp.items()}, max_steps=4, tc_tiles=tc_tiles)
    for s in range(4):
        a.run(s, 1)
    b.run(0, 4, one_launch=True)
    assert a.sync().code == 0 and b.sync().code == 0
    th = a.plan.export()[2]
    assert (b.counters() == 4 * th).all()
    exact = ("res_out", "qa", "sa") if tc_tiles == 0 else tuple(a.out)
    for k in exact:
        assert torch.equal(a.out[k], b.out[k]), k
    if tc_tiles == 0:
        for k in ("qkva", "gate", "ik"):
            x, y = a.out[k].double(), b.out[k].double()
            assert ((x - y).abs() <= 2.0 ** -7 * x.abs() + 1e-30).all(), k
        if not (torch.equal(a.out["qkva"], b.out["qkva"]) and torch.equal(a.out["ik"], b.out["ik"])):
            return
        for k in ("qb", "sb", "q", "iq"):
            assert torch.equal(a.out[k], b.out[k]), k
    assert torch.equal(a.latent, b.latent) and torch.equal(a.index, b.index)


def test_one_launch_trace_keeps_the_last_step():
    """With MK_RUN_TRACE a slot's stamps are those of its last step: in a
    3-step launch every first-layer QKV tile is handed its activation after
    the embedding of the same (last) step is done."""
    shape = synth.TINY
    dev = torch.device("cuda:0")
    w = synth.make_weights(shape, 52, device=dev)
    kc, vc = synth.make_cache(shape, 1, 80, 152, device=dev)
    sess = rt.Session(shape, w, kc, vc, [64], 4)
    sess.run(0, 3, trace=True, one_launch=True)
    assert sess.sync().code == 0
    t = sess.trace().astype(np.int64)
    tasks = sess.plan.export()[3]
    op = t[..., 0] & 0xFFFFFFFF
    tid = t[..., 0] >> 32
    emb_done = t[op == rt.OPCODE["embed"]][0][3]
    q0 = (op == rt.OPCODE["qkv"]) & (tasks[np.clip(tid, 0, len(tasks) - 1), 1] == 0) & (t[..., 13] > 0)
    assert q0.any() and (t[..., 13][q0] > emb_done).all()
