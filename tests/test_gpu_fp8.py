"""FP8 projections on the GPU against the oracle.

The seven projections stream as e4m3 rows with one fp32 scale per 128 x 128
block (the embedding, LM head and norms stay bf16); the batch-1 FP8 kernel
instance runs them as row-per-warp tiles of 32 rows to a 64 KB page.  The
oracle dequantises every weight in fp64 before its dot product.

* two layers of the Llama-3.2-1B shape (K = 2048 everywhere), 700 cached
  tokens, three steps;
* the full 16-layer Llama-3.2-1B shape, 1024 cached tokens (the benchmarked
  FP8 plan), one step;
* 256 teacher-forced steps of the two-layer model: at least 99 % identical
  argmax;
* several steps in one launch equal the same steps launched one by one.

Bars as for every path: per-layer residual stream, logits and the appended
K/V within 1e-2 normwise of the oracle; an argmax may differ only where the
oracle's top-2 gap is within 4x the measured logits error.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from persistent_megakernel_decode_gb300 import runtime as rt
from persistent_megakernel_decode_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_megakernel_decode_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _check(run, tol=1e-2):
    for r in run.reports:
        assert max(r.hidden_err) <= tol, (r.step, r.hidden_err)
        assert r.logits_err <= tol, (r.step, r.logits_err)
        assert r.kv_err <= tol, (r.step, r.kv_err)
        assert r.argmax_mismatches_explained(), (r.step, r.argmax_gpu, r.argmax_ref, r.gaps, r.logits_err)


def test_plan_takes_the_fp8_instance():
    p = rt.Plan.llama(replace(synth.LLAMA_1B, L=2), 1, [700], 3, 710, fp8=True)
    assert p.info()["weight_fp8"] == 1


def test_llama_width_two_layers():
    from harness import run_parity
    run = run_parity(replace(synth.LLAMA_1B, L=2), [700], 3, [0, 1, 2], seed=61, fp8=True)
    _check(run)


def test_llama1b_full_size_benchmarked_plan():
    from harness import run_parity
    run = run_parity(synth.LLAMA_1B, [1024], 1, [0], seed=62, fp8=True)
    _check(run)


def test_two_layers_argmax_over_256_steps():
    from harness import run_parity
    run = run_parity(replace(synth.LLAMA_1B, L=2), [300], 256, range(256), seed=63, fp8=True)
    _check(run)
    m, t = run.matches()
    assert t == 256 and m >= 0.99 * t, (m, t)


def test_one_launch_matches_step_launches():
    shape = replace(synth.LLAMA_1B, L=2)
    dev = torch.device("cuda:0")
    steps = 5

    def run(one_launch):
        w = synth.make_weights(shape, 64, device=dev, fp8=True)
        kc, vc = synth.make_cache(shape, 1, 700 + steps + 1, 164, device=dev)
        sess = rt.Session(shape, w, kc, vc, [700], steps, capture_hidden=True)
        sess.tokens[0] = torch.tensor([123], dtype=torch.int32, device=dev)
        if one_launch:
            sess.run(0, steps, one_launch=True)
        else:
            for s in range(steps):
                sess.run(s, 1)
        assert sess.sync().code == 0
        return sess

    a, b = run(False), run(True)
    assert np.array_equal(a.tokens.cpu().numpy(), b.tokens.cpu().numpy())
    la, lb = a.logits.cpu().numpy(), b.logits.cpu().numpy()
    assert np.max(np.abs(la - lb)) <= 1e-4 * np.max(np.abs(la))
    th = a.plan.export()[2]
    assert (a.counters() == steps * th).all() and (b.counters() == steps * th).all()
