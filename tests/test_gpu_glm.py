"""GLM FP8 pre-attention block on the GPU against the oracle (full size: M = 16
tokens, hidden 6144, 39.3 MB of e4m3 weights), with the GEMMs on tcgen05
tiles (the default at M = 16) and on the warp-level MMA tiles
(``tc_tiles=-1``); every test runs on both.

Each stage is checked on the device's own inputs to that stage (so one
rounding-boundary flip upstream cannot hide or fake an error downstream), and
the whole block end to end against the pure oracle.

Tolerances: GEMM outputs are exact products summed in fp32 per 128-wide K
block against fp64, then rounded to bf16 on both sides, so 99.9 % agree to
one bf16 unit in the last place (2^-8 relative) and every one within that
unit plus 2^-18 of the sum of its terms' magnitudes (fp32 accumulation error
where the terms cancel); RoPE outputs take one more rounding (two units),
plus a one-unit flip of either bf16 input.  An e4m3 code is an integer: the
device decides it in fp32, the oracle in fp64 from the same fp32-stored
scale, so a code may differ by one step where value / scale sits at a
rounding midpoint.  With bf16 inputs value / scale is 448 h / h_max, so exact
midpoints are common (about 0.3 % of the codes); every differing code must be
one step away and at a midpoint to within 2^-20.

End to end against the pure oracle, every output is within 1e-2 of the
largest reference value (normwise).  Q-B and Indexer-Q sit behind a second
quantisation, of bf16 QKV-A values in which the two sides differ by a unit
here and there; where that moves a block's maximum (its scale) or a value
across a midpoint, codes of the re-quantised q-lora differ by one e4m3 step.
For those two outputs the bar is: every re-quantised code within one step of
the oracle's where the two sides' q-lora inputs agree (where they differ, the
input explains the code); every element within 1e-2 (normwise) plus the change that the
differing codes and scales alone cause in the oracle's own second GEMMs; and
every element of a token row whose codes and scales all agree within 1e-2.

The tcgen05 plan splits the first GEMMs over K and adds the fp32 parts with
atomics, in whatever order they arrive: a repeated step agrees with the
first to the rounding of that sum (A0's outputs bit for bit, the first
GEMMs' outputs within one bf16 unit, everything behind them bit for bit
where those inputs agree).
"""
import numpy as np
import pytest
import torch

from oracle import glm
from persistent_megakernel_decode_gb300 import runtime as rt
from persistent_megakernel_decode_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

D = synth.GLM
SH = glm.GlmShape(R=D.R, T=D.T, H=D.H, qlora=D.qlora, kvlora=D.kvlora, rope=D.rope, q_heads=D.q_heads,
                  q_head_dim=D.q_head_dim, gate_heads=D.gate_heads, idx_heads=D.idx_heads, idx_dim=D.idx_dim,
                  slots=D.slots, eps=D.eps, theta=D.theta)


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def u8(t):
    return t.detach().cpu().numpy()


def host_weights(inp):
    w = {}
    for n in synth.GLM_MATS:
        w[n] = u8(inp["w_" + n])
        w[n + "_s"] = inp["s_" + n].cpu().numpy()
    return w


def ulp_ok(got, want, units, mag=None):
    """|got - want| <= units bf16 ulps of want (ulp = 2^(e - 7) for want in [2^e, 2^(e+1))), plus, for a
    GEMM output, 2^-18 of the sum of its terms' magnitudes `mag` (fp32 accumulation error where the
    terms cancel)."""
    want = np.asarray(want, np.float64)
    e = np.floor(np.log2(np.maximum(np.abs(want), 1e-30)))
    tol = units * np.ldexp(1.0, (e - 7).astype(np.int64)) + 1e-30
    if mag is not None:
        tol = tol + 2.0 ** -18 * mag
    return np.abs(np.asarray(got) - want) <= tol


def gemm_mag(qa, sa, qw, sw):
    """sum over k of |a_k w_k| with the block scales: the size of the terms a GEMM output sums."""
    return glm.fp8_gemm(qa & 0x7F, sa, qw & 0x7F, sw)


def codes_close(got, want):
    """Fraction of differing e4m3 codes, and whether every difference is one step."""
    g = glm.e4m3_decode(got)
    w = glm.e4m3_decode(want)
    diff = got != want
    step = np.abs(g - w) <= np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(w), 2.0 ** -6))) - 3).astype(int)) + 1e-12
    return diff.mean(), bool(step[diff].all()) if diff.any() else True


def flips_at_midpoints(got, want, quotient):
    """Every code where the device and the oracle differ sits at a rounding
    midpoint: the oracle's fp64 value / scale lies within 2^-20 (a few fp32
    roundings) of the midpoint between the two codes' values.  With bf16
    inputs value / scale is 448 h / h_max, a ratio of short numbers, so exact
    midpoints are common; the device's fp32 division lands on them exactly,
    the fp64 quotient with the fp32-stored scale just beside them."""
    diff = got != want
    if not diff.any():
        return True
    g = glm.e4m3_decode(got[diff])
    w = glm.e4m3_decode(want[diff])
    mid = (g + w) / 2
    q = np.asarray(quotient, np.float64)[diff]
    return bool((np.abs(q - mid) <= 2.0 ** -20 * np.abs(mid)).all())


def normwise(got, want):
    return np.abs(got - want).max() / np.abs(want).max()


@pytest.fixture(scope="module", params=[0, -1], ids=["tcgen05", "warp_mma"])
def run(request):
    dev = torch.device("cuda:0")
    inp_cpu = synth.make_glm_inputs(D)
    inp = {k: v.to(dev) for k, v in inp_cpu.items()}
    sess = rt.GlmSession(D, inp, max_steps=3, tc_tiles=request.param)
    assert sess.plan.info()["tc_tiles"] == (1 if request.param == 0 else 0)
    sess.run(0, 1)
    rec = sess.sync()
    assert rec.code == 0, rec.code
    out = {k: v.clone() for k, v in sess.out.items()}
    out["latent"] = sess.latent.clone()
    out["index"] = sess.index.clone()
    return sess, inp_cpu, out


def test_a0_add_norm_quant(run):
    _, inp, out = run
    h, q, s = glm.add_norm_quant(f64(inp["x"]), f64(inp["res"]), f64(inp["norm"]), SH.eps)
    assert ulp_ok(f64(out["res_out"]), h, 1).all()
    frac, one_step = codes_close(u8(out["qa"]), q)
    quot = (glm.rmsnorm(h, f64(inp["norm"]), SH.eps).reshape(SH.M, -1, 128) / s[:, :, None]).reshape(SH.M, -1)
    assert one_step and flips_at_midpoints(u8(out["qa"]), q, quot) and frac <= 1e-2, frac
    assert np.allclose(out["sa"].cpu().numpy(), s, rtol=1e-5, atol=0)


@pytest.mark.parametrize("name,mat", [("qkva", "qkva"), ("gate", "gate"), ("ik", "ik")])
def test_fan_out_gemms(run, name, mat):
    _, inp, out = run
    w = host_weights(inp)
    args = (u8(out["qa"]), out["sa"].cpu().numpy(), w[mat], w[mat + "_s"])
    ref = glm.fp8_gemm(*args)
    mag = gemm_mag(*args)
    got = f64(out[name])
    assert ulp_ok(got, ref, 1).mean() >= 0.999
    assert ulp_ok(got, ref, 1, mag).all()


def test_fin_requant_and_cache_rows(run):
    sess, inp, out = run
    qkva = f64(out["qkva"])
    q, s = glm.quant_blocks(qkva[:, :SH.qlora])
    frac, one_step = codes_close(u8(out["qb"]), q)
    quot = (qkva[:, :SH.qlora].reshape(SH.M, -1, 128) / s[:, :, None]).reshape(SH.M, -1)
    assert one_step and flips_at_midpoints(u8(out["qb"]), q, quot) and frac <= 1e-2, frac
    assert np.allclose(out["sb"].cpu().numpy(), s, rtol=1e-5, atol=0)
    pos = glm.positions(SH)
    kv_end = SH.qlora + SH.kvlora
    lat = f64(out["latent"])
    idx = f64(out["index"])
    lat0 = f64(inp["latent"])
    idx0 = f64(inp["index"])
    ik = f64(out["ik"])
    for m in range(SH.M):
        r, slot = m // SH.T, pos[m]
        assert np.array_equal(lat[r, slot, :SH.kvlora], qkva[m, SH.qlora:kv_end])
        kpe = glm.rope_half(qkva[m, kv_end:], pos[m], SH.theta)
        assert ulp_ok(lat[r, slot, SH.kvlora:], glm.bf16_round(kpe), 2).all()
        assert np.array_equal(idx[r, slot, :SH.idx_dim - SH.rope], ik[m, :SH.idx_dim - SH.rope])
        ikr = glm.rope_half(ik[m, SH.idx_dim - SH.rope:], pos[m], SH.theta)
        assert ulp_ok(idx[r, slot, SH.idx_dim - SH.rope:], glm.bf16_round(ikr), 2).all()
    # every other slot keeps its bytes
    mask = np.ones(lat.shape[:2], bool)
    for m in range(SH.M):
        mask[m // SH.T, pos[m]] = False
    assert np.array_equal(lat[mask], lat0[mask]) and np.array_equal(idx[mask], idx0[mask])


@pytest.mark.parametrize("name,mat,heads,hd", [("q", "qb", SH.q_heads, SH.q_head_dim),
                                                ("iq", "iq", SH.idx_heads, SH.idx_dim)])
def test_second_gemms_with_rope(run, name, mat, heads, hd):
    _, inp, out = run
    w = host_weights(inp)
    args = (u8(out["qb"]), out["sb"].cpu().numpy(), w[mat], w[mat + "_s"])
    ref = glm.fp8_gemm(*args).reshape(SH.M, heads, hd)
    mag = gemm_mag(*args).reshape(SH.M, heads, hd)
    r = hd - SH.rope
    rot = ref.copy()
    rot[:, :, r:] = glm.bf16_round(glm.rope_half(ref[:, :, r:], glm.positions(SH)[:, None], SH.theta))
    # a roped value mixes two bf16 GEMM outputs: besides their terms' size, a
    # one-unit flip of either input (2^-8 of it) moves it
    pair = lambda a: a[:, :, r:] + np.concatenate([a[:, :, r + 32:], a[:, :, r:r + 32]], axis=2)
    rtol_terms = pair(mag) + 2.0 ** 10 * pair(np.abs(ref))
    got = f64(out[name])
    assert ulp_ok(got[:, :, :r], ref[:, :, :r], 1).mean() >= 0.999
    assert ulp_ok(got[:, :, :r], ref[:, :, :r], 1, mag[:, :, :r]).all()
    assert ulp_ok(got[:, :, r:], rot[:, :, r:], 2).mean() >= 0.999
    assert ulp_ok(got[:, :, r:], rot[:, :, r:], 2, rtol_terms).all()


def second_gemms(qb, sb, w, mat, heads, hd):
    """The oracle's Q-B / Indexer-Q step (GEMM, then RoPE on each head's last
    `rope` columns) on the given re-quantised q-lora codes and scales."""
    y = glm.fp8_gemm(qb, sb, w[mat], w[mat + "_s"]).reshape(SH.M, heads, hd)
    r = hd - SH.rope
    y[:, :, r:] = glm.bf16_round(glm.rope_half(y[:, :, r:], glm.positions(SH)[:, None], SH.theta))
    return y


def test_end_to_end_against_the_oracle(run):
    _, inp, out = run
    w = host_weights(inp)
    ref = glm.forward(SH, f64(inp["x"]), f64(inp["res"]), f64(inp["norm"]), w)
    for k in ("res_out", "qkva", "gate", "ik"):
        assert normwise(f64(out[k]), ref[k]) <= 1e-2, k
    dq, ds = u8(out["qb"]), out["sb"].cpu().numpy()
    # where the two sides' bf16 q-lora inputs agree, their codes are within one
    # step (a block's scale may still move with another element); where the
    # inputs differ (a GEMM output near zero may even change sign) the code
    # difference traces to the input
    same_in = f64(out["qkva"])[:, :SH.qlora] == ref["qkva"][:, :SH.qlora]
    _, one_step = codes_close(dq[same_in], ref["qb"][same_in])
    assert one_step, "a re-quantised code differs from the oracle's by more than one e4m3 step on equal inputs"
    agree = (dq == ref["qb"]).all(axis=1) & (ds == ref["qb_s"]).all(axis=1)   # token rows
    for k, mat, heads, hd in (("q", "qb", SH.q_heads, SH.q_head_dim), ("iq", "iq", SH.idx_heads, SH.idx_dim)):
        got, want = f64(out[k]), ref[k]
        bar = 1e-2 * np.abs(want).max()
        explained = np.abs(second_gemms(dq, ds, w, mat, heads, hd) - want)
        err = np.abs(got - want)
        assert (err <= bar + explained).all(), k
        assert (err[agree] <= bar).all(), k
    pos = glm.positions(SH)
    lat = f64(out["latent"])
    idx = f64(out["index"])
    got_lat = np.stack([lat[m // SH.T, pos[m]] for m in range(SH.M)]).reshape(ref["latent"].shape)
    got_idx = np.stack([idx[m // SH.T, pos[m]] for m in range(SH.M)]).reshape(ref["index"].shape)
    assert normwise(got_lat, ref["latent"]) <= 1e-2 and normwise(got_idx, ref["index"]) <= 1e-2


def test_repeated_steps_are_identical_and_counters_add_up(run):
    sess, _, out = run
    sess.run(1, 2)
    assert sess.sync().code == 0
    th = sess.plan.export()[2]
    assert (sess.counters() == 3 * th).all()
    if sess.plan.info()["tc_tiles"] == 0:
        for k, v in sess.out.items():
            assert torch.equal(v, out[k]), k
        return
    for k in ("res_out", "qa", "sa"):
        assert torch.equal(sess.out[k], out[k]), k
    for k in ("qkva", "gate", "ik"):
        assert ulp_ok(f64(sess.out[k]), f64(out[k]), 1).all(), k
    if torch.equal(sess.out["qkva"], out["qkva"]):
        for k in ("qb", "sb", "q", "iq"):
            assert torch.equal(sess.out[k], out[k]), k
