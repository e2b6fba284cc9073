"""Pins of the C oracle's decoder forward.

Every check here is fixed by mathematics or by a library routine, not by
retyping the oracle: closed forms (RMSNorm with unit weight, RoPE rotation
angles read back with atan2), special cases that collapse to numpy (zeroed
projections, a single attended position, identity output projection with
per-head attention recomputed through numpy/scipy), invariants (norm
preservation, softmax weights summing to one) and exhaustive bf16 rounding.
"""
import math

import numpy as np
import pytest
import torch

from oracle import forward as orc
from persistent_megakernel_decode_gb300 import synth


def bf(x):
    return orc.to_bf16(np.asarray(x, np.float64))


def f64(u):
    return orc.bf16_to_f64(u)


# ---------------------------------------------------------------- bf16

def test_bf16_roundtrip_exhaustive():
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = f64(u)
    keep = ~np.isnan(v)
    assert np.array_equal(bf(v[keep]), u[keep])


def test_bf16_matches_torch_rounding():
    r = np.random.default_rng(1)
    x = np.concatenate([r.standard_normal(20000) * 10.0 ** r.integers(-30, 30, 20000),
                        [1.00390625, 1.01171875, -2.0 ** -130, 3e38]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf(x.astype(np.float64)), ref)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_form():
    r = np.random.default_rng(2)
    for n, eps in ((64, 1e-5), (256, 1e-6), (7, 0.5)):
        x = r.standard_normal(n) * 3
        y = orc.rmsnorm(x, bf(np.ones(n)), eps)
        ms = np.mean(x * x)
        # with unit weight, mean(y^2) = ms / (ms + eps)
        assert math.isclose(np.mean(y * y), ms / (ms + eps), rel_tol=1e-12)
        # direction is kept
        assert math.isclose(np.dot(x, y) / np.linalg.norm(x) / np.linalg.norm(y), 1.0, rel_tol=1e-12)
        w = r.standard_normal(n)
        yw = orc.rmsnorm(x, bf(w), eps)
        assert np.allclose(yw, y * f64(bf(w)), rtol=1e-14, atol=0)


# ---------------------------------------------------------------- matvec

def test_matvec_vs_numpy_and_onehot():
    r = np.random.default_rng(3)
    W = bf(r.standard_normal((37, 53)))
    x = r.standard_normal(53)
    assert np.allclose(orc.matvec(W, x), f64(W) @ x, rtol=1e-13, atol=1e-13)
    E = np.zeros((53, 53))
    E[np.arange(53), (np.arange(53) * 7) % 53] = 1
    assert np.array_equal(orc.matvec(bf(E), x), x[(np.arange(53) * 7) % 53])


# ---------------------------------------------------------------- RoPE

def test_rope_angles_and_invariants():
    D, theta = 64, 10000.0
    r = np.random.default_rng(4)
    v = r.standard_normal(D)
    assert np.array_equal(orc.rope(v, 0, theta), v)            # position 0: identity
    for pos in (1, 17, 1000):
        w = orc.rope(v, pos, theta)
        for i in range(D // 2):
            a, b = v[i], v[i + D // 2]
            c, d = w[i], w[i + D // 2]
            assert math.isclose(a * a + b * b, c * c + d * d, rel_tol=1e-12)   # pair norm kept
            ang = math.atan2(a * d - b * c, a * c + b * d)                     # rotation applied
            want = math.remainder(pos * theta ** (-2 * i / D), 2 * math.pi)
            assert abs(math.remainder(ang - want, 2 * math.pi)) < 1e-9
    # relative position: <rope(q, m), rope(k, n)> depends only on m - n
    q, k = r.standard_normal(D), r.standard_normal(D)
    s1 = np.dot(orc.rope(q, 40, theta), orc.rope(k, 30, theta))
    s2 = np.dot(orc.rope(q, 110, theta), orc.rope(k, 100, theta))
    assert math.isclose(s1, s2, rel_tol=1e-9)


# ---------------------------------------------------------------- attention

def test_attention_special_cases():
    from scipy.special import softmax
    r = np.random.default_rng(5)
    D = 64
    q = r.standard_normal(D)
    K = bf(r.standard_normal((1, D)))
    V = bf(r.standard_normal((1, D)))
    assert np.array_equal(orc.attend(q, K, V), f64(V)[0])               # one position: o = v
    K = bf(np.repeat(r.standard_normal((1, D)), 9, 0))
    V = bf(r.standard_normal((9, D)))
    assert np.allclose(orc.attend(q, K, V), f64(V).mean(0), rtol=1e-13, atol=1e-14)   # equal keys: mean
    K = bf(r.standard_normal((50, D)))
    Vones = bf(np.ones((50, D)))
    assert np.allclose(orc.attend(q, K, Vones), 1.0, rtol=1e-14)        # weights sum to one
    V = bf(r.standard_normal((50, D)))
    p = softmax(f64(K) @ q / math.sqrt(D))
    assert np.allclose(orc.attend(q, K, V), p @ f64(V), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- whole step

def _setup(B=1, pos=(5,), seed=0, s=synth.TINY):
    w = synth.make_weights(s, seed)
    kc, vc = synth.make_cache(s, B, 80, seed + 1)
    host = synth.host_weights(w)
    shape = orc.Shape(s.L, s.H, s.Hq, s.Hkv, s.D, s.F, s.V, s.qk_norm, s.eps, s.theta)
    return s, shape, host, synth.to_host_u16(kc).copy(), synth.to_host_u16(vc).copy()


def _rms(x, eps):
    return x / np.sqrt(np.mean(x * x) + eps)


def test_step_with_zeroed_output_projections():
    """Wo = Wd = 0: the residual stays the embedding; logits = W_lm RMSNorm(E[t])."""
    s, shape, w, kc, vc = _setup()
    w["wo"] = [np.zeros_like(a) for a in w["wo"]]
    w["wd"] = [np.zeros_like(a) for a in w["wd"]]
    tok = [77]
    logits, hidden, am = orc.decode_step(shape, w, kc, vc, [5], tok)
    e = f64(w["embed"][77])
    for l in range(s.L):
        assert np.array_equal(hidden[l, 0], e)
    ref = f64(w["lm_head"]) @ _rms(e, s.eps)
    assert np.allclose(logits[0], ref, rtol=1e-12, atol=1e-12)
    assert am[0] == np.argmax(ref.astype(np.float32))


def test_step_attention_block_through_identity_output():
    """Wo = I, Wd = 0: layer-0 hidden = E[t] + o, so o is read back and checked
    head by head against numpy softmax attention over its kv group (GQA), with
    the new position's K/V taken from the appended cache slot."""
    from scipy.special import softmax
    s, shape, w, kc, vc = _setup(pos=(40,))
    assert s.H == s.Hq * s.D
    w["wo"] = [bf(np.eye(s.H)) for _ in range(s.L)]
    w["wd"] = [np.zeros_like(a) for a in w["wd"]]
    kc0 = kc.copy()
    pos, tok = 40, 3
    logits, hidden, _ = orc.decode_step(shape, w, kc, vc, [pos], [tok])
    e = f64(w["embed"][tok])
    x = _rms(e, s.eps)
    q = f64(w["wq"][0]) @ x
    k = f64(w["wk"][0]) @ x
    v = f64(w["wv"][0]) @ x
    G = s.Hq // s.Hkv
    for g in range(s.Hkv):
        kr = orc.rope(k[g * s.D:(g + 1) * s.D], pos, s.theta)
        assert np.array_equal(kc[0, 0, g, pos], bf(kr))                 # appended at slot pos, layer 0
        assert np.array_equal(vc[0, 0, g, pos], bf(v[g * s.D:(g + 1) * s.D]))
        assert np.array_equal(kc[0, 0, g, :pos], kc0[0, 0, g, :pos])    # older slots untouched
    o = hidden[0, 0] - e
    for j in range(s.Hq):
        g = j // G
        qj = orc.rope(q[j * s.D:(j + 1) * s.D], pos, s.theta)
        Kg, Vg = f64(kc[0, 0, g, :pos + 1]), f64(vc[0, 0, g, :pos + 1])
        ref = softmax(Kg @ qj / math.sqrt(s.D)) @ Vg
        assert np.allclose(o[j * s.D:(j + 1) * s.D], ref, rtol=1e-9, atol=1e-12)


def test_step_mlp_block():
    """Wo = 0: layer-0 hidden = E[t] + Wd (silu(Wg x) * (Wu x)), x = RMSNorm(E[t])."""
    s, shape, w, kc, vc = _setup()
    w["wo"] = [np.zeros_like(a) for a in w["wo"]]
    _, hidden, _ = orc.decode_step(shape, w, kc, vc, [5], [9])
    e = f64(w["embed"][9])
    x = _rms(e, s.eps)
    g = f64(w["wg"][0]) @ x
    u = f64(w["wu"][0]) @ x
    a = g / (1 + np.exp(-g)) * u
    ref = e + f64(w["wd"][0]) @ a
    assert np.allclose(hidden[0, 0], ref, rtol=1e-11, atol=1e-13)


def test_step_batch_independence_and_precisions():
    s, shape, w, kc, vc = _setup(B=2)
    kc[:, 1] = kc[:, 0]
    vc[:, 1] = vc[:, 0]
    kc2, vc2 = kc.copy(), vc.copy()
    l64, h64, a64 = orc.decode_step(shape, w, kc, vc, [12, 12], [500, 500])
    assert np.array_equal(l64[0], l64[1])
    l32, h32, _ = orc.decode_step(shape, w, kc2, vc2, [12, 12], [500, 500], precision=32)
    assert np.max(np.abs(l32 - l64)) < 1e-4 * np.max(np.abs(l64))


def test_qk_norm_path():
    s = synth.ModelShape(L=1, H=256, Hq=2, Hkv=1, D=128, F=64, V=64, eps=1e-6, theta=1e6, qk_norm=True, tied=False)
    w = synth.make_weights(s, 3)
    host = synth.host_weights(w)
    host["wo"] = [bf(np.eye(256))]
    host["wd"] = [np.zeros((256, 64), np.uint16)]
    host["qnorm"] = [bf(np.linspace(0.5, 1.5, 128))]
    host["knorm"] = [bf(np.linspace(1.5, 0.5, 128))]
    kc, vc = synth.make_cache(s, 1, 8, 4)
    kc, vc = synth.to_host_u16(kc).copy(), synth.to_host_u16(vc).copy()
    shape = orc.Shape(s.L, s.H, s.Hq, s.Hkv, s.D, s.F, s.V, True, s.eps, s.theta)
    pos = 3
    host["norm_final"] = bf(np.linspace(0.8, 1.2, 256))
    logits, hidden, _ = orc.decode_step(shape, host, kc, vc, [pos], [1])
    # untied head: logits = W_lm (RMSNorm(h_L) * w_final), not the embedding
    ref = f64(host["lm_head"]) @ (_rms(hidden[-1, 0], s.eps) * f64(host["norm_final"]))
    assert np.allclose(logits[0], ref, rtol=1e-11, atol=1e-13)
    x = _rms(f64(host["embed"][1]), s.eps)
    k = f64(host["wk"][0]) @ x
    kn = _rms(k, s.eps) * f64(host["knorm"][0])
    assert np.array_equal(kc[0, 0, 0, pos], bf(orc.rope(kn, pos, s.theta)))
    # q: per-head RMSNorm with its own weights, then RoPE; read back through Wo = I
    from scipy.special import softmax
    q = f64(host["wq"][0]) @ x
    o = hidden[0, 0] - f64(host["embed"][1])
    K, V = f64(kc[0, 0, 0, :pos + 1]), f64(vc[0, 0, 0, :pos + 1])
    for j in range(s.Hq):
        qj = orc.rope(_rms(q[j * s.D:(j + 1) * s.D], s.eps) * f64(host["qnorm"][0]), pos, s.theta)
        ref = softmax(K @ qj / math.sqrt(s.D)) @ V
        assert np.allclose(o[j * s.D:(j + 1) * s.D], ref, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- FP8 projections

def _e4m3_codes(r, shape):
    c = r.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return c


def _e4m3_as_bf16(codes):
    """The codes' values as bf16 bit patterns (torch's own e4m3 cast; every e4m3 value is exact in bf16)."""
    return synth.to_host_u16(torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.bfloat16))


def test_e4m3_decode_matches_torch_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_matvec8_with_unit_scales_is_the_bf16_matvec():
    r = np.random.default_rng(5)
    N, K = 200, 384
    codes = _e4m3_codes(r, (N, K))
    x = r.standard_normal(K)
    ones = np.ones(((N + 127) // 128, K // 128), np.float32)
    assert np.array_equal(orc.matvec8(codes, ones, x), orc.matvec(_e4m3_as_bf16(codes), x))


@pytest.mark.parametrize("rb,kb,sv", [(0, 2, 0.5), (1, 0, 2.0), (1, 2, 0.25)])
def test_matvec8_block_scale_placement(rb, kb, sv):
    """One nonzero block scale (power of two, so scaling is exact): rows outside
    row block rb are zero; rows inside are sv x the bf16 matvec over column
    block kb alone (a transposed or shifted scale index fails this)."""
    r = np.random.default_rng(6)
    N, K = 200, 384
    codes = _e4m3_codes(r, (N, K))
    x = r.standard_normal(K)
    sc = np.zeros(((N + 127) // 128, K // 128), np.float32)
    sc[rb, kb] = sv
    y = orc.matvec8(codes, sc, x)
    xk = np.zeros(K)
    xk[kb * 128:(kb + 1) * 128] = x[kb * 128:(kb + 1) * 128]
    rows = np.arange(N) // 128 == rb
    assert (y[~rows] == 0).all()
    assert np.array_equal(y[rows], sv * orc.matvec(_e4m3_as_bf16(codes), xk)[rows])


def test_step_fp8_equals_the_bf16_step_on_the_same_values():
    """A whole decode step with e4m3 projections and block scales 2^-6 (a
    power of two: code x scale is exact in bf16) equals the bf16 step on the
    dequantised weights, bit for bit (ffn 512: whole 128-wide blocks)."""
    s, shape, w, kc, vc = _setup(s=synth.TINY_TC)
    r = np.random.default_rng(7)
    w8 = dict(w)
    w8["fp8"] = True
    for n in orc.PROJ:
        pairs = []
        for l in range(s.L):
            N, K = w[n][l].shape
            codes = _e4m3_codes(r, (N, K)) & 0xBF  # exponent field <= 7: values within +-1.875
            pairs.append((codes, np.full(((N + 127) // 128, K // 128), 2.0 ** -6, np.float32)))
            vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64) * 2.0 ** -6
            w[n][l] = synth.to_host_u16(vals.to(torch.bfloat16))
        w8[n] = pairs
    kc2, vc2 = kc.copy(), vc.copy()
    lb, hb, ab = orc.decode_step(shape, w, kc, vc, [5], [42])
    l8, h8, a8 = orc.decode_step(shape, w8, kc2, vc2, [5], [42])
    assert np.isfinite(lb).all() and np.abs(hb).max() < 1e3
    assert np.array_equal(lb, l8) and np.array_equal(hb, h8) and np.array_equal(ab, a8)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


def test_fp8_weights_recipe():
    """synth's FP8 projections: every block's largest code is +-448 (scale =
    amax / 448) and code x scale reproduces N(0, 0.02)-sized weights."""
    w = synth.make_weights(synth.TINY_TC, 11, fp8=True)
    assert w["fp8"] is True
    codes, scales = w["wq"][0]
    v = torch.from_numpy(codes.numpy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    N, K = codes.shape
    blocks = np.abs(v).reshape((N + 127) // 128, -1, K // 128, 128).max(axis=(1, 3)) if N % 128 == 0 else None
    if blocks is not None:
        assert (blocks == 448.0).all()
    deq = v * np.repeat(np.repeat(scales.numpy(), 128, axis=0)[:N], 128, axis=1)
    assert 0.015 < deq.std() < 0.025
