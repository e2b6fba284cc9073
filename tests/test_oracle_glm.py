"""Pins for the GLM FP8 block oracle (no GPU): the e4m3 format from its
definition, quantisation bounds, the blocked FP8 GEMM against brute force,
RoPE and RMSNorm invariants, bf16 rounding against torch's own conversion."""
import math

import numpy as np
import pytest
import torch

from oracle import glm


def test_e4m3_decode_known_codes():
    d = glm.e4m3_decode
    assert d(0x00) == 0.0
    assert d(0x01) == 2.0 ** -9                 # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert d(0x08) == 2.0 ** -6                 # smallest normal
    assert d(0x38) == 1.0                       # exponent field 7 = bias
    assert d(0x39) == 1.125
    assert d(0x7E) == 448.0                     # largest finite
    assert d(0xFE) == -448.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))


def test_e4m3_every_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    assert (glm.e4m3_encode(glm.e4m3_decode(codes)) == codes).all()


def test_e4m3_ties_to_even_and_saturation():
    enc = glm.e4m3_encode
    assert enc(1.0 + 1 / 16) == 0x38            # halfway 1.0 / 1.125 -> even mantissa 0
    assert enc(1.0 + 3 / 16) == 0x3A            # halfway 1.125 / 1.25 -> even mantissa 2
    assert enc(2.0 ** -10) == 0x00              # halfway 0 / 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02          # halfway 2^-9 / 2^-8 -> even
    assert enc(1000.0) == 0x7E and enc(-1e9) == 0xFE and enc(464.0) == 0x7E


def test_e4m3_relative_error_bound():
    rng = np.random.default_rng(3)
    x = rng.uniform(2.0 ** -6, 448.0, 20000) * rng.choice([-1, 1], 20000)
    err = np.abs(glm.e4m3_decode(glm.e4m3_encode(x)) - x)
    assert (err <= 2.0 ** -4 * np.abs(x)).all()


def test_e4m3_matches_torch_conversion():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.uniform(-448, 448, 20000), rng.normal(0, 0.01, 5000)])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = glm.e4m3_encode(x.astype(np.float32).astype(np.float64))
    same = ours == ref
    # -0.0 from torch for tiny negatives encodes as 0x80; ours gives 0x00 (both are zero)
    zero = (glm.e4m3_decode(ref) == 0) & (glm.e4m3_decode(ours) == 0)
    assert (same | zero).all()


def test_quant_blocks_scale_and_zero_block():
    rng = np.random.default_rng(5)
    y = rng.normal(0, 2, (3, 384))
    y[1, 128:256] = 0.0
    q, s = glm.quant_blocks(y)
    assert s.dtype == np.float32 and s.shape == (3, 3)
    assert s[1, 1] == 1.0 and (q[1, 128:256] == 0).all()
    dq = glm.e4m3_decode(q).reshape(3, 3, 128)
    for m in range(3):
        for b in range(3):
            if m == 1 and b == 1:
                continue
            assert np.abs(dq[m, b]).max() == 448.0   # the amax element lands on the largest code
    rel = np.abs(dq * s[:, :, None] - y.reshape(3, 3, 128))
    assert (rel <= 2.0 ** -4 * np.abs(y.reshape(3, 3, 128)) + s[:, :, None] * 2.0 ** -9).all()


def _brute_gemm(qa, sa, qw, sw):
    A, W = glm.e4m3_decode(qa), glm.e4m3_decode(qw)
    M, K = A.shape
    N = W.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):   # dequantise each element with its own scales, then multiply
                acc += (A[m, k] * sa[m, k // 128]) * (W[n, k] * sw[n // 128, k // 128])
            out[m, n] = acc
    return out


def test_fp8_gemm_matches_brute_force():
    rng = np.random.default_rng(6)
    M, N, K = 3, 130, 256
    qa = rng.integers(0, 256, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x38               # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0x38
    sa = rng.uniform(0.01, 2, (M, 2)).astype(np.float32)
    sw = rng.uniform(0.01, 2, (2, 2)).astype(np.float32)
    got = glm.fp8_gemm(qa, sa, qw, sw)
    ref = _brute_gemm(qa, sa, qw, sw)
    assert np.array_equal(got, glm.bf16_round(ref)) or np.allclose(got, ref, rtol=2 ** -8, atol=1e-6)


def test_fp8_gemm_one_hot_weights():
    rng = np.random.default_rng(7)
    qa = glm.e4m3_encode(rng.normal(0, 50, (4, 256)))
    sa = np.full((4, 2), 0.5, np.float32)
    qw = np.zeros((8, 256), np.uint8)
    for n in range(8):
        qw[n, 17 * n + 3] = 0x38                  # 1.0 at one position
    sw = np.ones((1, 2), np.float32)
    got = glm.fp8_gemm(qa, sa, qw, sw)
    want = glm.e4m3_decode(qa)[:, [17 * n + 3 for n in range(8)]] * 0.5
    assert np.array_equal(got, glm.bf16_round(want))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.normal(0, 1, 50000), rng.normal(0, 1e4, 1000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(glm.bf16_round(x.astype(np.float64)), ref)


def test_rope_half_invariants():
    rng = np.random.default_rng(9)
    x = rng.normal(0, 1, (5, 64))
    y = glm.rope_half(x, np.arange(5) * 1000 + 3, 1e4)
    lo, hi = x[:, :32], x[:, 32:]
    ylo, yhi = y[:, :32], y[:, 32:]
    assert np.allclose(lo ** 2 + hi ** 2, ylo ** 2 + yhi ** 2)      # each pair keeps its norm
    assert np.allclose(glm.rope_half(x, np.zeros(5), 1e4), x)       # position 0 is the identity
    q, k = rng.normal(0, 1, 64), rng.normal(0, 1, 64)
    d1 = glm.rope_half(q, 8191, 1e4) @ glm.rope_half(k, 8184, 1e4)
    d2 = glm.rope_half(q, 7, 1e4) @ glm.rope_half(k, 0, 1e4)
    assert math.isclose(d1, d2, rel_tol=1e-9, abs_tol=1e-9)          # depends on m - n only


def _rope_angles_ok(rope_fn, theta=1e4):
    """Each pair (i, i + 32) of a 64-wide slice is rotated by +pos * theta^(-i/32),
    read back with atan2 (direction and frequency, not just norms)."""
    rng = np.random.default_rng(11)
    x = rng.normal(0, 1, 64)
    for pos in (1, 9, 8191):
        y = rope_fn(x, pos, theta)
        for i in range(32):
            a, b, c, d = x[i], x[i + 32], y[i], y[i + 32]
            ang = math.atan2(a * d - b * c, a * c + b * d)
            want = math.remainder(pos * theta ** (-i / 32), 2 * math.pi)
            if abs(math.remainder(ang - want, 2 * math.pi)) > 1e-9:
                return False
    return True


def test_rope_half_rotation_direction_and_frequency():
    assert _rope_angles_ok(glm.rope_half)


def test_rope_angle_pin_catches_a_planted_sign_error():
    """The invariants above (pair norms, identity at 0, relative position) all
    hold for a rotation the wrong way; the angle pin does not."""
    def wrong_way(x, pos, theta):
        return glm.rope_half(x, -np.asarray(pos, dtype=np.float64), theta)
    assert not _rope_angles_ok(wrong_way)


def test_rmsnorm_unit_weight_invariant():
    rng = np.random.default_rng(10)
    h = rng.normal(0, 3, (4, 6144))
    ms = np.mean(h * h, axis=1)
    for eps in (1e-6, 0.5, 30.0):   # large eps values tell where eps sits in the formula
        y = glm.rmsnorm(h, np.ones(6144), eps)
        assert np.allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-12, atol=0)


def test_block_shapes_and_positions():
    sh = glm.GlmShape()
    assert sh.M == 16 and sh.qkva == 2112 and sh.pos0 == 8184
    assert list(glm.positions(sh)) == [8184 + j for j in range(8)] * 2
    # weight bytes of the five FP8 matrices: 39.32 MB
    n = sh.qkva * sh.H + sh.gate_heads * sh.H + sh.idx_dim * sh.H + \
        (sh.q_heads * sh.q_head_dim + sh.idx_heads * sh.idx_dim) * sh.qlora
    assert n == 39_321_600


@pytest.mark.parametrize("seed", [0, 1])
def test_forward_small_block_consistency(seed):
    """A shrunken block: every output agrees with its definition composed by hand."""
    sh = glm.GlmShape(R=1, T=2, H=256, qlora=128, kvlora=128, rope=64, q_heads=2, q_head_dim=192, gate_heads=8,
                      idx_heads=2, idx_dim=128, slots=16)
    rng = np.random.default_rng(seed)
    x = glm.bf16_round(rng.normal(0, 1, (sh.M, sh.H)))
    res = glm.bf16_round(rng.normal(0, 1, (sh.M, sh.H)))
    wts = {}
    for name, n, k in (("qkva", sh.qkva, sh.H), ("gate", sh.gate_heads, sh.H), ("ik", sh.idx_dim, sh.H),
                       ("qb", sh.q_heads * sh.q_head_dim, sh.qlora), ("iq", sh.idx_heads * sh.idx_dim, sh.qlora)):
        q = glm.e4m3_encode(rng.normal(0, 100, (n, k)))
        wts[name] = q
        wts[name + "_s"] = rng.uniform(1e-4, 1e-3, ((n + 127) // 128, k // 128)).astype(np.float32)
    out = glm.forward(sh, x, res, np.ones(sh.H), wts)
    assert np.array_equal(out["res_out"], glm.bf16_round(x + res))
    y = glm.rmsnorm(out["res_out"], np.ones(sh.H), sh.eps)
    assert np.allclose(glm.e4m3_decode(out["qa"]) * np.repeat(out["sa"], 128, axis=1), y, rtol=2 ** -4, atol=1e-3)
    kv_end = sh.qlora + sh.kvlora
    assert np.array_equal(out["latent"][0, :, :sh.kvlora], out["qkva"][:, sh.qlora:kv_end])
    # Q-B and Indexer-Q read the q-lora columns (the first qlora of QKV-A), re-quantised per 128
    dq = glm.e4m3_decode(out["qb"]) * np.repeat(out["qb_s"], 128, axis=1)
    assert np.allclose(dq, out["qkva"][:, :sh.qlora], rtol=2 ** -4, atol=np.max(out["qb_s"]) * 2.0 ** -9)
    assert np.array_equal(out["index"][0, :, :64], out["ik"][:, :64])
    # the roped slice keeps pair norms up to bf16 rounding
    a = out["qkva"][:, kv_end:]
    b = out["latent"][0, :, sh.kvlora:]
    assert np.allclose(a[:, :32] ** 2 + a[:, 32:] ** 2, b[:, :32] ** 2 + b[:, 32:] ** 2, rtol=2e-2, atol=1e-6)
    # Q-B and Indexer-Q: the GEMM of the re-quantised q-lora, RoPE on the last 64 of each head only
    for name, mat, heads, hd in (("q", "qb", sh.q_heads, sh.q_head_dim), ("iq", "iq", sh.idx_heads, sh.idx_dim)):
        g = glm.fp8_gemm(out["qb"], out["qb_s"], wts[mat], wts[mat + "_s"]).reshape(sh.M, heads, hd)
        r = hd - sh.rope
        assert np.array_equal(out[name][:, :, :r], g[:, :, :r])
        got, ref = out[name][:, :, r:], g[:, :, r:]
        assert not np.array_equal(got, ref)                     # the slice was rotated
        assert np.allclose(got[..., :32] ** 2 + got[..., 32:] ** 2, ref[..., :32] ** 2 + ref[..., 32:] ** 2,
                           rtol=2e-2, atol=1e-9)
