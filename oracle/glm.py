"""GLM FP8 pre-attention block, written out plainly (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module.  It shares no code with the CUDA path.

Source: "MegaRTP megakernel article" (GLM-5.2-FP8 decode, the computation
before sparse FlashMLA, M = 16 = 2 requests x 8 tokens, KV = 8192), section 1
(the Add+RMSNorm+Quant kernel, the GEMMs, RoPE and cache write-back) and
section 2 (the three independent branches QKV-A, Head-Gate and Indexer-K
after the first kernel; QKV-A feeding the main path and the Indexer-Q path).
Where the article is silent the plainest reading is taken:

* FP8 is e4m3 "fn" (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
  bits, no infinities, largest finite value 448).  Activations are quantised
  per (row, 128-column block): scale = amax / 448 (amax = 0 gives scale 1),
  code = round-to-nearest-even of value / scale, saturating at +-448.  The
  block scales are stored as fp32 (the workload states "fp32 block scales"),
  so the scale is amax / 448 rounded to fp32.  Neither the article nor the
  workload fixes the precision of the division and of the rounding decision;
  they are taken in fp64 here, like the rest of this oracle, on the fp64
  values and the fp32-stored scale.  A device that decides in fp32 may land
  one e4m3 step the other way where value / scale sits within an fp32
  rounding of a midpoint; the tests count such codes.
* Weights are e4m3 with one fp32 scale per 128 x 128 block (inputs).
* A GEMM output is sum over 128-wide K blocks of
  a_scale[m, kb] * w_scale[n // 128, kb] * sum_k a[m, k] * w[n, k], rounded to
  bf16.
* The Add of the residual gives the new residual stream in bf16; the RMSNorm
  (eps 1e-6, weight 1) reads those bf16 values.
* RoPE: rotate-half pairs (i, i + 32) of each 64-wide slice, angle
  pos * theta^(-2i/64), theta 1e4, applied to the bf16 GEMM output and
  rounded to bf16 again.  Slices: QKV-A columns 2048..2111 (k_pe), the last 64
  of each 192-wide Q-B head, the last 64 of each 128-wide Indexer-Q head and
  of Indexer-K.  Token j of request r is at position pos0 + j.
* QKV-A columns: q-lora 0..1535, kv-lora 1536..2047, k_pe 2048..2111.  The
  q-lora part is re-quantised per 128 columns and feeds Q-B and Indexer-Q.
* Caches: latent [R, S, 576] <- kv-lora || roped k_pe; index [R, S, 128] <-
  Indexer-K with its last 64 roped; token j of request r writes slot pos0 + j.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


@dataclass(frozen=True)
class GlmShape:
    R: int = 2            # requests
    T: int = 8            # new tokens per request
    H: int = 6144         # hidden
    qlora: int = 1536
    kvlora: int = 512
    rope: int = 64
    q_heads: int = 64
    q_head_dim: int = 192
    gate_heads: int = 64
    idx_heads: int = 32
    idx_dim: int = 128
    slots: int = 8192     # cache slots per request
    eps: float = 1e-6
    theta: float = 1e4

    @property
    def M(self):
        return self.R * self.T

    @property
    def pos0(self):
        return self.slots - self.T

    @property
    def qkva(self):
        return self.qlora + self.kvlora + self.rope


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 value (8 significand bits), ties to even."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3fn byte (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = np.ldexp(1.0 + man / 8.0, exp - 7)
    sub = np.ldexp(man / 8.0, -6)
    v = sign * np.where(exp == 0, sub, normal)
    return np.where((exp == 0xF) & (man == 0x7), np.nan, v)


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3fn code, ties to even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # quantum of the binade holding a: 2^(e - 3) for a in [2^e, 2^(e+1)),
    # e >= -6 (below 2^-6 the subnormal quantum 2^-9)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    q = np.ldexp(1.0, (e - 3).astype(np.int64))
    v = np.round(a / q) * q                  # np.round: ties to even
    v = np.minimum(v, E4M3_MAX)
    # encode v exactly
    ve = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    is_sub = v < 2.0 ** -6
    exp_field = np.where(is_sub, 0, ve + 7).astype(np.int64)
    man_field = np.where(is_sub, np.round(v / 2.0 ** -9), np.round((v / np.ldexp(1.0, ve.astype(np.int64)) - 1.0) * 8))
    code = (exp_field << 3) | man_field.astype(np.int64)
    code = np.where(v == 0, 0, code)
    code = np.where(np.signbit(x) & (v != 0), code | 0x80, code)
    return code.astype(np.uint8)


def quant_blocks(y) -> tuple:
    """Per (row, 128-column block) e4m3 quantisation of y [M, K]: (codes, fp32 scales [M, K/128])."""
    y64 = np.asarray(y, dtype=np.float64)
    M, K = y64.shape
    yb = y64.reshape(M, K // BLOCK, BLOCK)
    amax = np.abs(yb).max(axis=2)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)   # stored as fp32
    v = yb / scale.astype(np.float64)[:, :, None]
    return e4m3_encode(v).reshape(M, K), scale


# ---------------------------------------------------------------------------
# steps
# ---------------------------------------------------------------------------

def rmsnorm(h, w, eps) -> np.ndarray:
    h = np.asarray(h, dtype=np.float64)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * np.asarray(w, dtype=np.float64)


def rope_half(x, pos, theta) -> np.ndarray:
    """Rotate-half RoPE on the last axis (even width n): pairs (i, i + n/2),
    angle pos * theta^(-2i/n); pos broadcasts against the leading axes."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    half = n // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * i / n)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def add_norm_quant(x, res, w, eps):
    """Add + RMSNorm + Quant: (new residual bf16 values, codes, scales)."""
    h = bf16_round(np.asarray(x, np.float64) + np.asarray(res, np.float64))
    y = rmsnorm(h, w, eps)
    q, s = quant_blocks(y)
    return h, q, s


def fp8_gemm(qa, sa, qw, sw) -> np.ndarray:
    """sum over K blocks of sa[m,kb] * sw[n//128,kb] * (a_kb . w_kb), fp64, then bf16."""
    A = e4m3_decode(qa)
    W = e4m3_decode(qw)
    M, K = A.shape
    N = W.shape[0]
    KB = K // BLOCK
    out = np.zeros((M, N), dtype=np.float64)
    sa = np.asarray(sa, np.float64)
    sw = np.asarray(sw, np.float64)
    for kb in range(KB):
        ks = slice(kb * BLOCK, (kb + 1) * BLOCK)
        part = A[:, ks] @ W[:, ks].T                       # [M, N]
        out += part * sa[:, kb][:, None] * np.repeat(sw[:, kb], BLOCK)[:N][None, :]
    return bf16_round(out)


def positions(sh: GlmShape) -> np.ndarray:
    return sh.pos0 + (np.arange(sh.M) % sh.T)


def forward(sh: GlmShape, x, res, norm_w, w: dict) -> dict:
    """The whole block for one step.  ``w`` holds e4m3 codes and fp32 scales:
    qkva, qkva_s, gate, gate_s, ik, ik_s, qb, qb_s, iq, iq_s."""
    pos = positions(sh)
    h, qa, sa = add_norm_quant(x, res, norm_w, sh.eps)
    qkva = fp8_gemm(qa, sa, w["qkva"], w["qkva_s"])
    gate = fp8_gemm(qa, sa, w["gate"], w["gate_s"])
    ik = fp8_gemm(qa, sa, w["ik"], w["ik_s"])
    qb_q, qb_s = quant_blocks(qkva[:, :sh.qlora])
    q = fp8_gemm(qb_q, qb_s, w["qb"], w["qb_s"]).reshape(sh.M, sh.q_heads, sh.q_head_dim)
    r = sh.q_head_dim - sh.rope
    q[:, :, r:] = bf16_round(rope_half(q[:, :, r:], pos[:, None], sh.theta))
    iq = fp8_gemm(qb_q, qb_s, w["iq"], w["iq_s"]).reshape(sh.M, sh.idx_heads, sh.idx_dim)
    r = sh.idx_dim - sh.rope
    iq[:, :, r:] = bf16_round(rope_half(iq[:, :, r:], pos[:, None], sh.theta))
    kv = qkva[:, sh.qlora:sh.qlora + sh.kvlora]
    kpe = bf16_round(rope_half(qkva[:, sh.qlora + sh.kvlora:], pos, sh.theta))
    latent = np.concatenate([kv, kpe], axis=1).reshape(sh.R, sh.T, sh.kvlora + sh.rope)
    r = sh.idx_dim - sh.rope
    index = np.concatenate([ik[:, :r], bf16_round(rope_half(ik[:, r:], pos, sh.theta))], axis=1)
    index = index.reshape(sh.R, sh.T, sh.idx_dim)
    return dict(res_out=h, qa=qa, sa=sa, qkva=qkva, gate=gate, ik=ik, qb=qb_q, qb_s=qb_s, q=q, iq=iq,
                latent=latent, index=index)
