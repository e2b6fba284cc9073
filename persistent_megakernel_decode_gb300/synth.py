"""Model shapes and seeded synthetic inputs.

This module holds no arithmetic of the decode method: it only names the
workloads (shapes, step counts, cache lengths) and draws their random
weights, caches, tokens and lengths from seeded generators.  It serves both
the CUDA path and the CPU checks, which receive the same tensors.

Recipe: weights bf16 N(0, 0.02) (norm weights 1), KV caches bf16 N(0, 1),
tokens uniform over the vocabulary, batch-8 cache lengths uniform in
[512, 4096]; seeds 1234 + workload index for weights, +100 for caches,
+200 for tokens and lengths.  There are no trained weights and no dataset.

GLM pre-attention block (workload index 3): activations and residual bf16
N(0, 1); weights fp32 N(0, 0.02), stored as e4m3 bytes with one fp32 scale
per 128 x 128 block (scale = block amax / 448, bytes from torch's own
float8_e4m3fn conversion of weight / scale) -- the block's weights arrive
quantised, so this is input preparation, not a step of the block; caches
bf16 N(0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import torch


@dataclass(frozen=True)
class ModelShape:
    L: int
    H: int
    Hq: int
    Hkv: int
    D: int
    F: int
    V: int
    eps: float
    theta: float
    qk_norm: bool = False
    tied: bool = True


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    shape: ModelShape
    batch: int
    seq_len: int              # cached tokens per sequence before the first step
    steps: int
    len_range: Optional[tuple] = None   # (lo, hi) inclusive: per-sequence lengths drawn from a seed
    fp8: bool = False                   # projections e4m3 with 128 x 128 block scales (make_weights(fp8=True))

    @property
    def weight_seed(self):
        return 1234 + self.index

    @property
    def cache_seed(self):
        return 1234 + self.index + 100

    @property
    def token_seed(self):
        return 1234 + self.index + 200


TINY = ModelShape(L=2, H=256, Hq=4, Hkv=2, D=64, F=688, V=1024, eps=1e-5, theta=1e4)
LLAMA_1B = ModelShape(L=16, H=2048, Hq=32, Hkv=8, D=64, F=8192, V=128256, eps=1e-5, theta=5e5)
QWEN3_8B = ModelShape(L=36, H=4096, Hq=32, Hkv=8, D=128, F=12288, V=151936, eps=1e-6, theta=1e6,
                      qk_norm=True, tied=False)
# Small shapes for the tensor-core tiles' checks (every K and row count a
# multiple of 128): the tiny decoder with an ffn of 512, and a two-layer
# Qwen3-style decoder (head_dim 128, q/k norm, untied head).
TINY_TC = ModelShape(L=2, H=256, Hq=4, Hkv=2, D=64, F=512, V=1024, eps=1e-5, theta=1e4)
SMALL_QK = ModelShape(L=2, H=512, Hq=4, Hkv=2, D=128, F=512, V=2048, eps=1e-6, theta=1e6, qk_norm=True, tied=False)

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 0, TINY, 1, 64, 8),
    "llama1b_b1": Workload("llama1b_b1", 1, LLAMA_1B, 1, 1024, 128),
    # the same model and step with FP8 projections (SURVEY's next row: FP8 weight streaming)
    "llama1b_b1_fp8": Workload("llama1b_b1_fp8", 1, LLAMA_1B, 1, 1024, 128, fp8=True),
    "llama1b_b8": Workload("llama1b_b8", 2, LLAMA_1B, 8, 4096, 64, len_range=(512, 4096)),
    "qwen3_8b_b1": Workload("qwen3_8b_b1", 4, QWEN3_8B, 1, 2048, 32),
    "qwen3_8b_b16": Workload("qwen3_8b_b16", 4, QWEN3_8B, 16, 2048, 32),
}


def seq_lengths(w: Workload) -> List[int]:
    """Cached tokens per sequence before the first step."""
    if w.len_range is None:
        return [w.seq_len] * w.batch
    g = torch.Generator().manual_seed(w.token_seed)
    lo, hi = w.len_range
    return torch.randint(lo, hi + 1, (w.batch,), generator=g).tolist()


def first_tokens(w: Workload) -> List[int]:
    g = torch.Generator().manual_seed(w.token_seed + 1)
    return torch.randint(0, w.shape.V, (w.batch,), generator=g).tolist()


def _randn(shape, g, device, std=1.0):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def quant_e4m3_blocks(w: torch.Tensor):
    """FP8 weights from fp32 ones, the recipe the pages give for FP8 weights:
    per 128 x 128 block scale = amax / 448 (1 for an all-zero block), codes
    = e4m3 of w / scale (torch's float8_e4m3fn cast).  Returns (uint8 codes
    [N, K], fp32 scales [ceil(N/128), K/128])."""
    n, k = w.shape
    nb = (n + 127) // 128
    wp = torch.zeros((nb * 128, k), device=w.device)
    wp[:n] = w
    amax = wp.view(nb, 128, k // 128, 128).abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
    q = (wp.view(nb, 128, k // 128, 128) / scale[:, None, :, None]).view(nb * 128, k)[:n]
    return q.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), scale.contiguous()


def make_weights(shape: ModelShape, seed: int, device="cpu", std: float = 0.02, fp8: bool = False) -> Dict[str, object]:
    """Weights in the usual [out_features, in_features] row-major layout.
    Per-layer tensors are lists indexed by layer.  With tied embeddings
    ``lm_head`` is the same tensor as ``embed``.  ``fp8``: the seven
    projections are (e4m3 codes, 128 x 128 block scales) pairs drawn from
    fp32 N(0, std) (``quant_e4m3_blocks``), and ``w["fp8"]`` is True; the
    embedding, LM head and norm weights stay bf16."""
    g = torch.Generator(device=device).manual_seed(seed)
    s = shape
    w: Dict[str, object] = {"embed": _randn((s.V, s.H), g, device, std)}
    per = {k: [] for k in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "norm_attn", "norm_mlp")}
    if s.qk_norm:
        per["qnorm"], per["knorm"] = [], []
    ones_h = torch.ones(s.H, dtype=torch.bfloat16, device=device)

    def proj(shp):
        if not fp8:
            return _randn(shp, g, device, std)
        return quant_e4m3_blocks(torch.randn(shp, generator=g, device=device, dtype=torch.float32) * std)

    for _ in range(s.L):
        per["wq"].append(proj((s.Hq * s.D, s.H)))
        per["wk"].append(proj((s.Hkv * s.D, s.H)))
        per["wv"].append(proj((s.Hkv * s.D, s.H)))
        per["wo"].append(proj((s.H, s.Hq * s.D)))
        per["wg"].append(proj((s.F, s.H)))
        per["wu"].append(proj((s.F, s.H)))
        per["wd"].append(proj((s.H, s.F)))
        per["norm_attn"].append(ones_h.clone())
        per["norm_mlp"].append(ones_h.clone())
        if s.qk_norm:
            per["qnorm"].append(torch.ones(s.D, dtype=torch.bfloat16, device=device))
            per["knorm"].append(torch.ones(s.D, dtype=torch.bfloat16, device=device))
    w.update(per)
    w["fp8"] = fp8
    w["norm_final"] = ones_h.clone()
    w["lm_head"] = w["embed"] if s.tied else _randn((s.V, s.H), g, device, std)
    return w


def make_cache(shape: ModelShape, batch: int, smax: int, seed: int, device="cpu"):
    """K and V caches, [L, B, Hkv, smax, D] bf16, every slot N(0, 1)."""
    g = torch.Generator(device=device).manual_seed(seed)
    dims = (shape.L, batch, shape.Hkv, smax, shape.D)
    return _randn(dims, g, device), _randn(dims, g, device)


@dataclass(frozen=True)
class GlmDims:
    """GLM-5.2-FP8 decode before sparse attention: 2 requests x 8 new tokens,
    hidden 6144, QKV-A 1536 + 512 + 64, Head-Gate 64, Indexer-K 128, Q-B
    64 x 192, Indexer-Q 32 x 128, caches of 8192 slots."""
    R: int = 2
    T: int = 8
    H: int = 6144
    qlora: int = 1536
    kvlora: int = 512
    rope: int = 64
    q_heads: int = 64
    q_head_dim: int = 192
    gate_heads: int = 64
    idx_heads: int = 32
    idx_dim: int = 128
    slots: int = 8192
    eps: float = 1e-6
    theta: float = 1e4

    @property
    def M(self):
        return self.R * self.T

    @property
    def pos0(self):
        return self.slots - self.T


GLM = GlmDims()
GLM_INDEX = 3
GLM_MATS = ("qkva", "gate", "ik", "qb", "iq")


def glm_mat_shapes(d: GlmDims) -> Dict[str, tuple]:
    return {"qkva": (d.qlora + d.kvlora + d.rope, d.H), "gate": (d.gate_heads, d.H), "ik": (d.idx_dim, d.H),
            "qb": (d.q_heads * d.q_head_dim, d.qlora), "iq": (d.idx_heads * d.idx_dim, d.qlora)}


def make_glm_inputs(d: GlmDims, device="cpu", index: int = GLM_INDEX) -> Dict[str, torch.Tensor]:
    """x, res, norm, w_<mat> (uint8 e4m3 [N, K]), s_<mat> (fp32 [ceil(N/128), K/128]), latent, index caches."""
    gw = torch.Generator(device="cpu").manual_seed(1234 + index)
    ga = torch.Generator(device="cpu").manual_seed(1234 + index + 200)
    gc = torch.Generator(device="cpu").manual_seed(1234 + index + 100)
    out: Dict[str, torch.Tensor] = {}
    out["x"] = torch.randn((d.M, d.H), generator=ga).to(torch.bfloat16)
    out["res"] = torch.randn((d.M, d.H), generator=ga).to(torch.bfloat16)
    out["norm"] = torch.ones(d.H, dtype=torch.bfloat16)
    for name, (n, k) in glm_mat_shapes(d).items():
        out["w_" + name], out["s_" + name] = quant_e4m3_blocks(torch.randn((n, k), generator=gw) * 0.02)
    out["latent"] = torch.randn((d.R, d.slots, d.kvlora + d.rope), generator=gc).to(torch.bfloat16)
    out["index"] = torch.randn((d.R, d.slots, d.idx_dim), generator=gc).to(torch.bfloat16)
    return {k: v.to(device) for k, v in out.items()}


def to_host_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the CPU checks)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def host_weights(w: Dict[str, object]) -> Dict[str, object]:
    """A ``make_weights`` dict on the host: bf16 tensors as uint16 bit
    patterns, FP8 (codes, scales) pairs as (uint8, float32) arrays."""
    def one(t):
        if isinstance(t, tuple):
            return (t[0].detach().contiguous().cpu().numpy(), t[1].detach().contiguous().cpu().numpy())
        return to_host_u16(t)
    return {k: ([one(t) for t in v] if isinstance(v, list) else v if isinstance(v, bool) else one(v))
            for k, v in w.items()}
