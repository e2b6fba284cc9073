"""ctypes binding of libmk (argument marshalling only).

Every step of the decode path runs in the library's CUDA kernel; this module
converts Python / torch arguments to the C ABI of ``include/mk.h`` and keeps
the device buffers alive.  There is no CPU fallback: ``load()`` raises when
``libmk.so`` is missing or cannot be loaded.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmk.so")

# ---- constants mirrored from include/mk.h ----
MK_OK, MK_ERR_INVALID, MK_ERR_UNSUPPORTED, MK_ERR_DEADLOCK, MK_ERR_CUDA = 0, 1, 2, 3, 4
MK_ERR_RESIDENCY, MK_ERR_TIMEOUT, MK_ERR_DEVICE_CHECK, MK_ERR_UNBOUND = 5, 6, 7, 8
OP_NAMES = {0: "noop", 1: "counter", 2: "embed", 3: "qkv", 4: "attn", 5: "o", 6: "up", 7: "down", 8: "lm",
            9: "glm_a0", 10: "glm_gemm", 11: "glm_fin", 12: "norm", 13: "attn_pool"}
OPCODE = {v: k for k, v in OP_NAMES.items()}
MODE_MEGAKERNEL, MODE_PER_OP = 0, 1
SCHED_DEFAULT, SCHED_BYTES, SCHED_TIMED = 0, 1, 2
RUN_HOST_TOKENS, RUN_TRACE, RUN_ONE_LAUNCH = 1, 2, 4
PAIR_WHOLE, PAIR_TILE, PAIR_TILE_COVER, PAIR_TILE_REDUCE = 0, 1, 2, 3
TASK_FIELDS = 24
BIND = {n: i for i, n in enumerate([
    "embed", "lm_head", "norm_final", "wq", "wk", "wv", "wo", "wg", "wu", "wd", "norm_attn", "norm_mlp",
    "qnorm", "knorm", "kcache", "vcache", "tokens", "logits", "argmax", "hidden",
    # GLM pre-attention block
    "glm_x", "glm_res", "glm_norm", "glm_res_out", "glm_qa", "glm_sa", "glm_w_qkva", "glm_s_qkva", "glm_w_gate",
    "glm_s_gate", "glm_w_ik", "glm_s_ik", "glm_w_qb", "glm_s_qb", "glm_w_iq", "glm_s_iq", "glm_qkva", "glm_ik",
    "glm_qb", "glm_sb", "glm_gate", "glm_q", "glm_iq", "glm_latent", "glm_index",
    # FP8 projections: block scales of wq .. wd
    "sq", "sk", "sv", "so", "sg", "su", "sd"])}
SCALE_OF = {"wq": "sq", "wk": "sk", "wv": "sv", "wo": "so", "wg": "sg", "wu": "su", "wd": "sd"}
PER_LAYER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "norm_attn", "norm_mlp", "qnorm", "knorm")

EXPORTED = ["mk_plan", "mk_plan_graph", "mk_plan_info_get", "mk_plan_export", "mk_bind", "mk_run",
            "mk_sync_status", "mk_read_counters", "mk_read_trace", "mk_free", "mk_last_error", "mk_argmax_index",
            "mk_run_static", "mk_plan_glm", "mk_launch_probe", "mk_plan_export_attn_table"]
STATIC_WORKSPACE_BYTES = 64 << 20


class MkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmk error {code}: {msg}")
        self.code = code


class ModelDesc(C.Structure):
    _fields_ = [("layers", C.c_int), ("hidden", C.c_int), ("q_heads", C.c_int), ("kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("vocab", C.c_int), ("qk_norm", C.c_int),
                ("eps", C.c_float), ("rope_theta", C.c_float), ("weight_fp8", C.c_int)]


class StepDesc(C.Structure):
    _fields_ = [("batch", C.c_int), ("seq_len0", C.POINTER(C.c_int)), ("max_steps", C.c_int),
                ("cache_slots", C.c_int), ("capture_hidden", C.c_int)]


class TargetDesc(C.Structure):
    _fields_ = [("num_sms", C.c_int), ("smem_per_cta", C.c_int), ("mode", C.c_int), ("rows_qkv", C.c_int),
                ("rows_o", C.c_int), ("rows_up", C.c_int), ("rows_down", C.c_int), ("kchunk_down", C.c_int),
                ("rows_lm", C.c_int), ("attn_split", C.c_int), ("page_bytes", C.c_int),
                ("schedule", C.c_int), ("tc_tiles", C.c_int), ("attn_pool", C.c_int)]


class GlmDesc(C.Structure):
    _fields_ = [(n, C.c_int) for n in (
        "requests", "tokens", "hidden", "q_lora", "kv_lora", "rope", "q_heads", "q_head_dim", "gate_heads",
        "idx_heads", "idx_dim", "cache_slots", "pos0", "max_steps")] + [("eps", C.c_float), ("rope_theta", C.c_float)]


class PlanInfo(C.Structure):
    _fields_ = [(n, C.c_int) for n in (
        "num_workers", "lmax", "num_tasks", "num_events", "num_ops", "num_launches", "num_pages", "page_bytes",
        "smem_bytes", "act_bytes", "rows_qkv", "rows_o", "rows_up", "rows_down", "kchunk_down", "rows_lm",
        "attn_split", "total_slots")] + [("workspace_bytes", C.c_uint64), ("scratch_offset", C.c_uint64),
                                          ("algorithmic_bytes_step", C.c_uint64)] + [
        (n, C.c_int) for n in ("tc_tiles", "ksplit_qkv", "ksplit_o", "weight_fp8", "attn_table_rows")]


class GraphOp(C.Structure):
    _fields_ = [("grid", C.c_int * 3), ("cost", C.c_int)]


class GraphEdge(C.Structure):
    _fields_ = [("prod", C.c_int), ("cons", C.c_int), ("out_map", C.c_int * 3), ("in_map", C.c_int * 3)]


class GraphPub(C.Structure):
    _fields_ = [("prod", C.c_int), ("first_pub", C.c_int), ("num_pub", C.c_int), ("strategy", C.c_int),
                ("k", C.c_int), ("num_cons", C.c_int), ("cons", C.c_int * 4)]


class GraphDesc(C.Structure):
    _fields_ = [("num_ops", C.c_int), ("ops", C.POINTER(GraphOp)), ("num_edges", C.c_int),
                ("edges", C.POINTER(GraphEdge)), ("num_pubs", C.c_int), ("pubs", C.POINTER(GraphPub)),
                ("round_robin", C.c_int)]


class ErrorRecord(C.Structure):
    _fields_ = [("code", C.c_int32), ("worker", C.c_int32), ("slot", C.c_int32), ("event", C.c_int32),
                ("observed", C.c_uint32), ("needed", C.c_uint32), ("opcode", C.c_int32), ("role", C.c_int32)]


_lib = None


def load():
    """Load libmk.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmk.so not found at {LIB_PATH}; build it with "
                           "`python -m persistent_megakernel_decode_gb300.build`")
    lib = C.CDLL(LIB_PATH)
    P = C.c_void_p
    lib.mk_plan.argtypes = [C.POINTER(ModelDesc), C.POINTER(StepDesc), C.POINTER(TargetDesc), C.POINTER(P)]
    lib.mk_plan_graph.argtypes = [C.POINTER(GraphDesc), C.POINTER(TargetDesc), C.POINTER(P)]
    lib.mk_plan_glm.argtypes = [C.POINTER(GlmDesc), C.POINTER(TargetDesc), C.POINTER(P)]
    lib.mk_plan_info_get.argtypes = [P, C.POINTER(PlanInfo)]
    lib.mk_plan_export.argtypes = [P, P, P, P, P]
    lib.mk_plan_export_attn_table.argtypes = [P, P]
    lib.mk_bind.argtypes = [P, C.c_int, C.c_int, C.c_uint64]
    lib.mk_run.argtypes = [P, P, C.c_size_t, C.c_int, C.c_int, C.c_uint32, C.c_uint64, P]
    lib.mk_run_static.argtypes = [P, C.c_int, C.c_int, C.c_uint32, C.c_uint64, P, C.POINTER(C.c_uint64)]
    lib.mk_sync_status.argtypes = [P, P, P, C.POINTER(ErrorRecord)]
    lib.mk_read_counters.argtypes = [P, P, P]
    lib.mk_read_trace.argtypes = [P, P, P]
    lib.mk_launch_probe.argtypes = [C.c_int, C.c_int, P]
    lib.mk_free.argtypes = [P]
    lib.mk_free.restype = None
    lib.mk_last_error.restype = C.c_char_p
    lib.mk_argmax_index.argtypes = [C.c_uint64]
    lib.mk_argmax_index.restype = C.c_int32
    _lib = lib
    return lib


def _check(rc: int):
    if rc != MK_OK:
        raise MkError(rc, load().mk_last_error().decode())


def argmax_index(keys: np.ndarray) -> np.ndarray:
    """Token index of each packed argmax key, decoded by the library's
    ``mk_argmax_index``."""
    k = np.asarray(keys, dtype=np.uint64)
    f = load().mk_argmax_index
    return np.array([f(int(v)) for v in k.reshape(-1)], dtype=np.int64).reshape(k.shape)


def _target(num_sms=0, smem_per_cta=0, mode=MODE_MEGAKERNEL, **knobs) -> TargetDesc:
    t = TargetDesc()
    t.num_sms, t.smem_per_cta, t.mode = num_sms, smem_per_cta, mode
    for k, v in knobs.items():
        setattr(t, k, int(v))
    return t


def launch_probe(num_workers: int, cooperative: bool, stream) -> None:
    """Launch the empty probe kernel (see ``mk_launch_probe``) on a torch stream."""
    _check(load().mk_launch_probe(int(num_workers), int(cooperative), C.c_void_p(stream.cuda_stream)))


class Plan:
    """A host plan (owns host memory only)."""

    def __init__(self, handle):
        self.h = C.c_void_p(handle)
        self._info = None

    @classmethod
    def llama(cls, shape, batch: int, seq_len0: Sequence[int], max_steps: int, cache_slots: int,
              capture_hidden: bool = False, fp8: bool = False, **target):
        """``fp8``: the seven projections are e4m3 with 128 x 128 block scales."""
        lib = load()
        m = ModelDesc(shape.L, shape.H, shape.Hq, shape.Hkv, shape.D, shape.F, shape.V, int(shape.qk_norm),
                      shape.eps, shape.theta, int(fp8))
        lens = (C.c_int * batch)(*[int(x) for x in seq_len0])
        s = StepDesc(batch, lens, max_steps, cache_slots, int(capture_hidden))
        t = _target(**target)
        out = C.c_void_p()
        _check(lib.mk_plan(C.byref(m), C.byref(s), C.byref(t), C.byref(out)))
        return cls(out.value)

    @classmethod
    def graph(cls, ops: List[dict], edges: List[dict] = (), pubs: List[dict] = (), round_robin=False, **target):
        lib = load()
        o = (GraphOp * len(ops))(*[GraphOp((C.c_int * 3)(*op["grid"]), op.get("cost", 1)) for op in ops])
        e = (GraphEdge * max(1, len(edges)))(*[GraphEdge(x["prod"], x["cons"], (C.c_int * 3)(*x["out_map"]),
                                                         (C.c_int * 3)(*x["in_map"])) for x in edges])
        pb = (GraphPub * max(1, len(pubs)))(*[GraphPub(x["prod"], x.get("first_pub", 0), x["num_pub"], x["strategy"],
                                                       x.get("k", 1), len(x["cons"]),
                                                       (C.c_int * 4)(*(list(x["cons"]) + [0] * 4)[:4]))
                                              for x in pubs])
        g = GraphDesc(len(ops), o, len(edges), e, len(pubs), pb, int(round_robin))
        t = _target(**target)
        out = C.c_void_p()
        _check(lib.mk_plan_graph(C.byref(g), C.byref(t), C.byref(out)))
        return cls(out.value)

    @classmethod
    def glm(cls, dims, max_steps: int = 1, **target):
        """Plan the GLM pre-attention block; ``dims`` has the fields of ``mk_glm_desc``."""
        lib = load()
        d = GlmDesc(dims.R, dims.T, dims.H, dims.qlora, dims.kvlora, dims.rope, dims.q_heads, dims.q_head_dim,
                    dims.gate_heads, dims.idx_heads, dims.idx_dim, dims.slots, dims.pos0, max_steps, dims.eps,
                    dims.theta)
        t = _target(**target)
        out = C.c_void_p()
        _check(lib.mk_plan_glm(C.byref(d), C.byref(t), C.byref(out)))
        return cls(out.value)

    def attn_table(self) -> np.ndarray:
        """attn_pool plans: the attention task table, int32 [rows, 32]."""
        n = self.info()["attn_table_rows"]
        out = np.zeros((max(n, 1), 32), np.int32)
        _check(load().mk_plan_export_attn_table(self.h, C.c_void_p(out.ctypes.data)))
        return out[:n]

    def info(self) -> dict:
        if self._info is None:
            i = PlanInfo()
            _check(load().mk_plan_info_get(self.h, C.byref(i)))
            self._info = {f: getattr(i, f) for f, _ in PlanInfo._fields_}
        return self._info

    def export(self):
        i = self.info()
        W, Lm, E, T = i["num_workers"], i["lmax"], i["num_events"], i["num_tasks"]
        total_words = i["total_slots"] * 32
        q = np.zeros(total_words, np.int32)
        ids = np.zeros(total_words // 32, np.int32)
        th = np.zeros(max(E, 1), np.int32)
        tasks = np.zeros((max(T, 1), TASK_FIELDS), np.int32)
        _check(load().mk_plan_export(self.h, q.ctypes.data, ids.ctypes.data, th.ctypes.data, tasks.ctypes.data))
        if i["num_launches"] == 1:
            q = q.reshape(W, Lm, 32)
            ids = ids.reshape(W, Lm)
        return q, ids, th[:E], tasks[:T]

    def bind(self, name: str, ptr: int, layer: int = 0):
        _check(load().mk_bind(self.h, BIND[name], layer, int(ptr)))

    def free(self):
        if self.h and self.h.value:
            load().mk_free(self.h)
            self.h = C.c_void_p()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Session:
    """Device-resident decode state: weights, KV caches, outputs and the workspace.

    ``weights`` follows ``synth.make_weights`` naming (torch bf16 CUDA tensors;
    with ``weights["fp8"]`` the projections are (e4m3 codes, block scales) pairs);
    ``kcache`` / ``vcache`` are [L, B, Hkv, S_max, D] bf16 CUDA tensors, appended in place.
    """

    def __init__(self, shape, weights: Dict[str, object], kcache, vcache, seq_len0: Sequence[int], max_steps: int,
                 capture_hidden: bool = False, stream=None, **target):
        import torch
        self.torch = torch
        self.shape = shape
        self.B = len(seq_len0)
        self.max_steps = max_steps
        self.seq_len0 = list(seq_len0)
        dev = kcache.device
        fp8 = bool(weights.get("fp8", False))
        self.plan = Plan.llama(shape, self.B, seq_len0, max_steps, kcache.shape[3], capture_hidden, fp8=fp8, **target)
        info = self.plan.info()
        self.weights, self.kcache, self.vcache = weights, kcache, vcache
        self.tokens = torch.zeros((max_steps + 1, self.B), dtype=torch.int32, device=dev)
        self.logits = torch.zeros((self.B, shape.V), dtype=torch.float32, device=dev)
        self.argmax = torch.zeros((max_steps, self.B), dtype=torch.int64, device=dev)
        self.hidden = torch.zeros((shape.L, self.B, shape.H), dtype=torch.float32, device=dev) if capture_hidden else None
        self.workspace = torch.zeros(info["workspace_bytes"] + 256, dtype=torch.uint8, device=dev)
        off = (-self.workspace.data_ptr()) % 256
        self.ws_ptr = self.workspace.data_ptr() + off
        self.ws_bytes = info["workspace_bytes"]
        p = self.plan
        for n in ("embed", "lm_head", "norm_final"):
            p.bind(n, weights[n].data_ptr())
        for n in PER_LAYER:
            if n in weights:
                for l, t in enumerate(weights[n]):
                    if isinstance(t, tuple):  # FP8: codes, then their block scales
                        p.bind(n, t[0].data_ptr(), l)
                        p.bind(SCALE_OF[n], t[1].data_ptr(), l)
                    else:
                        p.bind(n, t.data_ptr(), l)
        p.bind("kcache", kcache.data_ptr())
        p.bind("vcache", vcache.data_ptr())
        p.bind("tokens", self.tokens.data_ptr())
        p.bind("logits", self.logits.data_ptr())
        p.bind("argmax", self.argmax.data_ptr())
        if self.hidden is not None:
            p.bind("hidden", self.hidden.data_ptr())
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)

    def run(self, first_step: int, num_steps: int = 1, host_tokens: bool = False, trace: bool = False,
            timeout_ns: int = 0, one_launch: bool = False):
        flags = (RUN_HOST_TOKENS if host_tokens else 0) | (RUN_TRACE if trace else 0) | \
            (RUN_ONE_LAUNCH if one_launch else 0)
        _check(load().mk_run(self.plan.h, C.c_void_p(self.ws_ptr), self.ws_bytes, first_step, num_steps, flags,
                             timeout_ns, C.c_void_p(self.stream.cuda_stream)))

    def sync(self) -> ErrorRecord:
        rec = ErrorRecord()
        rc = load().mk_sync_status(self.plan.h, C.c_void_p(self.ws_ptr), C.c_void_p(self.stream.cuda_stream),
                                   C.byref(rec))
        if rc != MK_OK:
            raise MkError(rc, load().mk_last_error().decode())
        return rec

    def run_static(self, first_step: int, num_steps: int = 1, host_tokens: bool = False, timeout_ns: int = 0) -> int:
        """Run through mk_run_static (library-owned workspace, no device allocation).
        Returns the device address of that workspace, for sync_static()."""
        addr = C.c_uint64(0)
        flags = RUN_HOST_TOKENS if host_tokens else 0
        _check(load().mk_run_static(self.plan.h, first_step, num_steps, flags, timeout_ns,
                                    C.c_void_p(self.stream.cuda_stream), C.byref(addr)))
        return addr.value

    def sync_static(self, addr: int) -> ErrorRecord:
        rec = ErrorRecord()
        rc = load().mk_sync_status(self.plan.h, C.c_void_p(addr), C.c_void_p(self.stream.cuda_stream), C.byref(rec))
        if rc != MK_OK:
            raise MkError(rc, load().mk_last_error().decode())
        return rec

    def step_tokens(self, step: int) -> np.ndarray:
        """Argmax token of every sequence at ``step`` (after sync)."""
        keys = self.argmax[step].cpu().numpy().view(np.uint64)
        return argmax_index(keys)

    def counters(self) -> np.ndarray:
        out = np.zeros(self.plan.info()["num_events"], np.uint32)
        _check(load().mk_read_counters(self.plan.h, C.c_void_p(self.ws_ptr), out.ctypes.data))
        return out

    def trace(self) -> np.ndarray:
        i = self.plan.info()
        out = np.zeros((i["num_workers"], i["lmax"], 16), np.uint64)
        _check(load().mk_read_trace(self.plan.h, C.c_void_p(self.ws_ptr), out.ctypes.data))
        return out


class GlmSession:
    """Device state of the GLM pre-attention block: inputs and FP8 weights from
    ``synth.make_glm_inputs`` (torch CUDA tensors), every output and
    intermediate, and the workspace."""

    OUTPUTS = ("res_out", "qa", "sa", "qkva", "ik", "qb", "sb", "gate", "q", "iq")

    def __init__(self, dims, inputs: Dict[str, object], max_steps: int = 1, stream=None, **target):
        import torch
        self.dims = dims
        dev = inputs["x"].device
        self.plan = Plan.glm(dims, max_steps, **target)
        info = self.plan.info()
        M, H, QL = dims.M, dims.H, dims.qlora
        NQKVA = dims.qlora + dims.kvlora + dims.rope
        bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=dev)
        self.out = dict(res_out=z((M, H), bf), qa=z((M, H), u8), sa=z((M, H // 128), f32), qkva=z((M, NQKVA), bf),
                        ik=z((M, dims.idx_dim), bf), qb=z((M, QL), u8), sb=z((M, QL // 128), f32),
                        gate=z((M, dims.gate_heads), bf), q=z((M, dims.q_heads, dims.q_head_dim), bf),
                        iq=z((M, dims.idx_heads, dims.idx_dim), bf))
        self.inputs = inputs
        self.latent = inputs["latent"]
        self.index = inputs["index"]
        self.workspace = torch.zeros(info["workspace_bytes"] + 256, dtype=torch.uint8, device=dev)
        self.ws_ptr = self.workspace.data_ptr() + (-self.workspace.data_ptr()) % 256
        self.ws_bytes = info["workspace_bytes"]
        p = self.plan
        for n in ("x", "res", "norm", "w_qkva", "s_qkva", "w_gate", "s_gate", "w_ik", "s_ik", "w_qb", "s_qb",
                  "w_iq", "s_iq", "latent", "index"):
            p.bind("glm_" + n, inputs[n].data_ptr())
        for n, t in self.out.items():
            p.bind("glm_" + n, t.data_ptr())
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)

    def run(self, first_step: int = 0, num_steps: int = 1, trace: bool = False, timeout_ns: int = 0,
            one_launch: bool = False):
        flags = (RUN_TRACE if trace else 0) | (RUN_ONE_LAUNCH if one_launch else 0)
        _check(load().mk_run(self.plan.h, C.c_void_p(self.ws_ptr), self.ws_bytes, first_step, num_steps, flags,
                             timeout_ns, C.c_void_p(self.stream.cuda_stream)))

    def sync(self) -> ErrorRecord:
        rec = ErrorRecord()
        rc = load().mk_sync_status(self.plan.h, C.c_void_p(self.ws_ptr), C.c_void_p(self.stream.cuda_stream),
                                   C.byref(rec))
        if rc != MK_OK:
            raise MkError(rc, load().mk_last_error().decode())
        return rec

    def counters(self) -> np.ndarray:
        out = np.zeros(self.plan.info()["num_events"], np.uint32)
        _check(load().mk_read_counters(self.plan.h, C.c_void_p(self.ws_ptr), out.ctypes.data))
        return out

    def trace(self) -> np.ndarray:
        i = self.plan.info()
        out = np.zeros((i["num_workers"], i["lmax"], 16), np.uint64)
        _check(load().mk_read_trace(self.plan.h, C.c_void_p(self.ws_ptr), out.ctypes.data))
        return out


class GraphSession:
    """Workspace for an explicit-graph plan (counter tasks only)."""

    def __init__(self, plan: Plan, device="cuda:0", stream=None):
        import torch
        self.plan = plan
        info = plan.info()
        self.workspace = torch.zeros(info["workspace_bytes"] + 256, dtype=torch.uint8, device=device)
        self.ws_ptr = self.workspace.data_ptr() + (-self.workspace.data_ptr()) % 256
        self.ws_bytes = info["workspace_bytes"]
        self.stream = stream if stream is not None else torch.cuda.current_stream(torch.device(device))

    def run(self, first_step: int, num_steps: int = 1, timeout_ns: int = 0):
        _check(load().mk_run(self.plan.h, C.c_void_p(self.ws_ptr), self.ws_bytes, first_step, num_steps, 0,
                             timeout_ns, C.c_void_p(self.stream.cuda_stream)))

    def sync(self) -> ErrorRecord:
        rec = ErrorRecord()
        rc = load().mk_sync_status(self.plan.h, C.c_void_p(self.ws_ptr), C.c_void_p(self.stream.cuda_stream),
                                   C.byref(rec))
        if rc not in (MK_OK, MK_ERR_TIMEOUT, MK_ERR_DEVICE_CHECK):
            raise MkError(rc, load().mk_last_error().decode())
        return rec

    def counters(self) -> np.ndarray:
        out = np.zeros(self.plan.info()["num_events"], np.uint32)
        _check(load().mk_read_counters(self.plan.h, C.c_void_p(self.ws_ptr), out.ctypes.data))
        return out
