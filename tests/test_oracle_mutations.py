"""Planted mistakes in the C oracle (no GPU): each test compiles a copy of the
oracle with one plausible error -- a sign, an index, a scale, a missing term --
and checks that one of the oracle's pins fails on it.  This is what makes the
pins a check of the oracle rather than of themselves."""
import os
import shutil
import subprocess

import pytest

import test_oracle_forward as pins
from oracle import forward as orc

HERE = os.path.dirname(os.path.abspath(orc.__file__))

_NORM_Q = "                for (int j = 0; j < Hq; j++) { FN(rmsnorm)(q + j * D, D, w->qnorm[l], sh->eps, tmp); " \
          "memcpy(q + j * D, tmp, sizeof(REAL) * D); }\n"
_NORM_K = "                for (int g = 0; g < Hkv; g++) { FN(rmsnorm)(k + g * D, D, w->knorm[l], sh->eps, tmp); " \
          "memcpy(k + g * D, tmp, sizeof(REAL) * D); }\n"
_ROPE = ("            for (int j = 0; j < Hq; j++) FN(rope)(q + j * D, D, p, sh->theta);\n"
         "            for (int g = 0; g < Hkv; g++) FN(rope)(k + g * D, D, p, sh->theta);\n")
_QK_BLOCK = "            if (sh->qk_norm) {\n" + _NORM_Q + _NORM_K + "            }\n" + _ROPE
_QK_SWAPPED = _ROPE + "            if (sh->qk_norm) {\n" + _NORM_Q + _NORM_K + "            }\n"

MUTATIONS = {
    # RoPE rotating the wrong way
    "rope_sign": ("        v[i] = a * c - b * s;\n        v[i + half] = a * s + b * c;",
                  "        v[i] = a * c + b * s;\n        v[i + half] = -a * s + b * c;",
                  pins.test_rope_angles_and_invariants),
    # RoPE frequencies theta^(-i/D) instead of theta^(-2i/D)
    "rope_freq": ("pow(theta, -2.0 * i / D)", "pow(theta, -1.0 * i / D)", pins.test_rope_angles_and_invariants),
    # scores scaled by 1/D instead of 1/sqrt(D)
    "softmax_scale": ("REAL inv = (REAL)(1.0 / sqrt((double)D));", "REAL inv = (REAL)(1.0 / (double)D);",
                      pins.test_attention_special_cases),
    # eps added outside the square root
    "rms_eps": ("sqrt((double)ss / n + eps)", "(sqrt((double)ss / n) + eps)", pins.test_rmsnorm_closed_form),
    # query head j reading kv head j mod Hkv instead of j / (Hq / Hkv)
    "gqa_map": ("int g = j / G;", "int g = j % Hkv;", pins.test_step_attention_block_through_identity_output),
    # attention over the cached tokens only, without the appended one
    "attn_len": ("FN(attend)(q + j * D, kcache + base, vcache + base, p + 1, D, o + j * D, scr);",
                 "FN(attend)(q + j * D, kcache + base, vcache + base, p, D, o + j * D, scr);",
                 pins.test_step_attention_block_through_identity_output),
    # SwiGLU without the SiLU
    "silu": ("gt[i] = g / (1 + (REAL)exp(-(double)g)) * ut[i];", "gt[i] = g * ut[i];", pins.test_step_mlp_block),
    # the attention output replacing the residual instead of adding to it
    "residual": ("            FN(project)(w, 3, w->wo, l, H, Hq * D, o, t1, nthreads);\n"
                 "            for (int i = 0; i < H; i++) h[i] += t1[i];",
                 "            FN(project)(w, 3, w->wo, l, H, Hq * D, o, t1, nthreads);\n"
                 "            for (int i = 0; i < H; i++) h[i] = t1[i];",
                 pins.test_step_attention_block_through_identity_output),
    # q normalised with the k-norm weights
    "qnorm_weights": ("FN(rmsnorm)(q + j * D, D, w->qnorm[l], sh->eps, tmp)", "FN(rmsnorm)(q + j * D, D, w->knorm[l], sh->eps, tmp)",
                      pins.test_qk_norm_path),
    # RoPE before the per-head RMSNorm instead of after
    "qk_norm_order": (_QK_BLOCK, _QK_SWAPPED, pins.test_qk_norm_path),
    # SwiGLU with gate and up exchanged
    "gate_up_swap": ("                REAL g = gt[i];\n                gt[i] = g / (1 + (REAL)exp(-(double)g)) * ut[i];",
                     "                REAL g = ut[i];\n                gt[i] = g / (1 + (REAL)exp(-(double)g)) * gt[i];",
                     pins.test_step_mlp_block),
    # new k and v appended into each other's cache
    "kv_swap": ("                    kcache[base + d] = double_to_bf16((double)k[g * D + d]);\n"
                "                    vcache[base + d] = double_to_bf16((double)v[g * D + d]);",
                "                    kcache[base + d] = double_to_bf16((double)v[g * D + d]);\n"
                "                    vcache[base + d] = double_to_bf16((double)k[g * D + d]);",
                pins.test_step_attention_block_through_identity_output),
    # the embedding used as the LM head of an untied model
    "untied_head": ("        FN(matvec)(w->lm_head, V, H, x, logits + (size_t)b * V, nthreads);",
                    "        FN(matvec)(w->embed, V, H, x, logits + (size_t)b * V, nthreads);",
                    pins.test_qk_norm_path),
    # the final norm's weights ignored
    "final_norm_weights": ("        FN(rmsnorm)(h, H, w->norm_final, sh->eps, x);", "        FN(rmsnorm)(h, H, w->norm_mlp[0], sh->eps, x);",
                           pins.test_qk_norm_path),
    # the final RMSNorm skipped before the LM head
    "final_norm": ("        FN(rmsnorm)(h, H, w->norm_final, sh->eps, x);\n        FN(matvec)(w->lm_head, V, H, x,",
                   "        memcpy(x, h, sizeof(REAL) * H);\n        FN(matvec)(w->lm_head, V, H, x,",
                   pins.test_step_with_zeroed_output_projections),
    # FP8 block scales indexed [column block][row block]
    "fp8_scale_transposed": ("(REAL)(e4m3_to_double(row[k]) * (double)srow[k / 128]) * x[k];",
                             "(REAL)(e4m3_to_double(row[k]) * (double)S[(size_t)(k / 128) * KB + n / 128]) * x[k];",
                             lambda: pins.test_matvec8_block_scale_placement(1, 0, 2.0)),
    # FP8 projections: the up matrix used for the gate
    "fp8_gate_matrix": ("FN(project)(w, 4, w->wg, l, F, H, x, gt, nthreads);",
                        "FN(project)(w, 5, w->wg, l, F, H, x, gt, nthreads);",
                        pins.test_step_fp8_equals_the_bf16_step_on_the_same_values),
}


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(HERE, "forward_impl.h")).read()
    assert src.count(old) == 1, old
    d = tmp_path / "src"
    d.mkdir()
    shutil.copy(os.path.join(HERE, "forward.c"), d / "forward.c")
    (d / "forward_impl.h").write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(d / "forward.c"), "-lm"])
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pin_catches_planted_mistake(name, tmp_path, monkeypatch):
    old, new, pin = MUTATIONS[name]
    pin()  # the pin holds on the real oracle
    so = _build_mutant(tmp_path, old, new)
    monkeypatch.setattr(orc, "_lib", None)
    monkeypatch.setattr(orc, "build", lambda force=False: so)
    with pytest.raises(AssertionError):
        pin()


# ---------------------------------------------------------------- planner rules
import importlib.util  # noqa: E402
import sys  # noqa: E402

import test_oracle_rules as rule_pins  # noqa: E402
from oracle import rules  # noqa: E402

RULE_MUTATIONS = {
    # the per-edge event partition by min instead of gcd
    "gcd_as_min": ("[math.gcd(a, b) for a, b in zip(pp, cp)]", "[min(a, b) for a, b in zip(pp, cp)]",
                   rule_pins.test_gcd_examples),
    # the fork/join normalisation by max instead of lcm (the F/A/B/G example
    # cannot tell them apart: its groups are 1 and 2; coprime groups can)
    "lcm_as_max": ("    return a * b // math.gcd(a, b)", "    return max(a, b)",
                   rule_pins.test_fork_with_coprime_consumer_groups_merges_to_one_event),
    # grid axes multiplying into the wrong tensor dimension
    "partition_axis": ("            part[d] *= grid[axis]", "            part[axis] *= grid[axis]",
                       rule_pins.test_build_partition_example),
    # counters reset every step instead of growing by epochs
    "counter_epochs": ("    return [steps * t for t in thresholds]", "    return list(thresholds)",
                       rule_pins.test_expected_counters),
}


def _load_rules_mutant(old, new):
    src = open(rules.__file__).read()
    assert src.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle_rules_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules["oracle_rules_mutant"] = mod  # dataclasses resolve their module by name
    try:
        exec(compile(src.replace(old, new), rules.__file__, "exec"), mod.__dict__)
    finally:
        del sys.modules["oracle_rules_mutant"]
    return mod


@pytest.mark.parametrize("name", sorted(RULE_MUTATIONS))
def test_rule_pin_catches_planted_mistake(name, monkeypatch):
    old, new, pin = RULE_MUTATIONS[name]
    pin()
    monkeypatch.setattr(rule_pins, "rules", _load_rules_mutant(old, new))
    with pytest.raises(AssertionError):
        pin()


# ---------------------------------------------------------------- GLM block
import test_oracle_glm as glm_pins  # noqa: E402
from oracle import glm  # noqa: E402

GLM_MUTATIONS = {
    # e4m3 rounding half up instead of to even
    "e4m3_ties": ("    v = np.round(a / q) * q                  # np.round: ties to even",
                  "    v = np.floor(a / q + 0.5) * q", glm_pins.test_e4m3_ties_to_even_and_saturation),
    # activation scale against the wrong format maximum
    "quant_max": ("scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)",
                  "scale = np.where(amax > 0, amax / 240.0, 1.0).astype(np.float32)",
                  glm_pins.test_quant_blocks_scale_and_zero_block),
    # the activation's block scale left out of the GEMM
    "gemm_scale": ("        out += part * sa[:, kb][:, None] * np.repeat(sw[:, kb], BLOCK)[:N][None, :]",
                   "        out += part * np.repeat(sw[:, kb], BLOCK)[:N][None, :]",
                   glm_pins.test_fp8_gemm_matches_brute_force),
    # RoPE rotating the wrong way
    "rope_sign": ("    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)",
                  "    return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)",
                  glm_pins.test_rope_half_rotation_direction_and_frequency),
    # bf16 by truncation
    "bf16_trunc": ("    return np.ldexp(np.round(m * 256.0) / 256.0, e)", "    return np.ldexp(np.trunc(m * 256.0) / 256.0, e)",
                   glm_pins.test_bf16_round_matches_torch),
    # eps outside the square root
    "rms_eps": ("    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * np.asarray(w, dtype=np.float64)",
                "    return h / (np.sqrt(np.mean(h * h, axis=-1, keepdims=True)) + eps) * np.asarray(w, dtype=np.float64)",
                glm_pins.test_rmsnorm_unit_weight_invariant),
    # the re-quantised q-lora taken from the wrong columns of QKV-A
    "qlora_cols": ("    qb_q, qb_s = quant_blocks(qkva[:, :sh.qlora])",
                   "    qb_q, qb_s = quant_blocks(qkva[:, sh.kvlora:sh.kvlora + sh.qlora])",
                   lambda: glm_pins.test_forward_small_block_consistency(0)),
    # latent cache rows as k_pe || kv-lora instead of kv-lora || k_pe
    "latent_order": ("    latent = np.concatenate([kv, kpe], axis=1).reshape(sh.R, sh.T, sh.kvlora + sh.rope)",
                     "    latent = np.concatenate([kpe, kv], axis=1).reshape(sh.R, sh.T, sh.kvlora + sh.rope)",
                     lambda: glm_pins.test_forward_small_block_consistency(0)),
    # every token of both requests at its own position (request index ignored)
    "positions": ("    return sh.pos0 + (np.arange(sh.M) % sh.T)", "    return sh.pos0 + np.arange(sh.M)",
                  glm_pins.test_block_shapes_and_positions),
}


def _load_glm_mutant(old, new):
    src = open(glm.__file__).read()
    assert src.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle_glm_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules["oracle_glm_mutant"] = mod
    try:
        exec(compile(src.replace(old, new), glm.__file__, "exec"), mod.__dict__)
    finally:
        del sys.modules["oracle_glm_mutant"]
    return mod


@pytest.mark.parametrize("name", sorted(GLM_MUTATIONS))
def test_glm_pin_catches_planted_mistake(name, monkeypatch):
    old, new, pin = GLM_MUTATIONS[name]
    pin()
    monkeypatch.setattr(glm_pins, "glm", _load_glm_mutant(old, new))
    with pytest.raises(AssertionError):
        pin()


# ---------------------------------------------------------------- queue simulator
import test_oracle_sim as sim_pins  # noqa: E402
from oracle import sim  # noqa: E402

SIM_MUTATIONS = {
    # counters compared with the bare threshold (as if reset every step)
    "no_epochs": ("                if counters[ev] < thr * (s + 1 + off):", "                if counters[ev] < thr:",
                  sim_pins.test_waits_target_the_current_epoch),
    # the epoch offset applied the wrong way
    "offset_sign": ("                if counters[ev] < thr * (s + 1 + off):",
                    "                if counters[ev] < thr * (s + 1 - off):", sim_pins.test_wait_one_epoch_back),
    # a stuck worker not reported
    "no_blocked": ("        if blocked:\n            return SimResult(False, counters, blocked, order)",
                   "        if False:\n            return SimResult(False, counters, blocked, order)",
                   sim_pins.test_deadlock_detected),
}


def _load_sim_mutant(old, new):
    src = open(sim.__file__).read()
    assert src.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle.sim_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"  # its relative imports resolve against the real package
    sys.modules["oracle.sim_mutant"] = mod
    try:
        exec(compile(src.replace(old, new), sim.__file__, "exec"), mod.__dict__)
    finally:
        del sys.modules["oracle.sim_mutant"]
    return mod


@pytest.mark.parametrize("name", sorted(SIM_MUTATIONS))
def test_sim_pin_catches_planted_mistake(name, monkeypatch):
    old, new, pin = SIM_MUTATIONS[name]
    pin()
    monkeypatch.setattr(sim_pins, "sim", _load_sim_mutant(old, new))
    with pytest.raises(AssertionError):
        pin()


# ---------------------------------------------------------------- plan builder
import test_oracle_rules as plan_pins  # noqa: E402  (its plan pins call plans.*)
from oracle import plans  # noqa: E402

PLAN_MUTATIONS = {
    # attention splits rounded down: the last partial split dropped
    "nsplit_floor": ("    nsplit = [_ceil(seq0[b] + max_steps, k.attn_split) for b in range(B)]",
                     "    nsplit = [(seq0[b] + max_steps) // k.attn_split for b in range(B)]",
                     plan_pins.test_attention_splits_cover_every_position),
    # MLP-down without its K chunks (one chunk of the whole F)
    "down_chunks": ("        ops.append(Op(down, (_ceil(shape.H, k.rows_down), shape.F // k.kchunk_down, 1),",
                    "        ops.append(Op(down, (_ceil(shape.H, k.rows_down), 1, 1),",
                    plan_pins.test_llama1b_layer_counts),
}


def _load_plans_mutant(old, new):
    src = open(plans.__file__).read()
    assert src.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle.plans_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    sys.modules["oracle.plans_mutant"] = mod
    try:
        exec(compile(src.replace(old, new), plans.__file__, "exec"), mod.__dict__)
    finally:
        del sys.modules["oracle.plans_mutant"]
    return mod


@pytest.mark.parametrize("name", sorted(PLAN_MUTATIONS))
def test_plan_pin_catches_planted_mistake(name, monkeypatch):
    old, new, pin = PLAN_MUTATIONS[name]
    pin()
    monkeypatch.setattr(plan_pins, "plans", _load_plans_mutant(old, new))
    with pytest.raises(AssertionError):
        pin()
