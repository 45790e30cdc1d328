"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a scratch copy of the oracle's C source (a
dropped term, a wrong sign, index or constant, an operation in the wrong
order, a rounding rule changed, a carry lost), rebuilds that copy and runs
the pin suite (tests/test_oracle_pins.py) against it: at least one pin must
fail.  The untouched copy must pass, so a failure is the mistake's doing.

The mistakes cover every function of the oracle: the layout and the memory
accounting, the reduce and unscale, the exact norm accumulator, the decision
(clipping, loss-scale state machine), AdamW with bias correction and
decoupled decay, the RNE casts and decodes, the micro-step accumulation, and
the int8 payload quantizer.

CPU only; the copies run in parallel subprocesses.  The two slowest cast pins
(every fp16 and bf16 rounding pattern) are left out of the mutant runs, except
for the mistakes in the casts and the decode."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SLOW_CASTS = ("tests/test_oracle_pins.py::test_cast_f16_matches_numpy",
              "tests/test_oracle_pins.py::test_cast_bf16_matches_torch")

# name -> (exact text in oracle/zero_oracle.c, its replacement)
MISTAKES = {
    # AdamW ("DeepSpeed 与 FSDP" §ZeRO-Offload equations; ZeRO reading §5.1)
    "m_drops_beta1_term": ("b1 * m[i] + omb1 * gc", "omb1 * gc"),
    "betas_swapped": ("const float b1 = (float)hp->beta1, b2 = (float)hp->beta2;",
                      "const float b2 = (float)hp->beta1, b1 = (float)hp->beta2;"),
    "bias_correction_t_plus_1": ("pow(hp->beta1, (double)t)", "pow(hp->beta1, (double)(t + 1))"),
    "update_sign": ("th = th - (lr * mh)", "th = th + (lr * mh)"),
    "decay_after_the_step": (
        "float th = theta[i] * decay;                        /* decoupled decay */\n"
        "        th = th - (lr * mh) / (sqrtf(vh) + eps);",
        "float th = theta[i] - (lr * mh) / (sqrtf(vh) + eps);\n"
        "        th = th * decay;"),
    "v_without_square": ("omb2 * (gc * gc)", "omb2 * gc"),
    # reduce, AVG, unscale, padding ("PyTorch FSDP …" §3.3; ZeRO reading §5.1)
    "avg_divisor": ("acc = acc / (float)n_contrib;", "acc = acc / (float)(n_contrib + 1);"),
    "unscale_by_multiply": ("g_out[i] = acc / scale;", "g_out[i] = acc * scale;"),
    "padding_not_zeroed": ("if (first_flat_index + i >= full_numel) {", "if (0) {"),
    "fp32_contributions_misread": ("if (grad_kind == 2) return ((const float *)grads)[idx];",
                                   "if (grad_kind == 3) return ((const float *)grads)[idx];"),
    # overflow and norm (ZeRO reading §5.3)
    "overflow_ignored": ("        if (!isfinite(g[i])) {\n            of = 1;\n",
                         "        if (!isfinite(g[i])) {\n"),
    "norm_without_sqrt": ("const double norm = sqrt(ora_norm_sum(&acc) + extra_norm_sq);",
                          "const double norm = ora_norm_sum(&acc) + extra_norm_sq;"),
    "norm_of_first_shard_only": (
        "        ora_norm_accumulate(g + (int64_t)j * shard_size, shard_size, &acc, &overflow);",
        "        if (j == 0) ora_norm_accumulate(g + (int64_t)j * shard_size, shard_size, &acc,"
        " &overflow);"),
    "norm_carry_lost": ("x = a->w[k] < before;               /* carry */",
                        "x = 0;"),
    "norm_merge_carry_lost": ("carry = c1 | c2;", "carry = 0;"),
    "norm_rounds_ties_up": ("if (round && (sticky || (mant & 1u))) mant += 1;",
                            "if (round) mant += 1;"),
    # decision: clipping and the loss-scale state machine (ZeRO reading §5.1, §5.3)
    "clip_inverted": ("const double q = hp->max_grad_norm / (norm + 1e-6);",
                      "const double q = (norm + 1e-6) / hp->max_grad_norm;"),
    "clip_applied_above_one": ("if (q < 1.0) c = (float)q;", "c = (float)q;"),
    "scale_grows_a_step_early": ("if (st->good_steps == hp->loss_scale_window)",
                                 "if (st->good_steps + 1 == hp->loss_scale_window)"),
    "scale_without_floor": ("st->scale = s < lo ? lo : s;", "st->scale = s;"),
    "skipped_step_counts": ("        *skip = 1;\n        *coef = 1.0f;",
                            "        *skip = 1;\n        *coef = 1.0f;\n        st->step_t += 1;"),
    # the fp16 cast: ties away from zero instead of to even
    "cast_ties_away": ("if (rem > half || (rem == half && (r & 1u))) r += 1u;",
                       "if (rem >= half) r += 1u;"),
    # micro-step accumulation ("DeepSpeed 与 FSDP" §实践要点)
    "accumulate_ignores_first": ("acc[j][i] = first ? r[i] : acc[j][i] + r[i];",
                                 "acc[j][i] = acc[j][i] + r[i];"),
    "accumulate_overwrites": ("acc[j][i] = first ? r[i] : acc[j][i] + r[i];",
                              "acc[j][i] = r[i];"),
    "accumulate_unscaled_early": ("rk * shard_size, full_numel, avg, 1.0f, r);",
                                  "rk * shard_size, full_numel, avg, 2.0f, r);"),
    "accumulator_not_unscaled": (
        "g_out[i] = first_flat_index + i >= full_numel ? 0.0f : acc[i] / scale;",
        "g_out[i] = first_flat_index + i >= full_numel ? 0.0f : acc[i];"),
    "accumulator_padding_kept": (
        "g_out[i] = first_flat_index + i >= full_numel ? 0.0f : acc[i] / scale;",
        "g_out[i] = acc[i] / scale;"),
    # the int8 payload ("DeepSpeed 与 FSDP" §ZeRO++; the reading in the oracle)
    "q8_scale_over_128": ("const float scale = amax / 127.0f;",
                          "const float scale = amax / 128.0f;"),
    "q8_rounds_half_away": ("const float r = rintf(v);", "const float r = roundf(v);"),
    "q8_truncates": ("const float r = rintf(v);", "const float r = truncf(v);"),
    "q8_nan_in_amax": ("if (a > amax) amax = a;", "if (!(a <= amax)) amax = a;"),
    # more of the casts and the decode (IEEE-754 binary16 / bfloat16)
    "cast_subnormal_cutoff": ("if (shift >= 25) {", "if (shift >= 24) {"),
    "cast_overflow_threshold": ("if (e > 15) return sign | 0x7c00u;",
                                "if (e > 16) return sign | 0x7c00u;"),
    "cast_nan_to_inf": ("return (uint16_t)(sign | 0x7e00u | (man >> 13));",
                        "return (uint16_t)(sign | 0x7c00u);"),
    "cast_bf16_ties_up": ("if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;",
                          "if (lo >= 0x8000u) hi += 1u;"),
    "decode_f16_subnormal_scale": ("mag = (float)ldexp((double)man, -24);",
                                   "mag = (float)ldexp((double)man, -25);"),
    # more of AdamW
    "decay_without_lr": ("const float decay = (float)(1.0 - hp->lr * hp->weight_decay);",
                         "const float decay = (float)(1.0 - hp->weight_decay);"),
    "eps_inside_sqrt": ("th = th - (lr * mh) / (sqrtf(vh) + eps);",
                        "th = th - (lr * mh) / sqrtf(vh + eps);"),
    "bc2_with_beta1": ("const float bc2 = (float)(1.0 - pow(hp->beta2, (double)t));",
                       "const float bc2 = (float)(1.0 - pow(hp->beta1, (double)t));"),
    # more of the reduce, the norm and the decision
    "contributors_reversed": (
        "for (int32_t c = 0; c < n_contrib; ++c)\n"
        "            acc = acc + contribution(grads, grad_kind, (int64_t)c * ld + rank_off + i);",
        "for (int32_t c = n_contrib - 1; c >= 0; --c)\n"
        "            acc = acc + contribution(grads, grad_kind, (int64_t)c * ld + rank_off + i);"),
    "unscale_before_avg": ("if (avg) acc = acc / (float)n_contrib;\n        g_out[i] = acc / scale;",
                           "acc = acc / scale;\n        if (avg) acc = acc / (float)n_contrib;\n"
                           "        g_out[i] = acc;"),
    "extra_norm_dropped": ("const double norm = sqrt(ora_norm_sum(&acc) + extra_norm_sq);",
                           "const double norm = sqrt(ora_norm_sum(&acc));"),
    "norm_bit_position": ("int off = q - 53 - ORA_ACC_UNIT_EXP;",
                          "int off = q - 52 - ORA_ACC_UNIT_EXP;"),
    "norm_high_part_shift": ("if (sh) acc_add_at(a, limb + 1, m >> (64 - sh));",
                             "if (sh) acc_add_at(a, limb + 1, m >> (63 - sh));"),
    "norm_sticky_skips_bit0": (
        "for (int i = low - 1; i >= 0 && !sticky; --i) sticky = acc_bit(a, i);",
        "for (int i = low - 1; i > 0 && !sticky; --i) sticky = acc_bit(a, i);"),
    "clip_epsilon": ("const double q = hp->max_grad_norm / (norm + 1e-6);",
                     "const double q = hp->max_grad_norm / (norm + 1e-5);"),
    "static_scale_ignored": (": (float)hp->static_loss_scale;", ": 1.0f;"),
    "overflow_not_counted": ("st->overflow_count += 1;", ""),
    # the layout ("PyTorch FSDP ..." §3.1, §3.3) and the memory accounting
    # ("DeepSpeed 与 FSDP" §逐步推导, §ZeRO-3 的数学总结)
    "shard_size_floor": ("int64_t s = total / world_size + (total % world_size != 0);",
                         "int64_t s = total / world_size;"),
    "layout_gap_accepted": ("if (starts[k] != total) return ORA_EINVAL;", ""),
    "zero2_grads_not_split": ("    {0, 1, 1},   /* ZeRO-2: + gradients */",
                              "    {0, 0, 1},   /* ZeRO-2: + gradients */"),
    "zero1_params_split": ("    {0, 0, 1},   /* ZeRO-1: optimizer states */",
                           "    {1, 0, 1},   /* ZeRO-1: optimizer states */"),
    "optimizer_8_bytes": ("const uint64_t per[3] = {2, 2, 12};",
                          "const uint64_t per[3] = {2, 2, 8};"),
    "memory_rounds_down": ("u128 q = num / den + (num % den != 0);", "u128 q = num / den;"),
}


def _copy_tree(dst):
    ignore = shutil.ignore_patterns("__pycache__", "*.so", "*.tmp*")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"), ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(dst, "tests"), ignore=ignore)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst)


def _run_pins(tmp, name, mistake):
    d = os.path.join(tmp, name)
    _copy_tree(d)
    src_path = os.path.join(d, "oracle", "zero_oracle.c")
    if mistake is not None:
        old, new = mistake
        with open(src_path) as f:
            src = f.read()
        assert src.count(old) == 1, "%s: the text to change is not found once" % name
        with open(src_path, "w") as f:
            f.write(src.replace(old, new))
    cmd = [sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
           "-p", "no:cacheprovider"]
    if not name.startswith(("cast_", "decode_")):
        for t in SLOW_CASTS:
            cmd += ["--deselect", t]
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run(cmd, cwd=d, capture_output=True, text=True, env=env, timeout=900)
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    return r.returncode, failed, r.stdout[-2000:] + r.stderr[-2000:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    tmp = str(tmp_path)
    base = _run_pins(tmp, "untouched", None)
    assert base[0] == 0, "the untouched copy must pass its pins:\n" + base[2]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {n: ex.submit(_run_pins, tmp, n, m) for n, m in MISTAKES.items()}
        results = {n: f.result() for n, f in futs.items()}
    missed = [n for n, (rc, _, _) in results.items() if rc == 0]
    errors = [n for n, (rc, failed, _) in results.items() if rc != 0 and not failed]
    assert not missed, "mistakes no pin catches: %s" % missed
    # a mutant that does not even build or collect is not a caught mistake
    assert not errors, "mutants that failed without a failing pin: %s\n%s" % (
        errors, "\n".join(results[n][2] for n in errors))
